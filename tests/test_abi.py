"""The C ABI on the host: the library loads, exports every symbol the header declares,
and rejects bad arguments with the documented status before touching the device.

Only invalid arguments are passed here, which the library rejects before it enqueues
anything, so these tests run the same with or without a GPU.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ob.h")


@pytest.fixture(scope="module")
def ob():
    from error_compensated_bit_gb300 import build
    build.build()
    from error_compensated_bit_gb300 import ob as mod
    mod.load()
    return mod


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ob_[a-z_0-9]+)\s*\(", text)))


def test_header_symbols_exported(ob):
    names = header_functions()
    assert len(names) >= 20
    lib = ob.load()
    for name in names:
        assert hasattr(lib, name), "symbol %s declared but not exported" % name
    assert sorted(ob.SIGNATURES) == names, "binding and header disagree"


def test_library_has_no_oracle_dependency():
    """The product library links nothing from the oracle."""
    import subprocess
    from error_compensated_bit_gb300 import build
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True, text=True).stdout
    assert "ora_" not in out
    src = "".join(open(os.path.join(build.CSRC, f)).read() for f in os.listdir(build.CSRC))
    assert "oracle" not in src.lower()


def _init(ob, n=1 << 20, W=4, chunk=1 << 18, b1=0.9, b2=0.999, eps=1e-8, lr=1e-4):
    h = ctypes.c_void_p()
    rc = ob.load().ob_init(n, W, chunk, b1, b2, eps, lr, ctypes.byref(h))
    return rc, h


@pytest.mark.parametrize("kw", [
    dict(W=0), dict(W=17), dict(n=1000), dict(n=(1 << 20) + 256), dict(chunk=300),
    dict(chunk=3 << 18), dict(n=0), dict(lr=float("nan")), dict(b1=1.0), dict(b2=-0.1),
    dict(eps=-1.0), dict(chunk=0), dict(n=1 << 36, W=16, chunk=1 << 20)])
def test_init_rejects(ob, kw):
    rc, h = _init(ob, **kw)
    assert rc == ob.OB_EINVAL and not h.value


def test_init_accepts_and_sizes_workspace(ob):
    rc, h = _init(ob)
    assert rc == ob.OB_OK and h.value
    lib = ob.load()
    n, W = 1 << 20, 4
    nbytes = lib.ob_workspace_bytes(h)
    # packed signs of W workers + server + mask, at least
    assert nbytes >= W * n // 8 + 2 * n // 8
    assert nbytes % 256 == 0
    assert lib.ob_loco_workspace_bytes(h, 4) >= W * n // 2
    assert lib.ob_loco_workspace_bytes(h, 3) == 0
    lib.ob_destroy(h)
    lib.ob_destroy(None)


def test_calls_reject_bad_arguments(ob):
    rc, h = _init(ob)
    lib = ob.load()
    good, odd = 1 << 20, (1 << 20) + 4      # never dereferenced: rejected first
    ws, ws_odd = 1 << 24, (1 << 24) + 16
    S = None
    assert lib.ob_compressed_step(h, good, 7, good, good, good, good, good, ws, S) == ob.OB_EINVAL
    assert lib.ob_compressed_step(h, odd, 0, good, good, good, good, good, ws, S) == ob.OB_EALIGN
    assert lib.ob_compressed_step(h, good, 0, good, odd, good, good, good, ws, S) == ob.OB_EALIGN
    assert lib.ob_compressed_step(h, good, 0, good, good, good, good, good, ws_odd, S) == ob.OB_EALIGN
    assert lib.ob_compressed_step(h, None, 0, good, good, good, good, good, ws, S) == ob.OB_EINVAL
    assert lib.ob_compressed_step(None, good, 0, good, good, good, good, good, ws, S) == ob.OB_EINVAL
    assert lib.ob_compressed_step(h, good, 1, good, good, None, good, good, ws, S) == ob.OB_EINVAL
    assert lib.ob_warmup_step(h, good, 2, good, good, odd, ws, S) == ob.OB_EALIGN
    assert lib.ob_warmup_step(h, good, -1, good, good, good, ws, S) == ob.OB_EINVAL
    assert lib.ob_loco_step(h, good, 2, good, good, good, good, 0.9, 3, ws, S) == ob.OB_ENOTIMPL
    assert lib.ob_loco_step(h, good, 2, good, good, good, good, 1.5, 4, ws, S) == ob.OB_EINVAL
    assert lib.ob_loco_step(h, good, 2, good, good, good, odd, 0.9, 4, ws, S) == ob.OB_EALIGN
    assert lib.ob_reset_errors(h, odd, good, ws, S) == ob.OB_EALIGN
    assert lib.ob_export_state(h, good, good, ws, good, None, S) == ob.OB_EINVAL
    assert lib.ob_set_mask(h, odd, ws, S) == ob.OB_EALIGN
    assert lib.ob_set_mask(h, None, ws, S) == ob.OB_OK          # clears, enqueues nothing
    assert lib.ob_compressed_step_host(h, None, good, 0, good, good, good, good, good, ws,
                                       good, good, S) == ob.OB_EINVAL
    assert lib.ob_set_options(h, -0.1, 0) == ob.OB_EINVAL
    assert lib.ob_set_options(h, 0.01, 1) == ob.OB_OK
    for bad in (-0.25, 1.5, float("nan"), float("inf")):
        assert lib.ob_set_loco_ratio(h, bad) == ob.OB_EINVAL
    for good_ratio in (0.0, 0.5, 1.0):
        assert lib.ob_set_loco_ratio(h, good_ratio) == ob.OB_OK
    for bad_keep in (-1, 2):
        assert lib.ob_set_loco_codes(h, bad_keep) == ob.OB_EINVAL
    assert lib.ob_set_loco_codes(h, 1) == ob.OB_OK and lib.ob_set_loco_codes(h, 0) == ob.OB_OK
    assert lib.ob_set_step(h, -1) == ob.OB_EINVAL
    assert lib.ob_set_step(h, 41) == ob.OB_OK and lib.ob_get_step(h) == 41
    assert lib.ob_set_lr(h, float("inf")) == ob.OB_EINVAL
    assert lib.ob_profile_read(h, 99, None, None) == ob.OB_EINVAL
    assert lib.ob_selftest_wait(h, ws, 0, S) == ob.OB_EINVAL
    assert lib.ob_selftest_wait(h, ws, 3 * 10 ** 9, S) == ob.OB_EINVAL
    assert lib.ob_selftest_wait(h, ws_odd, 1000, S) == ob.OB_EALIGN
    assert lib.ob_launch_count(h) == 0, "rejected calls launch nothing"
    lib.ob_destroy(h)


def test_strerror(ob):
    lib = ob.load()
    for code in (0, -1, -2, -3, -4, 5):
        assert lib.ob_strerror(code)


def test_product_path_fails_loudly_without_library(tmp_path, monkeypatch):
    """With the built library absent the binding raises instead of falling back."""
    import importlib
    from error_compensated_bit_gb300 import ob as mod
    monkeypatch.setattr(mod, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(mod, "_LIB", None)
    with pytest.raises(ImportError):
        mod.load()
