"""The worker pass that allocates nothing (ob_worker_compress_noalloc).

Some callers cannot allocate device memory: code running while a stream is captured
into a CUDA graph, or a runtime that owns all device memory up front. For them the
library offers one entry point whose scratch lives in a fixed array inside the library
instead of a caller-provided workspace. Its output must equal that of the worker pass
of ob_compressed_step (the existing entry point), call after call, even though every
call reuses the same scratch array.

This file is named to be collected last, so a run that stops at the first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from gpu_util import ATOL, RTOL, assert_close


def _ctx_args(n, W, C):
    return (n, W, C, 0.9, 0.999, 1e-8, 1e-4)


def test_rejects_sizes_beyond_the_fixed_scratch():
    """Many tiny chunks over a large buffer need more scratch than the array holds: the
    call returns OB_ESCRATCH before touching the device (the pointers are never used)."""
    from error_compensated_bit_gb300 import build, ob
    build.build()
    lib = ob.load()
    W, n, C = 16, 16 * 256 * 8192, 256
    h = ctypes.c_void_p()
    assert lib.ob_init(*_ctx_args(n, W, C), ctypes.byref(h)) == ob.OB_OK
    fake = 1 << 20
    rc = lib.ob_worker_compress_noalloc(h, fake, ob.OB_F16, fake, fake, fake, fake, fake + 4096, None)
    assert rc == ob.OB_ESCRATCH
    assert b"scratch" in lib.ob_strerror(rc)
    assert lib.ob_launch_count(h) == 0
    lib.ob_destroy(h)


@pytest.mark.gpu
def test_noalloc_worker_pass_matches_compressed_step():
    from error_compensated_bit_gb300 import build, ob
    if not torch.cuda.is_available():
        pytest.fail("needs a CUDA device")
    build.build()
    dev = torch.device("cuda", torch.cuda.current_device())
    rng = np.random.default_rng(4242)
    W, n = 8, 8 * 256 * 600
    C = n // W // 2
    nch = n // C
    f32 = dict(dtype=torch.float32, device=dev)

    # the existing entry point: two full compressed steps, workspace from the caller
    ref = ob.Context(*_ctx_args(n, W, C))
    x = torch.from_numpy((rng.standard_normal(n) * 0.02).astype(np.float32)).to(dev)
    v = torch.from_numpy(rng.uniform(1e-8, 1e-4, n).astype(np.float32)).to(dev)
    m = torch.zeros(n, **f32)
    ew = torch.zeros(W, n, **f32)
    es = torch.zeros(n, **f32)
    ws = torch.empty(ref.workspace_bytes(), dtype=torch.uint8, device=dev)
    ref.workspace_init(ws)
    wb_ptr, wsc_ptr, _, _ = ref.debug_views(ws)
    wb_off, wsc_off = wb_ptr - ws.data_ptr(), wsc_ptr - ws.data_ptr()

    grads = [torch.from_numpy((rng.standard_normal((W, n)) * 1e-3).astype(np.float16)).to(dev)
             for _ in range(2)]
    expected, m_before = [], []
    for g in grads:
        m_before.append(m.clone())
        ref.compressed_step(g, x, m, v, ew, es, ws)
        torch.cuda.synchronize()
        expected.append(dict(
            z=ew.cpu().numpy(),
            wbits=ws[wb_off:wb_off + W * n // 8].cpu().numpy().view(np.uint32).reshape(W, -1),
            wscale=ws[wsc_off:wsc_off + W * nch * 4].view(torch.float32).cpu().numpy().reshape(W, -1)))

    # the new entry point: two calls in a row, each given the same inputs as the step
    # above and its own previous outputs, no workspace at all
    ctx = ob.Context(*_ctx_args(n, W, C))
    z = torch.zeros(W, n, **f32)
    scales = [torch.zeros(W, nch, **f32), torch.empty(W, nch, **f32), torch.empty(W, nch, **f32)]
    wbits = torch.empty(W, n // 32, dtype=torch.int32, device=dev)
    for t, g in enumerate(grads):
        ctx.worker_compress_noalloc(g, m_before[t], z, scales[t], wbits, scales[t + 1])
        torch.cuda.synchronize()
        want = expected[t]
        assert np.array_equal(wbits.cpu().numpy().view(np.uint32), want["wbits"]), "call %d signs" % t
        assert_close("call %d scales" % t, scales[t + 1].cpu().numpy(), want["wscale"], RTOL, ATOL)
        assert_close("call %d z" % t, z.cpu().numpy(), want["z"], RTOL, ATOL)
    assert ctx.launch_count() == 2
