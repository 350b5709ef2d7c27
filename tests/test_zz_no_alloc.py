"""The worker pass that allocates nothing (ob_worker_compress_noalloc).

Some callers cannot allocate device memory themselves: a runtime that reserves all
device memory up front and hands it out from its own arena, or an embedding that only
receives buffers someone else owns. For them the library offers one entry point whose
scratch lives in a fixed array inside the library instead of a caller-provided
workspace. Its output must equal that of the worker pass of ob_compressed_step (the
existing entry point) bit for bit, call after call, even though every call reuses the
same scratch array, and a bounded wait that runs out must be reported through its own
status word.

This file is named to be collected last, so a run that stops at the first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch


def _ctx_args(n, W, C):
    return (n, W, C, 0.9, 0.999, 1e-8, 1e-4)


def _lib_ctx(n, W, C):
    from error_compensated_bit_gb300 import build, ob
    build.build()
    lib = ob.load()
    h = ctypes.c_void_p()
    assert lib.ob_init(*_ctx_args(n, W, C), ctypes.byref(h)) == ob.OB_OK
    return lib, h


def test_rejects_sizes_beyond_the_fixed_scratch():
    """Many tiny chunks over a large buffer need more scratch than the array holds: the
    call returns OB_ESCRATCH before touching the device (the pointers are never used)."""
    from error_compensated_bit_gb300 import ob
    W, n, C = 16, 16 * 256 * 8192, 256
    lib, h = _lib_ctx(n, W, C)
    base = 1 << 40
    g, m, z = base, base + (1 << 34), base + (2 << 34)
    sp, wb, so = base + (3 << 34), base + (4 << 34), base + (5 << 34)
    rc = lib.ob_worker_compress_noalloc(h, g, ob.OB_F16, m, z, sp, wb, so, None)
    assert rc == ob.OB_ESCRATCH
    assert b"scratch" in lib.ob_strerror(rc)
    assert lib.ob_launch_count(h) == 0
    lib.ob_destroy(h)


def test_rejects_outputs_that_overlap_another_buffer():
    """Each output must be disjoint from every other buffer: the kernel reads the
    previous scales and z while it writes the outputs. The sizes are those of the test
    above, whose scratch does not fit, so a call that passes the overlap check returns
    OB_ESCRATCH and nothing reaches the device (the pointers are fakes); moving one
    output onto a neighbour by a single 16-byte step is rejected first."""
    from error_compensated_bit_gb300 import ob
    W, n, C = 16, 16 * 256 * 8192, 256
    nch = n // C
    lib, h = _lib_ctx(n, W, C)
    base = 1 << 40
    gap = 1 << 32                                  # larger than any buffer here
    ptrs = dict(g=base, m=base + gap, z=base + 2 * gap, sp=base + 3 * gap,
                wb=base + 4 * gap, so=base + 5 * gap)
    sizes = dict(g=W * n * 2, m=n * 4, z=W * n * 4, sp=W * nch * 4, wb=W * n // 8, so=W * nch * 4)

    def call(p):
        return lib.ob_worker_compress_noalloc(h, p["g"], ob.OB_F16, p["m"], p["z"], p["sp"],
                                              p["wb"], p["so"], None)

    assert call(ptrs) == ob.OB_ESCRATCH
    for out in ("z", "wb", "so"):
        for other in ptrs:
            if other == out:
                continue
            p = dict(ptrs)
            # the output's last 16 bytes land on the other buffer's first 16
            p[out] = ptrs[other] - sizes[out] + 16
            assert call(p) == ob.OB_EINVAL, (out, other)
            # and ending exactly where the other begins is fine
            p[out] = ptrs[other] - sizes[out]
            if not any(q != out and q != other and
                       p[out] < ptrs[q] + sizes[q] and ptrs[q] < p[out] + sizes[out] for q in ptrs):
                assert call(p) == ob.OB_ESCRATCH, (out, other, "adjacent")
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
    # above and its own previous outputs, no workspace at all; same kernel and launch
    # shape, so every output is bit-identical
    ctx = ob.Context(*_ctx_args(n, W, C))
    z = torch.zeros(W, n, **f32)
    scales = [torch.zeros(W, nch, **f32), torch.empty(W, nch, **f32), torch.empty(W, nch, **f32)]
    wbits = torch.empty(W, n // 32, dtype=torch.int32, device=dev)
    for t, g in enumerate(grads):
        ctx.worker_compress_noalloc(g, m_before[t], z, scales[t], wbits, scales[t + 1])
        torch.cuda.synchronize()
        want = expected[t]
        assert np.array_equal(wbits.cpu().numpy().view(np.uint32), want["wbits"]), "call %d signs" % t
        assert np.array_equal(scales[t + 1].cpu().numpy(), want["wscale"]), "call %d scales" % t
        assert np.array_equal(z.cpu().numpy(), want["z"]), "call %d z" % t
    assert ctx.launch_count() == 2
    assert ctx.noalloc_read_status() == 0


@pytest.mark.gpu
def test_noalloc_status_reports_a_wait_that_ran_out():
    """A pipeline wait that gives up must not go unnoticed on this path either: the
    self-test's bounded wait (5 ms, on a barrier nothing completes) is pointed at the
    no-allocation status word, which reports it once and is then clear; the pass still
    works afterwards."""
    from error_compensated_bit_gb300 import build, ob
    if not torch.cuda.is_available():
        pytest.fail("needs a CUDA device")
    build.build()
    dev = torch.device("cuda", torch.cuda.current_device())
    W, n = 2, 2 * 256 * 64
    C = n // W // 2
    nch = n // C
    ctx = ob.Context(*_ctx_args(n, W, C))
    assert ctx.noalloc_read_status() == 0
    ctx.selftest_wait(None, limit_ns=5_000_000)
    assert ctx.noalloc_read_status() == 1
    assert ctx.noalloc_read_status() == 0
    f32 = dict(dtype=torch.float32, device=dev)
    g = torch.full((W, n), 1e-3, **f32)
    m = torch.zeros(n, **f32)
    z = torch.zeros(W, n, **f32)
    s_prev, s_out = torch.zeros(W, nch, **f32), torch.empty(W, nch, **f32)
    wbits = torch.empty(W, n // 32, dtype=torch.int32, device=dev)
    ctx.worker_compress_noalloc(g, m, z, s_prev, wbits, s_out)
    assert ctx.noalloc_read_status() == 0
    # from zero momentum and errors, z = c1*g with c1 = 1 - b1 in float32, the same
    # everywhere; every sign bit is set and each scale is |z|
    assert (wbits.cpu().numpy().view(np.uint32) == 0xFFFFFFFF).all()
    c1 = np.float32(np.float32(1.0) - np.float32(0.9))
    want = np.float32(c1 * np.float32(1e-3))
    assert np.array_equal(z.cpu().numpy(), np.full((W, n), want, np.float32))
    assert np.allclose(s_out.cpu().numpy(), want, rtol=1e-6, atol=0)
