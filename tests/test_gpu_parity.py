"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle, element by
element, on the same seeded inputs. Sign words bit-exact; float32 state within
1e-7 + 1e-5*|oracle| (see gpu_util for the tie-margin rule of multi-step runs)."""
import numpy as np
import pytest
import torch

import oracle as O
from gpu_util import CudaPath, Tracker, assert_close, exact_fraction, random_state, unpack_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from error_compensated_bit_gb300 import build
    build.build()


def _grads(rng, W, n, dtype, scale=1e-3):
    g = (rng.standard_normal((W, n)) * scale).astype(np.float32)
    if dtype == "f16":
        return g.astype(np.float16)
    if dtype == "bf16":
        return (g.view(np.uint32) >> 16).astype(np.uint16)     # truncated to bfloat16
    return g


def _free_run(ora, st, grads_fn, steps, mask=None):
    gpu = CudaPath(st, mask=mask)
    tr = Tracker(st.n, st.W, st.C)
    fracs = []
    for t in range(steps):
        g = grads_fn(t)
        out = ora.compressed_step(st, g)
        gpu.compressed_step(g)
        snap = gpu.snapshot()
        tr.compare(t, snap, out, st, check_mask=mask)
        fracs.append(exact_fraction(snap, out, st))
    return tr, fracs


def test_tiny_workload_ten_steps(ora):
    """The tiny workload: n = 2^20, W = 4, chunk = n/W, float32 grads, 10 steps."""
    from error_compensated_bit_gb300 import synth
    wl = synth.workload("tiny")
    st = O.OracleState(wl.n, wl.W, wl.C, x=synth.params(wl).numpy(), m=np.zeros(wl.n),
                       v=synth.variance(wl).numpy(), b1=wl.b1, b2=wl.b2, eps=wl.eps, lr=wl.lr)
    tr, fracs = _free_run(ora, st, lambda t: synth.to_numpy_grads(synth.grads(wl, t)), wl.steps)
    print("tiny: %d sign flips at %d near-ties; bit-identical float fraction per step %s"
          % (tr.flips, tr.near_ties, ["%.6f" % f for f in fracs]))
    assert tr.flips <= 2


# (W, grad dtype, groups of 256 per worker row, groups per chunk): ragged partitions
# (the group count is not a multiple of the warp count), several chunks per worker,
# chunk = 256 (every group its own chunk), one chunk per worker, prime sizes.
CASES = [
    (1, "f32", 64, 64),
    (2, "f16", 300, 100),
    (3, "bf16", 777, 259),
    (4, "f32", 1000, 1),
    (5, "bf16", 600, 600),
    (8, "f16", 1000, 250),
    (8, "f32", 1234, 617),
    (16, "f32", 173, 173),
    (16, "bf16", 96, 8),
    (7, "f16", 2000, 400),
    # short chunks with block ranges spanning many chunks: one range per warp, the chunks
    # inside a warp's range scaled by that warp alone (row counts padded to 2, 4, 8, 16)
    (1, "f32", 1000, 1),
    (2, "bf16", 10000, 2),
    (3, "f16", 6000, 2),
    (6, "f32", 700, 1),
    (9, "bf16", 500, 1),
    (11, "f16", 400, 1),
    (13, "f32", 1500, 2),
    # 16-bit gradients with W >= 11 and long chunks: the interleaved worker without the
    # block-level pre-combination of partials
    (12, "f16", 300, 300),
]


@pytest.mark.parametrize("W,dtype,groups,cgroups", CASES)
def test_compressed_step_parity(ora, W, dtype, groups, cgroups):
    rng = np.random.default_rng(1000 + W * 7 + groups)
    n = W * 256 * groups
    C = 256 * cgroups
    st = random_state(rng, n, W, C, lr=1e-4)
    tr, fracs = _free_run(ora, st, lambda t: _grads(rng, W, n, dtype), 4)
    print("W=%d %s: %d sign flips at %d near-ties; bit-identical float fraction %s"
          % (W, dtype, tr.flips, tr.near_ties, ["%.6f" % f for f in fracs]))
    assert tr.flips <= 2


def test_momentum_mask_parity(ora):
    """BERT-Base-like: 2% of positions have exactly-zero gradients and a zero mask."""
    rng = np.random.default_rng(77)
    W, n = 8, 8 * 256 * 700
    C = n // W
    zero = rng.random(n) < 0.02
    mask = (~zero).astype(np.float32)
    st = random_state(rng, n, W, C, v_dist="lognormal", mask=mask)

    def grads(t):
        g = _grads(rng, W, n, "f32")
        g[:, zero] = 0.0
        return g
    tr, _ = _free_run(ora, st, grads, 5, mask=mask)


def test_weight_decay_parity(ora):
    rng = np.random.default_rng(78)
    W, n = 4, 4 * 256 * 300
    st = random_state(rng, n, W, n // W, wd=0.01, lr=4e-4)
    _free_run(ora, st, lambda t: _grads(rng, W, n, "f16"), 3)


@pytest.mark.parametrize("C", [256 * 16, 256])
@pytest.mark.parametrize("case", ["zeros", "negzero", "single", "negative", "subnormal",
                                  "mask_all_zero", "huge_range", "overflow"])
def test_edge_cases(ora, case, C):
    """C = 4096 spreads every chunk over several warp ranges (partials combined by the
    last contributor); C = 256 puts every chunk inside one warp's range (scales formed by
    that warp alone). Degenerate chunks -- all zero, subnormal, or sums of squares that
    overflow float32 -- take the double-precision fallback in both."""
    rng = np.random.default_rng(5)
    # with 256-element chunks the buffer is long enough that a block's range spans many
    # chunks, so the worker runs one range per warp (at 64 groups per row it would not)
    W, n = 4, 4 * 256 * (1024 if C == 256 else 64)
    mask = None
    st = random_state(rng, n, W, C)
    g = np.zeros((W, n), np.float32)
    if case == "zeros":
        st.x[:] = 0.0
    elif case == "negzero":
        g[:] = -0.0
    elif case == "single":
        g[2, 12345] = 1e-3
    elif case == "negative":
        g[:] = -np.abs(_grads(rng, W, n, "f32"))
    elif case == "subnormal":
        g[:] = np.float32(1e-41) * rng.choice([-1.0, 1.0], (W, n)).astype(np.float32)
    elif case == "mask_all_zero":
        g = _grads(rng, W, n, "f32")
        mask = np.zeros(n, np.float32)
        st.mask = np.zeros(n, np.uint8)
    elif case == "huge_range":
        g = _grads(rng, W, n, "f32") * np.float32(10.0) ** rng.integers(-12, 6, (W, n)).astype(np.float32)
    elif case == "overflow":
        # |z| about 4e18: the squares fit float32 but a chunk's sum of them does not
        g = (rng.choice([-4e19, 4e19], (W, n)) * rng.uniform(0.5, 1.0, (W, n))).astype(np.float32)
        g[:, : n // 2] = _grads(rng, W, n // 2, "f32")
    gpu = CudaPath(st, mask=mask)
    tr = Tracker(n, W, C)
    for t in range(3):
        out = ora.compressed_step(st, g)
        gpu.compressed_step(g)
        tr.compare(t, gpu.snapshot(), out, st, check_mask=mask)
    if case in ("zeros", "negzero"):
        snap = gpu.snapshot()
        assert np.all(snap["wbits"] == 0xFFFFFFFF) and np.all(snap["wscale"] == 0)


@pytest.mark.parametrize("W", [3, 11])
def test_server_sum_order(ora, W):
    """Workers added in ascending order on the GPU too, where the order decides the
    rounding: b1 = 0 (z = g), worker 0's chunk all 1, the others all 2^-24 -- ascending,
    each 2^-24 rounds away against 1 (through the average table, and for W > 8 the
    workers after the eighth in order)."""
    n = W * 256
    C = 256
    g = np.full((W, n), 2.0 ** -24, np.float32)
    g[0] = 1.0
    st = O.OracleState(n, W, C, x=np.zeros(n), m=np.zeros(n), v=np.ones(n), b1=0.0, lr=1e-4)
    gpu = CudaPath(st)
    out = ora.compressed_step(st, g)
    gpu.compressed_step(g)
    snap = gpu.snapshot()
    assert np.array_equal(snap["y"], out["y"])
    assert np.array_equal(snap["sscale"], out["sscale"])
    assert np.array_equal(snap["m"], st.m)
    assert np.array_equal(snap["x"], st.x)


def test_warmup_and_loco_mean_orders(ora):
    """The warm-up and LoCo means add workers in ascending order on the GPU too (the
    cases where the order decides the rounding, b1 = 0 so m is the mean)."""
    from gpu_util import to_device_grads
    n, W = 3 * 256, 3
    g = np.stack([np.full(n, v, np.float32) for v in (1.0, 2.0 ** -24, 2.0 ** -24)])
    st = O.OracleState(n, W, n // W, x=np.zeros(n), m=np.zeros(n), v=np.zeros(n), b1=0.0, lr=1e-4)
    gpu = CudaPath(st)
    ora.warmup_step(st, g)
    gpu.warmup_step(g)
    torch.cuda.synchronize()
    assert np.array_equal(gpu.m.cpu().numpy(), st.m)
    assert np.array_equal(gpu.x.cpu().numpy(), st.x)

    g = np.full((W, n), 2.0 ** -22, np.float32)
    g[0] = 7.0
    g[1:, ::256] = 7.0 * 2.0 ** -22                  # sets the scale of every chunk
    st = O.OracleState(n, W, 256, x=np.zeros(n), m=np.zeros(n), v=np.zeros(n), b1=0.0, lr=1e-4)
    gpu = CudaPath(st)
    err = np.zeros((W, n), np.float32)
    err_d = torch.zeros(W, n, dtype=torch.float32, device="cuda")
    lws = torch.zeros(gpu.ctx.loco_workspace_bytes(4), dtype=torch.uint8, device="cuda")
    ora.loco_step(st, g, err, beta=0.0, bits=4)
    gpu.ctx.loco_step(to_device_grads(g, "cuda"), gpu.x, gpu.m, gpu.v, err_d, lws, 0.0, 4)
    torch.cuda.synchronize()
    assert np.array_equal(gpu.m.cpu().numpy(), st.m)
    assert np.array_equal(gpu.x.cpu().numpy(), st.x)


def test_deterministic(ora):
    rng = np.random.default_rng(9)
    W, n = 8, 8 * 256 * 500
    st = random_state(rng, n, W, n // W)
    g = _grads(rng, W, n, "f16")
    snaps = []
    for rep in range(2):
        gpu = CudaPath(st.copy())
        for t in range(3):
            gpu.compressed_step(g)
        snaps.append(gpu.snapshot())
    for k in snaps[0]:
        assert np.array_equal(np.asarray(snaps[0][k]).view(np.uint8), np.asarray(snaps[1][k]).view(np.uint8)), k


def test_reset_and_export(ora):
    """Errors reset as on checkpoint load: the next step equals one from zero errors."""
    rng = np.random.default_rng(10)
    W, n = 4, 4 * 256 * 200
    C = n // W // 2
    st = random_state(rng, n, W, C)
    gpu = CudaPath(st)
    tr = Tracker(n, W, C)
    for t in range(2):
        g = _grads(rng, W, n, "f32")
        out = ora.compressed_step(st, g)
        gpu.compressed_step(g)
        tr.compare(t, gpu.snapshot(), out, st)
    gpu.ctx.reset_errors(gpu.ew, gpu.es, gpu.ws)
    ew, es = gpu.errors()
    assert not ew.any() and not es.any()
    st.ew[:] = 0.0
    st.es[:] = 0.0
    g = _grads(rng, W, n, "f32")
    out = ora.compressed_step(st, g)
    gpu.compressed_step(g)
    tr.compare(2, gpu.snapshot(), out, st)


@pytest.mark.parametrize("W,dtype,bc,wd", [(8, "f32", False, 0.0), (4, "f16", True, 0.01),
                                           (3, "bf16", True, 0.0), (1, "f32", False, 0.01)])
def test_warmup_parity(ora, W, dtype, bc, wd):
    rng = np.random.default_rng(20 + W)
    n = W * 256 * 333
    st = random_state(rng, n, W, n // W, v_dist="lognormal", wd=wd)
    gpu = CudaPath(st)
    gpu.ctx.set_options(wd, bc)
    for t in range(4):
        g = _grads(rng, W, n, dtype)
        ora.warmup_step(st, g, bias_correction=bc)
        gpu.warmup_step(g)
        torch.cuda.synchronize()
        assert_close("warm-up %d m" % t, gpu.m.cpu().numpy(), st.m)
        assert_close("warm-up %d v" % t, gpu.v.cpu().numpy(), st.v)
        assert_close("warm-up %d x" % t, gpu.x.cpu().numpy(), st.x)
    assert np.array_equal(gpu.x.cpu().numpy(), st.x), "warm-up is element-wise: bit-exact"


def test_warmup_then_compressed(ora):
    """The BERT-Base recipe in small: warm-up steps, then compressed steps with a mask."""
    rng = np.random.default_rng(31)
    W, n = 8, 8 * 256 * 250
    zero = rng.random(n) < 0.02
    mask = (~zero).astype(np.float32)
    st = random_state(rng, n, W, n // W, v_dist="lognormal", mask=mask)
    gpu = CudaPath(st, mask=mask)
    tr = Tracker(n, W, n // W)
    for t in range(7):
        g = _grads(rng, W, n, "f32")
        g[:, zero] = 0.0
        if t < 3:
            ora.warmup_step(st, g)
            gpu.warmup_step(g)
        else:
            out = ora.compressed_step(st, g)
            gpu.compressed_step(g)
            tr.compare(t, gpu.snapshot(), out, st, check_mask=mask)


@pytest.mark.parametrize("W,dtype,bits,per_row,ratio,keep", [
    (4, "bf16", 4, 2, 1.0, False), (2, "f32", 8, 2, 1.0, True), (3, "f16", 4, 2, 1.0, False),
    (4, "bf16", 4, 400, 1.0, False), (2, "f32", 8, 25, 1.0, True),
    (4, "bf16", 4, 2, 0.5, True), (3, "f16", 8, 25, 0.0, False), (2, "f32", 4, 400, 0.3, True),
    (2, "bf16", 4, 200, 1.0, False), (3, "f32", 8, 100, 0.5, False), (2, "f16", 4, 400 // 3, 1.0, True),
    (2, "bf16", 8, 2, 0.5, True), (6, "f16", 4, 2, 1.0, True), (1, "bf16", 4, 2, 1.0, True)])
def test_loco_parity(ora, W, dtype, bits, per_row, ratio, keep):
    """per_row chunks per worker row: 400, 200 and 100 make chunks of one, two and four
    256-element groups (quantized in one pass from registers), 133 chunks of three groups
    and 25 chunks of 4096 elements (one pass, read twice through the L2), 2 long chunks
    (separate absmax pass, then one pass that quantizes every row and takes the Adam step,
    its codes in registers unless `keep` asks for them; short chunks store them anyway;
    16-bit gradients with W <= 4 stage each lane's rows in shared memory, the others
    keep them in registers).
    ratio: the share of the averaged error compensated into the gradient (1 is plain
    c = g + e~)."""
    from error_compensated_bit_gb300 import ob
    rng = np.random.default_rng(40 + W + per_row + int(ratio * 10))
    groups = 399 if per_row == 400 // 3 else 400      # 133 chunks of three groups
    n = W * 256 * groups
    C = n // W // per_row
    st = random_state(rng, n, W, C)
    st.v[:] = 0.0
    gpu = CudaPath(st)
    if ratio != 1.0:
        gpu.ctx.set_loco_ratio(ratio)
    gpu.ctx.set_loco_codes(keep)
    stored = keep or C <= 4096
    err_d = torch.zeros(W, n, dtype=torch.float32, device="cuda")
    lws = torch.zeros(gpu.ctx.loco_workspace_bytes(bits), dtype=torch.uint8, device="cuda")
    err = np.zeros((W, n), np.float32)
    code_bytes = W * n * bits // 8
    scale_off = (code_bytes + 255) // 256 * 256
    for t in range(4):
        g = _grads(rng, W, n, dtype)
        out = ora.loco_step(st, g, err, beta=0.9, bits=bits, ratio=ratio)
        from gpu_util import to_device_grads
        gpu.ctx.loco_step(to_device_grads(g, "cuda"), gpu.x, gpu.m, gpu.v, err_d, lws, 0.9, bits)
        torch.cuda.synchronize()
        codes = lws[:code_bytes].cpu().numpy().reshape(W, -1)
        scales = lws[scale_off:scale_off + W * (n // C) * 4].view(torch.float32).cpu().numpy().reshape(W, -1)
        if stored:
            assert np.array_equal(codes, out["codes"]), "step %d codes" % t
        else:
            assert not codes.any(), "long chunks without keep store no codes"
        assert np.array_equal(scales, out["scales"]), "step %d scales" % t
        assert_close("loco %d err" % t, err_d.cpu().numpy(), err)
        assert_close("loco %d m" % t, gpu.m.cpu().numpy(), st.m)
        assert_close("loco %d v" % t, gpu.v.cpu().numpy(), st.v)
        assert_close("loco %d x" % t, gpu.x.cpu().numpy(), st.x)
    assert np.array_equal(err_d.cpu().numpy(), err), "LoCo has no sums: bit-exact"


def test_contexts_in_host_threads(ora):
    """Two contexts created and driven from two host threads at once, each on its own
    stream (the worker kernels' shared-memory opt-in is set per context, not through a
    process-wide flag): both match the oracle."""
    import threading
    cases = [(4, "f16", 61), (8, "bf16", 62)]
    setups, results, errors = [], {}, []
    for W, dtype, seed in cases:
        rng = np.random.default_rng(seed)
        n = W * 256 * 96
        st = random_state(rng, n, W, n // W // 2)
        grads = [_grads(rng, W, n, dtype) for _ in range(3)]
        setups.append((W, st, grads))
    # the oracle's results first, on copies of the initial states
    starts = [st.copy() for _, st, _ in setups]
    want = []
    for W, st, grads in setups:
        outs = [ora.compressed_step(st, g) for g in grads]
        want.append((outs[-1], st))
    barrier = threading.Barrier(len(setups))

    def run(i):
        try:
            W, _, grads = setups[i]
            gpu = CudaPath(starts[i])
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            from gpu_util import to_device_grads
            gd = [to_device_grads(g, "cuda") for g in grads]
            torch.cuda.synchronize()
            barrier.wait()
            for g in gd:
                gpu.ctx.compressed_step(g, gpu.x, gpu.m, gpu.v, gpu.ew, gpu.es, gpu.ws, side)
            side.synchronize()
            results[i] = gpu.snapshot()
        except Exception as e:         # reported by the main thread
            errors.append(e)

    threads = [threading.Thread(target=run, args=(i,)) for i in range(len(setups))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for i, (out, st) in enumerate(want):
        got = results[i]
        assert np.array_equal(got["sbits"], out["sbits"]), "context %d server signs" % i
        assert_close("context %d params" % i, got["x"], st.x)
        assert_close("context %d momentum" % i, got["m"], st.m)


def test_stream_ordering():
    """Calls are asynchronous on the given stream: a step enqueued on a side stream is
    ordered after work already on that stream and visible after synchronizing it."""
    from error_compensated_bit_gb300.optimizer import OneBitAdam
    rng = np.random.default_rng(50)
    W, n = 2, 2 * 256 * 64
    opt = OneBitAdam(n, W, freeze_step=0)
    side = torch.cuda.Stream()
    g = torch.from_numpy(_grads(rng, W, n, "f32")).cuda()
    torch.cuda.synchronize()
    with torch.cuda.stream(side):
        g.mul_(2.0)              # queued on the side stream before the step
        opt.step(g)
    side.synchronize()
    ref = OneBitAdam(n, W, freeze_step=0)
    ref.step(g)
    torch.cuda.synchronize()
    assert torch.equal(opt.x, ref.x) and torch.equal(opt.m, ref.m)


def test_host_buffer_entry_point_matches_device_path():
    """ob_compressed_step_host (host gradients in, compressed message out, alternating
    device buffers so copies overlap earlier steps) computes exactly the device path."""
    from error_compensated_bit_gb300 import ob
    rng = np.random.default_rng(61)
    W, n = 4, 4 * 256 * 300
    C = n // W
    st = random_state(rng, n, W, C)
    a, b = CudaPath(st.copy()), CudaPath(st.copy())
    grads = [torch.from_numpy(_grads(rng, W, n, "f16")) for _ in range(3)]
    hosts = [g.pin_memory() for g in grads]
    dev_bufs = [torch.empty(W, n, dtype=torch.float16, device="cuda") for _ in range(2)]
    sb_host = torch.empty(n // 32, dtype=torch.int32).pin_memory()
    ss_host = torch.empty(n // C, dtype=torch.float32).pin_memory()
    for t in range(3):
        a.compressed_step(grads[t].cuda())
        b.ctx.compressed_step_host(hosts[t], dev_bufs[t % 2], b.x, b.m, b.v, b.ew, b.es, b.ws,
                                   sb_host, ss_host)
        torch.cuda.synchronize()
        sa, sb_ = a.snapshot(), b.snapshot()
        for k in ("wbits", "wscale", "sbits", "sscale", "x", "m", "z", "y"):
            assert np.array_equal(np.asarray(sa[k]).view(np.uint8), np.asarray(sb_[k]).view(np.uint8)), (t, k)
        assert np.array_equal(sb_host.numpy().view(np.uint32), sb_["sbits"])
        assert np.array_equal(ss_host.numpy(), sb_["sscale"])
    assert b.ctx.read_status(b.ws) == 0


def test_compressed_step_replays_from_a_cuda_graph(ora):
    """One compressed step captured into a CUDA graph and replayed gives, step for step,
    exactly what eager calls give (launch-bound small buffers can be run this way)."""
    rng = np.random.default_rng(80)
    W, n = 4, 4 * 256 * 128
    st = random_state(rng, n, W, n // W)
    g = torch.from_numpy(_grads(rng, W, n, "f16")).cuda()
    eager, graphed = CudaPath(st.copy()), CudaPath(st.copy())
    graphed.compressed_step(g)                    # first call outside the capture
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        graphed.ctx.compressed_step(g, graphed.x, graphed.m, graphed.v, graphed.ew, graphed.es, graphed.ws)
    eager.compressed_step(g)
    for t in range(3):
        graph.replay()
        eager.compressed_step(g)
        torch.cuda.synchronize()
        a, b = eager.snapshot(), graphed.snapshot()
        for k in ("wbits", "wscale", "sbits", "sscale", "x", "m", "z", "y"):
            assert np.array_equal(np.asarray(a[k]).view(np.uint8), np.asarray(b[k]).view(np.uint8)), (t, k)
