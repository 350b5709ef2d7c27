"""Full-size parity: every workload at its full size, in the launch configuration the
benchmark uses, checked against the oracle on sampled chunks.

Every quantity of a step depends only on its own chunk (element-wise arithmetic plus
per-chunk scales and, for LoCo, per-chunk maxima), so the oracle run on one chunk's slice
of the inputs reproduces exactly what the full-size run must produce for that chunk. The
first and the last chunk are checked (the last one holds the padding tail) over two
steps: sign words and LoCo codes bit-exact, float32 state within 1e-7 + 1e-5*|ref|.
"""
import gc

import numpy as np
import pytest
import torch

import oracle as O
from gpu_util import assert_close

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

# (workload, W, phase, chunk): chunk None is the workload's own (n/W); the short chunks
# run the worker with one range per warp, scales written by their only contributor and
# the separate scale-copy kernel, and LoCo's one-pass absmax + quantize kernels.
CASES = [
    ("bertL", 8, "compressed", None),
    ("bertL", 8, "compressed", 2048),
    ("bertB", 8, "compressed", None),
    ("sweep", 2, "compressed", None),
    ("sweep", 16, "compressed", None),
    ("sweep", 16, "compressed", 256),
    ("loco", 4, "loco", None),
    ("loco", 4, "compressed", None),
    ("loco", 4, "loco", 256),        # one-pass LoCo, chunks held in registers
    ("sweep", 4, "loco", 2048),      # one-pass LoCo, chunks read twice through the L2
]


def _np_grads(g):
    from error_compensated_bit_gb300 import synth
    return synth.to_numpy_grads(g)


def _view(ws, ptr, count, dtype):
    off = ptr - ws.data_ptr()
    size = torch.empty((), dtype=dtype).element_size()
    return ws[off:off + count * size].view(dtype)


@pytest.mark.parametrize("name,W,phase,chunk", CASES,
                         ids=["%s-W%d-%s%s" % (c[:3] + ("" if c[3] is None else "-C%d" % c[3],)) for c in CASES])
def test_full_size_sampled_chunks(ora, name, W, phase, chunk):
    from error_compensated_bit_gb300 import build, ob, synth
    if not torch.cuda.is_available():
        pytest.fail("needs a CUDA device")
    build.build()
    dev = torch.device("cuda", torch.cuda.current_device())
    wl = synth.workload(name, W=W, chunk=chunk)
    n, C = wl.n, wl.C
    nch = n // C
    ctx = ob.Context(n, W, C, wl.b1, wl.b2, wl.eps, wl.lr)
    x = synth.params(wl, dev)
    v = synth.variance(wl, dev)
    m = torch.zeros(n, dtype=torch.float32, device=dev)
    ew = torch.zeros(W, n, dtype=torch.float32, device=dev)
    es = torch.zeros(n, dtype=torch.float32, device=dev)
    ws = torch.empty(ctx.workspace_bytes(), dtype=torch.uint8, device=dev)
    ctx.workspace_init(ws)
    masked = wl.zero_frac > 0 and phase == "compressed"
    mask = synth.mask(wl, dev) if masked else None
    if masked:
        ctx.set_mask(mask, ws)
    lws = None
    if phase == "loco":
        v.zero_()
        lws = torch.zeros(ctx.loco_workspace_bytes(4), dtype=torch.uint8, device=dev)
    g = torch.empty(W, n, dtype=wl.grad_dtype, device=dev)

    # keep the oracle's share bounded: short chunks are cheap, so three are checked
    picks = [0, nch // 2, nch - 1] if C <= 4096 else ([0, nch - 1] if n < 10 ** 9 else [nch - 1])
    sl = {k: slice(k * C, (k + 1) * C) for k in picks}
    host = lambda t, k: t[sl[k]].cpu().numpy()
    states = {}
    for k in picks:
        states[k] = O.OracleState(C, W, C, x=host(x, k), m=host(m, k), v=host(v, k), b1=wl.b1,
                                  b2=wl.b2, eps=wl.eps, lr=wl.lr,
                                  mask=None if mask is None else host(mask, k))
    err = {k: np.zeros((W, C), np.float32) for k in picks}

    warm = wl.warmup_steps if (name == "bertB" and phase == "compressed") else 0
    warm = min(warm, 2)
    for t in range(warm + 2):
        synth.grads(wl, t, dev, out=g)
        gk = {k: _np_grads(g[:, sl[k]]) for k in picks}
        if t < warm:
            ctx.warmup_step(g, x, m, v, ws)
            for k in picks:
                ora.warmup_step(states[k], gk[k])
            torch.cuda.synchronize()
            for k in picks:
                assert np.array_equal(host(x, k), states[k].x), "warm-up %d chunk %d x" % (t, k)
            continue
        if phase == "loco":
            # long chunks keep their codes in registers; the first step stores them too,
            # to be compared, and the second runs as the benchmark does
            keep = t == warm
            ctx.set_loco_codes(keep)
            ctx.loco_step(g, x, m, v, ew, lws, 0.9, 4)
            outs = {k: ora.loco_step(states[k], gk[k], err[k], beta=0.9, bits=4) for k in picks}
            torch.cuda.synchronize()
            code_bytes = W * n // 2
            scale_off = (code_bytes + 255) // 256 * 256
            codes = lws[:code_bytes].view(W, n // 2)
            scales = lws[scale_off:scale_off + W * nch * 4].view(torch.float32).view(W, nch)
            for k in picks:
                st = states[k]
                if keep or C <= 4096:
                    assert np.array_equal(codes[:, k * C // 2:(k + 1) * C // 2].cpu().numpy(),
                                          outs[k]["codes"]), "step %d chunk %d codes" % (t, k)
                assert np.array_equal(scales[:, k].cpu().numpy(), outs[k]["scales"][:, 0])
                assert_close("loco %d err" % t, ew[:, sl[k]].cpu().numpy(), err[k])
                assert_close("loco %d x" % t, host(x, k), st.x)
                assert_close("loco %d m" % t, host(m, k), st.m)
                assert_close("loco %d v" % t, host(v, k), st.v)
            continue
        ctx.compressed_step(g, x, m, v, ew, es, ws)
        outs = {k: ora.compressed_step(states[k], gk[k]) for k in picks}
        torch.cuda.synchronize()
        wb, wsc, sb, ssc = ctx.debug_views(ws)
        wbits = _view(ws, wb, W * n // 32, torch.int32).view(W, n // 32)
        wscale = _view(ws, wsc, W * nch, torch.float32).view(W, nch)
        sbits = _view(ws, sb, n // 32, torch.int32)
        sscale = _view(ws, ssc, nch, torch.float32)
        e_w = torch.empty(W, C, dtype=torch.float32, device=dev)
        for k in picks:
            st, out = states[k], outs[k]
            words = slice(k * C // 32, (k + 1) * C // 32)
            assert np.array_equal(wbits[:, words].cpu().numpy().view(np.uint32), out["wbits"]), \
                "step %d chunk %d worker signs" % (t, k)
            assert np.array_equal(sbits[words].cpu().numpy().view(np.uint32), out["sbits"]), \
                "step %d chunk %d server signs" % (t, k)
            assert np.array_equal(wscale[:, k].cpu().numpy(), out["wscale"][:, 0])
            assert np.array_equal(sscale[k:k + 1].cpu().numpy(), out["sscale"])
            # the stored pre-compression buffers are the oracle's z and y
            assert np.array_equal(ew[:, sl[k]].cpu().numpy(), out["z"])
            assert np.array_equal(es[sl[k]].cpu().numpy(), out["y"])
            assert_close("step %d chunk %d x" % (t, k), host(x, k), st.x)
            assert_close("step %d chunk %d m" % (t, k), host(m, k), st.m)
            # the true residuals: e = z - S*sign(z)
            zk = ew[:, sl[k]]
            e_w.copy_(zk - torch.where(zk >= 0, wscale[:, k:k + 1], -wscale[:, k:k + 1]))
            assert_close("step %d chunk %d worker errors" % (t, k), e_w.cpu().numpy(), st.ew)
    assert ctx.read_status(ws) == 0
    del x, v, m, ew, es, ws, g, lws
    gc.collect()
    torch.cuda.empty_cache()
