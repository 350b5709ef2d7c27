"""Helpers for GPU-vs-oracle parity: run the same seeded inputs through the CUDA
library (via the C ABI binding) and through the CPU oracle, and compare.

Tolerances (float32 state): |gpu - oracle| <= 1e-7 + 1e-5*|oracle| element-wise;
packed sign words bit-exact. In free-running multi-step comparisons an element whose
sign decision was within a tie margin (|z| <= 1e-6 * S of its chunk, on the oracle's
own values) at some step is exempt from then on: a one-ulp difference in a chunk scale
(the chunk sums are accumulated in a different order on the two sides) may flip such
a sign legitimately, after which the element's trajectory differs.
"""
import numpy as np
import torch

import oracle as O

RTOL, ATOL = 1e-5, 1e-7
TIE = 1e-6


def to_device_grads(g, device):
    if g.dtype == np.uint16:
        return torch.from_numpy(g.view(np.int16).copy()).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(g)).to(device)


def close(got, want, rtol=RTOL, atol=ATOL, where=None):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    ok = np.abs(got - want) <= atol + rtol * np.abs(want)
    if where is not None:
        ok |= ~where
    return ok


def assert_close(name, got, want, rtol=RTOL, atol=ATOL, where=None):
    ok = close(got, want, rtol, atol, where)
    if not ok.all():
        idx = np.argwhere(~ok)[:5]
        g = np.asarray(got).reshape(ok.shape)
        w = np.asarray(want).reshape(ok.shape)
        raise AssertionError("%s: %d mismatches, first %s: gpu %s oracle %s" % (
            name, int((~ok).sum()), idx.tolist(), [g[tuple(i)] for i in idx],
            [w[tuple(i)] for i in idx]))


def unpack_bits(words, n):
    """[..., n/32] uint32 -> [..., n] bool (bit t of word k is element 32k+t)."""
    w = np.ascontiguousarray(words).view(np.uint32)
    b = (w[..., :, None] >> np.arange(32, dtype=np.uint32)) & 1
    return b.reshape(*w.shape[:-1], n).astype(bool)


class CudaPath:
    """The CUDA path on one device, holding the state as torch tensors."""

    def __init__(self, st, device="cuda", mask=None):
        from error_compensated_bit_gb300 import ob
        self.ob = ob
        self.n, self.W, self.C = st.n, st.W, st.C
        self.dev = torch.device(device)
        self.ctx = ob.Context(st.n, st.W, st.C, st.b1, st.b2, st.eps, st.lr)
        self.ctx.set_options(st.wd, False)
        f = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(self.dev)
        self.x, self.m, self.v = f(st.x), f(st.m), f(st.v)
        self.ew = torch.zeros(st.W, st.n, dtype=torch.float32, device=self.dev)
        self.es = torch.zeros(st.n, dtype=torch.float32, device=self.dev)
        self.ws = torch.empty(self.ctx.workspace_bytes(), dtype=torch.uint8, device=self.dev)
        self.ctx.workspace_init(self.ws)
        self.mask_t = None
        if mask is not None:
            self.mask_t = f(np.asarray(mask, np.float32))
            self.ctx.set_mask(self.mask_t, self.ws)

    def _view(self, ptr, count, dtype):
        off = ptr - self.ws.data_ptr()
        size = torch.empty((), dtype=dtype).element_size()
        return self.ws[off:off + count * size].view(dtype)

    def messages(self):
        wb, wsc, sb, ssc = self.ctx.debug_views(self.ws)
        nch = self.n // self.C
        return dict(
            wbits=self._view(wb, self.W * self.n // 32, torch.int32).cpu().numpy().view(np.uint32).reshape(self.W, -1),
            wscale=self._view(wsc, self.W * nch, torch.float32).cpu().numpy().reshape(self.W, -1),
            sbits=self._view(sb, self.n // 32, torch.int32).cpu().numpy().view(np.uint32),
            sscale=self._view(ssc, nch, torch.float32).cpu().numpy())

    def errors(self):
        ew = torch.empty_like(self.ew)
        es = torch.empty_like(self.es)
        self.ctx.export_state(self.ew, self.es, self.ws, ew, es)
        return ew.cpu().numpy(), es.cpu().numpy()

    def compressed_step(self, g):
        gd = g if isinstance(g, torch.Tensor) else to_device_grads(g, self.dev)
        self.ctx.compressed_step(gd, self.x, self.m, self.v, self.ew, self.es, self.ws)

    def warmup_step(self, g):
        gd = g if isinstance(g, torch.Tensor) else to_device_grads(g, self.dev)
        self.ctx.warmup_step(gd, self.x, self.m, self.v, self.ws)

    def snapshot(self):
        torch.cuda.synchronize(self.dev)
        out = self.messages()
        out["ew"], out["es"] = self.errors()
        out["x"] = self.x.cpu().numpy()
        out["m"] = self.m.cpu().numpy()
        out["z"] = self.ew.cpu().numpy()
        out["y"] = self.es.cpu().numpy()
        return out


class Tracker:
    """Free-running comparison with the tie-margin exemption described above.

    Only elements whose sign actually differs leave the comparison (they are counted in
    ``flips``); every flip must sit at a near-tie of the oracle's own values. Residual-
    type values (z, y and the errors) are differences of scale-sized terms, so their
    tolerance is taken relative to the chunk's scale: 1e-7 + 1e-5 * max(|ref|, scale).
    """

    def __init__(self, n, W, C):
        self.n, self.W, self.C = n, W, C
        self.div_w = np.zeros((W, n), bool)
        self.div_s = np.zeros(n, bool)
        self.flips = 0
        self.near_ties = 0

    def compare(self, step, gpu, ora_out, st, check_mask=None):
        n, W, C = self.n, self.W, self.C
        S = np.repeat(ora_out["wscale"], C, axis=1)
        T = np.repeat(ora_out["sscale"], C)
        near_w = np.abs(ora_out["z"]) <= TIE * S
        near_s = np.abs(ora_out["y"]) <= TIE * T
        self.near_ties += int(near_w.sum() + near_s.sum())
        gw = unpack_bits(gpu["wbits"], n)
        ow = unpack_bits(ora_out["wbits"], n)
        flip_w = (gw != ow) & ~self.div_w
        assert not (flip_w & ~near_w).any(), \
            "step %d: %d worker sign bits differ away from ties" % (step, (flip_w & ~near_w).sum())
        self.div_w |= flip_w
        any_w = self.div_w.any(0)
        gs = unpack_bits(gpu["sbits"], n)
        os_ = unpack_bits(ora_out["sbits"], n)
        flip_s = (gs != os_) & ~self.div_s & ~any_w
        assert not (flip_s & ~near_s).any(), \
            "step %d: %d server sign bits differ away from ties" % (step, (flip_s & ~near_s).sum())
        self.div_s |= flip_s
        self.flips += int(flip_w.sum() + flip_s.sum())
        ok_el = ~(self.div_s | self.div_w.any(0))
        ok_w = np.broadcast_to(ok_el, (W, n))
        assert_close("step %d worker scales" % step, gpu["wscale"], ora_out["wscale"])
        assert_close("step %d server scales" % step, gpu["sscale"], ora_out["sscale"])
        Sref = np.maximum(np.abs(st.ew), S)
        Tref = np.maximum(np.maximum(np.abs(st.es), T), S.max(0))
        assert_close("step %d worker errors" % step, gpu["ew"] - st.ew, 0 * S, atol=ATOL + RTOL * Sref, where=ok_w)
        assert_close("step %d server errors" % step, gpu["es"] - st.es, 0 * T, atol=ATOL + RTOL * Tref, where=ok_el)
        assert_close("step %d z" % step, gpu["z"] - ora_out["z"], 0 * S, atol=ATOL + RTOL * np.maximum(np.abs(ora_out["z"]), S), where=ok_w)
        assert_close("step %d y" % step, gpu["y"] - ora_out["y"], 0 * T, atol=ATOL + RTOL * np.maximum(np.abs(ora_out["y"]), Tref), where=ok_el)
        assert_close("step %d momentum" % step, gpu["m"], st.m, where=ok_el)
        assert_close("step %d params" % step, gpu["x"], st.x, where=ok_el)
        if check_mask is not None:
            assert np.all(gpu["m"][check_mask == 0] == 0.0)


def exact_fraction(gpu, ora_out, st):
    """Fraction of float outputs that agree bit-for-bit (reported, not asserted)."""
    want = dict(wscale=ora_out["wscale"], sscale=ora_out["sscale"], m=st.m, x=st.x)
    tot = same = 0
    for k, ref in want.items():
        a = np.asarray(gpu[k], np.float32).view(np.uint32)
        b = np.asarray(ref, np.float32).view(np.uint32)
        tot += a.size
        same += int((a == b).sum())
    return same / tot


def random_state(rng, n, W, C, v_dist="uniform", **kw):
    x = rng.standard_normal(n) * 0.02
    if v_dist == "lognormal":
        v = np.exp(rng.standard_normal(n) * 2.0 - 12.0)
    else:
        v = rng.uniform(1e-8, 1e-4, n)
    return O.OracleState(n, W, C, x=x, m=np.zeros(n), v=v, **kw)
