"""Pins of the CPU oracle: checks against facts fixed outside the oracle itself.

Each pin takes an ``oracle.Oracle`` and raises AssertionError on a mismatch. They are
collected by ``test_oracle_pins.py`` and re-run against deliberately broken copies of
the oracle's source by ``test_oracle_mutants.py`` (every broken copy must fail one).

What pins what:
  decode_*          numpy's / torch's own float16 / bfloat16 -> float32 casts, all 65536
                    bit patterns
  pack_exhaustive   every 16-bit sign pattern maps to the integer that spells it (bit t
                    <-> element t, 1 <-> non-negative)
  sign_of_zero      sign(0) = +1 for +0.0 and -0.0, subnormals keep their sign
  scale_*           closed forms of the RMS scale, exact-rational brute force for n <= 64,
                    power-of-two homogeneity
  onebit_identity   decompress(compress(z)) + residual == z (exactly where Sterbenz
                    applies), |residual| == ||z| - S|, norm preservation per chunk
  worked_example    a two-step, two-worker step derived by hand in exact binary
                    arithmetic (every intermediate is a small dyadic rational)
  identity_sgd      with the compressor replaced by the identity the compressed step is
                    momentum SGD preconditioned by the frozen variance:
                    torch.optim.SGD on g / (sqrt(v) + eps), with the weight decay applied
                    to the parameters before the step (decoupled, as AdamW does)
  w1_server         with one worker the server stage reproduces the worker's message
  server_sum_order  workers added in ascending order (a case where the order rounds
  mean_orders       differently); the same for the warm-up's and LoCo's means
  mask              masked momentum is exactly zero; unmasked values match the unmasked
                    run; errors are not masked
  warmup_adamw      the warm-up step is AdamW on the mean gradient (torch.optim.AdamW),
                    and from zero state it has the closed form -lr*c1*g/(sqrt(c2)|g|+eps)
  comm_bytes        the pages' 32x (97%) and "up to 5x" communication figures
  loco_*            LoCo codes for exactly representable inputs, nibble layout, 8-bit
                    codes as signed bytes (clamping, ties to even), the half-step error
                    bound, the moving average's closed form, the
                    dequantized mean driving a first Adam step (closed form), and with
                    exactly quantizable gradients the Adam part equal to the warm-up
                    step (itself pinned to AdamW) from non-zero state; the
                    compensation ratio: a case worked by hand in dyadic arithmetic at
                    ratio 1/2 (ties to even included), and ratio 0 making the codes,
                    scales and (beta = 0) new errors independent of the old errors
"""
import json
import math
import os
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np
import torch

import oracle as O

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _f32(a):
    return np.asarray(a, dtype=np.float32)


def _bits(a):
    return _f32(a).view(np.uint32)


def _same_bits(a, b):
    return np.array_equal(_bits(a), _bits(b))


# ---- gradient formats ---------------------------------------------------------------

def pin_decode_f16(ora):
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16).view(np.float16)
    got = ora.decode_grads(h)
    ref = h.astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert _same_bits(got[~nan], ref[~nan])


def pin_decode_bf16(ora):
    raw = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = ora.decode_grads(raw)
    ref = torch.from_numpy(raw.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert _same_bits(got[~nan], ref[~nan])


# ---- sign packing ---------------------------------------------------------------------

def _reverse16(p):
    r = np.zeros_like(p)
    for t in range(16):
        r |= ((p >> t) & 1) << (15 - t)
    return r


def pin_pack_exhaustive(ora):
    rng = np.random.default_rng(11)
    P = np.arange(65536, dtype=np.uint32)
    lo = ((P[:, None] >> np.arange(16, dtype=np.uint32)) & 1).astype(bool)
    signs = np.concatenate([lo, lo[:, ::-1]], axis=1)               # [65536, 32]
    mags = rng.uniform(1e-3, 10.0, size=signs.shape).astype(np.float32)
    z = np.where(signs, mags, -mags).astype(np.float32)
    words = ora.pack_signs(z.reshape(-1))
    expected = P | (_reverse16(P) << 16)
    assert np.array_equal(words, expected)


def pin_sign_of_zero(ora):
    tiny = np.float32(1e-45)          # smallest positive subnormal
    z = np.zeros(32, np.float32)
    z[0] = 0.0
    z[1] = -0.0
    z[2] = -tiny
    z[3] = tiny
    z[4] = -1.0
    z[5:] = -2.0
    word = int(ora.pack_signs(z)[0])
    assert word & 1 and word & 2, "sign(+0) and sign(-0) are +1"
    assert not word & 4 and word & 8, "subnormals keep their sign"
    assert word >> 4 == 0


# ---- the scale --------------------------------------------------------------------------

def _nearest_f32_sqrt(fr):
    """float32 nearest to sqrt(fr) for a non-negative Fraction, via 60-digit decimals."""
    getcontext().prec = 60
    root = (Decimal(fr.numerator) / Decimal(fr.denominator)).sqrt()
    lo = np.float32(float(root))
    cands = [np.nextafter(lo, np.float32(-np.inf)), lo, np.nextafter(lo, np.float32(np.inf))]
    best = min(cands, key=lambda c: abs(Decimal(float(c)) - root))
    return np.float32(best), root


def pin_scale_closed_forms(ora):
    rng = np.random.default_rng(5)
    for C, a in [(32, 1.0), (32, 0.1), (16, 3e-5), (32, 1e-40), (256, 0.75), (1024, 2.0 ** -7)]:
        s = np.where(rng.random(C) < 0.5, -1.0, 1.0)
        z = (s * np.float32(a)).astype(np.float32)
        assert ora.chunk_scale(z) == np.float32(a), (C, a)
    # sixteen values whose mean square is 4: 8 x (+1), 7 x (-1), one -7  ->  S = 2
    z = _f32([1] * 8 + [-1] * 7 + [-7])
    assert ora.chunk_scale(z) == np.float32(2.0)
    assert ora.chunk_scale(np.zeros(64, np.float32)) == 0.0
    assert ora.chunk_scale(_f32([0] * 15 + [4])) == np.float32(1.0)   # sqrt(16/16)


def pin_scale_bruteforce(ora):
    rng = np.random.default_rng(7)
    exact_hits = 0
    total = 0
    for n in range(1, 65):
        for trial in range(4):
            if trial == 0:
                z = rng.standard_normal(n)
            elif trial == 1:
                z = rng.standard_normal(n) * 10.0 ** rng.uniform(-30, 30)
            elif trial == 2:
                z = np.zeros(n)
                z[rng.integers(n)] = rng.standard_normal()
            else:
                z = -np.abs(rng.standard_normal(n)) * 1e-3
            z = z.astype(np.float32)
            got = ora.chunk_scale(z)
            ssq = sum(Fraction(float(v)) ** 2 for v in z)
            want, root = _nearest_f32_sqrt(ssq / n)
            total += 1
            if got == want:
                exact_hits += 1
                continue
            # only a value within a hair of a rounding midpoint may round the other way
            mid = (Decimal(float(got)) + Decimal(float(want))) / 2
            assert abs(mid - root) <= abs(root) * Decimal("1e-12"), (n, trial, got, want)
    assert exact_hits >= total - 2


def pin_scale_homogeneous(ora):
    rng = np.random.default_rng(3)
    z = rng.standard_normal(4096).astype(np.float32)
    s = ora.chunk_scale(z)
    for k in (-12, -1, 3, 20):
        assert ora.chunk_scale(z * np.float32(2.0 ** k)) == s * np.float32(2.0 ** k)


# ---- compressor identity ---------------------------------------------------------------

def pin_onebit_identity(ora):
    rng = np.random.default_rng(9)
    C, n = 64, 64 * 40
    z = (rng.standard_normal(n) * np.repeat(10.0 ** rng.uniform(-6, 2, n // C), C)).astype(np.float32)
    z[::97] = 0.0
    z[5] = -0.0
    words, scales, resid = ora.onebit_compress(z, C)
    S = np.repeat(scales, C)
    sigma = np.where(z >= 0, np.float32(1), np.float32(-1))
    sent = (S * sigma).astype(np.float32)
    # the decompressed message is +-S by the sign bit
    assert _same_bits(ora.unpack(words, scales, n, C), sent)
    # |residual| == ||z| - S| exactly (the same exact difference, rounded once)
    assert _same_bits(np.abs(resid), np.abs(np.abs(z) - S))
    # sent + residual == z exactly where Sterbenz's lemma makes the difference exact
    st = (np.abs(z) >= S / 2) & (np.abs(z) <= 2 * S)
    assert st.sum() > n // 4
    assert np.array_equal((sent[st] + resid[st]).astype(np.float32), z[st])
    # the residual points from the message to the value: sign(z - S*sigma)
    big = np.abs(z) > S * 1.01
    assert np.all(np.sign(resid[big]) == np.sign(z[big]))
    small = (np.abs(z) < S * 0.99) & (z != 0)
    assert np.all(np.sign(resid[small]) == -np.sign(z[small]))
    # the message keeps each chunk's 2-norm
    zn = np.sqrt((z.astype(np.float64) ** 2).reshape(-1, C).sum(1))
    sn = np.sqrt((sent.astype(np.float64) ** 2).reshape(-1, C).sum(1))
    assert np.allclose(sn, zn, rtol=2e-7, atol=0)


# ---- a step worked out by hand ---------------------------------------------------------

def pin_worked_example(ora):
    """W = 2, n = 32, C = 16, b1 = 1/2, v = 4, eps = 0, lr = 1/2, mask 0 on 16..19.

    Step 1 (m = e = 0, so z_w = g_w / 2):
      chunk 0  z0 = [1]*8 + [-1]*7 + [-7]      S0 = sqrt(64/16) = 2, e0 = [-1]*8 [1]*7 [-5]
               z1 = [2]*4 + [-2]*4 + [2]*8     S1 = 2,               e1 = 0
               a  = (s0 S0 + s1 S1)/2 = [2]*4 + [0]*12 ; y = a
               T = sqrt(4*4/16) = 1, all signs + (sign 0 = +1), es = [1]*4 + [-1]*12, m = 1
      chunk 1  z0 = [-3]*16   S0 = 3, e0 = 0 ;  z1 = [-1]*15 + [-7]  S1 = 2, e1 = [1]*15 [-5]
               a = (-3-2)/2 = -2.5 = y, T = 2.5, es = 0, m = -2.5 (masked: -0.0)
      x = 1 - lr*m/sqrt(4) = 1 - m/4  ->  0.75 | 1 (masked) | 1.625
    Step 2 (gradients chosen so every z is round):
      chunk 0  g0 = [5]*8 [-7]*7 [5]  p0 = 1/2 + g0/2, z0 = p0 + e0 = [2]*8 [-2]*8, S0 = 2
               g1 = [11]*16           z1 = [6]*16, S1 = 6
               a = [4]*8 + [2]*8 ; y = a + es = [5]*4 [3]*4 [1]*8 ; T = sqrt(144/16) = 3
               es = [2]*4 [0]*4 [-2]*8 ; m = 3
      chunk 1  g0 = [-2]*4 [0.5]*12   z0 = [-1]*16, S0 = 1
               g1 = [-8]*4 [-5.5]*11 [6.5]  p1 = [-4]*15 [2], z1 = p1 + e1 = [-3]*16, S1 = 3
               a = y = -2, T = 2, es = 0, m = -2 (masked: -0.0)
      x -> 0 | 1 (masked) | 2.125
    """
    n, W, C = 32, 2, 16
    mask = np.ones(n, np.uint8)
    mask[16:20] = 0
    st = O.OracleState(n, W, C, x=np.ones(n), m=np.zeros(n), v=np.full(n, 4.0),
                       b1=0.5, b2=0.999, eps=0.0, lr=0.5, mask=mask)
    g1 = np.zeros((W, n), np.float32)
    g1[0, :16] = 2 * _f32([1] * 8 + [-1] * 7 + [-7])
    g1[1, :16] = 2 * _f32([2] * 4 + [-2] * 4 + [2] * 8)
    g1[0, 16:] = 2 * _f32([-3] * 16)
    g1[1, 16:] = 2 * _f32([-1] * 15 + [-7])
    out = ora.compressed_step(st, g1)
    assert np.array_equal(out["wscale"], _f32([[2, 3], [2, 2]]))
    assert np.array_equal(out["sscale"], _f32([1, 2.5]))
    assert [int(w) for w in out["wbits"][:, 0]] == [0x000000FF, 0x0000FF0F]
    assert int(out["sbits"][0]) == 0x0000FFFF
    assert np.array_equal(out["y"], _f32([2] * 4 + [0] * 12 + [-2.5] * 16))
    assert np.array_equal(st.ew[0], _f32([-1] * 8 + [1] * 7 + [-5] + [0] * 16))
    assert np.array_equal(st.ew[1], _f32([0] * 16 + [1] * 15 + [-5]))
    assert np.array_equal(st.es, _f32([1] * 4 + [-1] * 12 + [0] * 16))
    assert _same_bits(st.m, _f32([1] * 16 + [-0.0] * 4 + [-2.5] * 12))
    assert np.array_equal(st.x, _f32([0.75] * 16 + [1] * 4 + [1.625] * 12))

    g2 = np.zeros((W, n), np.float32)
    g2[0, :16] = _f32([5] * 8 + [-7] * 7 + [5])
    g2[1, :16] = _f32([11] * 16)
    g2[0, 16:] = _f32([-2] * 4 + [0.5] * 12)
    g2[1, 16:] = _f32([-8] * 4 + [-5.5] * 11 + [6.5])
    out = ora.compressed_step(st, g2)
    assert np.array_equal(out["z"][0], _f32([2] * 8 + [-2] * 8 + [-1] * 16))
    assert np.array_equal(out["z"][1], _f32([6] * 16 + [-3] * 16))
    assert np.array_equal(out["wscale"], _f32([[2, 1], [6, 3]]))
    assert np.array_equal(out["sscale"], _f32([3, 2]))
    assert [int(w) for w in out["wbits"][:, 0]] == [0x000000FF, 0x0000FFFF]
    assert int(out["sbits"][0]) == 0x0000FFFF
    assert np.array_equal(out["y"], _f32([5] * 4 + [3] * 4 + [1] * 8 + [-2] * 16))
    assert not st.ew.any()
    assert np.array_equal(st.es, _f32([2] * 4 + [0] * 4 + [-2] * 8 + [0] * 16))
    assert _same_bits(st.m, _f32([3] * 16 + [-0.0] * 4 + [-2] * 12))
    assert np.array_equal(st.x, _f32([0] * 16 + [1] * 4 + [2.125] * 12))


# ---- special cases that reduce to library routines ----------------------------------------

def _rand_state(rng, n, W, C, **kw):
    x = rng.standard_normal(n) * 0.02
    v = rng.uniform(1e-8, 1e-4, n)
    return O.OracleState(n, W, C, x=x, m=np.zeros(n), v=v, **kw)


def pin_identity_sgd(ora):
    """Identity compressor: momentum SGD (torch.optim.SGD) on g / (sqrt(v) + eps); with a
    weight decay wd, the parameters are first scaled by (1 - lr*wd) (decoupled decay, as
    AdamW applies it), so the step is x - lr*(m/(sqrt(v)+eps) + wd*x)."""
    rng = np.random.default_rng(21)
    for W, wd in ((1, 0.0), (3, 0.0), (2, 0.01)):
        n, C = 1024, 256
        st = _rand_state(rng, n, W, C, b1=0.9, eps=1e-8, lr=1e-3, wd=wd)
        p = torch.nn.Parameter(torch.from_numpy(st.x.copy()).double())
        f = lambda a: float(np.float32(a))
        opt = torch.optim.SGD([p], lr=f(1e-3), momentum=f(0.9), dampening=f(0.9))
        opt.state[p]["momentum_buffer"] = torch.zeros_like(p)
        precond = torch.from_numpy(np.sqrt(st.v.astype(np.float64)) + f(1e-8))
        for step in range(5):
            g = (rng.standard_normal((W, n)) * 1e-3).astype(np.float32)
            ora.compressed_step(st, g, identity=True)
            p.grad = torch.from_numpy(g.astype(np.float64).mean(0)) / precond
            with torch.no_grad():
                p.mul_(1.0 - f(1e-3) * f(wd))
            opt.step()
            assert not st.ew.any() and not st.es.any()
            np.testing.assert_allclose(st.x, p.detach().numpy(), rtol=1e-5, atol=1e-7)
            mom = opt.state[p]["momentum_buffer"].numpy() * precond.numpy()
            np.testing.assert_allclose(st.m, mom, rtol=1e-5, atol=1e-9)


def pin_w1_server(ora):
    rng = np.random.default_rng(23)
    n, C = 2048, 512
    st = _rand_state(rng, n, 1, C)
    g = (rng.standard_normal((1, n)) * 1e-3).astype(np.float32)
    out = ora.compressed_step(st, g)
    sent = ora.unpack(out["wbits"][0], out["wscale"][0], n, C)
    assert np.array_equal(out["y"], sent)
    assert np.array_equal(out["sbits"], out["wbits"][0])
    np.testing.assert_allclose(out["sscale"], out["wscale"][0], rtol=1e-6)
    assert np.all(np.abs(st.es) <= 1e-6 * np.repeat(out["sscale"], C))
    assert np.array_equal(st.m, ora.unpack(out["sbits"], out["sscale"], n, C))


def pin_mask(ora):
    rng = np.random.default_rng(25)
    n, W, C = 4096, 4, 1024
    mask = (rng.random(n) > 0.3).astype(np.uint8)
    a = _rand_state(rng, n, W, C, mask=mask)
    b = a.copy()
    b.mask = None
    x0 = a.x.copy()
    for step in range(3):
        g = (rng.standard_normal((W, n)) * 1e-3).astype(np.float32)
        g[:, mask == 0] *= 0.5
        oa = ora.compressed_step(a, g)
        ob = ora.compressed_step(b, g)
        assert np.all(a.m[mask == 0] == 0.0)
        if step == 0:
            for k in ("z", "wbits", "wscale", "y", "sbits", "sscale"):
                assert np.array_equal(oa[k], ob[k]), k
            assert np.array_equal(a.m[mask == 1], b.m[mask == 1])
        assert np.array_equal(a.x[mask == 0], x0[mask == 0]), "masked momentum moves nothing"
    assert np.any(a.ew[:, mask == 0] != 0), "errors are not masked"


def pin_warmup_adamw(ora):
    rng = np.random.default_rng(27)
    for W, wd in ((1, 0.0), (4, 0.01)):
        n = 2048
        st = _rand_state(rng, n, W, 256, b1=0.9, b2=0.999, eps=1e-8, lr=1e-3, wd=wd)
        p = torch.nn.Parameter(torch.from_numpy(st.x.copy()).double())
        # the oracle's hyper-parameters are float32: hand torch the same rounded values
        f = lambda a: float(np.float32(a))
        opt = torch.optim.AdamW([p], lr=f(1e-3), betas=(f(0.9), f(0.999)), eps=f(1e-8),
                                weight_decay=f(wd))
        st.v[:] = 0.0
        for step in range(4):
            g = (rng.standard_normal((W, n)) * 1e-3).astype(np.float32)
            ora.warmup_step(st, g, bias_correction=True)
            p.grad = torch.from_numpy(g.astype(np.float64).mean(0))
            opt.step()
            np.testing.assert_allclose(st.x, p.detach().numpy(), rtol=1e-5, atol=1e-7)
            # m and v are sums of terms of size ~1e-4 and ~1e-9 that may cancel: compare
            # against float32 rounding of the terms, not of the (possibly tiny) result
            np.testing.assert_allclose(st.m, opt.state[p]["exp_avg"].numpy(), rtol=1e-5, atol=1e-10)
            np.testing.assert_allclose(st.v, opt.state[p]["exp_avg_sq"].numpy(), rtol=1e-5, atol=1e-15)
    # zero state, no bias correction: dx = -lr*c1*g / (sqrt(c2)*|g| + eps)
    n = 1024
    g = (rng.standard_normal((1, n)) * 10.0 ** rng.uniform(-9, -2, n)).astype(np.float32)
    st = O.OracleState(n, 1, 256, x=np.zeros(n), m=np.zeros(n), v=np.zeros(n), b1=0.9,
                       b2=0.999, eps=1e-8, lr=1e-4)
    ora.warmup_step(st, g)
    c1, c2 = 1 - np.float64(np.float32(0.9)), 1 - np.float64(np.float32(0.999))
    gd = g[0].astype(np.float64)
    want = -1e-4 * c1 * gd / (np.sqrt(c2) * np.abs(gd) + 1e-8)
    np.testing.assert_allclose(st.x, want, rtol=2e-6, atol=0)


# ---- communication volume (the pages' figures) -----------------------------------------------

def pin_comm_bytes(ora):
    claims = json.load(open(os.path.join(GOLDEN, "pages_claims.json")))
    n, W = 333_496_320, 8
    comp, dense16 = O.comm_bytes_per_worker(n, W, n // W, dense_bytes=2)
    _, dense32 = O.comm_bytes_per_worker(n, W, n // W, dense_bytes=4)
    r32 = dense32 / comp
    assert abs(r32 - claims["compressed_phase_reduction_vs_fp32"]["value"]) < 0.01
    saved = 100 * (1 - comp / dense32)
    assert round(saved) == claims["compressed_phase_reduction_vs_fp32"]["percent_saved"]
    r16 = dense16 / comp
    lo = claims["warmup_fraction_range"]["low"]
    hi = claims["warmup_fraction_range"]["high"]
    up_to = claims["whole_run_reduction_vs_uncompressed_adam"]["value_up_to"]
    for f in (lo, hi):
        whole = 1.0 / (f + (1.0 - f) / r16)
        assert whole <= up_to
    assert 1.0 / (lo + (1.0 - lo) / r16) > 0.9 * up_to
    assert r16 >= up_to


# ---- LoCo -------------------------------------------------------------------------------------

def pin_loco_codes(ora):
    n, W, C = 32, 1, 16
    q = np.array(list(range(-7, 8)) + [0] + list(range(7, -8, -1)) + [3], np.float32)
    s = np.float32(2.0 ** -10)
    g = (q * s).reshape(1, n)
    st = O.OracleState(n, W, C, x=np.zeros(n), m=np.zeros(n), v=np.zeros(n), lr=1e-4)
    err = np.zeros((W, n), np.float32)
    out = ora.loco_step(st, g, err, beta=0.0, bits=4)
    assert np.array_equal(out["scales"], _f32([[s, s]]))
    assert not err.any()
    nib = np.stack([out["codes"][0] & 0xF, out["codes"][0] >> 4], 1).reshape(-1).astype(np.int8)
    nib = np.where(nib > 7, nib - 16, nib)
    assert np.array_equal(nib, q.astype(np.int8))
    assert out["codes"][0][0] == ((-7 & 0xF) | ((-6 & 0xF) << 4))
    # the first Adam step on exactly-dequantized gradients: -lr*c1*g/(sqrt(c2)|g|+eps)
    c1, c2 = 1 - np.float64(np.float32(0.9)), 1 - np.float64(np.float32(0.999))
    gd = g[0].astype(np.float64)
    want = -1e-4 * c1 * gd / (np.sqrt(c2) * np.abs(gd) + 1e-8)
    np.testing.assert_allclose(st.x, want, rtol=2e-6, atol=1e-30)


def pin_loco_codes_8bit(ora):
    """8-bit codes: the levels are -127..127 (L = 2^7 - 1) and each code is one signed
    byte in element order. Inputs that are exact multiples of a power-of-two step with the
    largest magnitude 127 steps give exactly those levels, zero error, and scale = step."""
    n, W, C = 256, 1, 256
    q = np.concatenate([np.arange(-127, 128), [0]]).astype(np.float32)
    s = np.float32(2.0 ** -12)
    g = (q * s).reshape(1, n)
    st = O.OracleState(n, W, C, x=np.zeros(n), m=np.zeros(n), v=np.zeros(n), lr=1e-4)
    err = np.zeros((W, n), np.float32)
    out = ora.loco_step(st, g, err, beta=0.0, bits=8)
    assert np.array_equal(out["scales"], _f32([[s]]))
    assert np.array_equal(out["codes"][0].view(np.int8), q.astype(np.int8))
    assert not err.any()
    # above 127 steps the codes clamp: one element at 254 steps makes the step twice as
    # large, so level 127 now stands for 254 steps and odd multiples round to even ones
    g2 = g.copy()
    g2[0, 0] = np.float32(254) * s
    err = np.zeros((W, n), np.float32)
    out2 = ora.loco_step(O.OracleState(n, W, C, x=np.zeros(n), m=np.zeros(n), v=np.zeros(n), lr=1e-4),
                         g2, err, beta=0.0, bits=8)
    assert np.array_equal(out2["scales"], _f32([[2 * s]]))
    codes = out2["codes"][0].view(np.int8).astype(np.int32)
    assert codes[0] == 127
    halves = q[1:].astype(np.float64) / 2            # the other elements in units of 2s
    assert np.array_equal(codes[1:], np.rint(halves).astype(np.int32))   # ties to even


def pin_loco_error_bound(ora):
    rng = np.random.default_rng(31)
    n, W, C = 4096, 2, 512
    g = (rng.standard_normal((W, n)) * 1e-3).astype(np.float32)
    st = _rand_state(rng, n, W, C)
    err = np.zeros((W, n), np.float32)
    out = ora.loco_step(st, g, err, beta=0.0, bits=4)
    s = np.repeat(out["scales"], C, axis=1)
    amax = np.abs(g).reshape(W, -1, C).max(2)
    np.testing.assert_allclose(out["scales"], amax / 7, rtol=1e-7)
    assert np.all(np.abs(err) <= s / 2 * (1 + 1e-6))     # beta = 0: err = c - q*s
    # beta = 1/2: the moving average is the mean of the old average and the new error
    prev = err.copy()
    g2 = (rng.standard_normal((W, n)) * 1e-3).astype(np.float32)
    out2 = ora.loco_step(st, g2, err, beta=0.5, bits=4)
    c = (g2 + prev).astype(np.float32)
    s2 = np.repeat(out2["scales"], C, axis=1)
    codes = out2["codes"]
    nib = np.stack([codes & 0xF, codes >> 4], 2).reshape(W, n).astype(np.int16)
    qv = np.where(nib > 7, nib - 16, nib).astype(np.float32)
    e_new = (c - qv * s2).astype(np.float64)
    np.testing.assert_allclose(err, 0.5 * prev + 0.5 * e_new, rtol=1e-6, atol=1e-12)
    # rounding to the nearest level: the new error is at most half a step
    assert np.all(np.abs(e_new) <= s2 / 2 * (1 + 1e-6))


def pin_loco_mean(ora):
    """Two workers, exact levels: the Adam step sees the mean of the dequantized grads."""
    n, W, C = 16, 2, 16
    s = np.float32(2.0 ** -8)
    q0 = _f32([7, 1, -3, 0, 2, 2, -7, 5, 1, 1, 1, 1, -1, -1, 6, 0])
    q1 = _f32([7, 3, -1, 0, -2, 4, -7, 5, 1, 3, 5, 7, -3, 1, -6, 0])
    g = np.stack([q0 * s, q1 * s]).astype(np.float32)
    st = O.OracleState(n, W, C, x=np.zeros(n), m=np.zeros(n), v=np.zeros(n), lr=1e-4)
    err = np.zeros((W, n), np.float32)
    ora.loco_step(st, g, err, beta=0.9, bits=4)
    gbar = (q0.astype(np.float64) + q1) / 2 * float(s)
    c1, c2 = 1 - np.float64(np.float32(0.9)), 1 - np.float64(np.float32(0.999))
    want = -1e-4 * c1 * gbar / (np.sqrt(c2) * np.abs(gbar) + 1e-8)
    np.testing.assert_allclose(st.x, want, rtol=2e-6, atol=1e-30)
    np.testing.assert_allclose(st.m, c1 * gbar, rtol=1e-6, atol=0)


def pin_loco_ratio_half_by_hand(ora):
    """One worker, one chunk of four, 4-bit codes, beta = 1/2, ratio = 1/2, every value a
    small dyadic rational, worked out by hand:
      c   = g + e~/2         = [7/8, 0, 5/16, -3/16]
      s   = (7/8) / 7        = 1/8
      c/s                    = [7, 0, 5/2, -3/2] -> q = [7, 0, 2, -2] (ties to even)
      e   = c - q*s          = [0, 0, 1/16, 1/16]
      e~' = e~/2 + e/2       = [3/8, 1/4, 3/32, -1/32]."""
    n, W, C = 4, 1, 4
    g = _f32([[0.5, -0.25, 0.25, -0.125]])
    err = _f32([[0.75, 0.5, 0.125, -0.125]])
    st = O.OracleState(n, W, C, x=np.zeros(n), m=np.zeros(n), v=np.zeros(n), lr=1e-4)
    out = ora.loco_step(st, g, err, beta=0.5, bits=4, ratio=0.5)
    assert np.array_equal(out["scales"], _f32([[0.125]]))
    assert out["codes"].tolist() == [[0x07, (2 & 0xF) | ((-2 & 0xF) << 4)]]
    assert np.array_equal(err, _f32([[0.375, 0.25, 0.09375, -0.03125]]))


def pin_loco_ratio_zero(ora):
    """With ratio 0 the gradient is quantized as it is: codes and scales do not depend on
    the averaged errors, the scale is the chunk's max |g| / 7, and with beta = 0 the new
    average is the new error alone, the same whatever the old one was."""
    rng = np.random.default_rng(77)
    n, W, C = 2048, 2, 256
    g = (rng.standard_normal((W, n)) * 1e-3).astype(np.float32)
    outs, errs = [], []
    for scale in (0.0, 1e-3, -5e-3):
        st = _rand_state(rng, n, W, C)
        err = (rng.standard_normal((W, n)) * scale).astype(np.float32)
        outs.append(ora.loco_step(st, g, err, beta=0.0, bits=4, ratio=0.0))
        errs.append(err)
    for o, e in zip(outs[1:], errs[1:]):
        assert np.array_equal(o["codes"], outs[0]["codes"])
        assert np.array_equal(o["scales"], outs[0]["scales"])
        assert np.array_equal(e, errs[0])
    amax = np.abs(g).reshape(W, -1, C).max(2)
    np.testing.assert_allclose(outs[0]["scales"], amax / 7, rtol=1e-7)


def pin_server_sum_order(ora):
    """The server adds the W decompressed workers in ascending worker order, then divides
    by W. Three workers with b1 = 0 (so z = g) and constant chunks of 1, 2^-24, 2^-24:
    their scales are exactly those values; ascending, 1 + 2^-24 rounds back to 1 (a tie,
    to even) twice, so the average is rn(1/3); in the other order 2^-24 + 2^-24 = 2^-23
    survives and the average would be rn((1 + 2^-23)/3), a different float32."""
    n, W, C = 256, 3, 256
    vals = [1.0, 2.0 ** -24, 2.0 ** -24]
    g = np.stack([np.full(n, v, np.float32) for v in vals])
    st = O.OracleState(n, W, C, x=np.zeros(n), m=np.zeros(n), v=np.ones(n), b1=0.0, lr=1e-4)
    out = ora.compressed_step(st, g)
    assert np.array_equal(out["wscale"][:, 0], _f32(vals))
    third = np.float32(np.float32(1.0) / np.float32(3.0))
    other = np.float32(np.float32(1.0 + 2.0 ** -23) / np.float32(3.0))
    assert third != other
    assert np.all(out["y"] == third)
    assert np.all(st.m == third)                      # constant chunk: T = |y|, all signs +


def pin_mean_orders(ora):
    """The warm-up's gradient mean and LoCo's dequantized mean add the workers in
    ascending order too (cases where the order decides the rounding; b1 = 0, so m is the
    mean itself). Warm-up: 1, 2^-24, 2^-24 as in the server's case. LoCo: worker 0's
    chunk is all 7 (scale 1, level 7), workers 1 and 2 have level 1 at scale 2^-22 (one
    element at level 7 sets that scale); ascending, 7 + 2^-22 is a tie that rounds back
    to 7 twice; in the other order 2^-22 + 2^-22 = 2^-21 would survive."""
    n, W = 256, 3
    st = O.OracleState(n, W, n, x=np.zeros(n), m=np.zeros(n), v=np.zeros(n), b1=0.0, lr=1e-4)
    g = np.stack([np.full(n, v, np.float32) for v in (1.0, 2.0 ** -24, 2.0 ** -24)])
    ora.warmup_step(st, g)
    third = np.float32(np.float32(1.0) / np.float32(3.0))
    assert np.all(st.m == third)
    g = np.full((W, n), 2.0 ** -22, np.float32)
    g[0] = 7.0
    g[1:, 0] = 7.0 * 2.0 ** -22
    st = O.OracleState(n, W, n, x=np.zeros(n), m=np.zeros(n), v=np.zeros(n), b1=0.0, lr=1e-4)
    err = np.zeros((W, n), np.float32)
    out = ora.loco_step(st, g, err, beta=0.0, bits=4)
    assert np.array_equal(out["scales"][:, 0], _f32([1.0, 2.0 ** -22, 2.0 ** -22]))
    want = np.float32(np.float32(7.0) / np.float32(3.0))
    other = np.float32(np.float32(7.0 + 2.0 ** -21) / np.float32(3.0))
    assert want != other
    assert np.all(st.m[1:] == want)


def pin_loco_adam_is_the_warmup_step(ora):
    """With gradients that quantize exactly (every chunk has a level of +-7 steps and its
    own power-of-two step, so c = q*s with zero error and e~ stays zero), the dequantized
    mean equals the plain mean and the LoCo step's Adam part must equal the warm-up step
    (pinned against torch.optim.AdamW) bit for bit, from non-zero m and v, step after
    step: the same b1, b2, chunk-by-chunk scales and update."""
    rng = np.random.default_rng(88)
    n, W, C = 1024, 2, 256
    st_l = _rand_state(rng, n, W, C, b1=0.9, b2=0.999, eps=1e-8, lr=1e-3)
    st_l.m[:] = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    st_w = st_l.copy()
    err = np.zeros((W, n), np.float32)
    for step in range(3):
        q = rng.integers(-7, 8, (W, n)).astype(np.float32)
        q[:, ::C] = rng.choice([-7.0, 7.0], (W, n // C))                # a +-7 in every chunk
        steps = np.float32(2.0) ** rng.integers(-14, -8, (W, n // C)).astype(np.float32)
        g = (q * np.repeat(steps, C, axis=1)).astype(np.float32)
        out = ora.loco_step(st_l, g, err, beta=0.9, bits=4)
        ora.warmup_step(st_w, g)
        assert np.array_equal(out["scales"], steps)
        assert not err.any()
        for name in ("x", "m", "v"):
            assert _same_bits(getattr(st_l, name), getattr(st_w, name)), (step, name)


PINS = {name[4:]: fn for name, fn in sorted(globals().items())
        if name.startswith("pin_") and callable(fn)}
