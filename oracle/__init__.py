"""CPU oracle for the 1-bit Adam compression-stage step (numpy interface over plain C).

TEST INFRASTRUCTURE ONLY. Only the tests, the package's smoke check and the
benchmark's CPU-baseline leg may import this module. The product path (the CUDA
library and its binding) never imports, loads or calls anything here, and the two
share no code: only the seeded input generators feed both.

The arithmetic lives in ``ob_oracle.c`` (see its header for the passages it follows
and the readings taken where the pages are silent). This module only marshals numpy
arrays, plus the closed-form communication count below, which is not arithmetic of
the step itself.
"""
import ctypes

import numpy as np

from . import build as _build

F32, F16, BF16 = 0, 1, 2

_f32p = ctypes.POINTER(ctypes.c_float)
_u32p = ctypes.POINTER(ctypes.c_uint32)
_u8p = ctypes.POINTER(ctypes.c_uint8)
_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_i32 = ctypes.c_int32
_f = ctypes.c_float


def _p(a, ctype):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle buffers must be C-contiguous"
    return a.ctypes.data_as(ctype)


def grad_code(g):
    """Storage code of a gradient array: float32 -> F32, float16 -> F16, uint16 -> BF16."""
    if g.dtype == np.float32:
        return F32
    if g.dtype == np.float16:
        return F16
    if g.dtype == np.uint16:
        return BF16
    raise TypeError("gradients must be float32, float16 or raw bfloat16 (uint16)")


class Oracle:
    """Bound to one build of the oracle library (the default one, or a test variant)."""

    def __init__(self, lib_path=None):
        path = lib_path or _build.build()
        self.path = path
        lib = ctypes.CDLL(path)
        lib.ora_decode_grads.argtypes = [_vp, ctypes.c_int, _i64, _f32p]
        lib.ora_chunk_scale.argtypes = [_f32p, _i64]
        lib.ora_chunk_scale.restype = ctypes.c_float
        lib.ora_pack_signs.argtypes = [_f32p, _i64, _u32p]
        lib.ora_unpack.argtypes = [_u32p, _f32p, _i64, _i64, _f32p]
        lib.ora_onebit_compress.argtypes = [_f32p, _i64, _i64, _u32p, _f32p, _f32p]
        lib.ora_compressed_step.argtypes = [
            _i64, _i32, _i64, _f, _f, _f, _f, _vp, ctypes.c_int,
            _f32p, _f32p, _f32p, _f32p, _f32p, _u8p, ctypes.c_int,
            _f32p, _u32p, _f32p, _f32p, _u32p, _f32p]
        lib.ora_compressed_step.restype = ctypes.c_int
        lib.ora_warmup_step.argtypes = [
            _i64, _i32, _f, _f, _f, _f, _f, _f, _f, _vp, ctypes.c_int, _f32p, _f32p, _f32p]
        lib.ora_warmup_step.restype = ctypes.c_int
        lib.ora_loco_step.argtypes = [
            _i64, _i32, _i64, ctypes.c_int, _f, _f, _f, _f, _f, _f, _f, _vp, ctypes.c_int,
            _f32p, _f32p, _f32p, _f32p, _u8p, _f32p]
        lib.ora_loco_step.restype = ctypes.c_int
        self.lib = lib

    # -- building blocks -----------------------------------------------------------
    def decode_grads(self, g):
        g = np.ascontiguousarray(g)
        out = np.empty(g.shape, np.float32)
        self.lib.ora_decode_grads(g.ctypes.data, grad_code(g), g.size, _p(out, _f32p))
        return out

    def chunk_scale(self, z):
        z = np.ascontiguousarray(z, np.float32)
        return np.float32(self.lib.ora_chunk_scale(_p(z, _f32p), z.size))

    def pack_signs(self, z):
        z = np.ascontiguousarray(z, np.float32)
        assert z.size % 32 == 0
        out = np.empty(z.size // 32, np.uint32)
        self.lib.ora_pack_signs(_p(z, _f32p), z.size, _p(out, _u32p))
        return out

    def unpack(self, words, scales, n, C):
        words = np.ascontiguousarray(words, np.uint32)
        scales = np.ascontiguousarray(scales, np.float32)
        out = np.empty(n, np.float32)
        self.lib.ora_unpack(_p(words, _u32p), _p(scales, _f32p), n, C, _p(out, _f32p))
        return out

    def onebit_compress(self, z, C):
        z = np.ascontiguousarray(z, np.float32)
        n = z.size
        words = np.empty(n // 32, np.uint32)
        scales = np.empty(n // C, np.float32)
        resid = np.empty(n, np.float32)
        self.lib.ora_onebit_compress(_p(z, _f32p), n, C, _p(words, _u32p), _p(scales, _f32p),
                                     _p(resid, _f32p))
        return words, scales, resid

    # -- steps -----------------------------------------------------------------------
    def compressed_step(self, st, grads, identity=False):
        """One compression-stage step on ``st`` (an OracleState, updated in place).

        Returns the step's intermediate products: z [W,n], worker words [W,n/32],
        worker scales [W,n/C], y [n], server words [n/32], server scales [n/C].
        """
        n, W, C = st.n, st.W, st.C
        g = np.ascontiguousarray(grads)
        assert g.size == W * n
        z = np.empty((W, n), np.float32)
        ww = np.empty((W, n // 32), np.uint32)
        wsc = np.empty((W, n // C), np.float32)
        y = np.empty(n, np.float32)
        sw = np.empty(n // 32, np.uint32)
        ssc = np.empty(n // C, np.float32)
        rc = self.lib.ora_compressed_step(
            n, W, C, st.b1, st.eps, st.lr, st.wd, g.ctypes.data, grad_code(g),
            _p(st.x, _f32p), _p(st.m, _f32p), _p(st.v, _f32p), _p(st.ew, _f32p),
            _p(st.es, _f32p), _p(st.mask, _u8p), int(bool(identity)),
            _p(z, _f32p), _p(ww, _u32p), _p(wsc, _f32p), _p(y, _f32p), _p(sw, _u32p),
            _p(ssc, _f32p))
        if rc != 0:
            raise ValueError("ora_compressed_step rejected its arguments (%d)" % rc)
        st.step += 1
        return dict(z=z, wbits=ww, wscale=wsc, y=y, sbits=sw, sscale=ssc)

    def warmup_step(self, st, grads, bias_correction=False):
        g = np.ascontiguousarray(grads)
        assert g.size == st.W * st.n
        t = st.step + 1
        bc1, bc2 = bias_factors(st.b1, st.b2, t) if bias_correction else (1.0, 1.0)
        rc = self.lib.ora_warmup_step(st.n, st.W, st.b1, st.b2, st.eps, st.lr, st.wd, bc1, bc2,
                                      g.ctypes.data, grad_code(g), _p(st.x, _f32p),
                                      _p(st.m, _f32p), _p(st.v, _f32p))
        if rc != 0:
            raise ValueError("ora_warmup_step rejected its arguments (%d)" % rc)
        st.step += 1

    def loco_step(self, st, grads, loco_err, beta=0.9, bits=4, ratio=1.0):
        n, W, C = st.n, st.W, st.C
        g = np.ascontiguousarray(grads)
        assert g.size == W * n and loco_err.shape == (W, n)
        codes = np.empty((W, n * bits // 8), np.uint8)
        scales = np.empty((W, n // C), np.float32)
        rc = self.lib.ora_loco_step(n, W, C, bits, st.b1, st.b2, st.eps, st.lr, st.wd, beta, ratio,
                                    g.ctypes.data, grad_code(g), _p(st.x, _f32p),
                                    _p(st.m, _f32p), _p(st.v, _f32p), _p(loco_err, _f32p),
                                    _p(codes, _u8p), _p(scales, _f32p))
        if rc != 0:
            raise ValueError("ora_loco_step rejected its arguments (%d)" % rc)
        st.step += 1
        return dict(codes=codes, scales=scales)


def bias_factors(b1, b2, t):
    """Adam's bias-correction divisors (1 - b1^t, 1 - b2^t), as float32 values.

    Computed in double and rounded once; the CUDA library's host code derives the same
    two numbers the same way, so both sides divide by identical float32 values.
    """
    return (float(np.float32(1.0 - float(np.float32(b1)) ** t)),
            float(np.float32(1.0 - float(np.float32(b2)) ** t)))


class OracleState:
    """Host-side optimizer state in canonical form (errors are the true residuals)."""

    def __init__(self, n, W, C, x, m, v, b1=0.9, b2=0.999, eps=1e-8, lr=1e-4, wd=0.0,
                 ew=None, es=None, mask=None):
        self.n, self.W, self.C = int(n), int(W), int(C)
        self.b1, self.b2, self.eps, self.lr, self.wd = b1, b2, eps, lr, wd
        self.x = np.array(x, np.float32).reshape(n)
        self.m = np.array(m, np.float32).reshape(n)
        self.v = np.array(v, np.float32).reshape(n)
        self.ew = (np.zeros((W, n), np.float32) if ew is None
                   else np.array(ew, np.float32).reshape(W, n))
        self.es = np.zeros(n, np.float32) if es is None else np.array(es, np.float32).reshape(n)
        self.mask = None if mask is None else (np.asarray(mask).reshape(n) != 0).astype(np.uint8)
        self.step = 0

    def copy(self):
        c = OracleState(self.n, self.W, self.C, self.x, self.m, self.v, self.b1, self.b2,
                        self.eps, self.lr, self.wd, self.ew, self.es, self.mask)
        c.step = self.step
        return c


def comm_bytes_per_worker(n, W, C, dense_bytes=2):
    """Bytes one worker sends per step: compressed exchange vs. a dense ring AllReduce.

    The compressed exchange has two hops (worker -> server chunks, server -> all): in
    each a worker sends (W-1)/W of n sign bits plus (W-1) of its n/(W*C) chunk scales
    (float32). A ring AllReduce of dense values sends 2*(W-1)/W of n values.
    Returns (compressed_bytes, dense_bytes_sent).
    """
    hop_bits = (W - 1) / W * n / 8
    hop_scales = (W - 1) * (n // (W * C)) * 4
    compressed = 2 * (hop_bits + hop_scales)
    dense = 2 * (W - 1) / W * n * dense_bytes
    return compressed, dense


_DEFAULT = None


def default():
    """The oracle built from the committed source."""
    global _DEFAULT
    if _DEFAULT is None:
        _DEFAULT = Oracle()
    return _DEFAULT


__all__ = ["Oracle", "OracleState", "default", "comm_bytes_per_worker", "bias_factors",
           "grad_code", "F32", "F16", "BF16"]
