"""Python binding of the C ABI in include/ob.h (argument marshalling only).

Every function here forwards to the CUDA library ``_build/libob.so``; no step of the
method runs in Python. Tensors are passed as raw device pointers, the stream as the
current torch stream unless one is given. If the library is missing the import fails
loudly: there is no fallback.
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libob.so")

OB_OK, OB_EINVAL, OB_ECUDA, OB_ENOTIMPL, OB_EALIGN, OB_ESCRATCH = 0, -1, -2, -3, -4, -5
OB_NOALLOC_SCRATCH_BYTES = 4 << 20
OB_F32, OB_F16, OB_BF16 = 0, 1, 2
(OB_K_WORKER, OB_K_SERVER, OB_K_UPDATE, OB_K_WARMUP, OB_K_LOCO_ABSMAX, OB_K_LOCO_QUANT,
 OB_K_LOCO_SERVER, OB_K_MASK, OB_K_EXPORT, OB_K_SCALES, OB_K_COUNT) = range(11)
KERNEL_NAMES = {OB_K_WORKER: "worker", OB_K_SERVER: "server", OB_K_UPDATE: "update",
                OB_K_WARMUP: "warmup", OB_K_LOCO_ABSMAX: "loco_absmax",
                OB_K_LOCO_QUANT: "loco_quant", OB_K_LOCO_SERVER: "loco_server",
                OB_K_MASK: "mask", OB_K_EXPORT: "export", OB_K_SCALES: "scales"}

# Symbols the header declares, with their ctypes signatures.
_vp, _i64, _i32, _f, _int, _sz = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32,
                                  ctypes.c_float, ctypes.c_int, ctypes.c_size_t)
SIGNATURES = {
    "ob_init": (_int, [_i64, _i32, _i64, _f, _f, _f, _f, ctypes.POINTER(_vp)]),
    "ob_destroy": (None, [_vp]),
    "ob_workspace_bytes": (_sz, [_vp]),
    "ob_workspace_init": (_int, [_vp, _vp, _vp]),
    "ob_set_lr": (_int, [_vp, _f]),
    "ob_set_options": (_int, [_vp, _f, _int]),
    "ob_set_step": (_int, [_vp, _i64]),
    "ob_get_step": (_i64, [_vp]),
    "ob_set_mask": (_int, [_vp, _vp, _vp, _vp]),
    "ob_warmup_step": (_int, [_vp, _vp, _int, _vp, _vp, _vp, _vp, _vp]),
    "ob_compressed_step": (_int, [_vp, _vp, _int, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "ob_compressed_step_host": (_int, [_vp, _vp, _vp, _int, _vp, _vp, _vp, _vp, _vp, _vp,
                                       _vp, _vp, _vp]),
    "ob_loco_step": (_int, [_vp, _vp, _int, _vp, _vp, _vp, _vp, _f, _int, _vp, _vp]),
    "ob_loco_workspace_bytes": (_sz, [_vp, _int]),
    "ob_reset_errors": (_int, [_vp, _vp, _vp, _vp, _vp]),
    "ob_export_state": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "ob_debug_views": (_int, [_vp, _vp, ctypes.POINTER(_vp), ctypes.POINTER(_vp),
                              ctypes.POINTER(_vp), ctypes.POINTER(_vp)]),
    "ob_profile": (_int, [_vp, _int]),
    "ob_profile_read": (_int, [_vp, _int, ctypes.POINTER(ctypes.c_double),
                               ctypes.POINTER(_i64)]),
    "ob_launch_count": (_i64, [_vp]),
    "ob_read_status": (_int, [_vp, _vp, ctypes.POINTER(ctypes.c_uint), _vp]),
    "ob_selftest_wait": (_int, [_vp, _vp, ctypes.c_uint64, _vp]),
    "ob_strerror": (ctypes.c_char_p, [_int]),
    "ob_last_cuda_error": (_int, []),
    "ob_set_loco_ratio": (_int, [_vp, _f]),
    "ob_set_loco_codes": (_int, [_vp, _int]),
    "ob_worker_compress_noalloc": (_int, [_vp, _vp, _int, _vp, _vp, _vp, _vp, _vp, _vp]),
    "ob_noalloc_read_status": (_int, [_vp, ctypes.POINTER(ctypes.c_uint), _vp]),
}

_LIB = None


class ObError(RuntimeError):
    def __init__(self, name, code):
        msg = _lib().ob_strerror(code).decode()
        if code == OB_ECUDA:
            msg += " (cuda error %d)" % _lib().ob_last_cuda_error()
        super().__init__("%s failed: %s [%d]" % (name, msg, code))
        self.code = code


def _lib():
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError("the CUDA library %s is not built; run "
                              "`python -m error_compensated_bit_gb300.build`" % LIB_PATH)
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = lib
    return _LIB


def load():
    """Load the library (raises ImportError if it is not built)."""
    return _lib()


def _call(name, *args):
    rc = getattr(_lib(), name)(*args)
    if rc != OB_OK:
        raise ObError(name, rc)


def dtype_code(t):
    return {torch.float32: OB_F32, torch.float16: OB_F16, torch.bfloat16: OB_BF16}[t.dtype]


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream, device=None):
    if stream is None:
        return torch.cuda.current_stream(device).cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class Context:
    """Owns one ``ob_ctx`` (host memory only)."""

    def __init__(self, n, W, chunk, b1=0.9, b2=0.999, eps=1e-8, lr=1e-4):
        h = ctypes.c_void_p()
        _call("ob_init", n, W, chunk, b1, b2, eps, lr, ctypes.byref(h))
        self.h = h
        self.n, self.W, self.chunk = int(n), int(W), int(chunk)

    def close(self):
        if self.h:
            _lib().ob_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def nchunks(self):
        return self.n // self.chunk

    def workspace_bytes(self):
        return int(_lib().ob_workspace_bytes(self.h))

    def loco_workspace_bytes(self, bits=4):
        return int(_lib().ob_loco_workspace_bytes(self.h, bits))

    def workspace_init(self, ws, stream=None):
        _call("ob_workspace_init", self.h, _ptr(ws), _stream(stream))

    def set_lr(self, lr):
        _call("ob_set_lr", self.h, lr)

    def set_options(self, weight_decay=0.0, bias_correction=False):
        _call("ob_set_options", self.h, weight_decay, int(bool(bias_correction)))

    def set_loco_ratio(self, ratio):
        _call("ob_set_loco_ratio", self.h, float(ratio))

    def set_loco_codes(self, keep):
        _call("ob_set_loco_codes", self.h, int(bool(keep)))

    def set_step(self, step):
        _call("ob_set_step", self.h, step)

    def get_step(self):
        return int(_lib().ob_get_step(self.h))

    def set_mask(self, mask01, ws, stream=None):
        _call("ob_set_mask", self.h, _ptr(mask01), _ptr(ws), _stream(stream))

    def warmup_step(self, grads, x, m, v, ws, stream=None):
        _call("ob_warmup_step", self.h, _ptr(grads), dtype_code(grads), _ptr(x), _ptr(m),
              _ptr(v), _ptr(ws), _stream(stream))

    def compressed_step(self, grads, x, m, v, worker_err, server_err, ws, stream=None):
        _call("ob_compressed_step", self.h, _ptr(grads), dtype_code(grads), _ptr(x), _ptr(m),
              _ptr(v), _ptr(worker_err), _ptr(server_err), _ptr(ws), _stream(stream))

    def compressed_step_host(self, grads_host, grads_dev, x, m, v, worker_err, server_err, ws,
                             sbits_host, sscale_host, stream=None):
        _call("ob_compressed_step_host", self.h, _ptr(grads_host), _ptr(grads_dev),
              dtype_code(grads_dev), _ptr(x), _ptr(m), _ptr(v), _ptr(worker_err),
              _ptr(server_err), _ptr(ws), _ptr(sbits_host), _ptr(sscale_host), _stream(stream))

    def loco_step(self, grads, x, m, v, loco_err, loco_ws, beta=0.9, bits=4, stream=None):
        _call("ob_loco_step", self.h, _ptr(grads), dtype_code(grads), _ptr(x), _ptr(m), _ptr(v),
              _ptr(loco_err), beta, bits, _ptr(loco_ws), _stream(stream))

    def reset_errors(self, worker_err, server_err, ws, stream=None):
        _call("ob_reset_errors", self.h, _ptr(worker_err), _ptr(server_err), _ptr(ws),
              _stream(stream))

    def export_state(self, worker_err, server_err, ws, ew_out, es_out, stream=None):
        _call("ob_export_state", self.h, _ptr(worker_err), _ptr(server_err), _ptr(ws),
              _ptr(ew_out), _ptr(es_out), _stream(stream))

    def debug_views(self, ws):
        """Device addresses (ints) of worker bits, worker scales, server bits, server scales."""
        out = [ctypes.c_void_p() for _ in range(4)]
        _call("ob_debug_views", self.h, _ptr(ws), *[ctypes.byref(o) for o in out])
        return [o.value for o in out]

    def profile(self, enable=True):
        _call("ob_profile", self.h, int(bool(enable)))

    def profile_read(self, kernel):
        ms = ctypes.c_double()
        cnt = ctypes.c_int64()
        _call("ob_profile_read", self.h, kernel, ctypes.byref(ms), ctypes.byref(cnt))
        return ms.value, cnt.value

    def launch_count(self):
        return int(_lib().ob_launch_count(self.h))

    def read_status(self, ws, stream=None):
        """Synchronize and return the workspace status word (0 = every kernel finished)."""
        st = ctypes.c_uint()
        _call("ob_read_status", self.h, _ptr(ws), ctypes.byref(st), _stream(stream))
        return st.value

    def selftest_wait(self, ws, limit_ns=1_000_000, stream=None):
        """Enqueue a bounded wait that runs out (sets status 1 in the workspace; with
        ws None, in the no-allocation worker pass's status word)."""
        _call("ob_selftest_wait", self.h, _ptr(ws), int(limit_ns), _stream(stream))

    def worker_compress_noalloc(self, grads, m, worker_err, scale_prev, wbits, scale_out,
                                stream=None):
        """The worker pass with its scratch in the library's fixed array (no workspace)."""
        _call("ob_worker_compress_noalloc", self.h, _ptr(grads), dtype_code(grads), _ptr(m),
              _ptr(worker_err), _ptr(scale_prev), _ptr(wbits), _ptr(scale_out), _stream(stream))

    def noalloc_read_status(self, stream=None):
        """Synchronize, return and clear the no-allocation worker pass's status word."""
        st = ctypes.c_uint()
        _call("ob_noalloc_read_status", self.h, ctypes.byref(st), _stream(stream))
        return st.value
