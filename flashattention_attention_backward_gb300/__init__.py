"""Python binding of the GB300 attention-backward C library (libattnbwd.so).

The functions below carry the names and argument order of the C ABI in
``include/attnbwd.h`` and only marshal arguments: pointers may be given as
integers or as objects with ``data_ptr()`` (torch tensors), streams as an
integer handle, a ``torch.cuda.Stream`` or None (legacy default stream).
Each returns the C return code; ``check(rc)`` turns a non-zero code into an
``AttnError``. All computation happens in the library's CUDA kernels; if the
library has not been built, every call raises.
"""
import ctypes
import os

from .build import LIB_PATH

__all__ = [
    "AttnError", "check", "library", "attn_fwd", "attn_fwd_ref", "attn_bwd_preprocess", "attn_bwd",
    "attn_bwd_finalize", "attn_bwd_noalloc", "attn_device_status", "attn_strerror",
    "attn_selftest_wait_timeout", "attn_bwd_dq_partials_bytes", "attn_bwd_deterministic",
    "attn_bwd_finalize_partials", "attn_fwd_ref_dropout", "attn_bwd_dropout", "attn_fwd_local",
    "attn_fwd_ref_local", "attn_bwd_local", "attn_fwd_dropout",
    "ATTN_OK", "ATTN_ERR_NULL", "ATTN_ERR_SHAPE", "ATTN_ERR_UNSUPPORTED", "ATTN_ERR_ALIGN",
    "ATTN_ERR_LAUNCH", "ATTN_ERR_DEVICE_TIMEOUT", "ATTN_ERR_DEVICE", "ATTN_ERR_TOO_LARGE",
]

ATTN_OK = 0
ATTN_ERR_NULL = -1
ATTN_ERR_SHAPE = -2
ATTN_ERR_UNSUPPORTED = -3
ATTN_ERR_ALIGN = -4
ATTN_ERR_LAUNCH = -5
ATTN_ERR_DEVICE_TIMEOUT = -6
ATTN_ERR_DEVICE = -7
ATTN_ERR_TOO_LARGE = -8

_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float

_SIGNATURES = {
    "attn_fwd_ref": [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _F, _P],
    "attn_fwd": [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _F, _P],
    "attn_bwd_preprocess": [_P, _P, _P, _P, _I, _I, _I, _I, _P],
    "attn_bwd": [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _F, _P, _P],
    "attn_bwd_finalize": [_P, _P, _F, _I, _I, _I, _I, _P],
    "attn_device_status": [ctypes.POINTER(ctypes.c_int), _I, _P],
    "attn_selftest_wait_timeout": [ctypes.POINTER(ctypes.c_int), _P],
    "attn_bwd_deterministic": [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _F,
                               _P, _P],
    "attn_bwd_finalize_partials": [_P, _P, _F, _I, _I, _I, _I, _I, _P],
    "attn_fwd_ref_dropout": [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _F, _F,
                             ctypes.c_ulonglong, _P],
    "attn_bwd_dropout": [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _F, _P,
                         _F, ctypes.c_ulonglong, _P],
    "attn_fwd_dropout": [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _F, _F,
                         ctypes.c_ulonglong, _P],
    "attn_bwd_noalloc": [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _F, _P],
    "attn_fwd_local": [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _F, _I, _I, _P],
    "attn_fwd_ref_local": [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _F, _I, _I, _P],
    "attn_bwd_local": [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _F, _P,
                       _I, _I, _P],
}

_lib = None


class AttnError(RuntimeError):
    def __init__(self, code):
        super().__init__("attention library error %d: %s" % (code, attn_strerror(code)))
        self.code = code


def library():
    """The loaded ctypes library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                "libattnbwd.so is not built (%s missing); run "
                "flashattention_attention_backward_gb300.build.build()" % LIB_PATH)
        lib = ctypes.CDLL(LIB_PATH)
        for name, args in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        lib.attn_bwd_dq_partials_bytes.argtypes = [_I, _I, _I, _I, _I]
        lib.attn_bwd_dq_partials_bytes.restype = ctypes.c_longlong
        lib.attn_strerror.argtypes = [ctypes.c_int]
        lib.attn_strerror.restype = ctypes.c_char_p
        _lib = lib
    return _lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def check(rc):
    if rc != ATTN_OK:
        raise AttnError(rc)
    return rc


def attn_fwd_ref(q, k, v, o, lse, B, H, H_kv, N, d, scale, causal, softcap, stream=None):
    return library().attn_fwd_ref(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, H_kv, N,
                                  d, scale, int(causal), softcap, _stream(stream))


def attn_fwd(q, k, v, o, lse, B, H, H_kv, N, d, scale, causal, softcap, stream=None):
    return library().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, H_kv, N, d,
                              scale, int(causal), softcap, _stream(stream))


def attn_bwd_preprocess(o, dO, dpsum, dq_accum, B, H, N, d, stream=None):
    return library().attn_bwd_preprocess(_ptr(o), _ptr(dO), _ptr(dpsum), _ptr(dq_accum), B, H,
                                         N, d, _stream(stream))


def attn_bwd(q, k, v, o, dO, lse, dq_accum, dk, dv, B, H, H_kv, N, d, scale, causal, softcap,
             dpsum, stream=None):
    return library().attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), _ptr(lse),
                              _ptr(dq_accum), _ptr(dk), _ptr(dv), B, H, H_kv, N, d, scale,
                              int(causal), softcap, _ptr(dpsum), _stream(stream))


def attn_bwd_finalize(dq_accum, dq, scale, B, H, N, d, stream=None):
    return library().attn_bwd_finalize(_ptr(dq_accum), _ptr(dq), scale, B, H, N, d,
                                       _stream(stream))


def attn_bwd_noalloc(q, k, v, o, dO, lse, dq, dk, dv, B, H, H_kv, N, d, scale, causal, softcap,
                     stream=None):
    return library().attn_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), _ptr(lse),
                                      _ptr(dq), _ptr(dk), _ptr(dv), B, H, H_kv, N, d, scale,
                                      int(causal), softcap, _stream(stream))


def attn_fwd_ref_dropout(q, k, v, o, lse, B, H, H_kv, N, d, scale, causal, softcap, p_drop, seed,
                         stream=None):
    return library().attn_fwd_ref_dropout(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H,
                                          H_kv, N, d, scale, int(causal), softcap, p_drop,
                                          int(seed) & 0xFFFFFFFFFFFFFFFF, _stream(stream))


def attn_fwd_dropout(q, k, v, o, lse, B, H, H_kv, N, d, scale, causal, softcap, p_drop, seed,
                     stream=None):
    return library().attn_fwd_dropout(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, H_kv,
                                      N, d, scale, int(causal), softcap, p_drop,
                                      int(seed) & 0xFFFFFFFFFFFFFFFF, _stream(stream))


def attn_bwd_dropout(q, k, v, o, dO, lse, dq_accum, dk, dv, B, H, H_kv, N, d, scale, causal,
                     softcap, dpsum, p_drop, seed, stream=None):
    return library().attn_bwd_dropout(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), _ptr(lse), _ptr(dq_accum), _ptr(dk),
        _ptr(dv), B, H, H_kv, N, d, scale, int(causal), softcap, _ptr(dpsum), p_drop,
        int(seed) & 0xFFFFFFFFFFFFFFFF, _stream(stream))


def attn_fwd_local(q, k, v, o, lse, B, H, H_kv, N, d, scale, causal, softcap, window_left,
                   window_right, stream=None):
    return library().attn_fwd_local(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, H_kv, N,
                                    d, scale, int(causal), softcap, int(window_left),
                                    int(window_right), _stream(stream))


def attn_fwd_ref_local(q, k, v, o, lse, B, H, H_kv, N, d, scale, causal, softcap, window_left,
                       window_right, stream=None):
    return library().attn_fwd_ref_local(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H,
                                        H_kv, N, d, scale, int(causal), softcap,
                                        int(window_left), int(window_right), _stream(stream))


def attn_bwd_local(q, k, v, o, dO, lse, dq_accum, dk, dv, B, H, H_kv, N, d, scale, causal,
                   softcap, dpsum, window_left, window_right, stream=None):
    return library().attn_bwd_local(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), _ptr(lse), _ptr(dq_accum), _ptr(dk),
        _ptr(dv), B, H, H_kv, N, d, scale, int(causal), softcap, _ptr(dpsum), int(window_left),
        int(window_right), _stream(stream))


def attn_bwd_dq_partials_bytes(B, H, N, d, causal):
    return library().attn_bwd_dq_partials_bytes(B, H, N, d, int(causal))


def attn_bwd_deterministic(q, k, v, o, dO, lse, dq_partials, dk, dv, B, H, H_kv, N, d, scale,
                           causal, softcap, dpsum, stream=None):
    return library().attn_bwd_deterministic(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), _ptr(lse), _ptr(dq_partials), _ptr(dk),
        _ptr(dv), B, H, H_kv, N, d, scale, int(causal), softcap, _ptr(dpsum), _stream(stream))


def attn_bwd_finalize_partials(dq_partials, dq, scale, B, H, N, d, causal, stream=None):
    return library().attn_bwd_finalize_partials(_ptr(dq_partials), _ptr(dq), scale, B, H, N, d,
                                                int(causal), _stream(stream))


def attn_device_status(clear=True, stream=None):
    """Returns (rc, status): the library's device status word."""
    v = ctypes.c_int(0)
    rc = library().attn_device_status(ctypes.byref(v), int(clear), _stream(stream))
    return rc, v.value


def attn_selftest_wait_timeout(stream=None):
    """Returns (rc, status) of the device-side bounded-wait self test; the
    status is ATTN_ERR_DEVICE_TIMEOUT when waits give up as designed."""
    v = ctypes.c_int(0)
    rc = library().attn_selftest_wait_timeout(ctypes.byref(v), _stream(stream))
    return rc, v.value


def attn_strerror(code):
    return library().attn_strerror(int(code)).decode()
