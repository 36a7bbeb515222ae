"""ctypes binding of the C ABI in include/fa.h (argument marshalling only).

Every function here has the name and argument order of its C counterpart.
Pointer arguments accept an integer device address, ``None`` (NULL) or any
object with ``data_ptr()`` (a torch tensor); ``stream`` accepts an integer
handle, ``None`` (the legacy default stream) or a ``torch.cuda.Stream``.
All arithmetic runs in the CUDA library: if it is not built, loading fails
loudly -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
# ATTN_BWD_GB300_LIB may name another build of the same library (e.g. the bounds-checking
# debug build, libattn_bwd_gb300_bounds.so); it is read once, at import.
LIB_PATH = os.environ.get("ATTN_BWD_GB300_LIB") or os.path.join(_HERE, "libattn_bwd_gb300.so")

FA_OK = 0
FA_ERR_NULL = 1
FA_ERR_SHAPE = 2
FA_ERR_HEADDIM = 3
FA_ERR_GQA = 4
FA_ERR_ALIGN = 5
FA_ERR_WORKSPACE = 6
FA_ERR_DTYPE = 7
FA_ERR_CUDA = 8
FA_ERR_DEVICE_TIMEOUT = 9
FA_ERR_ARG = 10
FA_ERR_BOUNDS = 11
FA_F16 = 0
FA_BF16 = 1
FA_CAUSAL_NONE = 0
FA_CAUSAL_TOP_LEFT = 1
FA_CAUSAL_BOTTOM_RIGHT = 2

class fa_stride3(ctypes.Structure):
    _fields_ = [("b", ctypes.c_longlong), ("h", ctypes.c_longlong), ("n", ctypes.c_longlong)]


class fa_strides(ctypes.Structure):
    _fields_ = [(n, fa_stride3) for n in ("q", "k", "v", "o", "dO", "dq", "dk", "dv", "lse")]


class fa_bias(ctypes.Structure):
    _fields_ = [("bias", ctypes.c_void_p), ("bias_strides", fa_stride3), ("dbias", ctypes.c_void_p),
                ("dbias_strides", fa_stride3)]


_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_S = ctypes.c_size_t

_SIGNATURES = {
    "fa_fwd": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _I, _P]),
    "fa_bwd_workspace_size": (_S, [_I, _I, _I, _I, _I, _I, _I]),
    "fa_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _I, _I, _P, _S, _P]),
    "fa_bwd_preprocess": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _P, _S, _P]),
    "fa_bwd_main": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _I, _I, _P, _S, _P]),
    "fa_bwd_dq": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _I, _I, _P, _S, _P]),
    "fa_strerror": (ctypes.c_char_p, [_I]),
    "fa_last_device_error": (_I, [_P]),
    "fa_selftest_wait_timeout": (_I, [_I, _P]),
    "fa_bwd_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _I, _I, _P]),
    "fa_fwd_varlen": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _F, _I, _I, _P]),
    "fa_bwd_varlen_workspace_size": (_S, [_I, _I, _I, _I, _I, _I, _I]),
    "fa_bwd_varlen": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _F, _I, _I,
                           _I, _P, _S, _P]),
    "fa_fwd_strided": (_I, [_P, _P, _P, _P, _P, ctypes.POINTER(fa_strides), _P, _P, _I, _I, _I, _I, _I, _I, _I, _I,
                            _F, _I, _I, _P]),
    "fa_bwd_strided": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.POINTER(fa_strides), _P, _P, _I, _I, _I, _I,
                            _I, _I, _I, _I, _F, _I, _I, _I, _P, _S, _P]),
    "fa_bwd_host_staging_size": (_S, [_I, _I, _I, _I, _I, _I, _I, _I, _I]),
    "fa_bwd_host": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _I, _I, _I, _I, _P, _S,
                         _P]),
    "fa_fwd_bias": (_I, [_P, _P, _P, _P, _P, ctypes.POINTER(fa_bias), ctypes.POINTER(fa_strides), _P, _P, _I, _I,
                         _I, _I, _I, _I, _I, _I, _F, _I, _I, _P]),
    "fa_bwd_bias": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.POINTER(fa_bias), ctypes.POINTER(fa_strides),
                         _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _F, _I, _I, _I, _P, _S, _P]),
}

FA_STATIC_SCRATCH_BYTES = 64 << 20
FA_HOST_MAX_SLOTS = 8

_lib = None


def load():
    """Load the shared library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"CUDA library not built: {LIB_PATH} is missing "
                "(run `python -m attn_bwd_gb300.build` or __graft_entry__.build())")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _ptr(x):
    if x is None:
        return None
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    return int(x)


def _stream(s):
    if s is None:
        return None
    if hasattr(s, "cuda_stream"):
        return s.cuda_stream
    return int(s)


def fa_strerror(status: int) -> str:
    return load().fa_strerror(int(status)).decode()


def fa_fwd(q, k, v, o, lse, B, Hq, Hkv, Nq, Nkv, d, scale, causal, dtype, stream=None) -> int:
    return load().fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Nq, Nkv, d,
                         float(scale), int(causal), int(dtype), _stream(stream))


def fa_bwd_workspace_size(B, Hq, Hkv, Nq, Nkv, d, deterministic) -> int:
    return load().fa_bwd_workspace_size(B, Hq, Hkv, Nq, Nkv, d, int(deterministic))


def fa_bwd(q, k, v, o, dO, lse, dq, dk, dv, B, Hq, Hkv, Nq, Nkv, d, scale, causal, dtype, deterministic,
           workspace, workspace_bytes, stream=None) -> int:
    return load().fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
                         B, Hq, Hkv, Nq, Nkv, d, float(scale), int(causal), int(dtype), int(deterministic),
                         _ptr(workspace), int(workspace_bytes), _stream(stream))


def fa_bwd_preprocess(o, dO, lse, B, Hq, Hkv, Nq, Nkv, d, dtype, deterministic, workspace, workspace_bytes,
                      stream=None) -> int:
    return load().fa_bwd_preprocess(_ptr(o), _ptr(dO), _ptr(lse), B, Hq, Hkv, Nq, Nkv, d, int(dtype),
                                    int(deterministic), _ptr(workspace), int(workspace_bytes), _stream(stream))


def fa_bwd_main(q, k, v, dO, dk, dv, B, Hq, Hkv, Nq, Nkv, d, scale, causal, dtype, deterministic, workspace,
                workspace_bytes, stream=None) -> int:
    return load().fa_bwd_main(_ptr(q), _ptr(k), _ptr(v), _ptr(dO), _ptr(dk), _ptr(dv), B, Hq, Hkv, Nq, Nkv, d,
                              float(scale), int(causal), int(dtype), int(deterministic), _ptr(workspace),
                              int(workspace_bytes), _stream(stream))


def fa_bwd_dq(q, k, v, dO, dq, B, Hq, Hkv, Nq, Nkv, d, scale, causal, dtype, deterministic, workspace,
              workspace_bytes, stream=None) -> int:
    return load().fa_bwd_dq(_ptr(q), _ptr(k), _ptr(v), _ptr(dO), _ptr(dq), B, Hq, Hkv, Nq, Nkv, d, float(scale),
                            int(causal), int(dtype), int(deterministic), _ptr(workspace), int(workspace_bytes),
                            _stream(stream))


def fa_last_device_error(stream=None) -> int:
    return load().fa_last_device_error(_stream(stream))


def fa_selftest_wait_timeout(timeout_us, stream=None) -> int:
    return load().fa_selftest_wait_timeout(int(timeout_us), _stream(stream))


def fa_bwd_noalloc(q, k, v, o, dO, lse, dq, dk, dv, B, Hq, Hkv, Nq, Nkv, d, scale, causal, dtype, deterministic,
                   stream=None) -> int:
    """fa_bwd without a workspace argument, for callers that cannot allocate device memory
    (its scratch is a fixed FA_STATIC_SCRATCH_BYTES array inside the library)."""
    return load().fa_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), _ptr(lse), _ptr(dq), _ptr(dk),
                                 _ptr(dv), B, Hq, Hkv, Nq, Nkv, d, float(scale), int(causal), int(dtype),
                                 int(deterministic), _stream(stream))


def fa_fwd_varlen(q, k, v, o, lse, cu_q, cu_k, B, Hq, Hkv, total_q, total_k, max_q, max_k, d, scale, causal, dtype,
                  stream=None) -> int:
    """Packed variable-length forward: q [Hq, total_q, d], k/v [Hkv, total_k, d], cu_* int32 [B + 1] on the device."""
    return load().fa_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(cu_q), _ptr(cu_k), B, Hq, Hkv,
                                total_q, total_k, max_q, max_k, d, float(scale), int(causal), int(dtype),
                                _stream(stream))


def fa_bwd_varlen_workspace_size(B, Hq, Hkv, max_q, max_k, d, deterministic) -> int:
    return load().fa_bwd_varlen_workspace_size(B, Hq, Hkv, max_q, max_k, d, int(deterministic))


def fa_bwd_varlen(q, k, v, o, dO, lse, dq, dk, dv, cu_q, cu_k, B, Hq, Hkv, total_q, total_k, max_q, max_k, d, scale,
                  causal, dtype, deterministic, workspace, workspace_bytes, stream=None) -> int:
    return load().fa_bwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), _ptr(lse), _ptr(dq), _ptr(dk),
                                _ptr(dv), _ptr(cu_q), _ptr(cu_k), B, Hq, Hkv, total_q, total_k, max_q, max_k, d,
                                float(scale), int(causal), int(dtype), int(deterministic), _ptr(workspace),
                                int(workspace_bytes), _stream(stream))


def make_strides(**kw) -> fa_strides:
    """fa_strides from (b, h, n) element-stride triples keyed q, k, v, o, dO, dq, dk, dv, lse."""
    st = fa_strides()
    for name, (b, h, n) in kw.items():
        setattr(st, name, fa_stride3(int(b), int(h), int(n)))
    return st


def fa_fwd_strided(q, k, v, o, lse, strides, cu_q, cu_k, B, Hq, Hkv, Nq, Nkv, total_q, total_k, d, scale, causal,
                   dtype, stream=None) -> int:
    sp = ctypes.byref(strides) if strides is not None else None
    return load().fa_fwd_strided(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), sp, _ptr(cu_q), _ptr(cu_k), B, Hq,
                                 Hkv, Nq, Nkv, total_q, total_k, d, float(scale), int(causal), int(dtype),
                                 _stream(stream))


def fa_bwd_strided(q, k, v, o, dO, lse, dq, dk, dv, strides, cu_q, cu_k, B, Hq, Hkv, Nq, Nkv, total_q, total_k, d,
                   scale, causal, dtype, deterministic, workspace, workspace_bytes, stream=None) -> int:
    sp = ctypes.byref(strides) if strides is not None else None
    return load().fa_bwd_strided(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), _ptr(lse), _ptr(dq), _ptr(dk),
                                 _ptr(dv), sp, _ptr(cu_q), _ptr(cu_k), B, Hq, Hkv, Nq, Nkv, total_q, total_k, d,
                                 float(scale), int(causal), int(dtype), int(deterministic), _ptr(workspace),
                                 int(workspace_bytes), _stream(stream))


def make_bias(bias, bias_strides, dbias=None, dbias_strides=(0, 0, 0)) -> fa_bias:
    """fa_bias from a bias pointer and its (b, h, q) element strides (0 broadcasts), and an optional dBias."""
    return fa_bias(_ptr(bias), fa_stride3(*[int(x) for x in bias_strides]), _ptr(dbias),
                   fa_stride3(*[int(x) for x in dbias_strides]))


def fa_fwd_bias(q, k, v, o, lse, bias, strides, cu_q, cu_k, B, Hq, Hkv, Nq, Nkv, total_q, total_k, d, scale, causal,
                dtype, stream=None) -> int:
    bp = ctypes.byref(bias) if bias is not None else None
    sp = ctypes.byref(strides) if strides is not None else None
    return load().fa_fwd_bias(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), bp, sp, _ptr(cu_q), _ptr(cu_k), B, Hq,
                              Hkv, Nq, Nkv, total_q, total_k, d, float(scale), int(causal), int(dtype),
                              _stream(stream))


def fa_bwd_bias(q, k, v, o, dO, lse, dq, dk, dv, bias, strides, cu_q, cu_k, B, Hq, Hkv, Nq, Nkv, total_q, total_k, d,
                scale, causal, dtype, deterministic, workspace, workspace_bytes, stream=None) -> int:
    bp = ctypes.byref(bias) if bias is not None else None
    sp = ctypes.byref(strides) if strides is not None else None
    return load().fa_bwd_bias(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
                              bp, sp, _ptr(cu_q), _ptr(cu_k), B, Hq, Hkv, Nq, Nkv, total_q, total_k, d, float(scale),
                              int(causal), int(dtype), int(deterministic), _ptr(workspace), int(workspace_bytes),
                              _stream(stream))


def fa_bwd_host_staging_size(B, Hq, Hkv, Nq, Nkv, d, deterministic, chunk_groups, slots) -> int:
    return load().fa_bwd_host_staging_size(B, Hq, Hkv, Nq, Nkv, d, int(deterministic), int(chunk_groups), int(slots))


def fa_bwd_host(q, k, v, o, dO, lse, dq, dk, dv, B, Hq, Hkv, Nq, Nkv, d, scale, causal, dtype, deterministic,
                chunk_groups, slots, staging, staging_bytes, stream=None) -> int:
    """fa_bwd on HOST tensors (pinned for overlap), pipelined through device staging memory."""
    return load().fa_bwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
                              B, Hq, Hkv, Nq, Nkv, d, float(scale), int(causal), int(dtype), int(deterministic),
                              int(chunk_groups), int(slots), _ptr(staging), int(staging_bytes), _stream(stream))
