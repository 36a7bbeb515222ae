"""torch-tensor front end over the C ABI: checks, output allocation, stream.

PyTorch only supplies device memory and the current stream here; every
arithmetic step runs in the CUDA library through ``_lib``.
"""
from __future__ import annotations

import torch

from . import _lib

_DT = {torch.float16: _lib.FA_F16, torch.bfloat16: _lib.FA_BF16}


class FAError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {_lib.fa_strerror(status)} (fa_status {status})")
        self.status = status


def _check(status: int, where: str):
    if status != _lib.FA_OK:
        raise FAError(status, where)


def _dims(q, k):
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("expected [B, H, N, d] tensors")
    B, Hq, Nq, d = q.shape
    _, Hkv, Nkv, _ = k.shape
    return B, Hq, Hkv, Nq, Nkv, d


def _need(*ts):
    for t in ts:
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("tensors must be contiguous CUDA tensors")


def forward(q, k, v, scale: float, causal, stream=None):
    """Returns (O, L): O like q, L fp32 [B, Hq, Nq] (natural-log LSE of the scaled scores).

    ``causal``: False / True (top-left) or one of _lib.FA_CAUSAL_* (2 = bottom-right).
    """
    _need(q, k, v)
    B, Hq, Hkv, Nq, Nkv, d = _dims(q, k)
    o = torch.empty_like(q)
    lse = torch.empty(B, Hq, Nq, dtype=torch.float32, device=q.device)
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    _check(_lib.fa_fwd(q, k, v, o, lse, B, Hq, Hkv, Nq, Nkv, d, scale, causal, _DT[q.dtype], s), "fa_fwd")
    return o, lse


def workspace(q, k, deterministic: bool) -> torch.Tensor:
    B, Hq, Hkv, Nq, Nkv, d = _dims(q, k)
    n = _lib.fa_bwd_workspace_size(B, Hq, Hkv, Nq, Nkv, d, int(deterministic))
    if n == 0:
        raise ValueError("invalid shape for the backward")
    return torch.empty(n, dtype=torch.uint8, device=q.device)


def backward(q, k, v, o, do, lse, scale: float, causal, deterministic: bool = False, ws=None,
             out=None, stream=None):
    """Returns (dQ, dK, dV), freshly written (never accumulated)."""
    _need(q, k, v, o, do, lse)
    B, Hq, Hkv, Nq, Nkv, d = _dims(q, k)
    if ws is None:
        ws = workspace(q, k, deterministic)
    if out is None:
        out = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))
    dq, dk, dv = out
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    _check(_lib.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, B, Hq, Hkv, Nq, Nkv, d, scale, causal, _DT[q.dtype],
                       int(deterministic), ws, ws.numel(), s), "fa_bwd")
    return dq, dk, dv


# ------------------------------------------------------------ packed batches

def _cu(cu, device):
    """Offsets as a device int32 tensor, plus the lengths as host ints."""
    if isinstance(cu, torch.Tensor):
        host = [int(x) for x in cu.detach().cpu().tolist()]
    else:
        host = [int(x) for x in cu]
    dev = torch.tensor(host, dtype=torch.int32, device=device)
    lens = [b - a for a, b in zip(host, host[1:])]
    return dev, host, lens


def forward_varlen(q, k, v, cu_q, cu_k, scale: float, causal, max_q=None, max_k=None, stream=None):
    """Packed batch: q [Hq, total_q, d], k/v [Hkv, total_k, d]; cu_* are B + 1 offsets.
    Returns (O like q, L fp32 [Hq, total_q])."""
    _need(q, k, v)
    Hq, total_q, d = q.shape
    Hkv, total_k, _ = k.shape
    dq_, hq, lq = _cu(cu_q, q.device)
    dk_, hk, lk = _cu(cu_k, q.device)
    B = len(lq)
    max_q = max_q if max_q is not None else max(max(lq), 1)
    max_k = max_k if max_k is not None else max(max(lk), 1)
    o = torch.empty_like(q)
    lse = torch.empty(Hq, total_q, dtype=torch.float32, device=q.device)
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    _check(_lib.fa_fwd_varlen(q, k, v, o, lse, dq_, dk_, B, Hq, Hkv, total_q, total_k, max_q, max_k, d, scale,
                              causal, _DT[q.dtype], s), "fa_fwd_varlen")
    return o, lse


def backward_varlen(q, k, v, o, do, lse, cu_q, cu_k, scale: float, causal, deterministic: bool = False,
                    max_q=None, max_k=None, out=None, stream=None):
    """Packed-batch backward.  Returns (dQ, dK, dV) in the packed layouts."""
    _need(q, k, v, o, do, lse)
    Hq, total_q, d = q.shape
    Hkv, total_k, _ = k.shape
    dq_, hq, lq = _cu(cu_q, q.device)
    dk_, hk, lk = _cu(cu_k, q.device)
    B = len(lq)
    max_q = max_q if max_q is not None else max(max(lq), 1)
    max_k = max_k if max_k is not None else max(max(lk), 1)
    n = _lib.fa_bwd_varlen_workspace_size(B, Hq, Hkv, max_q, max_k, d, int(deterministic))
    if n == 0:
        raise ValueError("invalid shape for the backward")
    ws = torch.empty(n, dtype=torch.uint8, device=q.device)
    if out is None:
        out = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))
    dq, dk, dv = out
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    _check(_lib.fa_bwd_varlen(q, k, v, o, do, lse, dq, dk, dv, dq_, dk_, B, Hq, Hkv, total_q, total_k, max_q, max_k,
                              d, scale, causal, _DT[q.dtype], int(deterministic), ws, n, s), "fa_bwd_varlen")
    return dq, dk, dv


# ------------------------------------------------------------ strided tensors

def _str3(t):
    """(b, h, n) element strides of a [B, H, N, d] view, or of a [H, N] / [B, H, N] L."""
    st = t.stride()
    if t.dim() == 4:
        return st[0], st[1], st[2]
    if t.dim() == 3:
        return st[0], st[1], st[2]
    raise ValueError("expected a 3-D or 4-D tensor")


def _need_rows(*ts):
    for t in ts:
        if not t.is_cuda or t.stride(-1) != 1:
            raise ValueError("tensors must be CUDA tensors with a contiguous last (d) axis")


def forward_strided(q, k, v, scale: float, causal, stream=None):
    """Forward on [B, H, N, d] views with any strides (d contiguous), e.g. transposes of
    [B, N, H, d] tensors.  O is allocated with q's strides; L is contiguous [B, Hq, Nq]."""
    _need_rows(q, k, v)
    B, Hq, Nq, d = q.shape
    _, Hkv, Nkv, _ = k.shape
    o = torch.empty_like(q)
    lse = torch.empty(B, Hq, Nq, dtype=torch.float32, device=q.device)
    st = _lib.make_strides(q=_str3(q), k=_str3(k), v=_str3(v), o=_str3(o), dO=_str3(q), dq=_str3(q), dk=_str3(k),
                           dv=_str3(k), lse=_str3(lse))
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    _check(_lib.fa_fwd_strided(q, k, v, o, lse, st, None, None, B, Hq, Hkv, Nq, Nkv, 0, 0, d, scale, causal,
                               _DT[q.dtype], s), "fa_fwd_strided")
    return o, lse


def backward_strided(q, k, v, o, do, lse, scale: float, causal, deterministic: bool = False, out=None, stream=None):
    """Backward on [B, H, N, d] views with any strides (d contiguous); dQ, dK, dV are allocated
    like q, k, v unless ``out`` is given."""
    _need_rows(q, k, v, o, do)
    B, Hq, Nq, d = q.shape
    _, Hkv, Nkv, _ = k.shape
    if out is None:
        out = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))
    dq, dk, dv = out
    st = _lib.make_strides(q=_str3(q), k=_str3(k), v=_str3(v), o=_str3(o), dO=_str3(do), dq=_str3(dq),
                           dk=_str3(dk), dv=_str3(dv), lse=_str3(lse))
    n = _lib.fa_bwd_workspace_size(B, Hq, Hkv, Nq, Nkv, d, int(deterministic))
    if n == 0:
        raise ValueError("invalid shape for the backward")
    ws = torch.empty(n, dtype=torch.uint8, device=q.device)
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    _check(_lib.fa_bwd_strided(q, k, v, o, do, lse, dq, dk, dv, st, None, None, B, Hq, Hkv, Nq, Nkv, 0, 0, d, scale,
                               causal, _DT[q.dtype], int(deterministic), ws, n, s), "fa_bwd_strided")
    return dq, dk, dv


# ------------------------------------------------------------ additive bias

def _bias_strides(bias):
    """(b, h, q) element strides of a [B or 1, Hq or 1, Nq, Nkv] bias; size-1 axes broadcast (stride 0)."""
    if bias.dim() != 4 or bias.stride(-1) != 1:
        raise ValueError("bias must be a 4-D tensor with a contiguous key axis")
    st = bias.stride()
    return (0 if bias.shape[0] == 1 else st[0], 0 if bias.shape[1] == 1 else st[1],
            0 if bias.shape[2] == 1 else st[2])


def forward_bias(q, k, v, bias, scale: float, causal, stream=None):
    """Forward with an additive bias [B or 1, Hq or 1, Nq, Nkv] (same dtype as q; -inf masks a key)."""
    _need(q, k, v)
    B, Hq, Hkv, Nq, Nkv, d = _dims(q, k)
    o = torch.empty_like(q)
    lse = torch.empty(B, Hq, Nq, dtype=torch.float32, device=q.device)
    fb = _lib.make_bias(bias, _bias_strides(bias))
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    _check(_lib.fa_fwd_bias(q, k, v, o, lse, fb, None, None, None, B, Hq, Hkv, Nq, Nkv, 0, 0, d, scale, causal,
                            _DT[q.dtype], s), "fa_fwd_bias")
    return o, lse


def backward_bias(q, k, v, o, do, lse, bias, scale: float, causal, deterministic: bool = False, want_dbias=True,
                  stream=None):
    """Backward with an additive bias.  Returns (dQ, dK, dV, dBias); dBias [B, Hq, Nq, Nkv] is dS of every
    head (None unless ``want_dbias``); sum it over the axes the bias broadcasts."""
    _need(q, k, v, o, do, lse)
    B, Hq, Hkv, Nq, Nkv, d = _dims(q, k)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dbias = torch.empty(B, Hq, Nq, Nkv, dtype=q.dtype, device=q.device) if want_dbias else None
    fb = _lib.make_bias(bias, _bias_strides(bias), dbias, dbias.stride()[:3] if dbias is not None else (0, 0, 0))
    n = _lib.fa_bwd_workspace_size(B, Hq, Hkv, Nq, Nkv, d, int(deterministic))
    ws = torch.empty(n, dtype=torch.uint8, device=q.device)
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    _check(_lib.fa_bwd_bias(q, k, v, o, do, lse, dq, dk, dv, fb, None, None, None, B, Hq, Hkv, Nq, Nkv, 0, 0, d,
                            scale, causal, _DT[q.dtype], int(deterministic), ws, n, s), "fa_bwd_bias")
    return dq, dk, dv, dbias
