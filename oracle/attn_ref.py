"""fp64 CPU oracle for exact softmax attention and its analytic backward pass.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module:
only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` call it.  It shares no code with the
CUDA kernels (no helpers, tables or constants) and performs the full-matrix
computation with no tiling, fusion or reordering, so that each line can be
checked by eye against the definitions below.

Definitions (per batch b and query head h; the key/value head is
h_kv = h // (Hq // Hkv), i.e. consecutive groups of query heads share one
key/value head -- the plainest reading of the GQA support described in
"[Kernel] Flash attention 2" (Liger-Kernel #275), "Details"):

  S_ij  = scale * sum_c Q_ic K_jc, and S_ij = -inf when causal and j > i + delta
          (flash_attention_backward.cu, rustytorch rtx-flash-attention,
          blocks "Recompute attention scores" and "Apply causal mask", where
          delta = 0: the top-left alignment).  "[Kernel] Flash attention 2"
          (Liger-Kernel #275, "Details") lists causal masking together with
          different Q and KV lengths without fixing the alignment; the second
          option here, bottom-right, takes delta = Nkv - Nq so that the last
          query sees every key.  With Nq > Nkv its first Nq - Nkv rows see no
          key at all.
  L_i   = log sum_j exp(S_ij)         natural log of the *scaled* scores
          (same file, block "Compute softmax probabilities from scores and LSE");
          -inf for a row that sees no key (the log of an empty sum)
  P_ij  = exp(S_ij - L_i)             (same block); 0 wherever S_ij = -inf, so a
          row that sees no key has P = 0, O = 0, dS = 0 and dQ = 0
  O_i   = sum_j P_ij V_j
  dV_j  = sum_i P_ij dO_i             (same file, block "Compute dV")
  dP_ij = sum_c dO_ic V_jc            (same file, block "Compute dS", first step)
  D_i   = sum_j P_ij dP_ij            (equal to sum_c dO_ic O_ic, which is the
          form the pages precompute: same file, block "Compute row-wise dot
          product: dO * O"; the Triton kernel in triton #1806 takes it as D)
  dS_ij = P_ij (dP_ij - D_i)          (same file, block "Compute dS")
  dQ_i  = scale * sum_j dS_ij K_j     (same file, block "Compute dQ")
  dK_j  = scale * sum_i dS_ij Q_i     (same file, block "Compute dK")
  GQA:  dK, dV of a key/value head are summed over the query heads of its group.

All arithmetic is float64.  Inputs (16-bit on the CUDA side) are widened
exactly to float64 before use.  Matrix products use numpy's matmul as a
library primitive.
"""
from __future__ import annotations

import numpy as np


def _f64(x) -> np.ndarray:
    """Widen a torch tensor or array exactly to a float64 numpy array."""
    if hasattr(x, "detach"):
        import torch
        x = x.detach().cpu().to(torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def kv_head(h: int, Hq: int, Hkv: int) -> int:
    """Key/value head used by query head h: consecutive groups of Hq//Hkv."""
    if Hq % Hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    return h // (Hq // Hkv)


# Values of the ``causal`` argument (the same numbers the C interface takes;
# ``False`` / ``True`` mean none / top-left).
CAUSAL_NONE = 0
CAUSAL_TOP_LEFT = 1
CAUSAL_BOTTOM_RIGHT = 2


def causal_delta(causal, nq: int, nk: int):
    """delta of the mask rule "key j masked for query i when j > i + delta", or None (no mask)."""
    c = int(causal)
    if c == CAUSAL_NONE:
        return None
    if c == CAUSAL_TOP_LEFT:
        return 0
    if c == CAUSAL_BOTTOM_RIGHT:
        return nk - nq
    raise ValueError(f"unknown causal mode {causal!r}")


def scores(q: np.ndarray, k: np.ndarray, scale: float, causal, bias=None) -> np.ndarray:
    """S = scale * Q K^T (+ bias) for one head, [Nq, Nkv], with the causal mask applied.

    Top-left drops key j for query i whenever j > i (the literal rule of the
    pages' CUDA kernel); bottom-right whenever j > i + Nkv - Nq.  With
    Nq == Nkv both are the usual mask.  ``bias`` [Nq, Nkv] is added to the
    scaled scores before masking ("[Kernel] Flash attention 2", "Details":
    attention bias and attention masking); a boolean mask is the bias -inf
    at the dropped positions.
    """
    s = scale * (q @ k.T)
    if bias is not None:
        s = s + bias
    nq, nk = s.shape
    delta = causal_delta(causal, nq, nk)
    if delta is not None:
        i = np.arange(nq)[:, None]
        j = np.arange(nk)[None, :]
        s = np.where(j > i + delta, -np.inf, s)
    return s


def logsumexp_rows(s: np.ndarray) -> np.ndarray:
    """L_i = log sum_j exp(S_ij), evaluated stably as m_i + log sum_j exp(S_ij - m_i).

    A row whose scores are all -inf (it sees no key) gets -inf.
    """
    if s.shape[1] == 0:
        return np.full(s.shape[0], -np.inf)
    m = s.max(axis=1)
    out = np.full(s.shape[0], -np.inf)
    seen = np.isfinite(m)
    out[seen] = m[seen] + np.log(np.exp(s[seen] - m[seen, None]).sum(axis=1))
    return out


def probs(s: np.ndarray, lse: np.ndarray) -> np.ndarray:
    """P_ij = exp(S_ij - L_i), and exactly 0 where S_ij = -inf (masked)."""
    p = np.zeros_like(s)
    live = np.isfinite(s)
    p[live] = np.exp(s[live] - np.broadcast_to(lse[:, None], s.shape)[live])
    return p


def head_forward(q, k, v, scale, causal, bias=None):
    """Forward for one head: returns (O [Nq,d], L [Nq], P [Nq,Nkv])."""
    s = scores(q, k, scale, causal, bias)
    lse = logsumexp_rows(s)
    p = probs(s, lse)
    return p @ v, lse, p


def head_backward(q, k, v, do, scale, causal, lse=None, o=None, bias=None):
    """Backward for one head.

    Returns a dict with dq [Nq,d], dk [Nkv,d], dv [Nkv,d], D [Nq] (the
    rowsum(P * dP) form), D_rowdot [Nq] (the rowsum(dO * O) form, only when
    ``o`` is given or computed), and dS [Nq,Nkv], which is also the gradient of
    the loss with respect to an additive bias (the bias enters S with weight 1).

    ``lse`` / ``o``: when given, P is formed from that log-sum-exp and
    D_rowdot from that output (used to isolate the backward from forward
    rounding); otherwise both are recomputed here in fp64.
    """
    s = scores(q, k, scale, causal, bias)
    if lse is None:
        lse = logsumexp_rows(s)
    p = probs(s, lse)
    if o is None:
        o = p @ v
    dv = p.T @ do
    dp = do @ v.T
    D = (p * dp).sum(axis=1)
    D_rowdot = (do * o).sum(axis=1)
    ds = p * (dp - D[:, None])
    dq = scale * (ds @ k)
    dk = scale * (ds.T @ q)
    return {"dq": dq, "dk": dk, "dv": dv, "D": D, "D_rowdot": D_rowdot, "dS": ds, "P": p}


def _bias_of(bias, b, h):
    """The [Nq, Nkv] bias of (b, h) from a [B or 1, Hq or 1, Nq, Nkv] array (size-1 axes broadcast)."""
    if bias is None:
        return None
    return bias[b if bias.shape[0] > 1 else 0, h if bias.shape[1] > 1 else 0]


def forward(q, k, v, scale: float, causal: bool, bias=None):
    """Full forward over [B, Hq, Nq, d] / [B, Hkv, Nkv, d].  Returns (O, L) in fp64.

    ``bias``: optional additive bias [B or 1, Hq or 1, Nq, Nkv] (size-1 axes broadcast).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    bias = None if bias is None else _f64(bias)
    B, Hq, Nq, d = q.shape
    Hkv = k.shape[1]
    o = np.zeros((B, Hq, Nq, d))
    lse = np.zeros((B, Hq, Nq))
    for b in range(B):
        for h in range(Hq):
            hk = kv_head(h, Hq, Hkv)
            o[b, h], lse[b, h], _ = head_forward(q[b, h], k[b, hk], v[b, hk], scale, causal, _bias_of(bias, b, h))
    return o, lse


def backward(q, k, v, do, scale: float, causal: bool, lse=None, o=None, groups=None, bias=None):
    """Full backward.  Returns dict of fp64 arrays dq, dk, dv, D, D_rowdot, and dbias
    [B, Hq, Nq, Nkv] (= dS of every head) when ``bias`` is given.

    ``groups``: optional iterable of (b, h_kv) pairs; when given only those
    groups are computed (their query heads' dq/D and the group's dk/dv), the
    rest of the outputs are NaN.  Used for sampled parity at full size.
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    lse = None if lse is None else _f64(lse)
    o = None if o is None else _f64(o)
    bias = None if bias is None else _f64(bias)
    B, Hq, Nq, d = q.shape
    Hkv, Nkv = k.shape[1], k.shape[2]
    G = Hq // Hkv
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    fill = np.nan if groups is not None else 0.0
    dq = np.full((B, Hq, Nq, d), fill)
    dk = np.full((B, Hkv, Nkv, d), fill)
    dv = np.full((B, Hkv, Nkv, d), fill)
    D = np.full((B, Hq, Nq), fill)
    D_rowdot = np.full((B, Hq, Nq), fill)
    dbias = np.full((B, Hq, Nq, Nkv), fill) if bias is not None else None
    todo = groups if groups is not None else [(b, g) for b in range(B) for g in range(Hkv)]
    for b, g in todo:
        dk[b, g] = 0.0
        dv[b, g] = 0.0
        for h in range(g * G, (g + 1) * G):
            r = head_backward(q[b, h], k[b, g], v[b, g], do[b, h], scale, causal,
                              None if lse is None else lse[b, h],
                              None if o is None else o[b, h], _bias_of(bias, b, h))
            if dbias is not None:
                dbias[b, h] = r["dS"]
            dq[b, h] = r["dq"]
            dk[b, g] += r["dk"]
            dv[b, g] += r["dv"]
            D[b, h] = r["D"]
            D_rowdot[b, h] = r["D_rowdot"]
    out = {"dq": dq, "dk": dk, "dv": dv, "D": D, "D_rowdot": D_rowdot}
    if dbias is not None:
        out["dbias"] = dbias
    return out


# ------------------------------------------------------------ packed batches
#
# Variable-length batches: "[Kernel] Flash attention 2" (Liger-Kernel #275,
# "Details") supports different Q and KV lengths and places no restriction on
# the sequence length; a packed batch of sequences of different lengths is the
# plainest form of that for a batch.  Sequence b occupies rows
# [cu_q[b], cu_q[b+1]) of every query head of Q [Hq, total_q, d] and rows
# [cu_k[b], cu_k[b+1]) of every key/value head of K, V [Hkv, total_k, d], and
# attends only to its own keys, with the causal alignment taken per sequence.
# The definition is therefore the dense problem above applied to each
# sequence on its own.


def _check_cu(cu, total: int):
    cu = [int(x) for x in cu]
    if cu[0] != 0 or cu[-1] != total or any(b < a for a, b in zip(cu, cu[1:])):
        raise ValueError("cu_seqlens must start at 0, not decrease and end at the total")
    return cu


def forward_varlen(q, k, v, cu_q, cu_k, scale: float, causal):
    """Packed forward: q [Hq, total_q, d], k/v [Hkv, total_k, d].  Returns (O, L) in fp64."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    Hq, total_q, d = q.shape
    Hkv, total_k = k.shape[0], k.shape[1]
    cu_q, cu_k = _check_cu(cu_q, total_q), _check_cu(cu_k, total_k)
    o = np.zeros((Hq, total_q, d))
    lse = np.full((Hq, total_q), -np.inf)
    for b in range(len(cu_q) - 1):
        qs, ks = slice(cu_q[b], cu_q[b + 1]), slice(cu_k[b], cu_k[b + 1])
        for h in range(Hq):
            hk = kv_head(h, Hq, Hkv)
            o[h, qs], lse[h, qs], _ = head_forward(q[h, qs], k[hk, ks], v[hk, ks], scale, causal)
    return o, lse


def backward_varlen(q, k, v, do, cu_q, cu_k, scale: float, causal):
    """Packed backward.  Returns dict of fp64 arrays dq [Hq,total_q,d], dk, dv [Hkv,total_k,d], D."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    Hq, total_q, d = q.shape
    Hkv, total_k = k.shape[0], k.shape[1]
    cu_q, cu_k = _check_cu(cu_q, total_q), _check_cu(cu_k, total_k)
    dq = np.zeros((Hq, total_q, d))
    dk = np.zeros((Hkv, total_k, d))
    dv = np.zeros((Hkv, total_k, d))
    D = np.zeros((Hq, total_q))
    for b in range(len(cu_q) - 1):
        qs, ks = slice(cu_q[b], cu_q[b + 1]), slice(cu_k[b], cu_k[b + 1])
        for h in range(Hq):
            hk = kv_head(h, Hq, Hkv)
            r = head_backward(q[h, qs], k[hk, ks], v[hk, ks], do[h, qs], scale, causal)
            dq[h, qs] = r["dq"]
            dk[hk, ks] += r["dk"]
            dv[hk, ks] += r["dv"]
            D[h, qs] = r["D"]
    return {"dq": dq, "dk": dk, "dv": dv, "D": D}
