"""GPU parity of strided tensors: [B, N, H, d] storage used in place as [B, H, N, d]
views, rows with padding, and a token-major packed batch [total, H, d].

Same kernels and tiles as the contiguous path, so the deterministic results must be
bitwise equal to it; the oracle bound is checked as well.
"""
import numpy as np
import pytest
import torch

from attn_bwd_gb300 import _lib, inputs, torch_api
from oracle import attn_ref

pytestmark = pytest.mark.gpu


def _np(t):
    return t.detach().float().cpu().double().numpy()


def _bound_ok(got, ref):
    m = ~np.isneginf(ref)
    return np.abs(_np(got)[m] - ref[m]).max() <= 1e-2 * np.abs(ref[m]).max() + 1e-3


@pytest.mark.parametrize("causal", [0, 1, 2])
@pytest.mark.parametrize("d", [64, 128, 96])
def test_bshd_storage_matches_contiguous(d, causal):
    shape = inputs.Shape(2, 8, 2, 200, 260, d, causal, "bf16")
    q, k, v, do = (t.cuda() for t in inputs.draw(shape, 31))
    # the same values stored as [B, N, H, d], viewed as [B, H, N, d]
    qs, ks, vs, dos = (t.transpose(1, 2).contiguous().transpose(1, 2) for t in (q, k, v, do))
    assert not qs.is_contiguous()
    o, lse = torch_api.forward(q, k, v, shape.softmax_scale, causal)
    os_, lses = torch_api.forward_strided(qs, ks, vs, shape.softmax_scale, causal)
    ref = torch_api.backward(q, k, v, o, do, lse, shape.softmax_scale, causal, True)
    got = torch_api.backward_strided(qs, ks, vs, os_, dos, lses, shape.softmax_scale, causal, True)
    torch.cuda.synchronize()
    assert _lib.fa_last_device_error() == _lib.FA_OK
    assert torch.equal(os_, o) and torch.equal(lses, lse)
    assert got[0].stride() == qs.stride() and got[1].stride() == ks.stride()   # written in place, BSHD
    for a, b in zip(got, ref):
        assert torch.equal(a, b)
    g = attn_ref.backward(q.cpu(), k.cpu(), v.cpu(), do.cpu(), shape.softmax_scale, causal)
    assert _bound_ok(got[0], g["dq"]) and _bound_ok(got[1], g["dk"]) and _bound_ok(got[2], g["dv"])


def test_padded_rows_and_atomic_mode():
    """Rows with a stride larger than d (a slice of a wider buffer), atomic dQ."""
    shape = inputs.Shape(1, 4, 4, 150, 150, 64, 1, "f16")
    q, k, v, do = (t.cuda() for t in inputs.draw(shape, 32))
    wide = lambda t: torch.cat([t, torch.full_like(t, 7.0)], dim=-1)[..., :64]  # noqa: E731
    qs, ks, vs, dos = (wide(t) for t in (q, k, v, do))
    assert qs.stride(2) == 128
    o, lse = torch_api.forward_strided(qs, ks, vs, shape.softmax_scale, 1)
    dq, dk, dv = torch_api.backward_strided(qs, ks, vs, o, dos, lse, shape.softmax_scale, 1, False)
    torch.cuda.synchronize()
    o_ref, _ = attn_ref.forward(q.cpu(), k.cpu(), v.cpu(), shape.softmax_scale, 1)
    g = attn_ref.backward(q.cpu(), k.cpu(), v.cpu(), do.cpu(), shape.softmax_scale, 1)
    assert _bound_ok(o, o_ref)
    assert _bound_ok(dq, g["dq"]) and _bound_ok(dk, g["dk"]) and _bound_ok(dv, g["dv"])


@pytest.mark.parametrize("det", [False, True])
def test_token_major_packed_batch(det):
    """A packed batch stored token-major, [total, H, d], through the strided entry points,
    bitwise equal (deterministic mode) to the head-major packed path."""
    pk = inputs.Packed((70, 1, 190), (100, 9, 150), 4, 2, 128, 2, "bf16")
    q, k, v, do = (t.cuda() for t in inputs.draw_packed(pk, 33))
    o, lse = torch_api.forward_varlen(q, k, v, pk.cu_q, pk.cu_k, pk.softmax_scale, pk.causal)
    ref = torch_api.backward_varlen(q, k, v, o, do, lse, pk.cu_q, pk.cu_k, pk.softmax_scale, pk.causal, True)
    tm = lambda t: t.transpose(0, 1).contiguous().transpose(0, 1)  # noqa: E731  [total, H, d] storage
    qt, kt, vt, dot, ot = (tm(t) for t in (q, k, v, do, o))
    Hq, tq, d = q.shape
    Hkv, tk, _ = k.shape
    cu_q = torch.tensor(pk.cu_q, dtype=torch.int32, device="cuda")
    cu_k = torch.tensor(pk.cu_k, dtype=torch.int32, device="cuda")
    dq, dk, dv = (torch.empty_like(t) for t in (qt, kt, vt))
    o2 = torch.empty_like(qt)
    lse2 = torch.empty(Hq, tq, dtype=torch.float32, device="cuda")
    s3 = lambda t: (0, t.stride(0), t.stride(1))  # noqa: E731
    st = _lib.make_strides(q=s3(qt), k=s3(kt), v=s3(vt), o=s3(o2), dO=s3(dot), dq=s3(dq), dk=s3(dk), dv=s3(dv),
                           lse=(0, lse2.stride(0), 1))
    B, mq, mk = len(pk.lens_q), max(pk.lens_q), max(pk.lens_k)
    s = torch.cuda.current_stream()
    assert _lib.fa_fwd_strided(qt, kt, vt, o2, lse2, st, cu_q, cu_k, B, Hq, Hkv, mq, mk, tq, tk, d,
                               pk.softmax_scale, pk.causal, _lib.FA_BF16, s) == 0
    n = _lib.fa_bwd_workspace_size(B, Hq, Hkv, mq, mk, d, int(det))
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    st.o = _lib.fa_stride3(0, ot.stride(0), ot.stride(1))
    assert _lib.fa_bwd_strided(qt, kt, vt, ot, dot, lse, dq, dk, dv, st, cu_q, cu_k, B, Hq, Hkv, mq, mk, tq, tk, d,
                               pk.softmax_scale, pk.causal, _lib.FA_BF16, int(det), ws, n, s) == 0
    torch.cuda.synchronize()
    assert _lib.fa_last_device_error() == _lib.FA_OK
    assert torch.equal(o2, o) and torch.equal(lse2, lse)
    if det:
        for a, b in zip((dq, dk, dv), ref):
            assert torch.equal(a, b)
    g = attn_ref.backward_varlen(q.cpu(), k.cpu(), v.cpu(), do.cpu(), pk.cu_q, pk.cu_k, pk.softmax_scale, pk.causal)
    assert _bound_ok(dq, g["dq"]) and _bound_ok(dk, g["dk"]) and _bound_ok(dv, g["dv"])
