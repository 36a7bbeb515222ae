"""GPU parity of the additive bias (and -inf masks) against the fp64 oracle: O, L, dQ, dK,
dV and dBias = dS, for every broadcast shape of the bias and every causal mode.

Tolerance as elsewhere, per tensor: max|gpu - ref| <= 1e-2 * max|ref| + 1e-3, -inf exact.
"""
import numpy as np
import pytest
import torch

from attn_bwd_gb300 import _lib, inputs, torch_api
from oracle import attn_ref

pytestmark = pytest.mark.gpu


def _np(t):
    return t.detach().float().cpu().double().numpy()


def _check(pairs):
    bad = []
    for name, (got, ref) in pairs.items():
        ninf = np.isneginf(ref)
        if ninf.any() and not np.isneginf(got[ninf]).all():
            bad.append(f"{name}: -inf not reproduced")
            continue
        m = ~ninf
        err = float(np.abs(got[m] - ref[m]).max())
        bound = 1e-2 * float(np.abs(ref[m]).max()) + 1e-3
        if not (err <= bound and np.isfinite(got[m]).all()):
            bad.append(f"{name}: {err:.3e} > {bound:.3e}")
    assert not bad, "\n".join(bad)


def _run(shape, bias, seed, det):
    q, k, v, do = inputs.draw(shape, seed)
    o_ref, l_ref = attn_ref.forward(q, k, v, shape.softmax_scale, shape.causal, bias=bias)
    g = attn_ref.backward(q, k, v, do, shape.softmax_scale, shape.causal, bias=bias)
    qd, kd, vd, dod, bd = (t.cuda() for t in (q, k, v, do, bias))
    o, lse = torch_api.forward_bias(qd, kd, vd, bd, shape.softmax_scale, shape.causal)
    dq, dk, dv, db = torch_api.backward_bias(qd, kd, vd, o, dod, lse, bd, shape.softmax_scale, shape.causal, det)
    torch.cuda.synchronize()
    assert _lib.fa_last_device_error() == _lib.FA_OK
    _check({"O": (_np(o), o_ref), "L": (_np(lse), l_ref), "dQ": (_np(dq), g["dq"]), "dK": (_np(dk), g["dk"]),
            "dV": (_np(dv), g["dv"]), "dBias": (_np(db), g["dbias"])})


@pytest.mark.parametrize("det", [False, True])
@pytest.mark.parametrize("causal", [0, 1, 2])
@pytest.mark.parametrize("bshape", [(2, 4), (1, 4), (2, 1), (1, 1)])
def test_bias_broadcast_shapes(bshape, causal, det):
    shape = inputs.Shape(2, 4, 2, 130, 200, 64, causal, "bf16")
    g = torch.Generator().manual_seed(70)
    bias = (2.0 * torch.randn(bshape[0], bshape[1], 130, 200, generator=g)).to(torch.bfloat16)
    _run(shape, bias, 71, det)


@pytest.mark.parametrize("det", [False, True])
def test_minus_inf_bias_masks_keys_and_whole_rows(det):
    """A boolean mask as a -inf bias: random dropped keys, a row that keeps none, and a row
    whose first 150 keys (more than a tile) are dropped."""
    shape = inputs.Shape(1, 2, 1, 96, 256, 128, 0, "f16")
    g = torch.Generator().manual_seed(72)
    keep = torch.rand(1, 2, 96, 256, generator=g) > 0.3
    keep[0, 0, 5] = False
    keep[0, 1, 7, :150] = False
    bias = torch.zeros(1, 2, 96, 256).masked_fill(~keep, float("-inf")).to(torch.float16)
    _run(shape, bias, 73, det)


def test_bias_with_gqa_and_head_dim_128():
    shape = inputs.Shape(1, 8, 2, 257, 128, 128, 2, "bf16")
    g = torch.Generator().manual_seed(74)
    bias = torch.randn(1, 8, 257, 128, generator=g).to(torch.bfloat16)
    _run(shape, bias, 75, False)


@pytest.mark.parametrize("det", [False, True])
@pytest.mark.parametrize("causal", [0, 1, 2])
def test_bias_on_packed_batch(causal, det):
    """A per-sequence bias on a packed batch: [B, Hq, max_q, >= max_k] with a padded key axis.
    Sequence b reads and writes only rows [0, nq_b) x keys [0, nk_b) of its bias and dBias;
    the rest of the caller's dBias keeps its sentinel.  Lengths make some blocks lie inside a
    sequence and others cross its end in queries, keys or both."""
    lens_q, lens_k, Hq, Hkv, d = (77, 300, 16, 129), (200, 130, 16, 257), 4, 2, 128
    pk = inputs.Packed(lens_q, lens_k, Hq, Hkv, d, causal, "bf16")
    q, k, v, do = inputs.draw_packed(pk, 76)
    B, mq, mk, kpad = len(lens_q), max(lens_q), max(lens_k), 264     # key axis padded to a multiple of 8
    g = torch.Generator().manual_seed(77)
    bias = (1.5 * torch.randn(B, Hq, mq, kpad, generator=g)).to(torch.bfloat16)
    cu_q, cu_k = pk.cu_q, pk.cu_k
    qd, kd, vd, dod, bd = (t.cuda() for t in (q, k, v, do, bias))
    cq = torch.tensor(cu_q, dtype=torch.int32, device="cuda")
    ck = torch.tensor(cu_k, dtype=torch.int32, device="cuda")
    st_b = (Hq * mq * kpad, mq * kpad, kpad)
    o, lse = torch.empty_like(qd), torch.empty(Hq, cu_q[-1], dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream()
    assert _lib.fa_fwd_bias(qd, kd, vd, o, lse, _lib.make_bias(bd, st_b), None, cq, ck, B, Hq, Hkv, mq, mk,
                            cu_q[-1], cu_k[-1], d, pk.softmax_scale, causal, _lib.FA_BF16, s) == _lib.FA_OK
    sentinel = 7.0
    db = torch.full((B, Hq, mq, kpad), sentinel, dtype=torch.bfloat16, device="cuda")
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    n = _lib.fa_bwd_varlen_workspace_size(B, Hq, Hkv, mq, mk, d, int(det))
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    assert _lib.fa_bwd_bias(qd, kd, vd, o, dod, lse, dq, dk, dv, _lib.make_bias(bd, st_b, db, st_b), None, cq, ck, B,
                            Hq, Hkv, mq, mk, cu_q[-1], cu_k[-1], d, pk.softmax_scale, causal, _lib.FA_BF16, int(det),
                            ws, n, s) == _lib.FA_OK
    torch.cuda.synchronize()
    assert _lib.fa_last_device_error() == _lib.FA_OK
    dbh = db.cpu()
    untouched = torch.ones(B, Hq, mq, kpad, dtype=torch.bool)
    for b in range(B):
        nq, nk = lens_q[b], lens_k[b]
        untouched[b, :, :nq, :nk] = False
        sl_q, sl_k = slice(cu_q[b], cu_q[b + 1]), slice(cu_k[b], cu_k[b + 1])
        qb, kb, vb, dob = (t[:, sl][None] for t, sl in ((q, sl_q), (k, sl_k), (v, sl_k), (do, sl_q)))
        bb = bias[b:b + 1, :, :nq, :nk]
        o_ref, l_ref = attn_ref.forward(qb, kb, vb, pk.softmax_scale, causal, bias=bb)
        r = attn_ref.backward(qb, kb, vb, dob, pk.softmax_scale, causal, bias=bb)
        _check({f"O[{b}]": (_np(o[:, sl_q][None]), o_ref), f"L[{b}]": (_np(lse[:, sl_q][None]), l_ref),
                f"dQ[{b}]": (_np(dq[:, sl_q][None]), r["dq"]), f"dK[{b}]": (_np(dk[:, sl_k][None]), r["dk"]),
                f"dV[{b}]": (_np(dv[:, sl_k][None]), r["dv"]),
                f"dBias[{b}]": (_np(dbh[b:b + 1, :, :nq, :nk]), r["dbias"])})
    assert (dbh[untouched] == sentinel).all(), "dBias written outside a sequence"


@pytest.mark.parametrize("causal", [0, 1, 2])
def test_zero_bias_gives_the_same_bits(causal):
    """A zero bias adds exactly 0 to every exponent, so the backward's bias path (one CTA per
    work item) and its path without a bias (persistent kernels) must compute the same bits from
    the same O and L: dK and dV in both dQ modes, and the deterministic dQ, whose summation
    order both fix the same way.  (The forward is not compared: with a bias it steps over 128
    keys at a time instead of 64, which moves its running maxima.)"""
    shape = inputs.Shape(2, 4, 2, 300, 264, 128, causal, "bf16")   # bias rows need 16-byte strides
    q, k, v, do = (t.cuda() for t in inputs.draw(shape, 72))
    zero = torch.zeros(1, 1, 300, 264, dtype=torch.bfloat16, device="cuda")
    o, lse = torch_api.forward(q, k, v, shape.softmax_scale, causal)
    for det in (False, True):
        g0 = torch_api.backward(q, k, v, o, do, lse, shape.softmax_scale, causal, det)
        g1 = torch_api.backward_bias(q, k, v, o, do, lse, zero, shape.softmax_scale, causal, det)
        torch.cuda.synchronize()
        assert _lib.fa_last_device_error() == _lib.FA_OK
        assert torch.equal(g0[1], g1[1]) and torch.equal(g0[2], g1[2]), f"dK/dV det={det}"
        if det:
            assert torch.equal(g0[0], g1[0]), "deterministic dQ"
