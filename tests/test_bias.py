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
