"""GPU parity of packed variable-length batches against the fp64 oracle.

Same tolerance as the dense suite, per tensor: max|gpu - ref| <= 1e-2 * max|ref| + 1e-3,
with -inf (L of a row that sees no key) matched exactly.  The backward consumes the
GPU forward's 16-bit O and fp32 L.
"""
import numpy as np
import pytest
import torch

from attn_bwd_gb300 import _lib, inputs, torch_api
from oracle import attn_ref

pytestmark = pytest.mark.gpu

REL, ABS = 1e-2, 1e-3


def _np(t):
    return t.detach().float().cpu().double().numpy()


def _compare(pairs):
    fails, lines = [], []
    for name, (got, ref) in pairs.items():
        ninf = np.isneginf(ref)
        if ninf.any() and not np.isneginf(got[ninf]).all():
            fails.append(name)
            continue
        m = ~ninf
        err = float(np.abs(got[m] - ref[m]).max()) if m.any() else 0.0
        bound = REL * float(np.abs(ref[m]).max()) + ABS if m.any() else ABS
        ok = err <= bound and np.isfinite(got[m]).all()
        lines.append(f"{name}: max|err|={err:.3e} bound={bound:.3e} {'ok' if ok else 'FAIL'}")
        if not ok:
            fails.append(name)
    return fails, "\n".join(lines)


@pytest.mark.parametrize("det", [False, True])
@pytest.mark.parametrize("pk", inputs.packed_mix(), ids=lambda p: p.name())
def test_packed_batch(pk, det):
    q, k, v, do = inputs.draw_packed(pk, 21)
    o_ref, lse_ref = attn_ref.forward_varlen(q, k, v, pk.cu_q, pk.cu_k, pk.softmax_scale, pk.causal)
    g = attn_ref.backward_varlen(q, k, v, do, pk.cu_q, pk.cu_k, pk.softmax_scale, pk.causal)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = torch_api.forward_varlen(qd, kd, vd, pk.cu_q, pk.cu_k, pk.softmax_scale, pk.causal)
    dq, dk, dv = torch_api.backward_varlen(qd, kd, vd, o, dod, lse, pk.cu_q, pk.cu_k, pk.softmax_scale, pk.causal,
                                           det)
    torch.cuda.synchronize()
    assert _lib.fa_last_device_error() == _lib.FA_OK
    fails, rep = _compare({"O": (_np(o), o_ref), "L": (_np(lse), lse_ref), "dQ": (_np(dq), g["dq"]),
                           "dK": (_np(dk), g["dk"]), "dV": (_np(dv), g["dv"])})
    assert not fails, f"{pk.name()} det={det}\n{rep}"


def test_equal_lengths_match_the_dense_entry_points():
    """A packed batch of equal lengths runs the same kernels on the same values as the dense
    batch; the deterministic results are bitwise equal after repacking."""
    B, Hq, Hkv, N, d = 3, 4, 2, 200, 128
    shape = inputs.Shape(B, Hq, Hkv, N, N, d, True, "bf16")
    q, k, v, do = (t.cuda() for t in inputs.draw(shape, 22))
    pack = lambda t: t.transpose(0, 1).reshape(t.shape[1], -1, d).contiguous()  # noqa: E731
    cu = [b * N for b in range(B + 1)]
    o, lse = torch_api.forward(q, k, v, shape.softmax_scale, True)
    ref = torch_api.backward(q, k, v, o, do, lse, shape.softmax_scale, True, True)
    ov, lv = torch_api.forward_varlen(pack(q), pack(k), pack(v), cu, cu, shape.softmax_scale, True)
    got = torch_api.backward_varlen(pack(q), pack(k), pack(v), ov, pack(do), lv, cu, cu, shape.softmax_scale, True,
                                    True)
    torch.cuda.synchronize()
    assert torch.equal(ov, pack(o)) and torch.equal(lv, lse.transpose(0, 1).reshape(Hq, -1))
    for a, b in zip(got, ref):
        assert torch.equal(a, pack(b))


def test_out_of_range_offsets_are_reported_not_used():
    """Offsets that decrease are caught by the kernels' own checks: that sequence is skipped,
    FA_ERR_ARG is reported, the others are computed, and the context stays usable."""
    pk = inputs.Packed((40, 60), (40, 60), 2, 1, 64, 1, "bf16")
    q, k, v, do = (t.cuda() for t in inputs.draw_packed(pk, 23))
    bad = torch.tensor([0, 70, 60], dtype=torch.int32, device="cuda")     # sequence 1 ends before it starts
    good_k = torch.tensor([0, 40, 100], dtype=torch.int32, device="cuda")
    o = torch.zeros_like(q)
    lse = torch.zeros(2, 100, dtype=torch.float32, device="cuda")
    st = _lib.fa_fwd_varlen(q, k, v, o, lse, bad, good_k, 2, 2, 1, 100, 100, 100, 100, 64, pk.softmax_scale, 1,
                            _lib.FA_BF16, torch.cuda.current_stream())
    assert st == _lib.FA_OK
    assert _lib.fa_last_device_error() == _lib.FA_ERR_ARG
    assert (o[:, 70:] == 0).all()                                        # nothing written for the bad sequence
    o_ref, _ = attn_ref.forward_varlen(q[:, :70].cpu(), k[:, :40].cpu(), v[:, :40].cpu(), [0, 70], [0, 40],
                                       pk.softmax_scale, 1)
    # sequence 0 (rows 0..69 here, since its offsets read 0..70) was computed against keys 0..39
    assert np.abs(_np(o[:, :70]) - o_ref).max() <= REL * np.abs(o_ref).max() + ABS
    test_packed_batch(inputs.packed_mix()[1], False)                      # the context still works


def test_packed_batch_at_benchmark_scale_sampled():
    """The packed workload bench.py --feature varlen times (16 causal sequences of 768..7936
    tokens, Llama-3 heads): full run on the GPU, three sequences of one kv-head group checked
    exactly by the oracle."""
    import random
    rnd = random.Random(7)
    lens = [rnd.randrange(512, 8193, 64) for _ in range(16)]
    pk = inputs.Packed(tuple(lens), tuple(lens), 32, 8, 128, 1, "bf16")
    q, k, v, do = inputs.draw_packed(pk, 7, device="cuda")
    o, lse = torch_api.forward_varlen(q, k, v, pk.cu_q, pk.cu_k, pk.softmax_scale, 1)
    dq, dk, dv = torch_api.backward_varlen(q, k, v, o, do, lse, pk.cu_q, pk.cu_k, pk.softmax_scale, 1, False)
    torch.cuda.synchronize()
    assert _lib.fa_last_device_error() == _lib.FA_OK
    cu = pk.cu_q
    g, G = 3, 4
    hs = slice(g * G, (g + 1) * G)
    pairs = {}
    for b in (0, 12, 15):                       # lengths 3136, 7936 and 768
        rows = slice(cu[b], cu[b + 1])
        qs, dos = q[hs, rows].cpu()[None], do[hs, rows].cpu()[None]
        ks, vs = k[g:g + 1, rows].cpu()[None], v[g:g + 1, rows].cpu()[None]
        o_ref, l_ref = attn_ref.forward(qs, ks, vs, pk.softmax_scale, 1)
        r = attn_ref.backward(qs, ks, vs, dos, pk.softmax_scale, 1)
        pairs[f"O[{b}]"] = (_np(o[hs, rows])[None], o_ref)
        pairs[f"L[{b}]"] = (_np(lse[hs, rows])[None], l_ref)
        pairs[f"dQ[{b}]"] = (_np(dq[hs, rows])[None], r["dq"])
        pairs[f"dK[{b}]"] = (_np(dk[g:g + 1, rows])[None], r["dk"])
        pairs[f"dV[{b}]"] = (_np(dv[g:g + 1, rows])[None], r["dv"])
    fails, rep = _compare(pairs)
    assert not fails, rep
