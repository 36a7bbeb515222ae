"""GPU parity: the CUDA path against the fp64 oracle on the same seeded inputs.

Tolerance (per tensor): max|gpu - ref| <= 1e-2 * max|ref| + 1e-3, for O and L
of the forward and dQ, dK, dV of the backward.  The backward consumes the
GPU forward's 16-bit O and fp32 L; the oracle recomputes everything in fp64
from the 16-bit inputs, so the bound covers both passes' rounding.

Sizes: every workload in full where the oracle finishes in seconds; the
Llama-3 shaped sweep at N >= 2048 is checked on sampled (batch, kv-head)
groups, in the launch configuration the benchmark times (the whole problem
runs on the GPU; the oracle computes the sampled groups exactly).
"""
import functools

import numpy as np
import pytest
import torch

from attn_bwd_gb300 import _lib, inputs, torch_api
from oracle import attn_ref

pytestmark = pytest.mark.gpu

REL, ABS = 1e-2, 1e-3


def _np(t):
    return t.detach().float().cpu().double().numpy()


def errors(pairs):
    """pairs: name -> (gpu array, ref array). Returns (failures, report)."""
    fails, lines = [], []
    for name, (got, ref) in pairs.items():
        # -inf (L of a row that sees no key) must be matched exactly; the rest by the bound
        ninf = np.isneginf(ref)
        if ninf.any() and not np.isneginf(got[ninf]).all():
            fails.append(name)
            lines.append(f"{name}: -inf rows not reproduced FAIL")
            continue
        mask = ~np.isnan(ref) & ~ninf
        err = float(np.abs(got[mask] - ref[mask]).max()) if mask.any() else 0.0
        bound = REL * float(np.abs(ref[mask]).max()) + ABS if mask.any() else ABS
        ok = err <= bound and np.isfinite(got[mask]).all()
        lines.append(f"{name}: max|err|={err:.3e} bound={bound:.3e} {'ok' if ok else 'FAIL'}")
        if not ok:
            fails.append(name)
    return fails, "\n".join(lines)


@functools.lru_cache(maxsize=8)
def oracle_full(shape: inputs.Shape, seed: int):
    q, k, v, do = inputs.draw(shape, seed)
    o, lse = attn_ref.forward(q, k, v, shape.softmax_scale, shape.causal)
    g = attn_ref.backward(q, k, v, do, shape.softmax_scale, shape.causal)
    return (q, k, v, do), o, lse, g


def gpu_run(q, k, v, do, shape, deterministic):
    dev = torch.device("cuda")
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o, lse = torch_api.forward(qd, kd, vd, shape.softmax_scale, shape.causal)
    dq, dk, dv = torch_api.backward(qd, kd, vd, o, dod, lse, shape.softmax_scale, shape.causal, deterministic)
    torch.cuda.synchronize()
    assert _lib.fa_last_device_error() == _lib.FA_OK
    return o, lse, dq, dk, dv


def check_full(shape, seed, deterministic):
    (q, k, v, do), o_ref, lse_ref, g = oracle_full(shape, seed)
    o, lse, dq, dk, dv = gpu_run(q, k, v, do, shape, deterministic)
    fails, rep = errors({"O": (_np(o), o_ref), "L": (_np(lse), lse_ref),
                         "dQ": (_np(dq), g["dq"]), "dK": (_np(dk), g["dk"]), "dV": (_np(dv), g["dv"])})
    assert not fails, f"{shape.name()} det={deterministic}\n{rep}"


# ---------------------------------------------------------------- workloads

@pytest.mark.parametrize("det", [False, True])
def test_tiny_mha(det):
    check_full(inputs.tiny_mha()[0], 1, det)


@pytest.mark.parametrize("det", [False, True])
@pytest.mark.parametrize("shape", inputs.ragged(), ids=lambda s: s.name())
def test_ragged(shape, det):
    check_full(shape, 2, det)


@pytest.mark.parametrize("shape", inputs.mid_sweep(), ids=lambda s: s.name())
def test_mid_sweep(shape):
    check_full(shape, 3, False)


@pytest.mark.parametrize("shape", [s for s in inputs.mid_sweep() if s.d == 128 and s.Nq == 784],
                         ids=lambda s: s.name())
def test_mid_sweep_deterministic(shape):
    check_full(shape, 3, True)


@pytest.mark.parametrize("det", [False, True])
def test_long_uniform(det):
    check_full(inputs.long_uniform()[0], 4, det)


@pytest.mark.parametrize("n", [32, 64, 128, 256, 512, 1024])
def test_llama_gqa_full(n):
    check_full(inputs.llama_gqa(n), 5, False)


@pytest.mark.parametrize("n", [32, 96, 256, 512, 1000])
def test_llama_gqa_full_deterministic(n):
    check_full(inputs.llama_gqa(n), 5, True)


@pytest.mark.parametrize("n", [2048, 4096, 8192, 16384])
def test_llama_gqa_sampled(n):
    """Full-size run on the GPU; the oracle computes two (batch, kv-head) groups exactly."""
    shape = inputs.llama_gqa(n)
    q, k, v, do = inputs.draw(shape, 5, device="cuda")
    o, lse, dq, dk, dv = gpu_run(q, k, v, do, shape, False)
    G = shape.Hq // shape.Hkv
    groups = [(0, 0), (shape.B - 1, shape.Hkv - 1)]
    pairs = {}
    for b, g in groups:
        hs = slice(g * G, (g + 1) * G)
        sl = lambda t, h: t[b:b + 1, h].cpu()  # noqa: E731
        qs, dos = sl(q, hs), sl(do, hs)
        ks, vs = sl(k, slice(g, g + 1)), sl(v, slice(g, g + 1))
        o_ref, lse_ref = attn_ref.forward(qs, ks, vs, shape.softmax_scale, True)
        r = attn_ref.backward(qs, ks, vs, dos, shape.softmax_scale, True)
        pairs[f"O[{b},{g}]"] = (_np(o[b:b + 1, hs]), o_ref)
        pairs[f"L[{b},{g}]"] = (_np(lse[b:b + 1, hs]), lse_ref)
        pairs[f"dQ[{b},{g}]"] = (_np(dq[b:b + 1, hs]), r["dq"])
        pairs[f"dK[{b},{g}]"] = (_np(dk[b:b + 1, g:g + 1]), r["dk"])
        pairs[f"dV[{b},{g}]"] = (_np(dv[b:b + 1, g:g + 1]), r["dv"])
    fails, rep = errors(pairs)
    assert not fails, rep
    # A property that holds on every head: the sum of dK over the keys is exactly zero (each
    # row of dS sums to zero).  What remains on the GPU comes from rounding dS and dK to 16
    # bits.  On the sampled groups that residue must stay within 4x of the residue that
    # rounding the oracle's own dK to bf16 leaves; on every head within 0.1 of its max |dK|
    # (measured: at most 0.031 up to N = 16384).
    def residue(x):                      # max_c |sum_j x_jc| / max |x|, per (batch, kv head)
        x = torch.as_tensor(x).double()
        return x.sum(dim=-2).abs().amax(-1) / x.abs().amax((-2, -1))
    for b, g in groups:
        floor = residue(torch.from_numpy(pairs[f"dK[{b},{g}]"][1]).to(torch.bfloat16)).max().item()
        got = residue(dk[b:b + 1, g:g + 1].cpu()).max().item()
        assert got <= 4 * floor + 1e-3, (b, g, got, floor)
    assert residue(dk.cpu()).max().item() <= 0.1


# ------------------------------------------------------------ extra shapes

@pytest.mark.parametrize("det", [False, True])
@pytest.mark.parametrize("shape", [
    inputs.Shape(1, 4, 2, 77, 200, 64, True, "bf16"),      # Nq < Nkv, top-left causal
    inputs.Shape(1, 4, 2, 300, 130, 128, True, "f16"),     # Nq > Nkv
    inputs.Shape(2, 6, 3, 129, 257, 128, False, "bf16"),   # one past a tile on both sides
    inputs.Shape(1, 8, 1, 64, 64, 64, True, "bf16"),       # 8 query heads share one kv head
], ids=lambda s: s.name())
def test_extra_shapes(shape, det):
    check_full(shape, 6, det)


# ------------------------------------------------------------ step-level checks

def test_preprocess_rowdot_and_padding():
    """Step 1 alone: D = rowsum(dO o O) from the given O, -L*log2(e), and padding rows."""
    shape = inputs.Shape(2, 3, 3, 100, 100, 128, False, "bf16")
    q, k, v, do = (t.cuda() for t in inputs.draw(shape, 7))
    o, lse = torch_api.forward(q, k, v, shape.softmax_scale, False)
    ws = torch_api.workspace(q, k, False)
    ws.fill_(0xFF)
    st = _lib.fa_bwd_preprocess(o, do, lse, 2, 3, 3, 100, 100, 128, _lib.FA_BF16, 0, ws, ws.numel(),
                                torch.cuda.current_stream())
    assert st == 0
    torch.cuda.synchronize()
    rows = 2 * 3 * 128
    f = ws.view(torch.float32)[64:]           # after the call's 256-byte abort word
    nLg = f[:rows].view(2, 3, 128).cpu().double().numpy()
    Dv = f[rows:2 * rows].view(2, 3, 128).cpu().double().numpy()
    acc = f[2 * rows:2 * rows + rows * 128]
    D_ref = (_np(o) * _np(do)).sum(-1)
    np.testing.assert_allclose(Dv[:, :, :100], D_ref, rtol=1e-5, atol=1e-5)
    assert (Dv[:, :, 100:] == 0).all()
    np.testing.assert_allclose(nLg[:, :, :100], -_np(lse) * np.log2(np.e), rtol=1e-6, atol=1e-6)
    assert np.isinf(nLg[:, :, 100:]).all() and (nLg[:, :, 100:] < 0).all()
    assert (acc == 0).all()


@pytest.mark.parametrize("det", [False, True], ids=["atomic", "deterministic"])
@pytest.mark.parametrize("shape", [
    inputs.Shape(2, 4, 2, 300, 130, 128, 2, "f16"),     # rows that see no key
    inputs.Shape(2, 6, 3, 129, 257, 128, False, "bf16"),
    inputs.Shape(1, 4, 4, 200, 150, 40, True, "bf16"),
], ids=lambda s: s.name() if hasattr(s, "name") else str(s))
def test_stage_entry_points(shape, det):
    """fa_bwd_preprocess, fa_bwd_main and fa_bwd_dq called one at a time, on a workspace
    filled with garbage and outputs filled with 7.0: the gradients must match the oracle,
    and dK, dV (and, in deterministic mode, dQ) must equal fa_bwd's bit for bit."""
    (q, k, v, do), _, _, g = oracle_full(shape, 11)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = torch_api.forward(qd, kd, vd, shape.softmax_scale, shape.causal)
    B, Hq, Hkv, Nq, Nkv, d = shape.B, shape.Hq, shape.Hkv, shape.Nq, shape.Nkv, shape.d
    dt = _lib.FA_BF16 if shape.dtype == "bf16" else _lib.FA_F16
    s = torch.cuda.current_stream()
    ws = torch_api.workspace(qd, kd, det)
    ws.fill_(0x7F)                                   # contents on entry must not matter
    dq, dk, dv = torch.full_like(qd, 7.0), torch.full_like(kd, 7.0), torch.full_like(vd, 7.0)
    c = int(shape.causal)
    assert _lib.fa_bwd_preprocess(o, dod, lse, B, Hq, Hkv, Nq, Nkv, d, dt, det, ws, ws.numel(), s) == 0
    assert _lib.fa_bwd_main(qd, kd, vd, dod, dk, dv, B, Hq, Hkv, Nq, Nkv, d, shape.softmax_scale, c, dt, det,
                            ws, ws.numel(), s) == 0
    assert _lib.fa_bwd_dq(qd, kd, vd, dod, dq, B, Hq, Hkv, Nq, Nkv, d, shape.softmax_scale, c, dt, det,
                          ws, ws.numel(), s) == 0
    torch.cuda.synchronize()
    assert _lib.fa_last_device_error() == _lib.FA_OK
    fails, rep = errors({"dQ": (_np(dq), g["dq"]), "dK": (_np(dk), g["dk"]), "dV": (_np(dv), g["dv"])})
    assert not fails, rep
    ref = torch_api.backward(qd, kd, vd, o, dod, lse, shape.softmax_scale, shape.causal, det)
    torch.cuda.synchronize()
    assert torch.equal(ref[1], dk) and torch.equal(ref[2], dv)
    if det:
        assert torch.equal(ref[0], dq)


@pytest.mark.parametrize("det", [False, True], ids=["atomic", "deterministic"])
def test_workspace_reused_across_calls(det):
    """The persistent kernels hand out work items from counters in the workspace header and the
    last CTA of each launch resets them (and the preprocess kernel of each call clears them).
    One workspace, sized for the largest problem, serves several calls of different shapes and
    causal modes in a row; each result must match the oracle."""
    shapes = [inputs.Shape(1, 8, 2, 512, 512, 128, True, "bf16"), inputs.Shape(2, 4, 4, 200, 77, 64, 2, "f16"),
              inputs.Shape(1, 4, 1, 333, 333, 128, False, "bf16"), inputs.Shape(1, 8, 2, 512, 512, 128, True, "bf16")]
    big = max(_lib.fa_bwd_workspace_size(sh.B, sh.Hq, sh.Hkv, sh.Nq, sh.Nkv, sh.d, int(det)) for sh in shapes)
    ws = torch.empty(big, dtype=torch.uint8, device="cuda")
    for i, shape in enumerate(shapes):
        (q, k, v, do), _, _, g = oracle_full(shape, 12 + i)
        qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
        o, lse = torch_api.forward(qd, kd, vd, shape.softmax_scale, shape.causal)
        dq, dk, dv = torch_api.backward(qd, kd, vd, o, dod, lse, shape.softmax_scale, shape.causal, det, ws=ws)
        torch.cuda.synchronize()
        assert _lib.fa_last_device_error() == _lib.FA_OK
        fails, rep = errors({"dQ": (_np(dq), g["dq"]), "dK": (_np(dk), g["dk"]), "dV": (_np(dv), g["dv"])})
        assert not fails, f"call {i} {shape.name()}\n{rep}"


def test_deterministic_is_bitwise_reproducible():
    shape = inputs.llama_gqa(1000)
    q, k, v, do = (t.cuda() for t in inputs.draw(shape, 8))
    o, lse = torch_api.forward(q, k, v, shape.softmax_scale, True)
    a = torch_api.backward(q, k, v, o, do, lse, shape.softmax_scale, True, True)
    b = torch_api.backward(q, k, v, o, do, lse, shape.softmax_scale, True, True)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_atomic_mode_dk_dv_are_reproducible():
    """dK, dV never go through atomics, so they are bitwise stable in either mode."""
    shape = inputs.Shape(2, 8, 2, 700, 700, 128, True, "bf16")
    q, k, v, do = (t.cuda() for t in inputs.draw(shape, 9))
    o, lse = torch_api.forward(q, k, v, shape.softmax_scale, True)
    a = torch_api.backward(q, k, v, o, do, lse, shape.softmax_scale, True, False)
    b = torch_api.backward(q, k, v, o, do, lse, shape.softmax_scale, True, True)
    torch.cuda.synchronize()
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    assert (a[0].float() - b[0].float()).abs().max().item() <= 1e-2 * b[0].float().abs().max().item() + 1e-3


@pytest.mark.parametrize("det", [False, True])
@pytest.mark.parametrize("shape", [
    inputs.Shape(1, 4, 2, 77, 200, 64, 2, "bf16"),      # Nq < Nkv: every row sees a key
    inputs.Shape(2, 4, 2, 300, 130, 128, 2, "f16"),     # Nq > Nkv: the first 170 rows see none
    inputs.Shape(1, 2, 1, 450, 64, 128, 2, "bf16"),     # two whole 128-row query tiles see no key
    inputs.Shape(1, 2, 2, 129, 257, 128, 2, "bf16"),    # ragged on both sides
    inputs.Shape(1, 2, 1, 96, 96, 64, 2, "f16"),        # Nq == Nkv: same as top-left
], ids=lambda s: s.name())
def test_bottom_right_causal(shape, det):
    check_full(shape, 11, det)


@pytest.mark.parametrize("det", [False, True])
@pytest.mark.parametrize("shape", [
    inputs.Shape(1, 2, 1, 70, 90, 8, 1, "bf16"),
    inputs.Shape(2, 4, 2, 130, 130, 32, 0, "f16"),
    inputs.Shape(1, 4, 4, 200, 150, 40, 2, "bf16"),
    inputs.Shape(1, 6, 2, 129, 257, 72, 1, "bf16"),
    inputs.Shape(2, 2, 1, 256, 256, 96, 1, "f16"),
    inputs.Shape(1, 2, 2, 100, 300, 120, 0, "bf16"),
], ids=lambda s: s.name())
def test_other_head_dims(shape, det):
    """Head dims other than 64 / 128 run on those kernels with the missing columns read as zero."""
    check_full(shape, 12, det)


def test_outputs_are_overwritten_not_accumulated():
    shape = inputs.Shape(1, 2, 1, 150, 150, 64, True, "f16")
    q, k, v, do = (t.cuda() for t in inputs.draw(shape, 10))
    o, lse = torch_api.forward(q, k, v, shape.softmax_scale, True)
    ref = torch_api.backward(q, k, v, o, do, lse, shape.softmax_scale, True, False)
    out = tuple(torch.full_like(t, 7.0) for t in ref)
    got = torch_api.backward(q, k, v, o, do, lse, shape.softmax_scale, True, False, out=out)
    torch.cuda.synchronize()
    for x, y in zip(ref, got):
        assert (x.float() - y.float()).abs().max().item() <= 1e-2 * x.float().abs().max().item() + 1e-3


def test_bounded_wait_reports_timeout_and_context_survives():
    """Failure detection without a fault: a wait nobody satisfies gives up and reports."""
    s = torch.cuda.current_stream()
    assert _lib.fa_last_device_error(s) == _lib.FA_OK
    assert _lib.fa_selftest_wait_timeout(20000, s) == _lib.FA_OK
    assert _lib.fa_last_device_error(s) == _lib.FA_ERR_DEVICE_TIMEOUT
    assert _lib.fa_last_device_error(s) == _lib.FA_OK        # read-and-clear
    check_full(inputs.tiny_mha()[0], 1, False)              # the context still works


def test_llama_gqa_sampled_deterministic_headline():
    """The deterministic path at the benchmark's shape: full run on the GPU, two (batch, kv-head)
    groups computed exactly by the oracle; and a second run is bitwise identical."""
    shape = inputs.llama_gqa(8192)
    q, k, v, do = inputs.draw(shape, 15, device="cuda")
    o, lse, dq, dk, dv = gpu_run(q, k, v, do, shape, True)
    G = shape.Hq // shape.Hkv
    pairs = {}
    for b, g in [(1, 2), (shape.B - 1, 0)]:
        hs = slice(g * G, (g + 1) * G)
        sl = lambda t, h: t[b:b + 1, h].cpu()  # noqa: E731
        qs, dos = sl(q, hs), sl(do, hs)
        ks, vs = sl(k, slice(g, g + 1)), sl(v, slice(g, g + 1))
        r = attn_ref.backward(qs, ks, vs, dos, shape.softmax_scale, True)
        pairs[f"dQ[{b},{g}]"] = (_np(dq[b:b + 1, hs]), r["dq"])
        pairs[f"dK[{b},{g}]"] = (_np(dk[b:b + 1, g:g + 1]), r["dk"])
        pairs[f"dV[{b},{g}]"] = (_np(dv[b:b + 1, g:g + 1]), r["dv"])
    fails, rep = errors(pairs)
    assert not fails, rep
    again = torch_api.backward(q, k, v, o, do, lse, shape.softmax_scale, True, True)
    torch.cuda.synchronize()
    assert torch.equal(again[0], dq) and torch.equal(again[1], dk) and torch.equal(again[2], dv)
