"""Pins for the fp64 oracle, independent of the oracle itself.

The pages print no worked numeric example for the backward pass, so the
oracle is pinned by (1) hand-derived closed forms on two-key problems,
(2) central finite differences of the forward, (3) invariants that the
mathematics fixes, (4) special cases with known answers, (5) torch's own
fp64 autograd of scaled_dot_product_attention (a library routine), and
(6) planted mistakes that each of these must catch.
"""
import inspect
import math

import numpy as np
import pytest
import torch

from oracle import attn_ref


def _rand(shape, rng):
    return rng.standard_normal(shape)


# ---------------------------------------------------------------- closed forms

def test_two_key_closed_form_noncausal():
    """q=[1], keys 0 and ln3, scale 1: P=[1/4, 3/4] exactly.

    Hand derivation: S=[0, ln3], L=ln4, O = 2/4 + 18/4 = 5, dP = dO*V = [2, 6],
    D = 1/2 + 9/2 = 5 = dO*O, dS = P*(dP-D) = [-3/4, 3/4],
    dQ = sum_j dS_j K_j = (3/4) ln3, dK_j = dS_j * q = [-3/4, 3/4], dV = P = [1/4, 3/4].
    """
    q = np.array([[[[1.0]]]])
    k = np.array([[[[0.0], [math.log(3.0)]]]])
    v = np.array([[[[2.0], [6.0]]]])
    do = np.array([[[[1.0]]]])
    o, lse = attn_ref.forward(q, k, v, 1.0, False)
    assert o[0, 0, 0, 0] == pytest.approx(5.0, abs=1e-14)
    assert lse[0, 0, 0] == pytest.approx(math.log(4.0), abs=1e-14)
    g = attn_ref.backward(q, k, v, do, 1.0, False)
    assert g["dq"][0, 0, 0, 0] == pytest.approx(0.75 * math.log(3.0), abs=1e-14)
    np.testing.assert_allclose(g["dk"][0, 0, :, 0], [-0.75, 0.75], atol=1e-14)
    np.testing.assert_allclose(g["dv"][0, 0, :, 0], [0.25, 0.75], atol=1e-14)
    assert g["D"][0, 0, 0] == pytest.approx(5.0, abs=1e-14)


def test_two_key_closed_form_causal_with_scale():
    """Two queries q0=q1=[2], keys [0],[ln3/2], scale 1/2, causal.

    Row 0 sees key 0 only: P0=[1,0], O0=V0=2, L0=0, D0=dP00=2, dS0=[0,0], dQ0=0.
    Row 1 sees both keys; with q=2 and scale 1/2 the scaled score is q*k*scale = k,
    so S1 = [0, ln3/2], P1 = [1, sqrt3]/(1+sqrt3), L1 = ln(1+sqrt3).
    """
    r3 = math.sqrt(3.0)
    q = np.array([[[[2.0], [2.0]]]])
    k = np.array([[[[0.0], [math.log(3.0) / 2]]]])
    v = np.array([[[[2.0], [6.0]]]])
    do = np.array([[[[1.0], [1.0]]]])
    scale = 0.5
    p1 = np.array([1.0, r3]) / (1.0 + r3)
    o1 = p1 @ np.array([2.0, 6.0])
    dp1 = np.array([2.0, 6.0])
    d1 = p1 @ dp1
    ds1 = p1 * (dp1 - d1)
    kk = np.array([0.0, math.log(3.0) / 2])
    o, lse = attn_ref.forward(q, k, v, scale, True)
    np.testing.assert_allclose(o[0, 0, :, 0], [2.0, o1], atol=1e-14)
    np.testing.assert_allclose(lse[0, 0], [0.0, math.log(1.0 + r3)], atol=1e-14)
    g = attn_ref.backward(q, k, v, do, scale, True)
    np.testing.assert_allclose(g["dq"][0, 0, :, 0], [0.0, scale * ds1 @ kk], atol=1e-14)
    # dK_j = scale * sum_i dS_ij q_i ; only row 1 contributes
    np.testing.assert_allclose(g["dk"][0, 0, :, 0], scale * ds1 * 2.0, atol=1e-14)
    np.testing.assert_allclose(g["dv"][0, 0, :, 0], [1.0 + p1[0], p1[1]], atol=1e-14)


# --------------------------------------------------------- finite differences

def _loss(q, k, v, do, scale, causal):
    o, _ = attn_ref.forward(q, k, v, scale, causal)
    return float((o * do).sum())


def _fd_grad(x, f, h=1e-5):
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        idx = it.multi_index
        xp = x.copy(); xp[idx] += h
        xm = x.copy(); xm[idx] -= h
        g[idx] = (f(xp) - f(xm)) / (2 * h)
    return g


FD_CASES = [
    # B, Hq, Hkv, Nq, Nkv, d, causal
    (1, 1, 1, 1, 1, 2, False),
    (1, 1, 1, 2, 2, 2, True),
    (1, 2, 1, 3, 3, 4, False),
    (1, 2, 1, 5, 5, 4, True),
    (1, 2, 1, 3, 5, 2, True),     # Nq != Nkv, top-left causal
    (1, 4, 2, 4, 3, 2, False),    # GQA with two kv heads
    (2, 2, 2, 2, 3, 2, True),
    (1, 2, 1, 3, 5, 2, 2),        # bottom-right causal, Nq < Nkv
    (1, 2, 1, 5, 3, 2, 2),        # bottom-right causal, Nq > Nkv: two rows see no key
    (1, 4, 2, 4, 4, 2, 2),        # bottom-right causal, Nq == Nkv
]


@pytest.mark.parametrize("case", FD_CASES)
def test_finite_differences(case):
    B, Hq, Hkv, Nq, Nkv, d, causal = case
    rng = np.random.default_rng(hash(case) % 2**32)
    q = _rand((B, Hq, Nq, d), rng)
    k = _rand((B, Hkv, Nkv, d), rng)
    v = _rand((B, Hkv, Nkv, d), rng)
    do = _rand((B, Hq, Nq, d), rng)
    scale = 0.7
    g = attn_ref.backward(q, k, v, do, scale, causal)
    fq = _fd_grad(q, lambda x: _loss(x, k, v, do, scale, causal))
    fk = _fd_grad(k, lambda x: _loss(q, x, v, do, scale, causal))
    fv = _fd_grad(v, lambda x: _loss(q, k, x, do, scale, causal))
    for name, fd in (("dq", fq), ("dk", fk), ("dv", fv)):
        err = np.abs(g[name] - fd).max()
        assert err <= 1e-7 * max(1.0, np.abs(fd).max()), (name, err)


# ------------------------------------------------------------------ invariants

@pytest.mark.parametrize("causal", [False, True])
def test_invariants(causal):
    rng = np.random.default_rng(7)
    Nq, Nkv, d = 37, 29, 8
    q, k, v, do = (_rand((Nq, d), rng), _rand((Nkv, d), rng),
                   _rand((Nkv, d), rng), _rand((Nq, d), rng))
    r = attn_ref.head_backward(q, k, v, do, 0.4, causal)
    p, ds = r["P"], r["dS"]
    np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-13)
    assert np.abs(ds.sum(axis=1)).max() <= 1e-12 * np.abs(ds).max()
    np.testing.assert_allclose(r["D"], r["D_rowdot"], atol=1e-12)
    # sum over keys of dK = scale * sum_i (sum_j dS_ij) q_i = 0
    assert np.abs(r["dk"].sum(axis=0)).max() <= 1e-12 * max(1.0, np.abs(r["dk"]).max())
    if causal:
        assert np.all(p[np.triu_indices(min(Nq, Nkv), 1)] == 0.0)


# --------------------------------------------------------------- special cases

def test_single_key_and_query():
    rng = np.random.default_rng(1)
    q, k, v, do = (_rand((1, 2, 1, 4), rng), _rand((1, 2, 1, 4), rng),
                   _rand((1, 2, 1, 4), rng), _rand((1, 2, 1, 4), rng))
    for causal in (False, True):
        o, lse = attn_ref.forward(q, k, v, 0.3, causal)
        np.testing.assert_allclose(o, v, atol=1e-15)
        np.testing.assert_allclose(lse, 0.3 * (q * k).sum(-1), atol=1e-15)
        g = attn_ref.backward(q, k, v, do, 0.3, causal)
        assert np.all(g["dq"] == 0.0) and np.all(g["dk"] == 0.0)
        np.testing.assert_allclose(g["dv"], do, atol=1e-15)


def test_zero_queries_give_uniform_attention():
    rng = np.random.default_rng(2)
    q = np.zeros((1, 1, 6, 4))
    k, v = _rand((1, 1, 9, 4), rng), _rand((1, 1, 9, 4), rng)
    o, lse = attn_ref.forward(q, k, v, 1.0, False)
    np.testing.assert_allclose(o[0, 0], np.tile(v[0, 0].mean(axis=0), (6, 1)), atol=1e-14)
    np.testing.assert_allclose(lse, math.log(9.0), atol=1e-14)


def test_identical_value_rows_give_zero_dq_dk():
    rng = np.random.default_rng(3)
    q, k, do = _rand((1, 2, 7, 4), rng), _rand((1, 1, 7, 4), rng), _rand((1, 2, 7, 4), rng)
    v = np.tile(_rand((1, 1, 1, 4), rng), (1, 1, 7, 1))
    for causal in (False, True):
        g = attn_ref.backward(q, k, v, do, 0.5, causal)
        assert np.abs(g["dq"]).max() < 1e-14 and np.abs(g["dk"]).max() < 1e-14


def test_key_shift_invariance():
    """Adding one vector to every key adds a per-row constant to S: P, O, dV, dK, dQ unchanged."""
    rng = np.random.default_rng(4)
    q, k, v, do = (_rand((1, 2, 6, 4), rng), _rand((1, 2, 6, 4), rng),
                   _rand((1, 2, 6, 4), rng), _rand((1, 2, 6, 4), rng))
    c = _rand((1, 1, 1, 4), rng)
    for causal in (False, True):
        a = attn_ref.backward(q, k, v, do, 0.6, causal)
        b = attn_ref.backward(q, k + c, v, do, 0.6, causal)
        for name in ("dq", "dk", "dv"):
            np.testing.assert_allclose(a[name], b[name], atol=1e-12)


# ------------------------------------------------------ library cross-check

@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nkv,d,causal", [
    (2, 4, 4, 33, 33, 16, False),
    (2, 4, 4, 33, 33, 16, True),
    (1, 8, 2, 40, 40, 8, True),
    (1, 2, 1, 17, 31, 8, True),
])
def test_torch_sdpa_autograd(B, Hq, Hkv, Nq, Nkv, d, causal):
    """torch's fp64 math SDPA with autograd is an independent derivation of the gradients."""
    g = torch.Generator().manual_seed(11)
    q = torch.randn(B, Hq, Nq, d, generator=g, dtype=torch.float64)
    k = torch.randn(B, Hkv, Nkv, d, generator=g, dtype=torch.float64)
    v = torch.randn(B, Hkv, Nkv, d, generator=g, dtype=torch.float64)
    do = torch.randn(B, Hq, Nq, d, generator=g, dtype=torch.float64)
    scale = 0.3
    tq, tk, tv = (t.clone().requires_grad_(True) for t in (q, k, v))
    rep = Hq // Hkv
    out = torch.nn.functional.scaled_dot_product_attention(
        tq, tk.repeat_interleave(rep, dim=1), tv.repeat_interleave(rep, dim=1),
        is_causal=causal, scale=scale)
    out.backward(do)
    o, _ = attn_ref.forward(q, k, v, scale, causal)
    r = attn_ref.backward(q, k, v, do, scale, causal)
    np.testing.assert_allclose(o, out.detach().numpy(), atol=1e-12)
    np.testing.assert_allclose(r["dq"], tq.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(r["dk"], tk.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(r["dv"], tv.grad.numpy(), atol=1e-12)


def test_sampled_groups_match_full():
    rng = np.random.default_rng(5)
    q, do = _rand((2, 4, 9, 4), rng), _rand((2, 4, 9, 4), rng)
    k, v = _rand((2, 2, 9, 4), rng), _rand((2, 2, 9, 4), rng)
    full = attn_ref.backward(q, k, v, do, 0.5, True)
    part = attn_ref.backward(q, k, v, do, 0.5, True, groups=[(1, 0)])
    np.testing.assert_array_equal(part["dq"][1, 0:2], full["dq"][1, 0:2])
    np.testing.assert_array_equal(part["dk"][1, 0], full["dk"][1, 0])
    assert np.isnan(part["dq"][0]).all()


# ------------------------------------------------------------ planted mistakes

MUTANTS = [
    ("dropped scale on dQ", "dq = scale * (ds @ k)", "dq = (ds @ k)"),
    ("dropped scale on dK", "dk = scale * (ds.T @ q)", "dk = (ds.T @ q)"),
    ("wrong sign of D", "ds = p * (dp - D[:, None])", "ds = p * (dp + D[:, None])"),
    ("D dropped", "ds = p * (dp - D[:, None])", "ds = p * dp"),
    ("untransposed P in dV", "dv = p.T @ do", "dv = p @ do"),
    ("untransposed dS in dK", "dk = scale * (ds.T @ q)", "dk = scale * (ds @ q)"),
    ("D from the wrong axis", "D = (p * dp).sum(axis=1)", "D = (p * dp).sum(axis=0)"),
    ("dP from dO and K", "dp = do @ v.T", "dp = do @ k.T"),
]


@pytest.mark.parametrize("label,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistakes(label, old, new, monkeypatch):
    src = inspect.getsource(attn_ref.head_backward)
    assert old in src, label
    ns = dict(attn_ref.__dict__)
    exec(src.replace(old, new), ns)
    monkeypatch.setattr(attn_ref, "head_backward", ns["head_backward"])
    caught = False
    try:
        test_finite_differences((1, 2, 1, 3, 3, 4, False))
    except AssertionError:
        caught = True
    assert caught, f"finite-difference pin missed: {label}"


def test_pins_catch_wrong_causal_rule(monkeypatch):
    src = inspect.getsource(attn_ref.scores)
    ns = dict(attn_ref.__dict__)
    exec(src.replace("j > i", "j >= i + 1 + (i % 2)"), ns)
    monkeypatch.setattr(attn_ref, "scores", ns["scores"])
    with pytest.raises(AssertionError):
        test_torch_sdpa_autograd(2, 4, 4, 33, 33, 16, True)


def test_pins_catch_wrong_gqa_mapping(monkeypatch):
    monkeypatch.setattr(attn_ref, "kv_head", lambda h, Hq, Hkv: h % Hkv)
    src = inspect.getsource(attn_ref.backward)
    ns = dict(attn_ref.__dict__)
    exec(src.replace("range(g * G, (g + 1) * G)", "range(g, Hq, Hkv)"), ns)
    monkeypatch.setattr(attn_ref, "backward", ns["backward"])
    with pytest.raises(AssertionError):
        test_torch_sdpa_autograd(1, 8, 2, 40, 40, 8, True)


# ------------------------------------------------------------ golden record

def test_golden_regression_record():
    """The oracle still reproduces the record written by tests/golden/make_golden.py."""
    import json
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "oracle_small.json")
    rec = json.load(open(path))
    q, k, v, do = (np.array(rec[n]) for n in ("q", "k", "v", "do"))
    for c in rec["cases"]:
        o, lse = attn_ref.forward(q, k, v, c["scale"], c["causal"])
        g = attn_ref.backward(q, k, v, do, c["scale"], c["causal"])
        np.testing.assert_allclose(o, c["o"], rtol=0, atol=1e-15)
        np.testing.assert_allclose(lse, c["lse"], rtol=0, atol=1e-15)
        for n in ("dq", "dk", "dv", "D"):
            np.testing.assert_allclose(g[n], c[n], rtol=0, atol=1e-15)


# ------------------------------------------------------ causal alignment

BR = attn_ref.CAUSAL_BOTTOM_RIGHT


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nkv,d", [
    (1, 2, 1, 17, 31, 8),
    (2, 4, 2, 5, 40, 8),
    (1, 2, 2, 24, 24, 8),
])
def test_bottom_right_matches_torch_sdpa_with_explicit_mask(B, Hq, Hkv, Nq, Nkv, d):
    """Nq <= Nkv: every row sees a key, so torch's fp64 SDPA with the explicit
    bottom-right boolean mask (key j allowed for query i iff j <= i + Nkv - Nq)
    is an independent derivation of O, L and the gradients."""
    g = torch.Generator().manual_seed(23)
    q = torch.randn(B, Hq, Nq, d, generator=g, dtype=torch.float64)
    k = torch.randn(B, Hkv, Nkv, d, generator=g, dtype=torch.float64)
    v = torch.randn(B, Hkv, Nkv, d, generator=g, dtype=torch.float64)
    do = torch.randn(B, Hq, Nq, d, generator=g, dtype=torch.float64)
    scale = 0.4
    allowed = torch.ones(Nq, Nkv, dtype=torch.bool).tril(diagonal=Nkv - Nq)
    tq, tk, tv = (t.clone().requires_grad_(True) for t in (q, k, v))
    rep = Hq // Hkv
    out = torch.nn.functional.scaled_dot_product_attention(
        tq, tk.repeat_interleave(rep, dim=1), tv.repeat_interleave(rep, dim=1), attn_mask=allowed, scale=scale)
    out.backward(do)
    logits = scale * (q @ k.repeat_interleave(rep, dim=1).transpose(-1, -2))
    lse_t = torch.logsumexp(logits.masked_fill(~allowed, float("-inf")), dim=-1)
    o, lse = attn_ref.forward(q, k, v, scale, BR)
    r = attn_ref.backward(q, k, v, do, scale, BR)
    np.testing.assert_allclose(o, out.detach().numpy(), atol=1e-12)
    np.testing.assert_allclose(lse, lse_t.numpy(), atol=1e-12)
    np.testing.assert_allclose(r["dq"], tq.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(r["dk"], tk.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(r["dv"], tv.grad.numpy(), atol=1e-12)


@pytest.mark.parametrize("Nq,Nkv", [(7, 3), (12, 5), (4, 1)])
def test_bottom_right_with_more_queries_reduces_to_top_left(Nq, Nkv):
    """Nq > Nkv: the first m = Nq - Nkv rows see no key (O = 0, L = -inf, dQ = 0),
    and the rest is the top-left problem of the last Nkv queries, whose dK, dV
    are the whole problem's."""
    rng = np.random.default_rng(Nq * 100 + Nkv)
    q, do = _rand((1, 2, Nq, 4), rng), _rand((1, 2, Nq, 4), rng)
    k, v = _rand((1, 1, Nkv, 4), rng), _rand((1, 1, Nkv, 4), rng)
    m = Nq - Nkv
    o, lse = attn_ref.forward(q, k, v, 0.6, BR)
    r = attn_ref.backward(q, k, v, do, 0.6, BR)
    o_tl, lse_tl = attn_ref.forward(q[:, :, m:], k, v, 0.6, True)
    r_tl = attn_ref.backward(q[:, :, m:], k, v, do[:, :, m:], 0.6, True)
    assert (o[:, :, :m] == 0).all() and np.isneginf(lse[:, :, :m]).all()
    assert (r["dq"][:, :, :m] == 0).all() and (r["D"][:, :, :m] == 0).all()
    np.testing.assert_allclose(o[:, :, m:], o_tl, atol=1e-14)
    np.testing.assert_allclose(lse[:, :, m:], lse_tl, atol=1e-14)
    for n in ("dq",):
        np.testing.assert_allclose(r[n][:, :, m:], r_tl[n], atol=1e-14)
    for n in ("dk", "dv"):
        np.testing.assert_allclose(r[n], r_tl[n], atol=1e-14)


def test_bottom_right_single_key_closed_form():
    """Nq=3, Nkv=1, bottom-right: rows 0, 1 see nothing; row 2 sees the one key,
    so P = 1 there: O_2 = V_0, L_2 = S_20, dV_0 = dO_2, and dS = 0 gives dQ = dK = 0."""
    rng = np.random.default_rng(3)
    q, do = _rand((1, 1, 3, 2), rng), _rand((1, 1, 3, 2), rng)
    k, v = _rand((1, 1, 1, 2), rng), _rand((1, 1, 1, 2), rng)
    o, lse = attn_ref.forward(q, k, v, 0.5, BR)
    r = attn_ref.backward(q, k, v, do, 0.5, BR)
    np.testing.assert_array_equal(o[0, 0, :2], 0.0)
    np.testing.assert_allclose(o[0, 0, 2], v[0, 0, 0], atol=1e-15)
    assert np.isneginf(lse[0, 0, :2]).all()
    assert lse[0, 0, 2] == pytest.approx(0.5 * q[0, 0, 2] @ k[0, 0, 0], abs=1e-15)
    np.testing.assert_allclose(r["dv"][0, 0, 0], do[0, 0, 2], atol=1e-15)
    np.testing.assert_array_equal(r["dq"], 0.0)
    np.testing.assert_array_equal(r["dk"], 0.0)


def test_alignments_agree_when_lengths_are_equal():
    rng = np.random.default_rng(8)
    q, do = _rand((1, 2, 9, 4), rng), _rand((1, 2, 9, 4), rng)
    k, v = _rand((1, 1, 9, 4), rng), _rand((1, 1, 9, 4), rng)
    a = attn_ref.backward(q, k, v, do, 0.5, True)
    b = attn_ref.backward(q, k, v, do, 0.5, BR)
    for n in ("dq", "dk", "dv", "D"):
        np.testing.assert_array_equal(a[n], b[n])


def test_unknown_causal_mode_is_rejected():
    with pytest.raises(ValueError):
        attn_ref.causal_delta(3, 4, 4)


def test_pins_catch_wrong_bottom_right_offset(monkeypatch):
    src = inspect.getsource(attn_ref.causal_delta)
    ns = dict(attn_ref.__dict__)
    exec(src.replace("return nk - nq", "return nq - nk"), ns)
    monkeypatch.setattr(attn_ref, "causal_delta", ns["causal_delta"])
    with pytest.raises(AssertionError):
        test_bottom_right_matches_torch_sdpa_with_explicit_mask(1, 2, 1, 17, 31, 8)


# ------------------------------------------------------ packed batches

def _pack(x):
    """[B, H, N, d] -> [H, B*N, d] (sequence b at rows b*N .. b*N + N - 1)."""
    B, H, N, d = x.shape
    return np.ascontiguousarray(np.transpose(x, (1, 0, 2, 3)).reshape(H, B * N, d))


@pytest.mark.parametrize("causal", [0, 1, 2])
def test_varlen_equal_lengths_match_dense(causal):
    rng = np.random.default_rng(40 + causal)
    B, Hq, Hkv, Nq, Nkv, d = 3, 4, 2, 6, 9, 4
    q, do = _rand((B, Hq, Nq, d), rng), _rand((B, Hq, Nq, d), rng)
    k, v = _rand((B, Hkv, Nkv, d), rng), _rand((B, Hkv, Nkv, d), rng)
    cu_q, cu_k = [b * Nq for b in range(B + 1)], [b * Nkv for b in range(B + 1)]
    o, lse = attn_ref.forward(q, k, v, 0.5, causal)
    g = attn_ref.backward(q, k, v, do, 0.5, causal)
    ov, lv = attn_ref.forward_varlen(_pack(q), _pack(k), _pack(v), cu_q, cu_k, 0.5, causal)
    gv = attn_ref.backward_varlen(_pack(q), _pack(k), _pack(v), _pack(do), cu_q, cu_k, 0.5, causal)
    np.testing.assert_allclose(ov, _pack(o), atol=1e-14)
    np.testing.assert_allclose(lv, np.transpose(lse, (1, 0, 2)).reshape(Hq, B * Nq), atol=1e-14)
    for n in ("dq", "dk", "dv"):
        np.testing.assert_allclose(gv[n], _pack(g[n]), atol=1e-14)


def _sdpa_packed_mask(cu_q, cu_k, causal):
    """Allowed-key mask of the whole packed problem: same sequence, and the causal rule in local indices."""
    tq, tk = cu_q[-1], cu_k[-1]
    m = np.zeros((tq, tk), dtype=bool)
    for b in range(len(cu_q) - 1):
        nq, nk = cu_q[b + 1] - cu_q[b], cu_k[b + 1] - cu_k[b]
        i = np.arange(nq)[:, None]
        j = np.arange(nk)[None, :]
        delta = {0: None, 1: 0, 2: nk - nq}[causal]
        ok = np.ones((nq, nk), dtype=bool) if delta is None else (j <= i + delta)
        m[cu_q[b]:cu_q[b + 1], cu_k[b]:cu_k[b + 1]] = ok
    return m


@pytest.mark.parametrize("causal", [0, 1, 2])
def test_varlen_matches_torch_sdpa_on_the_packed_sequence(causal):
    """One packed sequence with a block-diagonal (and per-block causal) mask, through
    torch's fp64 SDPA and autograd: an independent construction of the packed batch."""
    lq = [3, 1, 7, 5]
    lk = [4, 1, 9, 5]                 # nq <= nk everywhere, so every row sees a key
    cu_q = list(np.cumsum([0] + lq))
    cu_k = list(np.cumsum([0] + lk))
    Hq, Hkv, d = 4, 2, 8
    g = torch.Generator().manual_seed(31 + causal)
    q = torch.randn(Hq, cu_q[-1], d, generator=g, dtype=torch.float64)
    k = torch.randn(Hkv, cu_k[-1], d, generator=g, dtype=torch.float64)
    v = torch.randn(Hkv, cu_k[-1], d, generator=g, dtype=torch.float64)
    do = torch.randn(Hq, cu_q[-1], d, generator=g, dtype=torch.float64)
    allowed = torch.from_numpy(_sdpa_packed_mask(cu_q, cu_k, causal))
    tq, tk, tv = (t.clone().requires_grad_(True) for t in (q, k, v))
    rep = Hq // Hkv
    out = torch.nn.functional.scaled_dot_product_attention(
        tq[None], tk.repeat_interleave(rep, dim=0)[None], tv.repeat_interleave(rep, dim=0)[None],
        attn_mask=allowed, scale=0.35)[0]
    out.backward(do)
    o, _ = attn_ref.forward_varlen(q, k, v, cu_q, cu_k, 0.35, causal)
    r = attn_ref.backward_varlen(q, k, v, do, cu_q, cu_k, 0.35, causal)
    np.testing.assert_allclose(o, out.detach().numpy(), atol=1e-12)
    np.testing.assert_allclose(r["dq"], tq.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(r["dk"], tk.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(r["dv"], tv.grad.numpy(), atol=1e-12)


def test_varlen_empty_sequences():
    """A sequence with queries but no keys: O = 0, L = -inf, dQ = 0; a sequence with keys
    but no queries: dK = dV = 0 for its keys."""
    rng = np.random.default_rng(9)
    cu_q, cu_k = [0, 2, 2, 5], [0, 3, 6, 6]     # seq 1: no queries; seq 2: no keys
    q, do = _rand((2, 5, 4), rng), _rand((2, 5, 4), rng)
    k, v = _rand((1, 6, 4), rng), _rand((1, 6, 4), rng)
    for causal in (0, 1, 2):
        o, lse = attn_ref.forward_varlen(q, k, v, cu_q, cu_k, 0.5, causal)
        r = attn_ref.backward_varlen(q, k, v, do, cu_q, cu_k, 0.5, causal)
        assert (o[:, 2:5] == 0).all() and np.isneginf(lse[:, 2:5]).all()
        assert (r["dq"][:, 2:5] == 0).all()
        assert (r["dk"][:, 3:6] == 0).all() and (r["dv"][:, 3:6] == 0).all()
        assert np.isfinite(lse[:, :2]).all()


def test_varlen_rejects_inconsistent_offsets():
    q = np.zeros((1, 4, 2))
    with pytest.raises(ValueError):
        attn_ref.forward_varlen(q, q, q, [0, 3, 2, 4], [0, 1, 2, 4], 1.0, 0)
    with pytest.raises(ValueError):
        attn_ref.forward_varlen(q, q, q, [0, 2, 3], [0, 2, 4], 1.0, 0)


def test_pins_catch_keys_leaking_across_sequences(monkeypatch):
    for fn in ("forward_varlen", "backward_varlen"):
        src = inspect.getsource(getattr(attn_ref, fn))
        assert "slice(cu_k[b], cu_k[b + 1])" in src
        ns = dict(attn_ref.__dict__)
        exec(src.replace("slice(cu_k[b], cu_k[b + 1])", "slice(0, cu_k[b + 1])"), ns)
        monkeypatch.setattr(attn_ref, fn, ns[fn])
    with pytest.raises(AssertionError):
        test_varlen_matches_torch_sdpa_on_the_packed_sequence(0)


# ------------------------------------------------------ additive bias

@pytest.mark.parametrize("bshape,causal", [
    ((2, 4), 0), ((1, 4), 1), ((2, 1), 2), ((1, 1), 0),
])
def test_bias_matches_torch_sdpa_float_mask(bshape, causal):
    """torch's fp64 SDPA adds a float attn_mask to the scaled scores and differentiates it:
    an independent derivation of O and of dBias (= dS) for every broadcast shape."""
    B, Hq, Hkv, Nq, Nkv, d = 2, 4, 2, 11, 19, 8
    g = torch.Generator().manual_seed(51 + causal)
    q = torch.randn(B, Hq, Nq, d, generator=g, dtype=torch.float64)
    k = torch.randn(B, Hkv, Nkv, d, generator=g, dtype=torch.float64)
    v = torch.randn(B, Hkv, Nkv, d, generator=g, dtype=torch.float64)
    do = torch.randn(B, Hq, Nq, d, generator=g, dtype=torch.float64)
    bias = torch.randn(bshape[0], bshape[1], Nq, Nkv, generator=g, dtype=torch.float64)
    scale = 0.45
    mask = bias.clone()
    delta = attn_ref.causal_delta(causal, Nq, Nkv)
    if delta is not None:
        allowed = torch.ones(Nq, Nkv, dtype=torch.bool).tril(diagonal=delta)
        mask = mask.masked_fill(~allowed, float("-inf"))
    tq, tk, tv, tb = (t.clone().requires_grad_(True) for t in (q, k, v, bias))
    tm = tb if delta is None else tb.masked_fill(~allowed, float("-inf"))
    rep = Hq // Hkv
    out = torch.nn.functional.scaled_dot_product_attention(
        tq, tk.repeat_interleave(rep, dim=1), tv.repeat_interleave(rep, dim=1), attn_mask=tm, scale=scale)
    out.backward(do)
    o, _ = attn_ref.forward(q, k, v, scale, causal, bias=bias)
    r = attn_ref.backward(q, k, v, do, scale, causal, bias=bias)
    np.testing.assert_allclose(o, out.detach().numpy(), atol=1e-12)
    np.testing.assert_allclose(r["dq"], tq.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(r["dk"], tk.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(r["dv"], tv.grad.numpy(), atol=1e-12)
    # dBias of a broadcast bias is dS summed over the broadcast axes
    db = r["dbias"]
    if bshape[0] == 1:
        db = db.sum(axis=0, keepdims=True)
    if bshape[1] == 1:
        db = db.sum(axis=1, keepdims=True)
    np.testing.assert_allclose(db, tb.grad.numpy(), atol=1e-12)


def test_minus_inf_bias_is_a_mask():
    """A -inf bias drops keys: equal to removing them, and a row with every key dropped
    sees none (O = 0, L = -inf)."""
    rng = np.random.default_rng(61)
    q, do = _rand((1, 2, 6, 4), rng), _rand((1, 2, 6, 4), rng)
    k, v = _rand((1, 1, 9, 4), rng), _rand((1, 1, 9, 4), rng)
    keep = np.array([1, 0, 1, 1, 0, 0, 1, 0, 1], dtype=bool)
    bias = np.where(keep, 0.0, -np.inf)[None, None, None, :].repeat(6, axis=2)
    bias[0, 0, 3, :] = -np.inf
    o, lse = attn_ref.forward(q, k, v, 0.5, 0, bias=bias)
    o2, lse2 = attn_ref.forward(q, k[:, :, keep], v[:, :, keep], 0.5, 0)
    rows = [0, 1, 2, 4, 5]          # row 3 drops every key (the bias broadcasts over both heads)
    np.testing.assert_allclose(o[0, :, rows], o2[0, :, rows], atol=1e-14)
    assert (o[0, :, 3] == 0).all() and np.isneginf(lse[0, :, 3]).all()
    r = attn_ref.backward(q, k, v, do, 0.5, 0, bias=bias)
    assert (r["dq"][0, :, 3] == 0).all()
    assert (r["dk"][0, 0, ~keep] == 0).all() and (r["dbias"][..., ~keep] == 0).all()


def test_pins_catch_bias_scaled_by_the_softmax_scale(monkeypatch):
    src = inspect.getsource(attn_ref.scores)
    ns = dict(attn_ref.__dict__)
    exec(src.replace("s = s + bias", "s = s + scale * bias"), ns)
    monkeypatch.setattr(attn_ref, "scores", ns["scores"])
    with pytest.raises(AssertionError):
        test_bias_matches_torch_sdpa_float_mask((2, 4), 0)
