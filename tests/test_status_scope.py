"""A device-side failure that nobody reads must not change the results of later calls.

Every bounded wait that gives up marks two places: the device's status word
(read and cleared by fa_last_device_error) and the abort word of its own call
(which stops the other CTAs of that call).  Kernels act only on their own
call's abort word.  These tests leave a failure pending in the status word,
on the host side and without any fault: a packed batch whose offsets decrease
(FA_ERR_ARG, caught by the kernels' own offset checks), and the wait self-test
(FA_ERR_DEVICE_TIMEOUT).  Without reading the word they then run fa_fwd and
fa_bwd in both dQ modes on the tiny and ragged workloads, and compare every
output with the fp64 oracle element by element.  Only after that is the word
read, and it must still hold the failure that was left in it.
Tolerance: max|gpu - ref| <= 1e-2 * max|ref| + 1e-3 per tensor.
"""
import pytest
import torch

from attn_bwd_gb300 import _lib, inputs, torch_api
from oracle import attn_ref
from test_parity import _np, errors, oracle_full

pytestmark = pytest.mark.gpu

WORKLOADS = [(inputs.tiny_mha()[0], 1)] + [(s, 2) for s in inputs.ragged() if s.Nq in (1, 33, 100)]


def _leave_arg_error():
    """A forward on a packed batch whose second sequence ends before it starts."""
    pk = inputs.Packed((40, 60), (40, 60), 2, 1, 64, 1, "bf16")
    q, k, v, _ = (t.cuda() for t in inputs.draw_packed(pk, 23))
    bad = torch.tensor([0, 70, 60], dtype=torch.int32, device="cuda")
    good_k = torch.tensor([0, 40, 100], dtype=torch.int32, device="cuda")
    o = torch.zeros_like(q)
    lse = torch.zeros(2, 100, dtype=torch.float32, device="cuda")
    st = _lib.fa_fwd_varlen(q, k, v, o, lse, bad, good_k, 2, 2, 1, 100, 100, 100, 100, 64, pk.softmax_scale, 1,
                            _lib.FA_BF16, torch.cuda.current_stream())
    assert st == _lib.FA_OK
    torch.cuda.synchronize()


def _check_unread(shape, seed, det):
    """Forward and backward through the C ABI and the oracle comparison, without reading the status."""
    (q, k, v, do), o_ref, lse_ref, g = oracle_full(shape, seed)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = torch_api.forward(qd, kd, vd, shape.softmax_scale, shape.causal)
    dq, dk, dv = torch_api.backward(qd, kd, vd, o, dod, lse, shape.softmax_scale, shape.causal, det)
    torch.cuda.synchronize()
    fails, rep = errors({"O": (_np(o), o_ref), "L": (_np(lse), lse_ref),
                         "dQ": (_np(dq), g["dq"]), "dK": (_np(dk), g["dk"]), "dV": (_np(dv), g["dv"])})
    assert not fails, f"{shape.name()} det={det} with a failure pending\n{rep}"


@pytest.mark.parametrize("det", [False, True], ids=["atomic", "deterministic"])
def test_pending_arg_error_leaves_later_calls_exact(det):
    s = torch.cuda.current_stream()
    assert _lib.fa_last_device_error(s) == _lib.FA_OK
    _leave_arg_error()
    for shape, seed in WORKLOADS:
        _check_unread(shape, seed, det)
    assert _lib.fa_last_device_error(s) == _lib.FA_ERR_ARG      # still the failure that was left
    assert _lib.fa_last_device_error(s) == _lib.FA_OK


def test_pending_timeout_leaves_later_calls_exact():
    s = torch.cuda.current_stream()
    assert _lib.fa_last_device_error(s) == _lib.FA_OK
    assert _lib.fa_selftest_wait_timeout(2000, s) == _lib.FA_OK
    torch.cuda.synchronize()
    for det in (False, True):
        for shape, seed in WORKLOADS:
            _check_unread(shape, seed, det)
    assert _lib.fa_last_device_error(s) == _lib.FA_ERR_DEVICE_TIMEOUT
    assert _lib.fa_last_device_error(s) == _lib.FA_OK


def test_pending_error_leaves_packed_and_host_paths_exact():
    """The same with the packed-batch backward and fa_bwd_host, which runs chunks on several streams."""
    s = torch.cuda.current_stream()
    assert _lib.fa_last_device_error(s) == _lib.FA_OK
    _leave_arg_error()
    pk = inputs.packed_mix()[1]
    q, k, v, do = inputs.draw_packed(pk, 24)
    o_ref, lse_ref = attn_ref.forward_varlen(q, k, v, pk.cu_q, pk.cu_k, pk.softmax_scale, pk.causal)
    g = attn_ref.backward_varlen(q, k, v, do, pk.cu_q, pk.cu_k, pk.softmax_scale, pk.causal)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = torch_api.forward_varlen(qd, kd, vd, pk.cu_q, pk.cu_k, pk.softmax_scale, pk.causal)
    dq, dk, dv = torch_api.backward_varlen(qd, kd, vd, o, dod, lse, pk.cu_q, pk.cu_k, pk.softmax_scale, pk.causal)
    torch.cuda.synchronize()
    fails, rep = errors({"O": (_np(o), o_ref), "L": (_np(lse), lse_ref),
                         "dQ": (_np(dq), g["dq"]), "dK": (_np(dk), g["dk"]), "dV": (_np(dv), g["dv"])})
    assert not fails, rep
    shape = inputs.Shape(2, 8, 2, 300, 300, 128, True, "bf16")
    (q, k, v, do), _, _, g = oracle_full(shape, 7)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = torch_api.forward(qd, kd, vd, shape.softmax_scale, True)
    host = [t.cpu().pin_memory() for t in (qd, kd, vd, o, dod, lse)]
    outs = [torch.empty_like(t).pin_memory() for t in (host[0], host[1], host[2])]
    n = _lib.fa_bwd_host_staging_size(2, 8, 2, 300, 300, 128, 0, 1, 3)
    staging = torch.empty(n, dtype=torch.uint8, device="cuda")
    st = _lib.fa_bwd_host(*host, *outs, 2, 8, 2, 300, 300, 128, shape.softmax_scale, 1, _lib.FA_BF16, 0, 1, 3,
                          staging, n, s)
    assert st == _lib.FA_OK
    torch.cuda.synchronize()
    fails, rep = errors({"dQ": (_np(outs[0]), g["dq"]), "dK": (_np(outs[1]), g["dk"]),
                         "dV": (_np(outs[2]), g["dv"])})
    assert not fails, rep
    assert _lib.fa_last_device_error(s) == _lib.FA_ERR_ARG
    assert _lib.fa_last_device_error(s) == _lib.FA_OK
