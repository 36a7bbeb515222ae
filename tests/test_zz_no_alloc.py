"""fa_bwd_noalloc: the backward for callers that cannot allocate device memory.

Some callers cannot hand the library a workspace (an engine plugin whose host
framework owns all device memory, or a serving loop that forbids cudaMalloc
after start-up).  fa_bwd_noalloc takes its scratch from a fixed array inside
the library instead.  These tests call it through the C ABI twice in a row and
compare each result with fa_bwd's (which uses a caller workspace): bitwise in
deterministic mode, where both run the same kernels in a fixed summation order,
and within the parity tolerance used everywhere else in atomic mode:
max|err| <= 1e-2 * max|ref| + 1e-3.
This file is collected last on purpose.
"""
import pytest
import torch

from attn_bwd_gb300 import _lib, inputs, torch_api

pytestmark = pytest.mark.gpu

REL, ABS = 1e-2, 1e-3
A = 0x100000  # fake, aligned, never dereferenced (the call is rejected before any launch)


@pytest.mark.parametrize("det", [False, True], ids=["atomic", "deterministic"])
def test_noalloc_matches_workspace_entry_point(det):
    shape = inputs.Shape(2, 8, 2, 1000, 1000, 128, True, "bf16")
    assert _lib.fa_bwd_workspace_size(2, 8, 2, 1000, 1000, 128, int(det)) <= _lib.FA_STATIC_SCRATCH_BYTES
    q, k, v, do = (t.cuda() for t in inputs.draw(shape, 21))
    o, lse = torch_api.forward(q, k, v, shape.softmax_scale, True)
    ref = torch_api.backward(q, k, v, o, do, lse, shape.softmax_scale, True, det)
    stream = torch.cuda.current_stream()
    for _ in range(2):
        out = tuple(torch.full_like(t, float("nan")) for t in (q, k, v))
        st = _lib.fa_bwd_noalloc(q, k, v, o, do, lse, *out, 2, 8, 2, 1000, 1000, 128, shape.softmax_scale, 1,
                                 _lib.FA_BF16, int(det), stream)
        assert st == _lib.FA_OK, _lib.fa_strerror(st)
        torch.cuda.synchronize()
        assert _lib.fa_last_device_error(stream) == _lib.FA_OK
        for name, got, want in zip(("dQ", "dK", "dV"), out, ref):
            if det:
                # the same kernels in a fixed summation order: bitwise the same result
                assert torch.equal(got, want), name
                continue
            err = (got.float() - want.float()).abs().max().item()
            bound = REL * want.float().abs().max().item() + ABS
            assert err <= bound, f"{name}: {err:.3e} > {bound:.3e}"


def test_noalloc_rejects_problems_beyond_the_static_scratch():
    need = _lib.fa_bwd_workspace_size(4, 32, 8, 8192, 8192, 128, 0)
    assert need > _lib.FA_STATIC_SCRATCH_BYTES
    st = _lib.fa_bwd_noalloc(A, A, A, A, A, A, A, A, A, 4, 32, 8, 8192, 8192, 128, 0.088, 1, _lib.FA_BF16, 0)
    assert st == _lib.FA_ERR_WORKSPACE
