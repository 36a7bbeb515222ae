"""fa_bwd_host: tensors in host memory, pipelined through a ring of device staging slots in
chunks of (batch, kv-head) groups.  Its results must be those of fa_bwd on the same values
(bitwise for everything that does not go through atomics)."""
import pytest
import torch

from attn_bwd_gb300 import _lib, inputs, torch_api

pytestmark = pytest.mark.gpu


# 5 sequences x 2 kv heads = 10 groups: one chunk per group on one slot, ragged last chunks,
# more slots than chunks, the whole problem as one chunk
@pytest.mark.parametrize("det", [False, True])
@pytest.mark.parametrize("chunk_groups,slots", [(1, 1), (3, 2), (4, 3), (3, 8), (10, 1)])
def test_host_pipeline_matches_device_call(chunk_groups, slots, det):
    shape = inputs.Shape(5, 4, 2, 300, 300, 128, 1, "bf16")
    q, k, v, do = (t.cuda() for t in inputs.draw(shape, 91))
    o, lse = torch_api.forward(q, k, v, shape.softmax_scale, 1)
    ref = torch_api.backward(q, k, v, o, do, lse, shape.softmax_scale, 1, det)
    hin = [t.cpu().pin_memory() for t in (q, k, v, o, do, lse)]
    hout = [torch.full(t.shape, 3.0, dtype=t.dtype).pin_memory() for t in ref]
    n = _lib.fa_bwd_host_staging_size(5, 4, 2, 300, 300, 128, int(det), chunk_groups, slots)
    assert n > 0
    staging = torch.empty(n, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream()
    for _ in range(2):      # a second call reuses the staging and the library's streams
        st = _lib.fa_bwd_host(*hin, *hout, 5, 4, 2, 300, 300, 128, shape.softmax_scale, 1, _lib.FA_BF16, int(det),
                              chunk_groups, slots, staging, n, s)
        assert st == _lib.FA_OK
        s.synchronize()
        assert _lib.fa_last_device_error() == _lib.FA_OK
        got = [t.cuda() for t in hout]
        assert torch.equal(got[1], ref[1]) and torch.equal(got[2], ref[2])          # dK, dV: no atomics
        if det:
            assert torch.equal(got[0], ref[0])
        else:
            err = (got[0].float() - ref[0].float()).abs().max().item()
            assert err <= 1e-2 * ref[0].float().abs().max().item() + 1e-3
        for t in hout:
            t.fill_(3.0)


def test_host_pipeline_gqa_groups_of_four():
    """Hq/Hkv = 4 (the Llama-3 grouping): a chunk's query heads are its groups' 4 heads each."""
    shape = inputs.Shape(2, 8, 2, 257, 257, 64, 0, "f16")
    q, k, v, do = (t.cuda() for t in inputs.draw(shape, 92))
    o, lse = torch_api.forward(q, k, v, shape.softmax_scale, 0)
    ref = torch_api.backward(q, k, v, o, do, lse, shape.softmax_scale, 0, True)
    hin = [t.cpu().pin_memory() for t in (q, k, v, o, do, lse)]
    hout = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in ref]
    n = _lib.fa_bwd_host_staging_size(2, 8, 2, 257, 257, 64, 1, 3, 2)
    staging = torch.empty(n, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream()
    assert _lib.fa_bwd_host(*hin, *hout, 2, 8, 2, 257, 257, 64, shape.softmax_scale, 0, _lib.FA_F16, 1, 3, 2,
                            staging, n, s) == _lib.FA_OK
    s.synchronize()
    for g, r in zip(hout, ref):
        assert torch.equal(g.cuda(), r)
