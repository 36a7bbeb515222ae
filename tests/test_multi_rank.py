"""The N > 1 path of bench.py on CPU: two gloo ranks, each a replica of the workload.

The backward shards into independent (batch, kv-head) groups with no exchange
step, so multi-GPU runs are replicas; the only cross-rank steps are the
barrier and the max over ranks of the timed region, tested here.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        ms = 10.0 + 5.0 * rank                     # rank 1 is the slow replica
        m = bench.max_over_ranks(ms, world)
        v = bench.whole_job_tflops(5e12, 4, world, m)
        q.put((rank, m, v))
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_whole_job_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, m, v in res:
        assert m == pytest.approx(15.0)                      # max over ranks
        assert v == pytest.approx(2 * 5e12 * 4 / 15e-3 / 1e12)  # both replicas' FLOPs / slowest time


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.whole_job_tflops(1e12, 10, 1, 1000.0) == pytest.approx(10.0)
