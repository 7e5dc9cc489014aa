"""The N>1 path of bench.py on CPU: two gloo ranks (no GPU).

bench.py runs one replica of the workload per GPU and reports the work of
all ranks over the slowest rank's time; these tests check that aggregation
with world_size 2 over gloo on 127.0.0.1."""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, result):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms_max = bench.max_over_ranks(times[rank], world, "cpu")
        result[rank] = (ms_max, bench.job_value(1e12, world, ms_max))
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("times", [(10.0, 12.5), (30.0, 3.0)])
def test_two_ranks_max_time_and_job_value(times):
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    result = mgr.dict()
    world, port = 2, _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, times, result)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    slow = max(times)
    for r in range(world):
        ms_max, value = result[r]
        assert ms_max == slow
        assert abs(value - world * 1e12 / (slow * 1e-3) / 1e12) < 1e-9


def test_single_rank_identity():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(7.5, 1, "cpu") == 7.5
    assert bench.job_value(2e12, 1, 1000.0) == 2.0
