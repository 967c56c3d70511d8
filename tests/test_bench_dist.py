"""bench.py's multi-rank path on the CPU: two gloo ranks, barrier, the
slowest rank's time, and the whole-job throughput (replicas only: each rank
runs its own copy of the job, so parameters add up over ranks)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist

    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        ms_local = 10.0 * (rank + 1)             # rank 1 is the slow one
        ms_step, value = bench.aggregate(ms_local, 1_000_000, 10, world)
        q.put((rank, ms_step, value))
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_max_over_ranks_and_whole_job_value(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(world))
    for rank, ms_step, value in got:
        assert ms_step == pytest.approx(2.0)               # the slowest rank: 20 ms over 10 steps
        assert value == pytest.approx(world * 1_000_000 / 2e-3 / 1e9)


def test_single_rank_aggregate():
    import bench
    assert bench.aggregate(5.0, 1000, 5, 1) == (1.0, pytest.approx(1000 / 1e-3 / 1e9))
