"""The benchmark's multi-rank path on CPU: two gloo ranks, barrier, slowest-rank timing.

With N ranks every rank runs its own replica of the workload (the (sequence, head)
units are independent, so there is no collective on the data path); the job's time is
the maximum over ranks and its throughput counts every rank's units.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    w, r, local, pg = bench.dist_setup(world)
    assert (w, r) == (world, rank) and pg is not None
    bench.barrier(pg)
    ms = 10.0 * (rank + 1)                       # rank 1 is the slow one
    ms_max = bench.max_over_ranks(pg, ms, torch.device("cpu"))
    rate = bench.aggregate_rate(w, 8192, ms_max)
    bench.barrier(pg)
    dist.destroy_process_group()
    q.put((rank, ms_max, rate))


def test_two_gloo_ranks_time_by_the_slowest_and_count_all_units():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    for rank, ms_max, rate in res:
        assert ms_max == pytest.approx(20.0)
        assert rate == pytest.approx(2 * 8192 / 0.020)


def test_aggregate_rate_single_rank():
    assert bench.aggregate_rate(1, 8192, 2.0) == pytest.approx(4_096_000.0)
