"""bench.py's replica accounting on N ranks, on CPU: two gloo ranks with different local
times both get the slowest rank's time, and the whole-job value counts every rank's
units over that time (replicas only: no data-path collective)."""

import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 100.0 + 25.0 * rank          # rank 1 is the slowest
        dist.barrier()
        m = bench.max_over_ranks(local_ms, world, torch.device("cpu"))
        out[rank] = (m, bench.job_gbs(world, 10, 1e9, m))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_time_and_the_job_total():
    world = 2
    port = _free_port()
    out = mp.Manager().dict()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_rank, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(world):
        m, gbs = out[r]
        assert m == 125.0
        # 2 ranks x 10 steps x 1 GB in 125 ms
        assert gbs == pytest.approx(2 * 10 * 1e9 / 0.125 / 1e9)


def test_one_rank_needs_no_collective():
    assert bench.max_over_ranks(42.0, 1, None) == 42.0
    assert bench.job_gbs(1, 4, 2e9, 1000.0) == pytest.approx(8.0)
