"""Replica aggregation of bench.py across ranks (gloo, world size 2, CPU):
the job's rate is the units of all ranks over the slowest rank's time."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    units = [1000.0, 3000.0][rank]
    ms = [10.0, 40.0][rank]
    rate, tmax = bench.whole_job_rate(units, ms, world, torch.device("cpu"))
    bench.barrier(world)
    q.put((rank, rate, tmax, bench.dist_env()))
    dist.destroy_process_group()


def test_whole_job_rate_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, rate, tmax, env in out:
        assert tmax == 40.0
        assert rate == pytest.approx(4000.0 / 0.040)
        assert env == (rank, 2, rank)


def test_single_rank_rate():
    import bench
    rate, tmax = bench.whole_job_rate(500.0, 5.0, 1, torch.device("cpu"))
    assert tmax == 5.0 and rate == pytest.approx(100000.0)
