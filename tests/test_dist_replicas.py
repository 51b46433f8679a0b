"""The N > 1 bench path on CPU (gloo, world size 2): every rank times its own replica, the
job takes each timing from the slowest rank, and the whole-job value counts all ranks'
units over that time (replicas only: no data-path collective)."""

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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r measured (r + 1) ms per step, 2 (r + 1) ms of attention, ...
        local = [0.001 * (rank + 1), 0.002 * (rank + 1), 0.0005 / (rank + 1), 0.004 + rank * 1e-4]
        got = bench.max_over_ranks(local, dist, "cpu")
        dist.barrier()
        q.put((rank, got, bench.job_value(37440, world, got[0])))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_value_gloo():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = dict((r, (g, v)) for r, g, v in (q.get(timeout=120) for _ in range(world)))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    expect = [0.002, 0.004, 0.0005, 0.0041]
    for r in range(world):
        g, v = res[r]
        assert g == pytest.approx(expect, rel=0, abs=1e-15)
        assert v == pytest.approx(2 * 37440 / 0.002)
