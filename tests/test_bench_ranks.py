"""The N-replica aggregation of bench.py on two gloo ranks (CPU): every rank
gets the slowest rank's time, divided over all the batches of the job."""
from __future__ import annotations

import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, totals, q) -> None:
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench.dist_env()
        q.put((r, w, local, bench.job_us_per_batch(totals[rank], 4, w, "cpu")))
    finally:
        dist.destroy_process_group()


def test_single_rank_is_the_plain_mean():
    assert bench.job_us_per_batch(2.0, 4, 1) == pytest.approx(500.0)


def test_two_ranks_take_the_slowest_over_all_batches():
    world, port = 2, _free_port()
    totals = [1.5, 2.5]                      # ms over 4 steps on each rank
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, totals, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    expect = max(totals) * 1000.0 / 4 / world    # 8 batches in the slowest rank's 2.5 ms
    assert [g[:3] for g in got] == [(0, 2, 0), (1, 2, 1)]
    assert all(g[3] == pytest.approx(expect) for g in got)
