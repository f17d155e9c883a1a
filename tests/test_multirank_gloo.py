"""The benchmark's multi-rank host logic on two CPU ranks (gloo, 127.0.0.1).

The path shards by token with no exchange step, so N GPUs run N independent replicas; the only
cross-rank logic is the barrier around the timed region and the maximum of the ranks' times.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    ws, r, local = bench.dist_env()
    bench.init_dist(ws, "gloo")
    try:
        bench.barrier(ws)
        my_ms = 10.0 + 5.0 * rank          # rank 1 is the slow one
        slowest = bench.max_over_ranks(my_ms, ws, torch.device("cpu"))
        rate = bench.whole_job_rate(ws, 16384, 20, slowest)
        q.put((r, local, slowest, rate))
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_rate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, local, slowest, rate in got:
        assert slowest == 15.0                       # the max over ranks, seen by every rank
        assert rate == pytest.approx(2 * 16384 * 20 / 0.015)
    assert [g[0] for g in got] == [0, 1]


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.5, 1, torch.device("cpu")) == 3.5
    assert bench.whole_job_rate(1, 100, 10, 1000.0) == pytest.approx(1000.0)
