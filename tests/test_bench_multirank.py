"""The benchmark's multi-rank plumbing on CPU: two gloo ranks, each an
independent replica (its own batch, no exchange on the data path).  The job's
time is the slowest rank's, and its rate counts every rank's sequences."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from workloads import make_linear


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, lr, w = bench.dist_env()
        elapsed = 1.0 + 0.5 * rank                     # rank 1 is the slow one
        slowest = bench.max_over_ranks(elapsed)
        d = make_linear(1, 1.0, B=2, K=2, V=64, seed=1001 + 7 * r)   # each replica's own batch
        q.put((r, lr, w, slowest, d["target"].sum().item()))
    finally:
        dist.destroy_process_group()


def test_two_rank_replicas_take_the_slowest_time():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for pr in procs:
        pr.start()
    for pr in procs:
        pr.join(120)
    assert all(pr.exitcode == 0 for pr in procs)
    got = sorted(q.get(timeout=10) for _ in range(world))
    assert [g[0] for g in got] == [0, 1] and all(g[2] == world for g in got)
    assert all(g[3] == pytest.approx(1.5) for g in got)     # max over ranks, seen by both
    assert got[0][4] != got[1][4]                            # independent batches per rank


def test_job_rate_counts_every_rank():
    assert bench.job_rate(1, 64, 100, 2.0) == pytest.approx(3200.0)
    assert bench.job_rate(4, 64, 100, 2.0) == pytest.approx(4 * 3200.0)


def test_single_process_max_is_identity():
    assert bench.max_over_ranks(3.25) == 3.25
