"""Host-side logic of the multi-GPU bench (replicas: one process per GPU):
two gloo ranks on CPU agree on the slowest rank's step time, and the job
throughput counts every rank's tokens.  No GPU is used."""
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench

    d = bench.Dist(world, backend="gloo")
    d.barrier()
    ms = d.max(1.0 + rank)  # rank 1 is the slower one
    d.barrier()
    q.put((rank, ms, d.n, bench.job_tokens_per_s(d.n, 4, ms)))
    d.close()


def test_two_gloo_ranks_take_the_slowest_rank_and_sum_the_tokens():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(world))
    for rank, ms, n, tok_s in got:
        assert ms == pytest.approx(2.0)  # max over ranks
        assert n == 2
        assert tok_s == pytest.approx(2 * 4 / 2e-3)  # all ranks' tokens / slowest time


def test_single_process_needs_no_group():
    import bench

    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        os.environ.pop(k, None)
    d = bench.Dist(1, backend="gloo")
    assert d.pg is None and d.max(3.5) == 3.5 and d.n == 1
    assert bench.job_tokens_per_s(1, 1, 0.5) == pytest.approx(2000.0)
