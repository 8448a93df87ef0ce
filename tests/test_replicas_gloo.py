"""Replica aggregation of bench.py over two ranks (gloo on the CPU).

Under torchrun every rank runs its own replica of the layer; the step time is
the slowest rank's and the throughput counts every rank's tokens.
"""
from __future__ import annotations

import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = 1.0 + rank  # rank 1 is the slower replica
    got = bench.max_over_ranks(ms, world)
    q.put((rank, got, bench.job_tokens_per_s(4096, world, got)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_max_and_throughput():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [2.0, 2.0]
    assert res[0][2] == pytest.approx(2 * 4096 / 2e-3)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_tokens_per_s(100, 1, 1.0) == pytest.approx(1e5)
