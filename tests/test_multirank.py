"""Host logic of the multi-rank bench path on CPU (gloo, world size 2).

Every GPU runs its own copy of the workload (weak scaling, no collective on the
data path); the only cross-rank steps are the barrier around the timed region
and the max-over-ranks of the elapsed time, which these tests exercise.
"""
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


def _worker(rank: int, world: int, port: int, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    d = bench.Dist("gloo")
    try:
        d.barrier()
        slowest = d.max(10.0 + 5.0 * rank)           # rank 1 is the slow one
        value = bench.aggregate(per_rank_flops=2.0e12, steps=10, max_ms=slowest, world=world)
        q.put((rank, slowest, value, d.active))
    finally:
        d.close()


def test_max_over_ranks_and_whole_job_aggregate():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, slowest, value, active in got:
        assert active
        assert slowest == 15.0                        # every rank sees the max
        # 2 ranks x 2e12 FLOP x 10 steps over 15 ms = 2666.67 TFLOP/s
        assert value == pytest.approx(2 * 2.0e12 * 10 / 15e-3 / 1e12)


def test_single_rank_needs_no_process_group():
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        os.environ.pop(k, None)
    d = bench.Dist("gloo")
    assert not d.active
    assert d.max(3.5) == 3.5
    assert bench.aggregate(1e12, 4, 2.0, 1) == pytest.approx(2000.0)
