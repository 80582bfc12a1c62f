"""The multi-rank plumbing of bench.py (replicas: barrier + max over ranks),
run as two gloo ranks on the CPU."""

from __future__ import annotations

import os
import socket

import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, out):
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        slowest = bench.max_over_ranks(10.0 + rank * 5.0, world)
        out[rank] = slowest
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert dict(out) == {0: 15.0, 1: 15.0}


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    bench.barrier(1)


def test_dist_env_defaults(monkeypatch):
    import bench
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (1, 0, 0)
    monkeypatch.setenv("WORLD_SIZE", "4")
    monkeypatch.setenv("RANK", "2")
    monkeypatch.setenv("LOCAL_RANK", "2")
    assert bench.dist_env() == (4, 2, 2)


def test_algorithmic_byte_counts():
    import bench
    assert bench.bytes_quant(2, 16) == 3 * 32 + 8
    assert bench.bytes_w8a16(1, 4, 16) == 64 + 16 + 32 + 8
    assert bench.bytes_w8a8(1, 4, 16, True) == 16 + 64 + 20 + 8 + 8
    import numpy as np
    assert bench.bytes_grouped(np.array([0, 3, 1], np.int32), 4, 16) == 2 * (64 + 16) + 2 * 4 * 20
