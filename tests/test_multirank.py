"""The benchmark's multi-GPU host logic on CPU ranks (gloo, world size 2):
every rank times its own shard, the job time is the slowest rank's, and the
whole-job throughput counts every rank's bytes (weak scaling)."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, ms_per_rank, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(ms_per_rank[rank], world, torch.device("cpu"))
        q.put((rank, ms, bench.weak_scaling_value(1_000_000, world, ms)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_weak_scaling_value():
    world = 2
    ms_per_rank = [0.25, 0.5]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, ms_per_rank, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, ms, value in got:
        assert ms == 0.5                                  # the slowest rank sets the job time
        assert value == pytest.approx(2 * 1_000_000 / 0.5e-3 / 1e9)


def test_single_rank_is_identity():
    assert bench.max_over_ranks(0.3, 1) == 0.3
    assert bench.weak_scaling_value(2_000_000, 1, 1.0) == pytest.approx(2.0)       # 2 MB in 1 ms
