"""The benchmark's multi-rank bookkeeping on CPU with gloo, world size 2: every rank runs its own
batch, the job's time is the slowest rank's, and the throughput counts every rank's tokens."""

import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [120.0, 150.0][rank]                      # rank 1 is the slow one
    m = bench.max_over_ranks(ms, world, torch.device("cpu"))
    out[rank] = (m, bench.tokens_per_second(world, 32768, m))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_weak_scaling_throughput():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    for r in range(world):
        ms, tps = out[r]
        assert ms == 150.0
        assert abs(tps - 2 * 32768 / 0.150) < 1e-6


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.5, 1, torch.device("cpu")) == 3.5
    assert bench.tokens_per_second(1, 1000, 500.0) == 2000.0
