"""Host-side logic of the multi-process benchmark path, on CPU with gloo (world size 2).

Each rank runs its own independent (batch, head) shard; the job's throughput is all
ranks' work divided by the slowest rank's time.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        my_ms = 2.0 + rank          # rank 1 is the slow one
        ms = bench.max_over_ranks(my_ms, dist, "cpu")
        out[rank] = ms
        out[world + rank] = bench.job_throughput(1e12, world, ms)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_weak_scaling_throughput_gloo():
    world = 2
    out = mp.get_context("spawn").Manager().list([0.0] * (2 * world))
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, start_method="spawn", join=True)
    assert list(out[:world]) == [3.0, 3.0]                      # every rank sees the slowest time
    assert out[world] == pytest.approx(1e12 * 2 / 3e-3 / 1e12)  # 2 ranks x 1 TFLOP in 3 ms


def test_single_process_helpers():
    assert bench.max_over_ranks(1.5) == 1.5
    assert bench.job_throughput(2e12, 1, 1000.0) == pytest.approx(2.0)
    B, H, N, d = 1, 32, 8192, 128
    assert bench.flops_fwd(B, H, N, d, True) == pytest.approx(549.76e9, rel=1e-3)
    assert bench.flops_bwd(B, H, N, d, True) == pytest.approx(2.5 * 549.76e9, rel=1e-3)
