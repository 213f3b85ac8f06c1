"""The multi-GPU path of bench.py is replicas only (the layer has no exchange
step): every rank times its own copy, the job takes the slowest rank's time
and counts every rank's tokens.  This checks that host logic with two gloo
ranks on the CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    bench.barrier(world)
    slowest = bench.max_over_ranks(1.5 + rank, world)         # rank 1 is the slow one
    out[rank] = slowest
    out[world + rank] = bench.job_throughput(128, world, slowest)
    bench.barrier(world)
    dist.destroy_process_group()


def test_two_replicas_agree_on_the_slowest_rank():
    world = 2
    out = torch.zeros(2 * world, dtype=torch.float64).share_memory_()
    mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
    assert out[0].item() == out[1].item() == 2.5
    # 2 ranks x 128 tokens in 2.5 ms
    assert out[2].item() == out[3].item() == pytest.approx(2 * 128 / 2.5e-3)


def test_single_process_path_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.0, 1) == 3.0
    assert bench.job_throughput(100, 1, 2.0) == pytest.approx(5e4)
