"""The multi-GPU path of the benchmark is N independent replicas: a barrier
and the slowest rank's time, no collective on the data path. Checked here
with two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def rank_main(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        ms = [12.5, 40.25][rank]  # rank 1 is the slow replica
        out[rank] = bench.max_over_ranks(ms, world)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    world, port = 2, free_port()
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(rank_main, args=(world, port, out), nprocs=world, join=True,
                       start_method="spawn")
    assert dict(out) == {0: 40.25, 1: 40.25}


def test_single_rank_and_replica_throughput():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    # two replicas of 2e12 FLOPs in 1 s (the slowest rank): 4 TFLOP/s in all
    assert bench.replicas_value(2e12, 2, 1000.0) == pytest.approx(4.0)
