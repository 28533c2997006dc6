"""The multi-rank host logic of bench.py on CPU (gloo, world size 2).

A convolution layer is one problem, so `bench.py --gpus N` runs N
independent replicas (no data exchange): each rank times its own steps, the
job's time is the slowest rank's, and the throughput counts every rank's
FLOP. Two gloo ranks on 127.0.0.1 check that reduction and the arithmetic;
no GPU is involved.
"""
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


def _rank(rank, world, port, times, out):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slowest = bench.max_over_ranks(times[rank], world)
        out[rank] = (slowest, bench.job_tflops(1e12, 10, world, slowest))
    finally:
        dist.destroy_process_group()


def test_replicas_take_the_slowest_rank_and_count_every_rank():
    world, times = 2, [4.0, 5.0]
    out = mp.Manager().dict()
    mp.spawn(_rank, args=(world, _free_port(), times, out), nprocs=world, join=True)
    for r in range(world):
        slowest, tflops = out[r]
        assert slowest == 5.0
        # 2 ranks x 10 steps x 1 TFLOP in 5 ms
        assert tflops == pytest.approx(2 * 10 * 1.0 / 5e-3)


def test_single_rank_needs_no_process_group():
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_tflops(2e12, 4, 1, 8.0) == pytest.approx(2 * 4 / 8e-3)
