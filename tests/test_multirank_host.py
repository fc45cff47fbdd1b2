"""The N > 1 path of bench.py on the CPU: two gloo ranks, each a replica with
its own timing; the job time is the slowest rank's and the throughput counts
both replicas' work."""
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


def _worker(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        out[rank] = bench.max_over_ranks(times[rank], torch.device("cpu"))
    finally:
        dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    world, port = 2, _free_port()
    times = [3.25, 4.5]
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(world, port, times, out), nprocs=world, join=True)
    assert out[0] == out[1] == 4.5


def test_aggregate_counts_every_replica():
    step_flop = 2.0e12
    assert bench.aggregate_tflops(step_flop, 4.0, 1) == pytest.approx(500.0)
    assert bench.aggregate_tflops(step_flop, 4.0, 2) == pytest.approx(1000.0)
