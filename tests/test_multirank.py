"""The N > 1 host path of the bench on CPU: two gloo ranks (replicas with their own
tokens, no collective on the data path; one all-reduce of the timing result)."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import workloads


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        ms = [12.5, 20.0][rank]                               # the slower rank sets the time
        out[rank] = bench.max_over_ranks(ms, world)
        x = workloads.gen_x(workloads.TINY, base_seed=rank)   # each replica its own tokens
        out[2 + rank] = float(x.float().sum())
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_distinct_tokens():
    world = 2
    out = mp.get_context("spawn").Manager().list([0.0] * 4)
    mp.start_processes(_rank, args=(world, _free_port(), out), nprocs=world, join=True,
                       start_method="spawn")
    assert out[0] == out[1] == 20.0
    assert out[2] != out[3]
    # whole-job value: every rank's tokens over the slowest rank's time
    assert bench.weak_scaling_value(256, 10, world, 20.0) == pytest.approx(256 * 2 * 10 / 0.02)
