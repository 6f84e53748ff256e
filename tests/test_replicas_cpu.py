"""The benchmark's multi-rank host logic on CPU ranks (gloo, world size 2).

Replicas process independent batches, so the only cross-rank step is the
timing: a barrier and the max of the ranks' elapsed times; whole-job tokens/s
is all ranks' tokens over the slowest rank's time.
"""
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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        elapsed = [0.5, 0.8][rank]  # rank 1 is the straggler
        value, slowest = bench.replica_tokens_per_second(4096, 10, elapsed, world, device="cpu")
        out[rank] = (value, slowest)
    finally:
        dist.destroy_process_group()


def test_replica_throughput_uses_the_slowest_rank():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
    for rank in range(world):
        value, slowest = out[rank]
        assert slowest == pytest.approx(0.8)
        assert value == pytest.approx(2 * 4096 * 10 / 0.8)


def test_single_rank_needs_no_process_group():
    value, slowest = bench.replica_tokens_per_second(100, 4, 2.0, 1, device="cpu")
    assert (value, slowest) == (200.0, 2.0)
