"""bench.py's multi-rank host logic on two gloo ranks (CPU only).

Each rank runs an independent replica of the workload; the job is timed by
the slowest rank and its value is the work of all ranks over that time.
"""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        elapsed = [3.0, 5.0][rank]  # rank 1 is the slow one
        out[rank] = bench.max_over_ranks(elapsed, dist, "cpu")
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    port = _free_port()
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    assert out[0] == 5.0 and out[1] == 5.0


def test_job_value_counts_every_rank():
    flops = 4.0 * 4 * 16 * 4096 ** 2 * 128
    one = bench.job_tflops(flops, 1, 0.4)
    assert bench.job_tflops(flops, 2, 0.4) == pytest.approx(2 * one)
    assert bench.max_over_ranks(1.25) == 1.25
