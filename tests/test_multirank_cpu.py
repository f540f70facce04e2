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


def test_head_ranges_cover_every_slice_once():
    from tiled_attention_forward_fa2_gb300.sharding import head_range
    for bh in (0, 1, 5, 16, 64, 257):
        for world in (1, 2, 3, 8):
            ranges = [head_range(bh, r, world) for r in range(world)]
            assert ranges[0][0] == 0 and ranges[-1][1] == bh
            assert all(a[1] == b[0] for a, b in zip(ranges, ranges[1:]))
            sizes = [b - a for a, b in ranges]
            assert max(sizes) - min(sizes) <= 1


def _shard_worker(rank, world, port, out):
    """Each rank computes its block of (batch, head) slices -- the CPU oracle stands in for
    the GPU kernel here -- and the blocks are gathered on every rank."""
    import numpy as np
    import torch

    import oracle
    from tiled_attention_forward_fa2_gb300.inputs import make_qkv
    from tiled_attention_forward_fa2_gb300.sharding import head_range

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        B, H, N, D = 2, 3, 96, 16
        q, k, v = make_qkv(B, H, N, D, seed=31)
        fl = lambda a: a.reshape(B * H, 1, N, D)  # noqa: E731
        a, b = head_range(B * H, rank, world)
        o, lse = oracle.attn_fwd(fl(q)[a:b].reshape(1, b - a, N, D), fl(k)[a:b].reshape(1, b - a, N, D),
                                 fl(v)[a:b].reshape(1, b - a, N, D), True, 0.25)
        # pad to the largest block for all_gather, then cut back
        m = B * H // world + 1
        t = torch.zeros(m, N, D + 1, dtype=torch.float64)
        t[: b - a, :, :D] = torch.from_numpy(o.reshape(b - a, N, D))
        t[: b - a, :, D] = torch.from_numpy(lse.reshape(b - a, N))
        parts = [torch.zeros_like(t) for _ in range(world)]
        dist.all_gather(parts, t)
        full = torch.cat([parts[r][: head_range(B * H, r, world)[1] - head_range(B * H, r, world)[0]]
                          for r in range(world)])
        o_ref, lse_ref = oracle.attn_fwd(q, k, v, True, 0.25)
        out[rank] = (bool(np.array_equal(full[..., :D].numpy(), o_ref.reshape(B * H, N, D))) and
                     bool(np.array_equal(full[..., D].numpy(), lse_ref.reshape(B * H, N))))
    finally:
        dist.destroy_process_group()


def test_two_ranks_each_compute_their_head_block():
    port = _free_port()
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_shard_worker, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    assert out[0] and out[1]
