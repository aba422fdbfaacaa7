"""The multi-GPU host logic on CPU with two gloo ranks.

Every (batch, head) problem is independent, so N ranks split the units with no
data-path collective; only the timing max-reduction talks between ranks.  Here
two processes each take their contiguous share of a small batch, run the fp64
oracle on it, and the gathered shares must equal the single-process result.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def test_shard_range_partitions_exactly():
    for total in (0, 1, 5, 8, 33):
        for world in (1, 2, 3, 8):
            spans = [bench.shard_range(total, world, r) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == total
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
            sizes = [hi - lo for lo, hi in spans]
            assert max(sizes) - min(sizes) <= 1


def _inputs():
    g = torch.Generator().manual_seed(77)
    B, H, N, d, m, dv = 5, 2, 40, 16, 8, 6
    q = torch.randn((B, H, N, d), generator=g, dtype=torch.float64)
    k = torch.randn((B, H, N, d), generator=g, dtype=torch.float64)
    v = torch.randn((B, H, N, dv), generator=g, dtype=torch.float64)
    P = torch.randn((H, d, m), generator=g, dtype=torch.float64) / 8 ** 0.5
    return q, k, v, P


def _worker(rank, world, port, out_path):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    q, k, v, P = _inputs()
    lo, hi = bench.shard_range(q.shape[0], world, rank)
    part = oracle.attention(q[lo:hi], k[lo:hi], v[lo:hi], P, causal=True)
    shares = [None] * world
    dist.all_gather_object(shares, (lo, hi, part))
    t_max = bench.max_over_ranks(1.0 + rank, dist)
    if rank == 0:
        full = np.concatenate([s[2] for s in sorted(shares, key=lambda s: s[0])], axis=0)
        np.save(out_path, full)
        with open(out_path + ".tmax", "w") as f:
            f.write(repr(t_max))
    dist.barrier()
    dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_reproduce_the_single_process_result(tmp_path):
    out = str(tmp_path / "full.npy")
    mp.start_processes(_worker, args=(2, _free_port(), out), nprocs=2, start_method="spawn")
    import oracle
    q, k, v, P = _inputs()
    ref = oracle.attention(q, k, v, P, causal=True)
    assert np.array_equal(np.load(out), ref)
    assert float(open(out + ".tmax").read()) == 2.0   # max over ranks of 1 + rank
