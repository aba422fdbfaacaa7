"""The multi-GPU host logic on CPU with two gloo ranks.

Every (batch, head) pair is independent, so N ranks split the B*H pairs of one
problem with no data-path collective (shard.shard_pairs, the helper bench.py
and spa_attention_fwd_shard use); only the timing max-reduction talks between
ranks.  Here two processes each take their share of a small problem whose
pairs do not divide evenly, run the fp64 oracle on it, and the gathered shares
must equal the single-process result.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from projected_feature_efficient_gb300.shard import gather_pairs, shard_pairs, shard_range


def test_shard_range_partitions_exactly():
    for total in (0, 1, 5, 8, 33):
        for world in (1, 2, 3, 8):
            spans = [shard_range(total, world, r) for r in range(world)]
            assert spans == [bench.shard_range(total, world, r) for r in range(world)]
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
    lo, hi, q_r, k_r, v_r, P_r = shard_pairs(q, k, v, P, world, rank)
    part = oracle.attention(q_r, k_r, v_r, P_r, causal=True)
    shares = [None] * world
    dist.all_gather_object(shares, (lo, hi, part))
    t_max = bench.max_over_ranks(1.0 + rank, dist)
    if rank == 0:
        full = gather_pairs(shares, q.shape[0], q.shape[1])
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


def test_shard_pairs_keeps_each_pairs_projection():
    q, k, v, P = _inputs()
    B, H = q.shape[:2]
    for world in (1, 3, 4):
        got = []
        for r in range(world):
            lo, hi, q_r, k_r, v_r, P_r = shard_pairs(q, k, v, P, world, r)
            assert q_r.shape == (1, hi - lo) + tuple(q.shape[2:])
            for j in range(hi - lo):
                b, h = divmod(lo + j, H)
                assert torch.equal(q_r[0, j], q[b, h]) and torch.equal(v_r[0, j], v[b, h])
                assert torch.equal(P_r[j], P[h])
            got.append((lo, hi, v_r))
        assert torch.equal(gather_pairs(got, B, H), v)
    with pytest.raises(ValueError):
        gather_pairs([(0, 3, v.reshape(1, B * H, *v.shape[2:])[:, :3])], B, H)
