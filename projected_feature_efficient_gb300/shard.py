"""Partition of one forward problem across ranks (one process per GPU).

Every (batch b, head h) pair of projected-feature attention is independent:
its output rows depend on q[b, h], k[b, h], v[b, h] and P_h only ("Sparse
Projection Attention", Sec. 3.1.2-3.1.3: the projection and the softmax act
per head).  So N ranks split the B*H pairs of one problem into contiguous
shares and each computes its share with no data-path collective; the shares
put side by side are the whole output.

This module only selects and reorders data (slices, gathers, concatenation);
it does no arithmetic of the method.
"""
from __future__ import annotations


def shard_range(total: int, world: int, rank: int):
    """Contiguous share [lo, hi) of `total` independent units owned by `rank`;
    the shares of ranks 0 .. world-1 tile [0, total) in order and differ in
    size by at most one."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside a world of {world}")
    base, extra = divmod(total, world)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


def shard_pairs(q, k, v, P, world: int, rank: int):
    """This rank's share of the problem (q, k [B,H,N,d], v [B,H,N,d_v],
    P [H,d,m]) as a problem of its own with B = 1 and H = hi - lo: pair
    j = b*H + h of [lo, hi) becomes head j - lo, with its own copy of P_h.

    Returns (lo, hi, q_r, k_r, v_r, P_r), each tensor contiguous."""
    import torch

    B, H = q.shape[0], q.shape[1]
    lo, hi = shard_range(B * H, world, rank)

    def rows(t):
        return t.reshape(B * H, *t.shape[2:])[lo:hi].unsqueeze(0).contiguous()

    heads = torch.arange(lo, hi, dtype=torch.long, device=P.device) % H
    return lo, hi, rows(q), rows(k), rows(v), P.index_select(0, heads).contiguous()


def gather_pairs(shares, B: int, H: int):
    """Inverse of shard_pairs for the outputs: `shares` is a list of
    (lo, hi, out_r) with out_r [1, hi-lo, N, d_v] (torch tensors or numpy
    arrays); returns the whole [B, H, N, d_v] output."""
    shares = sorted(shares, key=lambda s: s[0])
    if not shares or shares[0][0] != 0 or shares[-1][1] != B * H or \
            any(a[1] != b[0] for a, b in zip(shares, shares[1:])):
        raise ValueError("the shares do not tile the (batch, head) pairs")
    parts = [s[2].reshape(s[1] - s[0], *s[2].shape[2:]) for s in shares if s[1] > s[0]]
    import numpy as np
    if isinstance(parts[0], np.ndarray):
        whole = np.concatenate(parts, axis=0)
    else:
        import torch
        whole = torch.cat(parts, dim=0)
    return whole.reshape(B, H, *whole.shape[1:])


def spa_attention_fwd_shard(q, k, v, P, world: int, rank: int, causal: bool = False,
                            out=None, stream=None):
    """The forward of this rank's share through spa_attention_fwd: returns
    (lo, hi, out_r) with out_r [1, hi-lo, N, d_v] fp32 on q's device."""
    from . import _binding

    lo, hi, q_r, k_r, v_r, P_r = shard_pairs(q, k, v, P, world, rank)
    if hi == lo:
        return lo, hi, None
    return lo, hi, _binding.spa_attention_fwd(q_r, k_r, v_r, P_r, causal=causal, out=out,
                                              stream=stream)
