"""Sparse Feature Attention on the GPU: the Top-k prologue is bit-exact
against the oracle's Top-k (ties included), and the forward on the sparsified
rows matches the oracle's attention of Topk(q), Topk(k) with P = I."""
import numpy as np
import pytest
import torch

import oracle
import spa_inputs as si
from helpers import assert_parity, spa

pytestmark = pytest.mark.gpu


def rows_with_ties(n, d, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((n, d), generator=g, dtype=torch.float64)
    # a third of the rows from a tiny value set: many ties at the k-th magnitude
    few = torch.tensor([-2.0, -1.0, -0.0, 0.0, 1.0, 2.0], dtype=torch.float64)
    idx = torch.randint(0, len(few), (n // 3, d), generator=g)
    x[: n // 3] = few[idx]
    return x.to(dtype)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("d", [32, 64, 128, 256])
def test_topk_is_bit_exact(dtype, d):
    pkg = spa()
    x = rows_with_ties(300, d, dtype, seed=d)
    for k in sorted({1, 7, 16, d - 1, d} - {0}):
        got = pkg.spa_topk_features(x.cuda(), k).cpu()
        want = torch.from_numpy(oracle.topk_features(x, k)).to(dtype)
        # compare bit patterns (signed zeros included)
        view = torch.int16 if dtype == torch.bfloat16 else torch.int32
        assert torch.equal(got.view(view), want.view(view)), f"d={d} k={k}"


def test_topk_full_size_sampled():
    """The Top-k of q at the SFA measurement's size (B=1 H=32 N=32768 d=128,
    k=16: 2^20 rows, the launch the bench times), a third of the rows from a
    tiny value set; sampled rows, the first and the last, bit for bit."""
    pkg = spa()
    rows, d, k = 1 << 20, 128, 16
    x = rows_with_ties(rows, d, torch.bfloat16, seed=7)
    got = pkg.spa_topk_features(x.cuda(), k).cpu()
    g = torch.Generator().manual_seed(8)
    idx = torch.cat([torch.tensor([0, rows // 3 - 1, rows // 3, rows - 1]),
                     torch.randint(0, rows, (3000,), generator=g)])
    want = torch.from_numpy(oracle.topk_features(x[idx], k)).to(torch.bfloat16)
    assert torch.equal(got[idx].view(torch.int16), want.view(torch.int16))


@pytest.mark.parametrize("d", [64, 128])
def test_topk_in_place_matches(d):
    """Writing the sparsified rows over the input gives the same bits as a
    separate output (each block of rows is read before it is written)."""
    pkg = spa()
    x = rows_with_ties(70_000, d, torch.bfloat16, seed=3 + d).cuda()
    want = pkg.spa_topk_features(x, 9)
    y = x.clone()
    got = pkg.spa_topk_features(y, 9, out=y)
    assert got.data_ptr() == y.data_ptr()
    assert torch.equal(y.view(torch.int16), want.view(torch.int16))


@pytest.mark.parametrize("shape", [
    # (B, H, N, d, dv, topk, causal)
    (1, 2, 300, 128, 128, 16, False),
    (1, 2, 300, 128, 128, 16, True),
    (2, 2, 129, 64, 64, 8, True),
    (1, 3, 257, 32, 64, 4, False),
])
def test_sfa_forward_matches_oracle(shape):
    pkg = spa()
    B, H, N, d, dv, topk, causal = shape
    w = si.WORKLOADS["C3"].scaled(B=B, H=H, N=N, d=d, m=d, dv=dv, causal=causal)
    q, k, v = si.make_qkv(w, seed=50 + N)
    got = pkg.spa_sfa_attention_fwd(q.cuda(), k.cuda(), v.cuda(), topk, causal=causal).cpu()
    qs = torch.from_numpy(oracle.topk_features(q, topk)).to(torch.bfloat16)
    ks = torch.from_numpy(oracle.topk_features(k, topk)).to(torch.bfloat16)
    eye = torch.eye(d, dtype=torch.bfloat16).expand(H, d, d).contiguous()
    ref = oracle.attention(qs, ks, v, eye, causal=causal)
    assert_parity(got.numpy(), ref, "bf16", f"SFA {shape}")
