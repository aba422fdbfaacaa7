"""Decode with the projected key cache against the oracle: one query per
(batch, head) attending to every cached key is the last row of the causal
forward over the same keys, so the fp64 oracle's causal attention at row L-1
is the reference."""
import numpy as np
import pytest
import torch

import oracle
import spa_inputs as si
from helpers import assert_parity, spa

pytestmark = pytest.mark.gpu


def build_cache(pkg, k, P, v, cap, pieces=None):
    B, H, L, _ = k.shape
    m, dv = P.shape[2], v.shape[3]
    kc, kmul = pkg.kcache_new(B, H, cap, m)
    vc = torch.zeros((B, H, cap, dv), dtype=v.dtype, device="cuda")
    vc[:, :, :L] = v.cuda()
    bounds = [0] + list(pieces or []) + [L]
    for a, b in zip(bounds[:-1], bounds[1:]):
        pkg.spa_kcache_append(k[:, :, a:b].contiguous().cuda(), P.cuda(), kc, kmul, a)
    return kc, kmul, vc


SHAPES = [
    # (B, H, L, d, m, dv)
    (1, 1, 1, 64, 32, 64),        # one key: the output is that key's value row
    (2, 3, 100, 64, 16, 64),
    (1, 2, 1000, 128, 32, 128),
    (2, 2, 777, 128, 64, 128),
    (1, 1, 5000, 128, 128, 128),
    (3, 2, 9000, 64, 32, 64),     # more keys than one chunk holds: several chunks, ragged last
    (2, 8, 20000, 128, 32, 128),
]


@pytest.mark.parametrize("shape", SHAPES)
def test_decode_matches_oracle(shape):
    pkg = spa()
    B, H, L, d, m, dv = shape
    w = si.WORKLOADS["C3"].scaled(B=B, H=H, N=L, d=d, m=m, dv=dv, causal=True)
    q, k, v = si.make_qkv(w, seed=31 + L)
    P = si.make_P(w, seed=41 + m)
    cap = L + 9
    kc, kmul, vc = build_cache(pkg, k, P, v, cap)
    got = pkg.spa_attention_decode(q[:, :, L - 1].contiguous().cuda(), P.cuda(), kc, kmul, vc, L)
    ref = oracle.attention(q, k, v, P, causal=True, rows=[L - 1])[:, :, 0]
    assert_parity(got.cpu().numpy(), ref, "bf16", f"decode {shape}")
    if L == 1:  # softmax of one score is 1
        assert np.allclose(got.cpu().numpy(), v[:, :, 0].double().numpy(), rtol=0, atol=1e-6)


@pytest.mark.parametrize("m", [32, 64])
def test_append_in_pieces_is_bitwise_one_append(m):
    """Appending at any row offset writes the same bits as one append (m = 64
    goes through the warp-specialised projection kernel, m = 32 through the
    per-CTA one)."""
    pkg = spa()
    w = si.WORKLOADS["C3"].scaled(B=2, H=2, N=1500, d=128, m=m, dv=128)
    q, k, v = si.make_qkv(w, seed=5)
    P = si.make_P(w, seed=6)
    a = build_cache(pkg, k, P, v, 1600)
    b = build_cache(pkg, k, P, v, 1600, pieces=[300, 301, 1024])
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_cache_rows_follow_the_projection():
    """Every cached row times its multiplier is K P_h within fp16 rounding of
    the row max (the multiplier puts the row max in [2^13, 2^14))."""
    pkg = spa()
    w = si.WORKLOADS["C3"].scaled(B=1, H=3, N=257, d=64, m=64, dv=64)
    _, k, v = si.make_qkv(w, seed=9)
    P = si.make_P(w, seed=10)
    kc, kmul, _ = build_cache(pkg, k, P, v, 257)
    rows = kc.cpu().view(torch.float16).double() * kmul.cpu().double()[..., None]
    exact = torch.einsum("bhnl,hlk->bhnk", k.double(), P.double())
    amax = exact.abs().amax(dim=-1, keepdim=True)
    assert torch.all((rows - exact).abs() <= amax * 2.0 ** -10 + 1e-30)
    scaled_max = (kc.cpu().view(torch.float16).double().abs().amax(dim=-1))
    # fp16 rounding may carry a maximum just below 2^14 up to 2^14
    assert torch.all((scaled_max >= 2.0 ** 13) & (scaled_max <= 2.0 ** 14))
