"""SPA's sparse random projection (Definition 1): the input recipe draws the
stated distribution, and the forward with such a P matches the oracle (the
dense projection kernels take a sparse P as it is; its cost is that of any P,
since the projection reads X in full either way)."""
import math

import numpy as np
import pytest
import torch

import oracle
import spa_inputs as si
from helpers import assert_parity, spa


@pytest.mark.parametrize("s", [1.0, 3.0, math.sqrt(128)])
def test_entries_follow_definition_1(s):
    w = si.WORKLOADS["C4"].scaled(H=16, d=128, m=64, dtype="f32")
    P = si.make_sparse_P(w, s, seed=1).double().numpy()
    scale = math.sqrt(s / w.m)
    vals = np.unique(np.round(P / scale, 6))
    assert set(vals) <= {-1.0, 0.0, 1.0}
    n = P.size
    for target, frac in ((1.0, 0.5 / s), (-1.0, 0.5 / s), (0.0, 1.0 - 1.0 / s)):
        got = np.mean(np.isclose(P / scale, target))
        assert abs(got - frac) <= 5 * math.sqrt(frac * (1 - frac) / n) + 1e-12
    # E[S_ij^2] = 1/m, so E ||u S||^2 = ||u||^2 (the JL normalisation)
    assert abs(np.mean(P * P) * w.m - 1.0) < 0.05


def test_inner_products_are_preserved_on_average():
    """Over many independent draws, <uS, vS> averages to <u, v> (the sparse
    JL property of the pages, Proposition 1, at the level of the mean)."""
    rng = np.random.default_rng(3)
    u, v = rng.standard_normal(128), rng.standard_normal(128)
    w = si.WORKLOADS["C4"].scaled(H=4000, d=128, m=32, dtype="f32")
    S = si.make_sparse_P(w, 3.0, seed=7).double().numpy()     # 4000 draws of a 128 x 32 matrix
    ips = np.einsum("l,hlk,j,hjk->h", u, S, v, S)
    assert abs(ips.mean() - u @ v) < 5 * ips.std() / math.sqrt(len(ips))


@pytest.mark.gpu
@pytest.mark.parametrize("s,causal", [(1.0, False), (3.0, True), (math.sqrt(128), False)])
def test_forward_with_sparse_projection_matches_oracle(s, causal):
    pkg = spa()
    w = si.WORKLOADS["C3"].scaled(B=1, H=2, N=700, d=128, m=32, dv=128, causal=causal)
    q, k, v = si.make_qkv(w, seed=91)
    P = si.make_sparse_P(w, s, seed=92)
    got = pkg.spa_attention_fwd(q.cuda(), k.cuda(), v.cuda(), P.cuda(), causal=causal).cpu()
    ref = oracle.attention(q, k, v, P, causal=causal)
    assert_parity(got.numpy(), ref, "bf16", f"sparse P s={s:.2f}")
