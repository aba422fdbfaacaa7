"""Gradients on the GPU against the oracle's (pinned) gradients, through
spa_attention_bwd (the forward run once more for its log-sum-exp).

Tolerance, from the arithmetic: bf16 shapes of the tensor-core backward round
the probabilities and dS once to bf16 for their products (fp32 accumulation),
a few 2^-9 roundings per term: rel-F 1e-2.  fp32 inputs (and the other
shapes) take the CUDA-core backward, fp32 arithmetic throughout, whose
rounding errors grow with the sums' lengths (N, m, d_v of a few hundred):
rel-F 1e-4.  max |err| is bounded relative to the tensor's largest entry."""
import numpy as np
import pytest
import torch

import oracle
import spa_inputs as si
from helpers import spa

pytestmark = pytest.mark.gpu

TOL = {"bf16": 1e-2, "f32": 1e-4}


def rel_errors(got, ref):
    got = np.asarray(got, dtype=np.float64)
    diff = got - ref
    den = np.sqrt((ref * ref).sum())
    scale = np.abs(ref).max()
    rel_f = np.sqrt((diff * diff).sum()) / den if den > 0 else np.sqrt((diff * diff).sum())
    rel_max = np.abs(diff).max() / scale if scale > 0 else np.abs(diff).max()
    return rel_f, rel_max


SHAPES = [
    # (B, H, N, d, m, dv, causal, dtype)
    (1, 2, 100, 64, 32, 64, False, "bf16"),
    (2, 2, 257, 128, 32, 128, True, "bf16"),
    (1, 2, 300, 128, 16, 128, True, "bf16"),
    (1, 3, 300, 64, 64, 64, True, "f32"),
    (2, 1, 129, 96, 16, 32, False, "f32"),
]


@pytest.mark.parametrize("shape", SHAPES)
def test_gradients_match_oracle(shape):
    pkg = spa()
    B, H, N, d, m, dv, causal, dt = shape
    w = si.WORKLOADS["C3"].scaled(B=B, H=H, N=N, d=d, m=m, dv=dv, causal=causal, dtype=dt)
    q, k, v = si.make_qkv(w, seed=60 + N)
    P = si.make_P(w, seed=70 + m)
    g = torch.Generator().manual_seed(80 + N)
    dO = torch.randn((B, H, N, dv), generator=g, dtype=torch.float64).to(w.torch_dtype)
    q_, k_, v_, P_, dO_ = (t.cuda() for t in (q, k, v, P, dO))
    out = pkg.spa_attention_fwd(q_, k_, v_, P_, causal=causal)
    got = pkg.spa_attention_bwd(q_, k_, v_, P_, out, dO_, causal=causal)
    ref = oracle.attention_bwd(q, k, v, P, dO, causal=causal)
    for name, gg, rr in zip(("dq", "dk", "dv", "dP"), got, ref):
        rel_f, rel_max = rel_errors(gg.cpu().numpy(), rr)
        assert rel_f <= TOL[dt] and rel_max <= 2 * TOL[dt], f"{name} {shape}: rel-F {rel_f:.2e}, rel-max {rel_max:.2e}"


def test_single_key_has_no_score_gradient():
    """N = 1: the softmax is constant, so dq = dk = dP = 0 and dv = dO."""
    pkg = spa()
    w = si.WORKLOADS["C3"].scaled(B=1, H=2, N=1, d=64, m=16, dv=64, causal=True)
    q, k, v = (t.cuda() for t in si.make_qkv(w, seed=1))
    P = si.make_P(w, seed=2).cuda()
    dO = torch.randn((1, 2, 1, 64), dtype=torch.float32).to(torch.bfloat16).cuda()
    out = pkg.spa_attention_fwd(q, k, v, P, causal=True)
    dq, dk, dv, dP = pkg.spa_attention_bwd(q, k, v, P, out, dO, causal=True)
    for t_ in (dq, dk, dP):
        assert float(t_.abs().max()) < 1e-3 * float(dO.float().abs().max()) + 1e-6
    assert torch.allclose(dv, dO.float(), rtol=0, atol=1e-6)
