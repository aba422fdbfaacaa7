"""Pins of the oracle's gradients (CPU only).  They do not re-derive the
oracle's formulas: central finite differences of the oracle's own forward,
automatic differentiation of a plain fp64 restatement of the forward, and
exact sum rules of softmax attention.  tests/test_oracle_mutants.py checks
that these pins catch plausible mistakes in the gradient code."""
import math

import numpy as np
import pytest
import torch

import oracle


def _inputs(B=2, H=2, N=5, d=4, m=3, dv=3, seed=0):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((B, H, N, d), generator=g, dtype=torch.float64)
    k = torch.randn((B, H, N, d), generator=g, dtype=torch.float64)
    v = torch.randn((B, H, N, dv), generator=g, dtype=torch.float64)
    P = torch.randn((H, d, m), generator=g, dtype=torch.float64) / math.sqrt(m)
    dO = torch.randn((B, H, N, dv), generator=g, dtype=torch.float64)
    return q, k, v, P, dO


def finite_difference_pins(lib=None, causal=False, h=1e-5, tol=1e-7) -> bool:
    """Every gradient element against the central difference of
    L = sum(dO * O) computed with the oracle's forward."""
    q, k, v, P, dO = _inputs()
    grads = oracle.attention_bwd(q, k, v, P, dO, causal=causal, _lib=lib)
    w = dO.numpy()

    def loss(q_, k_, v_, P_):
        return float((oracle.attention(q_, k_, v_, P_, causal=causal, _lib=lib) * w).sum())

    tensors = [q, k, v, P]
    for which, g in enumerate(grads):
        t = tensors[which]
        flat = t.view(-1)
        gflat = g.reshape(-1)
        for idx in range(flat.numel()):
            old = float(flat[idx])
            flat[idx] = old + h
            lp = loss(*tensors)
            flat[idx] = old - h
            lm = loss(*tensors)
            flat[idx] = old
            if abs((lp - lm) / (2 * h) - gflat[idx]) > tol:
                return False
    return True


def torch_reference(q, k, v, P, dO, causal):
    """Autograd of a plain restatement of the forward (independent code path)."""
    q, k, v, P = (t.clone().requires_grad_(True) for t in (q, k, v, P))
    m = P.shape[-1]
    qp = torch.einsum("bhnl,hlk->bhnk", q, P)
    kp = torch.einsum("bhnl,hlk->bhnk", k, P)
    s = qp @ kp.transpose(-1, -2) / math.sqrt(m)
    if causal:
        N = s.shape[-1]
        s = s.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), float("-inf"))
    o = torch.softmax(s, dim=-1) @ v
    o.backward(dO)
    return q.grad, k.grad, v.grad, P.grad


@pytest.mark.parametrize("causal", [False, True])
def test_gradients_match_finite_differences(causal):
    assert finite_difference_pins(causal=causal)


@pytest.mark.parametrize("causal", [False, True])
def test_gradients_match_autograd_of_the_forward(causal):
    q, k, v, P, dO = _inputs(B=2, H=3, N=40, d=8, m=4, dv=5, seed=3)
    got = oracle.attention_bwd(q, k, v, P, dO, causal=causal)
    ref = torch_reference(q, k, v, P, dO, causal)
    for g, r in zip(got, ref):
        np.testing.assert_allclose(g, r.numpy(), rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_sum_rules(causal):
    """sum over keys of dK is 0 (each softmax row's gradient sums to 0), and
    sum over keys of dV equals sum over queries of dO (each row sums to 1)."""
    q, k, v, P, dO = _inputs(B=1, H=2, N=30, d=6, m=4, dv=5, seed=7)
    dq, dk, dv, dP = oracle.attention_bwd(q, k, v, P, dO, causal=causal)
    assert np.abs(dk.sum(axis=2)).max() < 1e-12 * (1 + np.abs(dk).max())
    np.testing.assert_allclose(dv.sum(axis=2), dO.numpy().sum(axis=2), rtol=1e-12, atol=1e-12)


def test_equal_value_rows_give_no_score_gradient():
    """If every value row is the same, the output does not depend on the scores:
    dQ, dK and dP vanish, and dV_j = sum_i A_ij dO_i still sums to sum dO."""
    q, k, v, P, dO = _inputs(B=1, H=2, N=12, d=5, m=3, dv=4, seed=9)
    v = v[:, :, :1].expand_as(v).contiguous()
    dq, dk, dv, dP = oracle.attention_bwd(q, k, v, P, dO, causal=True)
    for g in (dq, dk, dP):
        assert np.abs(g).max() < 1e-13
    np.testing.assert_allclose(dv.sum(axis=2), dO.numpy().sum(axis=2), rtol=1e-12, atol=1e-12)


def test_bf16_inputs_are_read_exactly():
    q, k, v, P, dO = _inputs(B=1, H=1, N=9, d=4, m=3, dv=3, seed=11)
    qb, kb, vb, Pb, dOb = (t.to(torch.bfloat16) for t in (q, k, v, P, dO))
    got = oracle.attention_bwd(qb, kb, vb, Pb, dOb, causal=True)
    ref = oracle.attention_bwd(*(t.double() for t in (qb, kb, vb, Pb, dOb)), causal=True)
    for g, r in zip(got, ref):
        np.testing.assert_array_equal(g, r)
