"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Each case draws seeded inputs once (spa_inputs), runs spa_attention_fwd on the
GPU and the oracle on the CPU, and compares element by element:
  fp32 inputs: max |err| <= 1e-5;  bf16 inputs: rel-Frobenius <= 1e-2 and
  max |err| <= 2e-2.
Small shapes are compared in full (several 128-row tiles and a ragged tail);
the full-size workloads are compared on sampled rows (row 0, N-1, tile
boundaries +-1 and random rows), which the oracle computes one by one.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import spa_inputs as si
from helpers import assert_parity, errors, sample_rows, spa

pytestmark = pytest.mark.gpu


def run_gpu(q, k, v, P, causal):
    pkg = spa()
    dev = torch.device("cuda:0")
    out = pkg.spa_attention_fwd(q.to(dev), k.to(dev), v.to(dev), P.to(dev), causal=causal)
    torch.cuda.synchronize()
    assert pkg.device_error() == 0
    return out.cpu().numpy()


def check(w, rows=None, seed=None):
    q, k, v = si.make_qkv(w, seed=seed)
    P = si.make_P(w)
    got = run_gpu(q, k, v, P, w.causal)
    if rows is None:
        ref = oracle.attention(q, k, v, P, causal=w.causal)
    else:
        ref = oracle.attention(q, k, v, P, causal=w.causal, rows=rows)
        got = got[:, :, rows]
    return assert_parity(got, ref, w.dtype, w.name)


# ------------------------------------------------------------ named workloads
def test_c1_fp32_full():
    check(si.WORKLOADS["C1"])


def test_c2_bf16_full():
    check(si.WORKLOADS["C2"])


def test_c3_bf16_causal_sampled():
    w = si.WORKLOADS["C3"]
    check(w, rows=sample_rows(w.N, 96, seed=3))


@pytest.mark.parametrize("m", [16, 32, 64])
def test_c4_bf16_sweep_sampled(m):
    w = si.WORKLOADS["C4"].with_m(m)
    check(w, rows=sample_rows(w.N, 48, seed=4))


def test_c5_bf16_causal_and_control_sampled():
    w = si.WORKLOADS["C5"]
    rows = sample_rows(w.N, 24, seed=5)
    q, k, v = si.make_qkv(w)
    for wc in (w, si.WORKLOADS["C5ctl"]):
        P = si.make_P(wc)
        got = run_gpu(q, k, v, P, True)[:, :, rows]
        ref = oracle.attention(q, k, v, P, causal=True, rows=rows)
        assert_parity(got, ref, "bf16", wc.name)


# ------------------------------------------------------------ shapes and tails
SMALL = [
    # (B, H, N, d, m, dv, causal)
    (1, 1, 1, 64, 32, 64, False),
    (1, 1, 2, 64, 32, 64, True),
    (1, 2, 127, 128, 32, 128, False),
    (1, 2, 128, 128, 32, 128, True),
    (2, 1, 129, 64, 16, 64, True),
    (1, 3, 1000, 128, 64, 128, True),
    (1, 2, 1000, 96, 128, 64, False),
    (2, 2, 384, 64, 16, 128, False),
    (1, 1, 777, 128, 128, 128, True),
    (1, 1, 300, 256, 32, 64, False),
    (1, 2, 200, 60, 32, 64, True),     # d not a multiple of 8: SIMT projection
    (1, 1, 333, 72, 16, 128, False),   # ragged 64-column box in the TMA projection
    # an odd number of 128-row tiles leaves the last CTA with one query tile,
    # with two- (m=128) and three-stage (m<128) key/value rings
    (2, 2, 777, 64, 128, 64, False),
    (1, 1, 1281, 128, 32, 128, False),
    (1, 2, 1281, 128, 64, 128, True),
    # more work items than SMs: each persistent CTA walks several query-tile
    # pairs of different heads, among them pairs without a second tile (odd
    # tile count), and projection ranges that cross heads and the q/k boundary
    (3, 60, 300, 64, 32, 64, True),
    (2, 90, 300, 128, 64, 128, False),
    (2, 80, 260, 64, 16, 64, True),
    # the warp-specialised projection (m != 32) with several tiles per CTA:
    # ranges that cross heads and the q/k boundary, the X-tile ring and the
    # four TMEM accumulators wrapping around
    (2, 10, 1000, 128, 64, 128, True),
    (3, 10, 2000, 64, 16, 64, False),
    (1, 12, 1000, 128, 128, 128, False),
    # ... and ranges of five or six tiles over three-tile heads, so that a CTA
    # stages P_h for three heads (the most that kernel takes)
    (1, 103, 300, 128, 64, 128, True),
    (1, 97, 500, 64, 16, 64, False),
    # its other (m, d) instantiations: one, three and four 64-column boxes of
    # X per tile (the last with two ring slots at m = 64)
    (2, 3, 500, 64, 64, 64, True),
    (1, 2, 300, 192, 16, 128, False),
    (1, 2, 300, 256, 64, 64, True),
    (1, 2, 300, 256, 16, 64, False),
]


@pytest.mark.parametrize("shape", SMALL)
def test_bf16_small_shapes_full(shape):
    B, H, N, d, m, dv, causal = shape
    w = si.WORKLOADS["C3"].scaled(B=B, H=H, N=N, d=d, m=m, dv=dv, causal=causal, qk="norm")
    check(w, seed=17 + N)


@pytest.mark.parametrize("shape", [(1, 1, 256, 64, 16, 64, False), (2, 3, 77, 7, 5, 33, True),
                                   (1, 2, 300, 128, 128, 256, False), (1, 1, 1, 3, 1, 1, True)])
def test_fp32_shapes_full(shape):
    B, H, N, d, m, dv, causal = shape
    w = si.WORKLOADS["C1"].scaled(B=B, H=H, N=N, d=d, m=m, dv=dv, causal=causal)
    check(w, seed=29 + N)


@pytest.mark.parametrize("scale_exp", [24, -24])
@pytest.mark.parametrize("m", [16, 32])
def test_bf16_extreme_input_ranges(scale_exp, m):
    """q scaled by 2^e and k by 2^-e (both exact in bf16) leaves every logit
    unchanged but pushes the projected operands far past fp16's largest value
    and below its smallest subnormal: the range exponents must absorb both."""
    w = si.WORKLOADS["C2"].scaled(B=1, H=2, N=300, m=m)
    q, k, v = si.make_qkv(w, seed=91)
    s = 2.0 ** scale_exp
    q = (q.double() * s).to(torch.bfloat16)
    k = (k.double() / s).to(torch.bfloat16)
    P = si.make_P(w)
    got = run_gpu(q, k, v, P, False)
    ref = oracle.attention(q, k, v, P)
    assert_parity(got, ref, "bf16", f"scale 2^{scale_exp}")


def test_projection_matches_oracle():
    """spa_project: fp32 sums of exact products, |err| <= 1e-5 * sum_l |x_l P_lk|."""
    pkg = spa()
    for dtype in (torch.bfloat16, torch.float32):
        w = si.WORKLOADS["C3"].scaled(B=2, H=3, N=300, d=128, m=32)
        w = w.scaled(dtype="bf16" if dtype == torch.bfloat16 else "f32")
        x, _, _ = si.make_qkv(w, seed=5)
        P = si.make_P(w)
        got = pkg.spa_project(x.cuda(), P.cuda()).cpu().numpy()
        ref = oracle.project(x, P)
        bound = 1e-5 * np.einsum("bhnl,hlk->bhnk", np.abs(x.double().numpy()),
                                 np.abs(P.double().numpy()))
        assert np.all(np.abs(got - ref) <= bound)


def test_workspace_and_host_forms_agree_bitwise():
    pkg = spa()
    w = si.WORKLOADS["C2"].scaled(B=2, H=2, N=700)
    q, k, v = si.make_qkv(w)
    P = si.make_P(w)
    dq, dk, dv_, dP = (t.cuda() for t in (q, k, v, P))
    a = pkg.spa_attention_fwd(dq, dk, dv_, dP, causal=True)
    n = pkg.spa_attention_workspace_size(2, 2, 700, 64, 32, 64, pkg.SPA_BF16)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    b = pkg.spa_attention_fwd_ws(dq, dk, dv_, dP, ws, causal=True)
    c = pkg.spa_attention_fwd_host(q.pin_memory(), k.pin_memory(), v.pin_memory(),
                                   P.pin_memory(), causal=True)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert torch.equal(a.cpu(), c)
    # repeated calls are deterministic
    assert torch.equal(a, pkg.spa_attention_fwd(dq, dk, dv_, dP, causal=True))


@pytest.mark.parametrize("B,H,causal", [(2, 8, True), (1, 7, False)])
def test_host_form_chunked_matches_device_bitwise(B, H, causal):
    """Large enough that the host form copies and computes in chunks of heads
    (several chunks per stream slot, a short last chunk when H does not
    divide): every head is computed alone, so the result is bit for bit the
    device form's."""
    pkg = spa()
    w = si.WORKLOADS["C2"].scaled(B=B, H=H, N=16384, causal=causal)
    g = torch.Generator().manual_seed(11)
    q = torch.randn((B, H, w.N, w.d), generator=g).to(torch.bfloat16)
    k = torch.randn((B, H, w.N, w.d), generator=g).to(torch.bfloat16)
    v = torch.randn((B, H, w.N, w.dv), generator=g).to(torch.bfloat16)
    P = (torch.randn((H, w.d, w.m), generator=g) / w.m ** 0.5).to(torch.bfloat16)
    a = pkg.spa_attention_fwd(q.cuda(), k.cuda(), v.cuda(), P.cuda(), causal=causal).cpu()
    c = pkg.spa_attention_fwd_host(q.pin_memory(), k.pin_memory(), v.pin_memory(),
                                   P.pin_memory(), causal=causal)
    assert torch.equal(a, c)


def test_rows_sum_to_one_through_constant_values():
    """V = 1 gives O = 1 exactly up to the bf16 rounding of the probabilities."""
    w = si.WORKLOADS["C3"].scaled(B=1, H=2, N=513, causal=True)
    q, k, _ = si.make_qkv(w)
    v = torch.ones((1, 2, 513, 128), dtype=torch.bfloat16)
    got = run_gpu(q, k, v, si.make_P(w), True)
    assert np.abs(got - 1.0).max() < 2e-2
    max_abs, _ = errors(got, np.ones_like(got))
    assert max_abs < 2e-2


@pytest.mark.parametrize("m", [16, 32])
def test_bf16_large_values_scale_exactly(m):
    """The softmax accumulates probabilities up to 2^40 times the running max
    between rescales; the header promises finite results for |v| below
    2^(87 - log2 N).  Values scaled by 2^60 (exact in bf16, N = 1000 allows
    up to about 2^77) must give the output scaled by exactly 2^60: every
    product and sum of the value path scales by the power of two, so the
    bits match unless something overflowed."""
    pkg = spa()
    w = si.WORKLOADS["C2"].scaled(B=1, H=2, N=1000, m=m, causal=True)
    q, k, v = si.make_qkv(w, seed=73)
    P = si.make_P(w)
    dev = torch.device("cuda:0")
    s = 2.0 ** 60
    big = (v.double() * s).to(torch.bfloat16)
    assert torch.equal(big.double() / s, v.double())
    a = pkg.spa_attention_fwd(q.to(dev), k.to(dev), v.to(dev), P.to(dev), causal=True)
    b = pkg.spa_attention_fwd(q.to(dev), k.to(dev), big.to(dev), P.to(dev), causal=True)
    torch.cuda.synchronize()
    assert pkg.device_error() == 0
    assert torch.isfinite(b).all()
    assert torch.equal(b, a * s)
