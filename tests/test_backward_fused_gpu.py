"""The fused tensor-core backward and the forward's log-sum-exp output, on the
GPU against the oracle.

Gradient tolerance, from the arithmetic of the fused path: the scores use the
forward's own operands (fp16 with range multipliers, or the split-bf16 sum at
m = 16), the probabilities and dS are rounded once to bf16 (relative 2^-9)
for their products, fp32 accumulation throughout, and dQp / dKp reach dq, dk,
dP as bf16 hi + lo pairs (16 significant bits).  A few 2^-9 roundings per
term stay well inside rel-F 1e-2, and max |err| inside 2e-2 of the tensor's
largest entry.

Log-sum-exp tolerance: lse_i - ref_i is the A-weighted mean of the score
errors; with score operands at fp16 precision that is below 1e-3 for these
inputs, so 5e-3 absolute (bf16); fp32 inputs 1e-5 relative to max(1, |lse|).
"""
import numpy as np
import pytest
import torch

import oracle
import spa_inputs as si
from helpers import spa

pytestmark = pytest.mark.gpu

REL_F = 1e-2


def rel_errors(got, ref):
    got = np.asarray(got, dtype=np.float64)
    diff = got - ref
    den = np.sqrt((ref * ref).sum())
    scale = np.abs(ref).max()
    rel_f = np.sqrt((diff * diff).sum()) / den if den > 0 else np.sqrt((diff * diff).sum())
    rel_max = np.abs(diff).max() / scale if scale > 0 else np.abs(diff).max()
    return rel_f, rel_max


def _problem(B, H, N, d, m, dv, causal, dt, seed):
    w = si.WORKLOADS["C3"].scaled(B=B, H=H, N=N, d=d, m=m, dv=dv, causal=causal, dtype=dt)
    q, k, v = si.make_qkv(w, seed=seed)
    P = si.make_P(w, seed=seed + 1)
    g = torch.Generator().manual_seed(seed + 2)
    dO = torch.randn((B, H, N, dv), generator=g, dtype=torch.float64).to(w.torch_dtype)
    return q, k, v, P, dO


LSE_SHAPES = [
    # (B, H, N, d, m, dv, causal, dtype)
    (1, 2, 300, 128, 32, 128, True, "bf16"),
    (2, 1, 200, 64, 16, 64, False, "bf16"),
    (1, 1, 129, 64, 64, 64, True, "bf16"),
    (1, 2, 77, 32, 16, 32, True, "f32"),
]


@pytest.mark.parametrize("shape", LSE_SHAPES)
def test_forward_lse_matches_oracle(shape):
    pkg = spa()
    B, H, N, d, m, dv, causal, dt = shape
    q, k, v, P, _ = _problem(*shape, seed=300 + N)
    out, lse = pkg.spa_attention_fwd_lse(q.cuda(), k.cuda(), v.cuda(), P.cuda(), causal=causal)
    ref_out, ref_lse = oracle.attention(q, k, v, P, causal=causal, return_lse=True)
    got = lse.cpu().numpy().astype(np.float64)
    if dt == "f32":
        assert np.abs(got - ref_lse).max() <= 1e-5 * max(1.0, np.abs(ref_lse).max())
    else:
        assert np.abs(got - ref_lse).max() <= 5e-3
    # the output is the plain forward's, bit for bit
    plain = pkg.spa_attention_fwd(q.cuda(), k.cuda(), v.cuda(), P.cuda(), causal=causal)
    assert torch.equal(out, plain)


FUSED_SHAPES = [
    # (B, H, N, d, m, dv, causal)
    (1, 2, 100, 64, 32, 64, False),     # one ragged tile
    (2, 2, 257, 128, 32, 128, True),    # three tiles, ragged, causal
    (1, 2, 300, 128, 16, 128, True),    # m = 16: split-bf16 scores
    (1, 3, 384, 64, 32, 128, False),    # whole tiles
    (2, 1, 129, 96, 16, 64, False),     # d = 96, d_v = 64: the CUDA-core backward
    (4, 16, 512, 64, 32, 64, True),     # 256 items: several per CTA
    (2, 40, 256, 64, 16, 128, False),   # 160 items, non-causal order
    # the projection gradients in one tensor-core pass
    (1, 3, 50, 128, 32, 128, True),     # one partial tile per (side, b, h)
    (3, 5, 700, 128, 32, 64, False),    # dP_h summed over three batch entries, ragged
    (2, 24, 1024, 128, 32, 128, True),  # 768 units: CTA ranges cross heads
    (2, 3, 333, 64, 16, 64, True),      # d = 64 (zero half of X^T), m = 16 (padded G rows)
    # m = 64: P^T over S^T in tensor memory at d_v = 128, single-buffered Qp
    # tiles, dQp in four 16-column slabs
    (1, 2, 300, 128, 64, 128, True),
    (2, 2, 257, 64, 64, 128, False),
    (1, 3, 200, 128, 64, 64, True),     # d_v = 64: P^T in columns of its own
    (1, 6, 1100, 128, 64, 128, True),   # several items per CTA, ragged
]


@pytest.mark.parametrize("shape", FUSED_SHAPES)
def test_fused_gradients_match_oracle(shape):
    pkg = spa()
    B, H, N, d, m, dv, causal = shape
    q, k, v, P, dO = _problem(B, H, N, d, m, dv, causal, "bf16", seed=400 + N + H)
    q_, k_, v_, P_, dO_ = (t.cuda() for t in (q, k, v, P, dO))
    out, lse = pkg.spa_attention_fwd_lse(q_, k_, v_, P_, causal=causal)
    got = pkg.spa_attention_bwd_lse(q_, k_, v_, P_, out, lse, dO_, causal=causal)
    ref = oracle.attention_bwd(q, k, v, P, dO, causal=causal)
    for name, gg, rr in zip(("dq", "dk", "dv", "dP"), got, ref):
        g_ = gg.cpu().numpy()
        assert np.all(np.isfinite(g_)), f"{name}: non-finite"
        rel_f, rel_max = rel_errors(g_, rr)
        assert rel_f <= REL_F and rel_max <= 2 * REL_F, \
            f"{name} {shape}: rel-F {rel_f:.2e}, rel-max {rel_max:.2e}"
    # without the log-sum-exp the library runs the forward again: the same
    # lse, so dk and dv agree bit for bit (dq and dP sum reduce-adds whose
    # order may vary)
    again = pkg.spa_attention_bwd(q_, k_, v_, P_, out, dO_, causal=causal)
    assert torch.equal(got[1], again[1]) and torch.equal(got[2], again[2])
    for a, b in ((got[0], again[0]), (got[3], again[3])):
        assert torch.allclose(a, b, rtol=1e-4, atol=1e-5 * float(a.abs().max()))


def test_fused_backward_is_deterministic_up_to_dq_order():
    """dv, dk are written once per key row: bit-identical across runs.  dq
    sums per-key-tile shares with float reduce-adds, whose order may vary."""
    pkg = spa()
    q, k, v, P, dO = (t.cuda() for t in _problem(2, 8, 640, 64, 32, 64, True, "bf16", seed=77))
    out, lse = pkg.spa_attention_fwd_lse(q, k, v, P, causal=True)
    a = pkg.spa_attention_bwd_lse(q, k, v, P, out, lse, dO, causal=True)
    b = pkg.spa_attention_bwd_lse(q, k, v, P, out, lse, dO, causal=True)
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    assert torch.allclose(a[0], b[0], rtol=1e-5, atol=1e-6 * float(a[0].abs().max()))


def test_fused_backward_full_size_sampled_heads():
    """The C3 backward shape (B=2 H=16 N=8192 d=128 m=32 d_v=128, causal) on the
    GPU, checked against the oracle on head 5 of both batch entries (dP_5 sums
    over the batch, so both entries are needed)."""
    pkg = spa()
    w = si.WORKLOADS["C3"]
    q, k, v = si.make_qkv(w, seed=91)
    P = si.make_P(w, seed=92)
    g = torch.Generator().manual_seed(93)
    dO = torch.randn((w.B, w.H, w.N, w.dv), generator=g, dtype=torch.float64).to(w.torch_dtype)
    q_, k_, v_, P_, dO_ = (t.cuda() for t in (q, k, v, P, dO))
    out, lse = pkg.spa_attention_fwd_lse(q_, k_, v_, P_, causal=True)
    dq, dk, dv, dP = pkg.spa_attention_bwd_lse(q_, k_, v_, P_, out, lse, dO_, causal=True)
    h = 5
    sl = slice(h, h + 1)
    ref = oracle.attention_bwd(q[:, sl].contiguous(), k[:, sl].contiguous(), v[:, sl].contiguous(),
                               P[sl].contiguous(), dO[:, sl].contiguous(), causal=True)
    for name, gg, rr in zip(("dq", "dk", "dv", "dP"),
                            (dq[:, sl], dk[:, sl], dv[:, sl], dP[sl]), ref):
        rel_f, rel_max = rel_errors(gg.cpu().numpy(), rr)
        assert rel_f <= REL_F and rel_max <= 2 * REL_F, \
            f"{name}: rel-F {rel_f:.2e}, rel-max {rel_max:.2e}"


def test_fused_backward_c4_m64_full_size_sampled_head():
    """The C4 backward at m = 64 (B=1 H=32 N=32768 d=128 d_v=128, non-causal),
    the shape and launch bench.py --backward --config C4 --m 64 times, on the
    GPU, checked against the oracle on one head (B = 1, so dP_h is that
    head's alone).  The oracle's gradients of one full head take about a
    minute on the host cores."""
    pkg = spa()
    w = si.WORKLOADS["C4"].with_m(64)
    q, k, v = si.make_qkv(w, seed=94)
    P = si.make_P(w, seed=95)
    g = torch.Generator().manual_seed(96)
    dO = torch.randn((w.B, w.H, w.N, w.dv), generator=g, dtype=torch.float64).to(w.torch_dtype)
    q_, k_, v_, P_, dO_ = (t.cuda() for t in (q, k, v, P, dO))
    out, lse = pkg.spa_attention_fwd_lse(q_, k_, v_, P_, causal=False)
    dq, dk, dv, dP = pkg.spa_attention_bwd_lse(q_, k_, v_, P_, out, lse, dO_, causal=False)
    torch.cuda.synchronize()
    h = 19
    sl = slice(h, h + 1)
    ref = oracle.attention_bwd(q[:, sl].contiguous(), k[:, sl].contiguous(), v[:, sl].contiguous(),
                               P[sl].contiguous(), dO[:, sl].contiguous(), causal=False)
    for name, gg, rr in zip(("dq", "dk", "dv", "dP"),
                            (dq[:, sl], dk[:, sl], dv[:, sl], dP[sl]), ref):
        rel_f, rel_max = rel_errors(gg.cpu().numpy(), rr)
        assert rel_f <= REL_F and rel_max <= 2 * REL_F, \
            f"{name}: rel-F {rel_f:.2e}, rel-max {rel_max:.2e}"
    assert pkg.device_error() == 0


@pytest.mark.parametrize("m,dv", [(128, 128), (128, 64)])
def test_cuda_core_backward_serves_m128(m, dv):
    """m = 128 does not fit the fused kernel's tensor memory: the CUDA-core
    backward (flash-style, nothing N x N stored) answers, and agrees with the
    oracle; with and without the forward's log-sum-exp it gives the same bits
    for dk and dv."""
    pkg = spa()
    q, k, v, P, dO = _problem(1, 2, 150, 128, m, dv, True, "bf16", seed=55)
    q_, k_, v_, P_, dO_ = (t.cuda() for t in (q, k, v, P, dO))
    out, lse = pkg.spa_attention_fwd_lse(q_, k_, v_, P_, causal=True)
    got = pkg.spa_attention_bwd_lse(q_, k_, v_, P_, out, lse, dO_, causal=True)
    ref = oracle.attention_bwd(q, k, v, P, dO, causal=True)
    for name, gg, rr in zip(("dq", "dk", "dv", "dP"), got, ref):
        rel_f, rel_max = rel_errors(gg.cpu().numpy(), rr)
        assert rel_f <= REL_F and rel_max <= 2 * REL_F, f"{name}: {rel_f:.2e} {rel_max:.2e}"
    again = pkg.spa_attention_bwd(q_, k_, v_, P_, out, dO_, causal=True)
    for a, b in zip(got, again):
        assert torch.equal(a, b)


def test_staged_backward_gives_the_entry_points_bits_m64():
    """prepare + apply + finish on a caller workspace gives the allocating
    entry point's dk and dv bit for bit at m = 64 (dq, dP within reduce-add
    order)."""
    pkg = spa()
    B, H, N, d, m, dv = 2, 3, 400, 128, 64, 128
    q, k, v, P, dO = (t.cuda() for t in _problem(B, H, N, d, m, dv, True, "bf16", seed=66))
    out, lse = pkg.spa_attention_fwd_lse(q, k, v, P, causal=True)
    want = pkg.spa_attention_bwd_lse(q, k, v, P, out, lse, dO, causal=True)
    ws = torch.empty(pkg.spa_attention_bwd_workspace_size(B, H, N, d, m, dv, pkg.SPA_BF16),
                     dtype=torch.uint8, device="cuda")
    dq = torch.empty((B, H, N, d), dtype=torch.float32, device="cuda")
    dk, dvo = torch.empty_like(dq), torch.empty((B, H, N, dv), dtype=torch.float32, device="cuda")
    dP = torch.empty((H, d, m), dtype=torch.float32, device="cuda")
    pkg.spa_attention_bwd_prepare(q, k, P, out, lse, dO, ws)
    pkg.spa_attention_bwd_apply(v, dO, dvo, ws, B, H, N, d, m, causal=True)
    pkg.spa_attention_bwd_finish(q, k, P, dq, dk, dP, dv, ws)
    torch.cuda.synchronize()
    assert torch.equal(dk, want[1]) and torch.equal(dvo, want[2])
    for a, b in ((dq, want[0]), (dP, want[3])):
        assert torch.allclose(a, b, rtol=1e-4, atol=1e-5 * float(b.abs().max()))
    assert pkg.device_error() == 0
