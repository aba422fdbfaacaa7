"""Pins for the fp64 oracle: facts fixed by the pages and by mathematics.

The oracle is checked here against things other than itself:
  * a library attention routine (torch SDPA in fp64) applied to Q P, K P, V;
  * the identity projection, which must give standard attention (SPA paper,
    Sec. 3.1.1 recap vs Sec. 3.1.3);
  * closed forms (N = 1, N = 2, causal first row, constant V, V = identity);
  * the scaling law of the logits under P -> cP;
  * permutation equivariance;
  * the softmax stability facts the pages prove (SPA Lemma 2, Frobenius
    Lipschitz; PDA Lemma 3.4, l_inf -> l_1 with constant 2; PDA Theorems
    3.4/3.7 on the output error);
  * the Johnson-Lindenstrauss inner-product tail bound 4 exp(-m eps^2 / 8)
    (PDA Theorem 3.1) and the Gaussian moments behind it;
  * the predicted 1/sqrt(m) decay of the score error (PDA Sec. 5.2 item 1).
A mutated copy of the oracle (tests/test_oracle_mutants.py) must fail these.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import spa_inputs as si


def _rand(shape, seed, dtype=torch.float64):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=torch.float64).to(dtype)


def _sdpa_projected(q, k, v, P, causal):
    qd, kd, vd, Pd = (t.double() for t in (q, k, v, P))
    # per-head projection: [B,H,N,d] @ [H,d,m] broadcasts over B
    return F.scaled_dot_product_attention(qd @ Pd, kd @ Pd, vd, is_causal=causal).numpy()


# ------------------------------------------------------------------ library pins
@pytest.mark.parametrize("shape", [(1, 1, 7, 5, 3), (2, 3, 33, 16, 8), (1, 2, 130, 64, 16)])
def test_project_matches_library_matmul(shape):
    B, H, N, d, m = shape
    x = _rand((B, H, N, d), 1)
    P = _rand((H, d, m), 2) / math.sqrt(m)
    ref = (x @ P).numpy()
    got = oracle.project(x, P)
    assert got.shape == (B, H, N, m)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(1, 1, 1, 4, 2, 3), (2, 2, 37, 16, 8, 12), (1, 3, 129, 32, 16, 24)])
def test_attention_matches_library_sdpa(shape, causal):
    B, H, N, d, m, dv = shape
    q = _rand((B, H, N, d), 3)
    k = _rand((B, H, N, d), 4)
    v = _rand((B, H, N, dv), 5)
    P = _rand((H, d, m), 6) / math.sqrt(m)
    got = oracle.attention(q, k, v, P, causal=causal)
    ref = _sdpa_projected(q, k, v, P, causal)
    np.testing.assert_allclose(got, ref, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_attention_reads_narrow_inputs_exactly(dtype):
    """bf16 / fp32 inputs are widened exactly: same answer as feeding the widened values."""
    q = _rand((1, 2, 40, 16), 7, dtype)
    k = _rand((1, 2, 40, 16), 8, dtype)
    v = _rand((1, 2, 40, 8), 9, dtype)
    P = (_rand((2, 16, 8), 10) / math.sqrt(8)).to(dtype)
    a = oracle.attention(q, k, v, P, causal=True)
    b = oracle.attention(q.double(), k.double(), v.double(), P.double(), causal=True)
    assert np.array_equal(a, b)


def test_row_sampling_matches_full():
    q = _rand((2, 2, 50, 8), 11)
    k = _rand((2, 2, 50, 8), 12)
    v = _rand((2, 2, 50, 6), 13)
    P = _rand((2, 8, 4), 14) / 2
    rows = [0, 1, 17, 48, 49]
    full = oracle.attention(q, k, v, P, causal=True)
    part = oracle.attention(q, k, v, P, causal=True, rows=rows)
    assert np.array_equal(part, full[:, :, rows])


def test_lse_is_log_sum_exp_of_scaled_scores():
    q = _rand((1, 1, 9, 4), 15)
    k = _rand((1, 1, 9, 4), 16)
    v = _rand((1, 1, 9, 3), 17)
    P = _rand((1, 4, 2), 18) / math.sqrt(2)
    _, lse = oracle.attention(q, k, v, P, return_lse=True)
    s = ((q @ P) @ (k @ P).transpose(-1, -2) / math.sqrt(2)).numpy()
    ref = np.log(np.exp(s).sum(-1))
    np.testing.assert_allclose(lse, ref, rtol=1e-12)


# ------------------------------------------------------------------ special cases
def test_identity_projection_is_standard_attention():
    """m = d and P = I gives softmax(Q K^T / sqrt(d)) V, the standard attention
    recapped in the SPA paper, Sec. 3.1.1 (the exact-attention control run)."""
    B, H, N, d = 1, 2, 65, 16
    q, k, v = _rand((B, H, N, d), 19), _rand((B, H, N, d), 20), _rand((B, H, N, d), 21)
    P = torch.eye(d, dtype=torch.float64).expand(H, d, d).contiguous()
    for causal in (False, True):
        got = oracle.attention(q, k, v, P, causal=causal)
        ref = F.scaled_dot_product_attention(q, k, v, is_causal=causal).numpy()
        np.testing.assert_allclose(got, ref, rtol=1e-11, atol=1e-12)


def test_single_token_returns_its_value():
    q, k, v = _rand((1, 3, 1, 8), 22), _rand((1, 3, 1, 8), 23), _rand((1, 3, 1, 5), 24)
    P = _rand((3, 8, 4), 25)
    for causal in (False, True):
        assert np.allclose(oracle.attention(q, k, v, P, causal=causal), v.numpy(), rtol=0,
                           atol=1e-15)


def test_two_tokens_closed_form():
    """N = 2: o_0 = sigmoid(s00 - s01) v_0 + sigmoid(s01 - s00) v_1."""
    d, m = 3, 2
    q = torch.tensor([[[[0.5, -1.0, 2.0], [1.5, 0.25, -0.5]]]], dtype=torch.float64)
    k = torch.tensor([[[[1.0, 0.0, -1.0], [-2.0, 1.0, 0.5]]]], dtype=torch.float64)
    v = torch.tensor([[[[1.0, 2.0], [-3.0, 0.5]]]], dtype=torch.float64)
    P = torch.tensor([[[0.3, -0.7], [1.1, 0.2], [-0.4, 0.9]]], dtype=torch.float64)
    qp = [[sum(q[0, 0, i, l].item() * P[0, l, c].item() for l in range(d)) for c in range(m)]
          for i in range(2)]
    kp = [[sum(k[0, 0, j, l].item() * P[0, l, c].item() for l in range(d)) for c in range(m)]
          for j in range(2)]
    got = oracle.attention(q, k, v, P)[0, 0]
    for i in range(2):
        s0 = (qp[i][0] * kp[0][0] + qp[i][1] * kp[0][1]) / math.sqrt(m)
        s1 = (qp[i][0] * kp[1][0] + qp[i][1] * kp[1][1]) / math.sqrt(m)
        w0 = 1.0 / (1.0 + math.exp(s1 - s0))
        w1 = 1.0 / (1.0 + math.exp(s0 - s1))
        for c in range(2):
            assert got[i, c] == pytest.approx(w0 * v[0, 0, 0, c].item() + w1 * v[0, 0, 1, c].item(),
                                              rel=1e-14, abs=1e-15)
    # causal: row 0 sees only key 0, row 1 both
    gc = oracle.attention(q, k, v, P, causal=True)[0, 0]
    assert np.allclose(gc[0], v[0, 0, 0].numpy(), atol=1e-15)
    assert np.allclose(gc[1], got[1], atol=1e-15)


def test_constant_value_column_passes_through():
    q, k = _rand((1, 2, 31, 8), 26), _rand((1, 2, 31, 8), 27)
    v = torch.ones((1, 2, 31, 3), dtype=torch.float64) * torch.tensor([1.0, -2.5, 7.0],
                                                                      dtype=torch.float64)
    P = _rand((2, 8, 4), 28)
    for causal in (False, True):
        np.testing.assert_allclose(oracle.attention(q, k, v, P, causal=causal), v.numpy(),
                                   rtol=1e-13)


def _softmax_matrix(q, k, P, causal):
    """V = I_N exposes the attention matrix: O = A_tilde."""
    B, H, N, _ = q.shape
    eye = torch.eye(N, dtype=torch.float64).expand(B, H, N, N).contiguous()
    return oracle.attention(q, k, eye.to(q.dtype), P, causal=causal)


def test_identity_values_expose_a_row_stochastic_matrix():
    q, k = _rand((1, 1, 24, 6), 29), _rand((1, 1, 24, 6), 30)
    P = _rand((1, 6, 3), 31) / math.sqrt(3)
    for causal in (False, True):
        A = _softmax_matrix(q, k, P, causal)[0, 0]
        np.testing.assert_allclose(A.sum(-1), 1.0, rtol=0, atol=1e-13)
        assert (A >= 0).all()
        if causal:
            assert np.all(np.triu(A, 1) == 0.0)
        # row i of A is a softmax of a vector whose differences are score differences
        qp, kp = (q @ P)[0, 0].numpy(), (k @ P)[0, 0].numpy()
        s = qp @ kp.T / math.sqrt(3)
        for i in (0, 5, 23):
            n = i + 1 if causal else 24
            np.testing.assert_allclose(np.log(A[i, :n] / A[i, 0]), s[i, :n] - s[i, 0],
                                       rtol=1e-9, atol=1e-11)


def test_scaling_projection_scales_logits_quadratically():
    """P -> cP multiplies every logit by c^2: A(cP) = softmax(c^2 * log A(P))."""
    q, k = _rand((1, 1, 20, 5), 32), _rand((1, 1, 20, 5), 33)
    P = _rand((1, 5, 4), 34) / 2
    c = 1.7
    A1 = _softmax_matrix(q, k, P, False)[0, 0]
    Ac = _softmax_matrix(q, k, c * P, False)[0, 0]
    z = c * c * np.log(A1)
    z -= z.max(-1, keepdims=True)
    ref = np.exp(z) / np.exp(z).sum(-1, keepdims=True)
    np.testing.assert_allclose(Ac, ref, rtol=1e-9, atol=1e-13)


def test_permutation_equivariance():
    q, k, v = _rand((1, 2, 30, 8), 35), _rand((1, 2, 30, 8), 36), _rand((1, 2, 30, 4), 37)
    P = _rand((2, 8, 4), 38) / 2
    base = oracle.attention(q, k, v, P)
    perm = torch.randperm(30, generator=torch.Generator().manual_seed(39))
    # permuting keys and values together leaves every row unchanged
    np.testing.assert_allclose(oracle.attention(q, k[:, :, perm], v[:, :, perm], P), base,
                               rtol=1e-12, atol=1e-14)
    # permuting queries permutes the rows of the output
    np.testing.assert_allclose(oracle.attention(q[:, :, perm], k, v, P), base[:, :, perm.numpy()],
                               rtol=1e-12, atol=1e-14)


def test_tiny_brute_force_against_log_sum_exp_form():
    """Second formulation: O_i = sum_j exp(s_ij - lse_i) v_j, enumerated in Python."""
    q, k, v = _rand((1, 1, 4, 3), 40), _rand((1, 1, 4, 3), 41), _rand((1, 1, 4, 2), 42)
    P = _rand((1, 3, 2), 43)
    got = oracle.attention(q, k, v, P, causal=True)[0, 0]
    Q, K, V, Pm = q[0, 0].tolist(), k[0, 0].tolist(), v[0, 0].tolist(), P[0].tolist()
    proj = lambda x: [sum(x[l] * Pm[l][c] for l in range(3)) for c in range(2)]
    for i in range(4):
        qi = proj(Q[i])
        s = [sum(a * b for a, b in zip(qi, proj(K[j]))) / math.sqrt(2) for j in range(i + 1)]
        lse = math.log(math.fsum(math.exp(x) for x in s))
        for c in range(2):
            ref = math.fsum(math.exp(s[j] - lse) * V[j][c] for j in range(i + 1))
            assert got[i, c] == pytest.approx(ref, rel=1e-13, abs=1e-15)


# ------------------------------------------------------------------ page invariants
def _exact_and_projected(seed, N=48, d=32, m=8, dv=5):
    q = _rand((1, 1, N, d), seed)
    k = _rand((1, 1, N, d), seed + 1)
    v = _rand((1, 1, N, dv), seed + 2)
    P = _rand((1, d, m), seed + 3) / math.sqrt(m)
    eye = torch.eye(d, dtype=torch.float64).expand(1, d, d).contiguous()
    S = (q[0, 0] @ k[0, 0].T).numpy() / math.sqrt(d)
    St = ((q[0, 0] @ P[0]) @ (k[0, 0] @ P[0]).T).numpy() / math.sqrt(m)
    A = _softmax_matrix(q, k, eye, False)[0, 0]
    At = _softmax_matrix(q, k, P, False)[0, 0]
    O = oracle.attention(q, k, v, eye)[0, 0]
    Ot = oracle.attention(q, k, v, P)[0, 0]
    return S, St, A, At, O, Ot, v[0, 0].numpy()


@pytest.mark.parametrize("seed", [100, 200, 300])
def test_softmax_stability_bounds_from_the_pages(seed):
    S, St, A, At, O, Ot, V = _exact_and_projected(seed)
    # SPA Lemma 2: ||softmax(A) - softmax(B)||_F <= ||A - B||_F
    assert np.linalg.norm(A - At) <= np.linalg.norm(S - St) + 1e-12
    # PDA Lemma 3.4 per row: ||a_i - a~_i||_1 <= 2 ||S_i - S~_i||_inf
    eps_rows = np.abs(S - St).max(-1)
    assert np.all(np.abs(A - At).sum(-1) <= 2 * eps_rows + 1e-12)
    # PDA Theorem 3.4: ||o_i - o~_i||_2 <= ||a_i - a~_i||_1 ||V||_2 <= 2 eps ||V||_F
    V2 = np.linalg.norm(V, 2)
    VF = np.linalg.norm(V)
    row_err = np.linalg.norm(O - Ot, axis=-1)
    assert np.all(row_err <= np.abs(A - At).sum(-1) * V2 + 1e-12)
    eps = np.abs(S - St).max()
    assert np.all(row_err <= 2 * eps * VF + 1e-12)
    # PDA Theorem 3.7: ||O - O~||_F <= 2 eps sqrt(L) ||V||_F
    assert np.linalg.norm(O - Ot) <= 2 * eps * math.sqrt(S.shape[0]) * VF + 1e-12
    # and the output error really is a consequence of A - A~ (O - O~ = (A - A~) V)
    np.testing.assert_allclose(O - Ot, (A - At) @ V, rtol=1e-9, atol=1e-12)


def _unit(x):
    return x / np.linalg.norm(x)


@pytest.mark.parametrize("m", [128, 256])
def test_jl_inner_product_tail_bound(m):
    """PDA Theorem 3.1: P(|<uP, vP> - <u, v>| >= eps) <= 4 exp(-m eps^2 / 8) for unit
    u, v and P_ij ~ N(0, 1/m).  The bound is vacuous for m <= 32, so it is checked
    at the m the page recommends (128, 256)."""
    d, T, eps = 64, 2000, 0.45
    rng = np.random.default_rng(7 + m)
    u = _unit(rng.standard_normal(d))
    v = _unit(u + 0.8 * rng.standard_normal(d))
    x = torch.tensor(np.stack([u, v]), dtype=torch.float64).reshape(1, 1, 2, d)
    g = torch.Generator().manual_seed(1234 + m)
    devs, ips = [], []
    for _ in range(T // 100):
        P = torch.randn((100, d, m), generator=g, dtype=torch.float64) / math.sqrt(m)
        xp = oracle.project(x.expand(1, 100, 2, d).contiguous(), P)[0]   # [100, 2, m]
        ip = (xp[:, 0] * xp[:, 1]).sum(-1)
        ips.append(ip)
    ips = np.concatenate(ips)
    frac = float(np.mean(np.abs(ips - u @ v) >= eps))
    bound = 4 * math.exp(-m * eps * eps / 8)
    assert frac <= bound
    # the moments behind the bound: E<uP,vP> = <u,v>, Var = (|u|^2|v|^2 + <u,v>^2) / m
    var = (1.0 + (u @ v) ** 2) / m
    assert abs(ips.mean() - u @ v) < 5 * math.sqrt(var / T)
    assert abs(ips.var() / var - 1.0) < 5 * math.sqrt(2.0 / T)


def test_score_error_decays_like_inverse_sqrt_m():
    """PDA Sec. 5.2 item 1: max |<q~_i, k~_j> - <q_i, k_j>| shrinks like m^(-1/2)."""
    d, N = 256, 64
    rng = np.random.default_rng(5)
    Q = np.stack([_unit(r) for r in rng.standard_normal((N, d))])
    K = np.stack([_unit(r) for r in rng.standard_normal((N, d))])
    exact = Q @ K.T
    ms = [16, 32, 64, 128, 256]
    errs = []
    g = torch.Generator().manual_seed(99)
    for m in ms:
        e = 0.0
        for _ in range(20):
            P = torch.randn((1, d, m), generator=g, dtype=torch.float64) / math.sqrt(m)
            qp = oracle.project(torch.tensor(Q).reshape(1, 1, N, d), P)[0, 0]
            kp = oracle.project(torch.tensor(K).reshape(1, 1, N, d), P)[0, 0]
            e += np.abs(qp @ kp.T - exact).max()
        errs.append(e / 20)
    slope = np.polyfit(np.log(ms), np.log(errs), 1)[0]
    assert -0.65 <= slope <= -0.35, slope


# ------------------------------------------------------------ Top-k features
def test_topk_worked_example_with_ties():
    """|x| = 1, 2, 2, 2, 0.5: the top two are the first two of the three tied 2s."""
    x = np.array([[1.0, -2.0, 2.0, 2.0, 0.5]])
    np.testing.assert_array_equal(oracle.topk_features(x, 2), [[0.0, -2.0, 2.0, 0.0, 0.0]])
    np.testing.assert_array_equal(oracle.topk_features(x, 1), [[0.0, -2.0, 0.0, 0.0, 0.0]])
    np.testing.assert_array_equal(oracle.topk_features(x, 5), x)


def test_topk_brute_force_on_small_rows():
    """Against brute force over every k-subset: the kept set has the largest
    sum of magnitudes, and among equal sums the lexicographically smallest
    index set (lowest indices first)."""
    import itertools
    rng = np.random.default_rng(4)
    for _ in range(60):
        d = int(rng.integers(1, 7))
        k = int(rng.integers(1, d + 1))
        x = rng.choice([-2.0, -1.0, -0.5, 0.5, 1.0, 2.0, 3.0], size=d)
        best = None
        for sub in itertools.combinations(range(d), k):
            key = (-sum(abs(x[i]) for i in sub), sub)
            if best is None or key < best:
                best = key
        want = np.zeros(d)
        want[list(best[1])] = x[list(best[1])]
        np.testing.assert_array_equal(oracle.topk_features(x[None], k)[0], want)


def test_topk_invariants_on_random_rows():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((50, 128))
    for k in (1, 16, 127, 128):
        y = oracle.topk_features(x, k)
        kept = y != 0
        assert np.all(kept.sum(axis=1) == k)
        assert np.all(y[kept] == x[kept])
        for r in range(x.shape[0]):
            if k < 128:
                assert np.abs(x[r][~kept[r]]).max() <= np.abs(x[r][kept[r]]).min()
