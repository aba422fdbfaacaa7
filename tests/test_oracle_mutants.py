"""The oracle's pins have teeth: copies of the oracle with one planted mistake
(compiled on the CPU into a temporary directory) must fail them.  The planted
mistakes are the plausible ones: a wrong score scale, an off-by-one causal
mask, a transposed projection, a missing normalisation, a wrong value row; and
in the gradients, a softmax Jacobian without its row term, a key gradient
built from the wrong operand, a value gradient with the wrong weight, masked
rows leaking into the key gradients, a projection gradient missing the keys."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

MUTANTS = {
    "scale_uses_d": ("const double inv_sqrt_m = 1.0 / sqrt((double)m);",
                     "const double inv_sqrt_m = 1.0 / sqrt((double)d);"),
    "causal_sees_next_key": ("long nkeys = causal ? i + 1 : N;",
                             "long nkeys = causal ? (i + 2 < N ? i + 2 : N) : N;"),
    "projection_transposed": ("orc_load(P, dt, p_off + (size_t)l * m + k);",
                              "orc_load(P, dt, p_off + ((size_t)k * d + l) % ((size_t)d * m));"),
    "missing_normalisation": ("dst[c] = o[c] / l;", "dst[c] = o[c];"),
    "value_row_of_query": ("size_t voff = (bh * N + j) * dv;", "size_t voff = (bh * N + i) * dv;"),
}


def _inputs(seed=0):
    g = torch.Generator().manual_seed(seed)
    B, H, N, d, m, dv = 1, 2, 33, 12, 5, 7
    q = torch.randn((B, H, N, d), generator=g, dtype=torch.float64)
    k = torch.randn((B, H, N, d), generator=g, dtype=torch.float64)
    v = torch.randn((B, H, N, dv), generator=g, dtype=torch.float64)
    P = torch.randn((H, d, m), generator=g, dtype=torch.float64) / math.sqrt(m)
    return q, k, v, P


def pins_pass(lib) -> bool:
    """The library-routine pins of test_oracle_pins, run against a given build."""
    q, k, v, P = _inputs()
    if not np.allclose(oracle.project(q, P, _lib=lib), (q @ P).numpy(), rtol=1e-12, atol=1e-12):
        return False
    for causal in (False, True):
        got = oracle.attention(q, k, v, P, causal=causal, _lib=lib)
        ref = F.scaled_dot_product_attention(q @ P, k @ P, v, is_causal=causal).numpy()
        if not np.allclose(got, ref, rtol=1e-11, atol=1e-12):
            return False
    return True


def test_unmodified_copy_passes(tmp_path):
    lib = oracle.compile_variant(oracle.source(), str(tmp_path))
    assert pins_pass(lib)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = oracle.source()
    assert src.count(old) == 1, f"mutation site for {name} not found"
    lib = oracle.compile_variant(src.replace(old, new), str(tmp_path))
    assert not pins_pass(lib), f"pins did not catch mutant {name}"


# ---------------------------------------------------------------- gradients
BWD_MUTANTS = {
    "softmax_grad_without_row_dot": ("(out_ds) = a_ * (da_ - rdot[i]);", "(out_ds) = a_ * da_;"),
    "key_grad_from_keys": ("g[c] += ds * qp[(size_t)i * m + c] * rsm;",
                           "g[c] += ds * kp[(size_t)i * m + c] * rsm;"),
    "value_grad_weighted_by_ds": ("gv[c] += a * orc_load(dO, dt, (bh * N + i) * dv + c);",
                                  "gv[c] += ds * orc_load(dO, dt, (bh * N + i) * dv + c);"),
    "masked_rows_in_key_grads": ("for (long i = causal ? j : 0; i < N; ++i) {",
                                 "for (long i = 0; i < N; ++i) {"),
    "projection_grad_misses_keys": ("orc_load(k, dt, (bh * N + i) * d + l) * dkp[(size_t)i * m + c];",
                                    "0.0 * dkp[(size_t)i * m + c];"),
}


def bwd_pins_pass(lib) -> bool:
    from test_oracle_bwd import finite_difference_pins
    return all(finite_difference_pins(lib, causal=c) for c in (False, True))


def test_unmodified_copy_passes_gradient_pins(tmp_path):
    lib = oracle.compile_variant(oracle.source(), str(tmp_path))
    assert bwd_pins_pass(lib)


@pytest.mark.parametrize("name", sorted(BWD_MUTANTS))
def test_planted_gradient_mistake_is_caught(name, tmp_path):
    old, new = BWD_MUTANTS[name]
    src = oracle.source()
    assert src.count(old) == 1, f"mutation site for {name} not found"
    lib = oracle.compile_variant(src.replace(old, new), str(tmp_path))
    assert not bwd_pins_pass(lib), f"gradient pins did not catch mutant {name}"
