"""Shared test helpers: library loading and the parity metrics."""
import os

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# Tolerances of the forward against the fp64 oracle (stated for the method):
#   fp32 inputs: max |err| <= 1e-5
#   bf16 inputs (fp32 accumulation): relative Frobenius <= 1e-2 and max |err| <= 2e-2
F32_MAX_ABS = 1e-5
BF16_REL_F = 1e-2
BF16_MAX_ABS = 2e-2


def ensure_built():
    from projected_feature_efficient_gb300 import build as b
    return b.build()


def spa():
    ensure_built()
    import projected_feature_efficient_gb300 as pkg
    return pkg


def errors(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    diff = got - ref
    max_abs = float(np.abs(diff).max()) if diff.size else 0.0
    den = float(np.sqrt((ref * ref).sum()))
    rel_f = float(np.sqrt((diff * diff).sum()) / den) if den > 0 else 0.0
    return max_abs, rel_f


def assert_parity(got, ref, dtype: str, what: str = ""):
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    max_abs, rel_f = errors(got, ref)
    if dtype == "f32":
        assert max_abs <= F32_MAX_ABS, f"{what}: max-abs {max_abs:.3e} > {F32_MAX_ABS}"
    else:
        assert rel_f <= BF16_REL_F and max_abs <= BF16_MAX_ABS, \
            f"{what}: rel-F {rel_f:.3e}, max-abs {max_abs:.3e}"
    return max_abs, rel_f


def sample_rows(N: int, n_random: int = 64, seed: int = 0):
    """Row 0, N-1, every 128-row tile boundary +-1 near both ends, and random rows."""
    rows = {0, N - 1}
    for b in (128, 256, N // 2, N - 128, N - 256):
        for r in (b - 1, b, b + 1):
            if 0 <= r < N:
                rows.add(r)
    rng = np.random.default_rng(seed)
    rows.update(int(r) for r in rng.integers(0, N, size=min(n_random, N)))
    return np.array(sorted(rows), dtype=np.int64)

