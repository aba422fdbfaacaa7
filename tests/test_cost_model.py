"""The FLOP model used for throughput, pinned to the pages' cost model.

SPA paper, Sec. 4.1.1: T_SPA = O(N d_k d_k'/s) + O(N^2 d_k') + O(N^2 d_v) against
T_std = O(N^2 d_k) + O(N^2 d_v); the score term shrinks by d_k / d_k' and the
end-to-end ratio tends to (d_k + d_v) / (d_k' + d_v).  The golden file holds
the numbers the page prints for d_k = d_v = 512, d_k' = 64.
"""
import os

import pytest

import bench

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "spa_cost_model.txt")


def golden():
    vals = {}
    for line in open(GOLDEN):
        line = line.split("#", 1)[0].strip()
        if line:
            k, v = (x.strip() for x in line.split("="))
            vals[k] = float(v)
    return vals


def test_score_term_speedup_matches_the_page():
    g = golden()
    d, m, N = int(g["d_k"]), int(g["d_k_proj"]), 4096
    # score FLOPs alone: attention FLOPs with d_v = 0, standard (m = d) vs projected
    ratio = bench.attn_flops(1, 1, N, d, 0, False) / bench.attn_flops(1, 1, N, m, 0, False)
    assert ratio == g["score_speedup"]


def test_end_to_end_ratio_tends_to_the_page_formula():
    g = golden()
    d, dv, m = int(g["d_k"]), int(g["d_v"]), int(g["d_k_proj"])
    limit = bench.speedup_vs_standard(d, m, dv)
    assert limit == pytest.approx((d + dv) / (m + dv))
    assert limit == pytest.approx(16 / 9)
    # finite N approaches the limit from below (the projection term vanishes)
    prev = 0.0
    for N in (512, 4096, 65536, 1 << 20):
        r = bench.speedup_vs_standard(d, m, dv, N)
        assert prev < r < limit
        prev = r
    assert limit - prev < 1e-3
    # the page's printed "approximately 1.9x" overstates its own formula
    assert abs(g["e2e_speedup_printed"] - limit) > 0.1


@pytest.mark.parametrize("B,H,N,d,m,dv,causal,gflops", [
    (1, 32, 32768, 128, 16, 128, False, 9904.194584576),
    (1, 32, 32768, 128, 32, 128, False, 11012.296146944),
    (1, 32, 32768, 128, 64, 128, False, 13228.49927168),
    (2, 16, 8192, 128, 32, 128, True, 347.892350976),
    (1, 8, 131072, 128, 32, 128, True, 22007.412424704),
    (1, 8, 131072, 128, 128, 128, True, 35253.091565568),
])
def test_workload_flops(B, H, N, d, m, dv, causal, gflops):
    """4 B H N d m + 2 B H N^2 (m + d_v), N^2 term halved when causal, counted
    independently here as multiply-adds x 2."""
    proj_macs = 2 * B * H * N * d * m                 # Q P and K P
    pair_macs = B * H * (N * (N + 1) // 2 if causal else N * N) * (m + dv)
    exact_causal = 2 * (proj_macs + pair_macs)
    assert bench.flops(B, H, N, d, m, dv, causal) == pytest.approx(gflops * 1e9, rel=1e-12)
    # the convention halves N^2 instead of counting N(N+1)/2 pairs
    assert bench.flops(B, H, N, d, m, dv, causal) == pytest.approx(exact_causal,
                                                                   rel=2.0 / N if causal else 0)


def test_decode_bytes_per_step():
    """A decode step reads, per cached key, m fp16 values and one fp32 multiplier
    of the projected key cache plus d_v bf16 values: 324 bytes at m=32, d_v=128,
    against 512 for a cache of K and V at d=128."""
    assert bench.decode_bytes(1, 1, 1, 32, 128) == 324
    assert bench.decode_bytes(8, 32, 32768, 32, 128) == 8 * 32 * 32768 * 324
    ratio = bench.decode_bytes(1, 1, 1, 32, 128) / (2 * 128 + 2 * 128)
    assert abs(ratio - 0.6328125) < 1e-12


def test_backward_flop_and_byte_models():
    # per head and N^2 term: S (2m), dA (2 d_v), dQp (2m), dKp (2m), dV (2 d_v)
    assert bench.bwd_flops(1, 1, 10, 4, 3, 5, False) == 2 * 100 * (9 + 10) + 12 * 10 * 4 * 3
    assert bench.bwd_flops(1, 1, 10, 4, 3, 5, True) == 100 * (9 + 10) + 12 * 10 * 4 * 3
    # one fused kernel launch: the five N^2 products only (projections outside)
    assert bench.bwd_kernel_flops(1, 1, 10, 3, 5, False) == 2 * 100 * (9 + 10)
    assert bench.bwd_kernel_flops(2, 16, 8192, 32, 128, True) == \
        2 * 32 * 8192 * 8192 * (96 + 256) / 2
