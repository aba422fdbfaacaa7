"""Failure detection on the GPU without a GPU fault: a bounded wait is made to
run out (a barrier arrival that the kernel withholds on purpose), the kernel
reports it through the device error word, and the device stays usable."""
import time

import pytest
import torch

import oracle
import spa_inputs as si
from helpers import assert_parity, spa

pytestmark = pytest.mark.gpu


def test_withheld_barrier_is_reported_and_the_device_stays_usable():
    pkg = spa()
    assert pkg.device_error() == 0  # nothing pending from earlier tests
    t0 = time.perf_counter()
    status = pkg.selftest_wait_timeout(50)
    elapsed = time.perf_counter() - t0
    assert status == pkg.SPA_ERR_TIMEOUT, pkg.status_str(status)
    # the waits gave up after about their limit, not after the 2 s default
    assert elapsed < 1.5, f"self-test took {elapsed:.2f} s"
    # the self-test read and cleared the error word
    assert pkg.device_error() == 0
    # a normal forward on the same device afterwards is still correct
    w = si.WORKLOADS["C2"].scaled(B=1, H=2, N=300)
    q, k, v = si.make_qkv(w)
    P = si.make_P(w)
    got = pkg.spa_attention_fwd(q.cuda(), k.cuda(), v.cuda(), P.cuda()).cpu().numpy()
    ref = oracle.attention(q, k, v, P, causal=False)
    assert_parity(got, ref, w.dtype, "after the self-test")
    assert pkg.device_error() == 0


def test_backward_kernel_reports_a_withheld_barrier():
    """The fused backward kernel's bounded waits: its first "scores ready" is
    withheld, the gradient warpgroups give up after 50 ms, every role (the
    copy thread, the issuer, the epilogue warpgroup with its named barriers)
    leaves through its abort path, and the device error word reports it.  A full backward afterwards is still correct."""
    pkg = spa()
    assert pkg.device_error() == 0
    t0 = time.perf_counter()
    status = pkg.selftest_bwd_wait_timeout(50)
    elapsed = time.perf_counter() - t0
    assert status == pkg.SPA_ERR_TIMEOUT, pkg.status_str(status)
    assert elapsed < 1.5, f"self-test took {elapsed:.2f} s"
    assert pkg.device_error() == 0
    w = si.WORKLOADS["C3"].scaled(B=1, H=2, N=200, d=64, m=32, dv=64)
    q, k, v = si.make_qkv(w, seed=5)
    P = si.make_P(w, seed=6)
    dO = torch.randn((1, 2, 200, 64), generator=torch.Generator().manual_seed(7)).to(torch.bfloat16)
    q_, k_, v_, P_, dO_ = (x.cuda() for x in (q, k, v, P, dO))
    out = pkg.spa_attention_fwd(q_, k_, v_, P_, causal=True)
    got = pkg.spa_attention_bwd(q_, k_, v_, P_, out, dO_, causal=True)
    ref = oracle.attention_bwd(q, k, v, P, dO, causal=True)
    for gg, rr in zip(got, ref):
        g = gg.cpu().numpy().astype("float64")
        rel = ((g - rr) ** 2).sum() ** 0.5 / ((rr ** 2).sum() ** 0.5)
        assert rel < 1e-2
    assert pkg.device_error() == 0


@pytest.mark.parametrize("m", [32, 64])
def test_projection_kernels_report_a_withheld_barrier(m):
    """The tensor-core projection kernels' bounded waits (m = 32: the per-CTA
    kernel, whose 128 threads decide together at each barrier; m = 64: the
    warp-specialised kernel, whose loader, issuer and two epilogue warpgroups
    each take their abort path): CTA 0's first "product done" is withheld,
    its waits give up after 50 ms, and the other CTAs finish normally."""
    pkg = spa()
    assert pkg.device_error() == 0
    t0 = time.perf_counter()
    status = pkg.selftest_proj_wait_timeout(50, m)
    elapsed = time.perf_counter() - t0
    assert status == pkg.SPA_ERR_TIMEOUT, pkg.status_str(status)
    assert elapsed < 1.5, f"self-test took {elapsed:.2f} s"
    assert pkg.device_error() == 0
    # the projection and a whole forward through the same kernel afterwards
    w = si.WORKLOADS["C3"].scaled(B=1, H=8, N=640, d=64, m=m, dv=64)
    q, k, v = si.make_qkv(w, seed=11)
    P = si.make_P(w, seed=12)
    got = pkg.spa_attention_fwd(q.cuda(), k.cuda(), v.cuda(), P.cuda(), causal=True).cpu().numpy()
    ref = oracle.attention(q, k, v, P, causal=True)
    assert_parity(got, ref, w.dtype, "after the projection self-test")
    assert pkg.device_error() == 0


@pytest.mark.parametrize("kernel", [0, 1, 2])
def test_copy_waiting_kernels_report_a_withheld_barrier(kernel):
    """The kernels that wait on their own TMA copies (0: the fused backward's
    row statistics, 1: its tensor-core finish, 2: the SFA Top-k): CTA 0 arms a
    copy barrier without starting the copies (0, 2) or withholds its first
    "products done" (1); its 128 threads give up together after 50 ms and
    drain what they started, and the other CTAs finish normally."""
    pkg = spa()
    assert pkg.device_error() == 0
    t0 = time.perf_counter()
    status = pkg.selftest_copy_wait_timeout(50, kernel)
    elapsed = time.perf_counter() - t0
    assert status == pkg.SPA_ERR_TIMEOUT, pkg.status_str(status)
    assert elapsed < 1.5, f"self-test took {elapsed:.2f} s"
    assert pkg.device_error() == 0
    if kernel == 2:  # the Top-k afterwards, bit for bit
        x = torch.randn((3000, 128), generator=torch.Generator().manual_seed(13)).to(torch.bfloat16)
        got = pkg.spa_topk_features(x.cuda(), 16).cpu()
        want = torch.from_numpy(oracle.topk_features(x, 16)).to(torch.bfloat16)
        assert torch.equal(got.view(torch.int16), want.view(torch.int16))
    else:  # a whole fused backward afterwards (statistics, kernel, finish)
        w = si.WORKLOADS["C3"].scaled(B=1, H=2, N=300, d=64, m=32, dv=128)
        q, k, v = si.make_qkv(w, seed=15)
        P = si.make_P(w, seed=16)
        dO = torch.randn((1, 2, 300, 128), generator=torch.Generator().manual_seed(17)).to(torch.bfloat16)
        q_, k_, v_, P_, dO_ = (t.cuda() for t in (q, k, v, P, dO))
        out = pkg.spa_attention_fwd(q_, k_, v_, P_, causal=True)
        got = pkg.spa_attention_bwd(q_, k_, v_, P_, out, dO_, causal=True)
        ref = oracle.attention_bwd(q, k, v, P, dO, causal=True)
        for gg, rr in zip(got, ref):
            g = gg.cpu().numpy().astype("float64")
            rel = ((g - rr) ** 2).sum() ** 0.5 / ((rr ** 2).sum() ** 0.5)
            assert rel < 1e-2
    assert pkg.device_error() == 0
