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
