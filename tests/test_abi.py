"""The C ABI boundary, on the host: the library loads, exports every function
include/spa.h declares, and rejects bad arguments with the documented status
codes before touching the GPU (no kernel runs in these tests)."""
import ctypes
import os
import re

import pytest

from helpers import ROOT, spa

HEADER = os.path.join(ROOT, "include", "spa.h")

OK, NULL, SHAPE, DTYPE, ALIGN, UNSUPPORTED, NOMEM = 0, 1, 2, 3, 4, 5, 6
F32, BF16 = 0, 1
A = 0x100000  # a 16-byte-aligned dummy address; never dereferenced by validation


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(spa_[a-z_0-9]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    return spa().lib


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("spa_project", "spa_attention_fwd", "spa_status_str"):
        assert required in names


def test_every_declared_function_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} not exported by libspa.so"
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings(lib):
    for code in range(9):
        assert spa().status_str(code).startswith("SPA_")
    assert spa().status_str(12345) == "SPA_ERR_UNKNOWN"
    assert lib.spa_version() >= 100


def fwd(lib, q=A, k=A, v=A, P=A, out=A, B=1, H=2, N=256, d=128, m=32, dv=128, causal=0,
        dtype=BF16):
    return lib.spa_attention_fwd(q, k, v, P, out, B, H, N, d, m, dv, causal, dtype, None)


def test_forward_rejects_bad_arguments(lib):
    assert fwd(lib, q=None) == NULL
    assert fwd(lib, out=None) == NULL
    assert fwd(lib, P=None) == NULL
    assert fwd(lib, N=-1) == SHAPE
    assert fwd(lib, B=-2) == SHAPE
    assert fwd(lib, dtype=7) == DTYPE
    assert fwd(lib, k=A + 8) == ALIGN
    assert fwd(lib, out=A + 4) == ALIGN
    assert fwd(lib, B=300, H=300) == SHAPE            # B*H above 65535
    assert fwd(lib, d=0) == UNSUPPORTED
    assert fwd(lib, d=257) == UNSUPPORTED
    assert fwd(lib, m=129) == UNSUPPORTED
    # bf16 tensor-core path: m in {16,32,64,128}, d_v in {64,128}
    assert fwd(lib, m=24) == UNSUPPORTED
    assert fwd(lib, dv=96) == UNSUPPORTED
    # fp32 path accepts any m <= 128 and d_v <= 256 (still validated before any launch)
    assert fwd(lib, m=24, dv=96, dtype=F32, q=None) == NULL


def test_empty_problem_is_a_no_op(lib):
    # nothing is read or written, so even NULL pointers are fine
    assert fwd(lib, q=None, k=None, v=None, P=None, out=None, N=0) == OK
    assert fwd(lib, q=None, k=None, v=None, P=None, out=None, B=0) == OK
    assert lib.spa_project(None, None, None, 1, 1, 0, 64, 16, BF16, None) == OK


def test_project_rejects_bad_arguments(lib):
    assert lib.spa_project(None, A, A, 1, 1, 8, 64, 16, BF16, None) == NULL
    assert lib.spa_project(A, A, A + 2, 1, 1, 8, 64, 16, BF16, None) == ALIGN
    assert lib.spa_project(A, A, A, 1, 1, 8, 300, 16, BF16, None) == UNSUPPORTED
    assert lib.spa_project(A, A, A, 1, 1, 8, 64, 16, 9, None) == DTYPE


def ws_size(lib, B, H, N, d, m, dv, dtype):
    n = ctypes.c_size_t(0)
    st = lib.spa_attention_workspace_size(B, H, N, d, m, dv, dtype, ctypes.byref(n))
    return st, n.value


def _r(x):
    return (x + 255) // 256 * 256


@pytest.mark.parametrize("m,KD", [(16, 48), (32, 32), (64, 64), (128, 128)])
def test_workspace_size_bf16(lib, m, KD):
    B, H, N = 1, 32, 32768 + 5
    NT = (N + 127) // 128
    tiles = B * H * NT * 128 * KD * 2
    expect = _r(_r(_r(tiles) + tiles) + B * H * NT * 128 * 4) + _r(B * H * NT * 4)
    st, n = ws_size(lib, B, H, N, 128, m, 128, BF16)
    assert st == OK and n == expect


def test_workspace_size_f32_and_empty(lib):
    st, n = ws_size(lib, 1, 1, 256, 64, 16, 64, F32)
    assert st == OK and n == 2 * _r(256 * 16 * 4)
    assert ws_size(lib, 1, 1, 0, 64, 16, 64, F32) == (OK, 0)
    assert ws_size(lib, 1, 1, 8, 64, 24, 64, BF16)[0] == UNSUPPORTED
    assert lib.spa_attention_workspace_size(1, 1, 8, 64, 16, 64, F32, None) == NULL


def test_workspace_entry_point_checks_its_buffer(lib):
    st, need = ws_size(lib, 1, 2, 256, 128, 32, 128, BF16)
    args = (A, A, A, A, A, 1, 2, 256, 128, 32, 128, 0, BF16)
    assert lib.spa_attention_fwd_ws(*args, None, need, None) == NULL
    assert lib.spa_attention_fwd_ws(*args, A + 16, need, None) == ALIGN
    assert lib.spa_attention_fwd_ws(*args, A, need - 1, None) == NOMEM


def test_noalloc_entry_point_validates_first(lib):
    """The allocation-free forward checks its arguments before it looks up its
    scratch array (no CUDA call happens in any of these cases)."""
    def call(q=A, k=A, v=A, P=A, out=A, B=1, H=2, N=256, d=128, m=32, dv=128, dtype=BF16):
        return lib.spa_attention_fwd_noalloc(q, k, v, P, out, B, H, N, d, m, dv, 0, dtype, None)
    assert call(q=None) == NULL
    assert call(P=None) == NULL
    assert call(out=None) == NULL
    assert call(v=A + 8) == ALIGN
    assert call(out=A + 4) == ALIGN
    assert call(N=-1) == SHAPE
    assert call(B=300, H=300) == SHAPE
    assert call(dtype=5) == DTYPE
    assert call(m=24) == UNSUPPORTED
    assert call(dv=96) == UNSUPPORTED
    # an empty problem returns before the scratch is looked up
    assert call(q=None, k=None, v=None, P=None, out=None, N=0) == OK
    assert call(q=None, k=None, v=None, P=None, out=None, B=0) == OK
    # a workspace larger than the 64 MiB array
    assert call(H=64, N=131072) == NOMEM


def test_host_entry_point_validates_first(lib):
    assert lib.spa_attention_fwd_host(None, A, A, A, A, 1, 1, 8, 64, 16, 64, 0, BF16, None) == NULL
    assert lib.spa_attention_fwd_host(A, A, A, A, A, 1, 1, 8, 64, 20, 64, 0, BF16, None) == \
        UNSUPPORTED
    assert lib.spa_device_error(None) == NULL


def test_binding_marshals_shapes():
    import torch
    pkg = spa()
    q = torch.zeros((1, 2, 8, 16), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        pkg.spa_attention_fwd(q, q, q, torch.zeros((3, 16, 16), dtype=torch.bfloat16))
    with pytest.raises(TypeError):
        pkg.spa_attention_fwd(q, q, q.float(), torch.zeros((2, 16, 16), dtype=torch.bfloat16))


def append(lib, k=A, P=A, kc=A, kmul=A, B=1, H=2, T=4, d=128, m=32, pos=0, cap=16, dtype=BF16):
    return lib.spa_kcache_append(k, P, kc, kmul, B, H, T, d, m, pos, cap, dtype, None)


def decode(lib, q=A, P=A, kc=A, kmul=A, v=A, out=A, B=1, H=2, L=8, d=128, m=32, dv=128, cap=16,
           dtype=BF16):
    return lib.spa_attention_decode(q, P, kc, kmul, v, out, B, H, L, d, m, dv, cap, dtype, None)


def test_cache_append_rejects_bad_arguments(lib):
    assert append(lib, k=None) == NULL
    assert append(lib, kmul=None) == NULL
    assert append(lib, pos=13, T=4, cap=16) == SHAPE   # rows past the capacity
    assert append(lib, pos=-1) == SHAPE
    assert append(lib, dtype=F32) == UNSUPPORTED       # the fp16 cache is for bf16 inputs
    assert append(lib, dtype=9) == DTYPE
    assert append(lib, m=24) == UNSUPPORTED
    assert append(lib, d=300) == UNSUPPORTED
    assert append(lib, kc=A + 2) == ALIGN
    assert append(lib, k=None, P=None, kc=None, kmul=None, T=0) == OK  # nothing to append


def test_decode_rejects_bad_arguments(lib):
    assert decode(lib, q=None) == NULL
    assert decode(lib, v=None) == NULL
    assert decode(lib, L=0) == SHAPE                    # no key to attend to
    assert decode(lib, L=17, cap=16) == SHAPE           # more keys than the cache holds
    assert decode(lib, dtype=F32) == UNSUPPORTED
    assert decode(lib, dv=96) == UNSUPPORTED
    assert decode(lib, m=48) == UNSUPPORTED
    assert decode(lib, out=A + 4) == ALIGN
    assert decode(lib, B=300, H=300) == SHAPE
    assert decode(lib, q=None, P=None, kc=None, kmul=None, v=None, out=None, B=0) == OK


def test_topk_and_sfa_reject_bad_arguments(lib):
    assert lib.spa_topk_features(A, A, 10, 96, 4, BF16, None) == UNSUPPORTED   # d not 32/64/128/256
    assert lib.spa_topk_features(A, A, 10, 128, 0, BF16, None) == SHAPE       # k < 1
    assert lib.spa_topk_features(A, A, 10, 128, 129, BF16, None) == SHAPE     # k > d
    assert lib.spa_topk_features(None, A, 10, 128, 4, BF16, None) == NULL
    assert lib.spa_topk_features(A, A + 2, 10, 128, 4, BF16, None) == ALIGN
    assert lib.spa_topk_features(None, None, 0, 128, 4, BF16, None) == OK     # no rows
    sfa = lib.spa_sfa_attention_fwd
    assert sfa(A, A, A, A, 1, 2, 64, 256, 128, 8, 0, BF16, None) == UNSUPPORTED  # m = d = 256
    assert sfa(A, A, A, A, 1, 2, 64, 128, 128, 0, 0, BF16, None) == SHAPE
    assert sfa(A, None, A, A, 1, 2, 64, 128, 128, 8, 0, BF16, None) == NULL
    assert sfa(None, None, None, None, 1, 2, 0, 128, 128, 8, 0, BF16, None) == OK


def test_forward_lse_validates_first(lib):
    def f(lse=A, **kw):
        a = dict(q=A, k=A, v=A, P=A, out=A, B=1, H=2, N=256, d=128, m=32, dv=128, causal=1,
                 dtype=BF16)
        a.update(kw)
        return lib.spa_attention_fwd_lse(a["q"], a["k"], a["v"], a["P"], a["out"], lse, a["B"],
                                         a["H"], a["N"], a["d"], a["m"], a["dv"], a["causal"],
                                         a["dtype"], None)
    assert f(lse=None) == NULL
    assert f(lse=A + 2) == ALIGN
    assert f(q=None) == NULL
    assert f(N=-1) == SHAPE
    assert f(N=0, lse=None) == OK  # empty: nothing to write


def bwd_lse(lib, lse=A, dO=A, dq=A, dk=A, dv_=A, dP=A, B=1, H=2, N=256, d=128, m=32, dv=128,
            dtype=BF16):
    return lib.spa_attention_bwd_lse(A, A, A, A, A, lse, dO, dq, dk, dv_, dP, B, H, N, d, m, dv,
                                     1, dtype, None)


def test_backward_entry_points_validate_first(lib):
    assert bwd_lse(lib, lse=None) == NULL          # the _lse form needs the log-sum-exp
    assert bwd_lse(lib, dq=None) == NULL
    assert bwd_lse(lib, N=-3) == SHAPE
    assert bwd_lse(lib, d=192) == UNSUPPORTED     # d <= 128 for both backward versions
    assert bwd_lse(lib, dO=A + 8) == ALIGN        # the tensor-core path loads dO with TMA
    assert bwd_lse(lib, dO=A + 8, m=128) == ALIGN  # the CUDA-core path checks the same
    assert bwd_lse(lib, dO=A + 8, dtype=F32) == ALIGN
    assert bwd_lse(lib, N=0, dP=None) == NULL     # empty problem: dP is still zeroed
    # spa_attention_bwd (no lse) checks the same way
    assert lib.spa_attention_bwd(A, A, A, A, A, A, A, A, A, None, 1, 2, 256, 128, 32, 128, 1, BF16,
                                 None) == NULL


def bwd_ws_size(lib, B=1, H=2, N=256, d=128, m=32, dv=128, dtype=BF16):
    n = ctypes.c_size_t(12345)
    st = lib.spa_attention_bwd_workspace_size(B, H, N, d, m, dv, dtype, ctypes.byref(n))
    return st, n.value


@pytest.mark.parametrize("m,d", [(16, 128), (32, 128), (64, 128), (16, 64), (64, 64)])
def test_backward_workspace_size(lib, m, d):
    st, small = bwd_ws_size(lib, N=256, m=m, d=d)
    assert st == OK
    st, big = bwd_ws_size(lib, N=4096, m=m, d=d)
    assert st == OK and big > small
    # at least the forward's operands, the bf16 Qp / Kp tiles, the statistics
    # and the fp32 dQp and dKp accumulators of the problem (N = 4096, B*H = 2)
    rows = 2 * 4096
    KD = 3 * m if m == 16 else m
    assert big >= rows * (2 * 2 * KD + 4 + 2 * 2 * m + 16 + 2 * 4 * m)


def test_backward_workspace_size_rejects(lib):
    assert bwd_ws_size(lib, m=128)[0] == UNSUPPORTED  # outside the fused TMEM plan
    assert bwd_ws_size(lib, d=96)[0] == UNSUPPORTED   # the one-pass finish: d in {64, 128}
    assert bwd_ws_size(lib, dtype=F32)[0] == UNSUPPORTED
    assert bwd_ws_size(lib, dv=96)[0] == UNSUPPORTED
    assert bwd_ws_size(lib, N=0) == (OK, 0)
    assert lib.spa_attention_bwd_workspace_size(1, 1, 8, 64, 32, 64, BF16, None) == NULL


def test_backward_stages_check_their_workspace(lib):
    st, need = bwd_ws_size(lib)
    prep = lambda ws, nb, m=32: lib.spa_attention_bwd_prepare(A, A, A, A, A, A, 1, 2, 256, 128, m,
                                                              128, BF16, ws, nb, None)
    assert prep(None, need) == NULL
    assert prep(A + 16, need) == ALIGN      # 256-byte alignment for the workspace
    assert prep(A, need - 1) == NOMEM
    assert prep(A, need, m=128) == UNSUPPORTED
    app = lambda ws, nb: lib.spa_attention_bwd_apply(A, A, A, 1, 2, 256, 128, 32, 128, 1, BF16,
                                                     ws, nb, None)
    assert app(None, need) == NULL
    assert app(A, 16) == NOMEM
    fin = lambda dP: lib.spa_attention_bwd_finish(A, A, A, A, A, dP, 1, 2, 256, 128, 32, 128, BF16,
                                                  A, need, None)
    assert fin(None) == NULL
    assert fin(A + 4) == ALIGN


def test_self_tests_validate_first(lib):
    """The failure-detection self-tests check their arguments before touching
    the GPU: a time limit outside 1..2000 ms, or an m or a kernel number with
    no kernel to test."""
    assert lib.spa_selftest_wait_timeout(0) == SHAPE
    assert lib.spa_selftest_bwd_wait_timeout(2001) == SHAPE
    assert lib.spa_selftest_proj_wait_timeout(0, 64) == SHAPE
    assert lib.spa_selftest_proj_wait_timeout(3000, 32) == SHAPE
    assert lib.spa_selftest_proj_wait_timeout(50, 48) == UNSUPPORTED
    assert lib.spa_selftest_proj_wait_timeout(50, 16) == UNSUPPORTED
    assert lib.spa_selftest_copy_wait_timeout(0, 0) == SHAPE
    assert lib.spa_selftest_copy_wait_timeout(50, 3) == UNSUPPORTED
    assert lib.spa_selftest_copy_wait_timeout(50, -1) == UNSUPPORTED
