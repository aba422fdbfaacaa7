"""ctypes binding of libspa.so: argument marshalling only.

Torch tensors supply data pointers, shapes and the current CUDA stream; the
functions raise ``SpaError`` on any non-zero status.  Names follow the C ABI.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
lib_path = os.path.join(_PKG, "libspa.so")

if not os.path.exists(lib_path):
    raise ImportError(
        f"libspa.so is not built ({lib_path}); build it with "
        "`python -m projected_feature_efficient_gb300.build` (needs nvcc)")

lib = ctypes.CDLL(lib_path)

SPA_F32, SPA_BF16 = 0, 1
SPA_OK, SPA_ERR_TIMEOUT = 0, 8  # spa_status values (include/spa.h)
_vp, _i, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t

lib.spa_status_str.argtypes = [_i]
lib.spa_status_str.restype = ctypes.c_char_p
lib.spa_version.argtypes = []
lib.spa_version.restype = _i
lib.spa_project.argtypes = [_vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp]
lib.spa_project.restype = _i
lib.spa_attention_fwd.argtypes = [_vp] * 5 + [_i] * 8 + [_vp]
lib.spa_attention_fwd.restype = _i
lib.spa_attention_workspace_size.argtypes = [_i] * 7 + [ctypes.POINTER(_sz)]
lib.spa_attention_workspace_size.restype = _i
lib.spa_attention_fwd_ws.argtypes = [_vp] * 5 + [_i] * 8 + [_vp, _sz, _vp]
lib.spa_attention_fwd_ws.restype = _i
lib.spa_attention_fwd_host.argtypes = [_vp] * 5 + [_i] * 8 + [_vp]
lib.spa_attention_fwd_host.restype = _i
lib.spa_attention_prepare.argtypes = [_vp] * 3 + [_i] * 7 + [_vp, _sz, _vp]
lib.spa_attention_prepare.restype = _i
lib.spa_attention_apply.argtypes = [_vp] * 2 + [_i] * 8 + [_vp, _sz, _vp]
lib.spa_attention_apply.restype = _i
lib.spa_attention_fwd_noalloc.argtypes = [_vp] * 5 + [_i] * 8 + [_vp]
lib.spa_attention_fwd_noalloc.restype = _i
lib.spa_device_error.argtypes = [ctypes.POINTER(_i)]
lib.spa_device_error.restype = _i
lib.spa_selftest_wait_timeout.argtypes = [_i]
lib.spa_selftest_wait_timeout.restype = _i
lib.spa_selftest_bwd_wait_timeout.argtypes = [_i]
lib.spa_selftest_bwd_wait_timeout.restype = _i
lib.spa_selftest_proj_wait_timeout.argtypes = [_i, _i]
lib.spa_selftest_proj_wait_timeout.restype = _i
lib.spa_selftest_copy_wait_timeout.argtypes = [_i, _i]
lib.spa_selftest_copy_wait_timeout.restype = _i
lib.spa_attention_bwd.argtypes = [_vp] * 10 + [_i] * 8 + [_vp]
lib.spa_attention_bwd.restype = _i
lib.spa_host_pool_trim.argtypes = []
lib.spa_host_pool_trim.restype = _i
lib.spa_attention_bwd_lse.argtypes = [_vp] * 11 + [_i] * 8 + [_vp]
lib.spa_attention_bwd_lse.restype = _i
lib.spa_attention_fwd_lse.argtypes = [_vp] * 6 + [_i] * 8 + [_vp]
lib.spa_attention_fwd_lse.restype = _i
lib.spa_attention_bwd_workspace_size.argtypes = [_i] * 7 + [ctypes.POINTER(_sz)]
lib.spa_attention_bwd_workspace_size.restype = _i
lib.spa_attention_bwd_prepare.argtypes = [_vp] * 6 + [_i] * 7 + [_vp, _sz, _vp]
lib.spa_attention_bwd_prepare.restype = _i
lib.spa_attention_bwd_apply.argtypes = [_vp] * 3 + [_i] * 8 + [_vp, _sz, _vp]
lib.spa_attention_bwd_apply.restype = _i
lib.spa_attention_bwd_finish.argtypes = [_vp] * 6 + [_i] * 7 + [_vp, _sz, _vp]
lib.spa_attention_bwd_finish.restype = _i
lib.spa_topk_features.argtypes = [_vp, _vp, ctypes.c_longlong, _i, _i, _i, _vp]
lib.spa_topk_features.restype = _i
lib.spa_sfa_attention_fwd.argtypes = [_vp] * 4 + [_i] * 8 + [_vp]
lib.spa_sfa_attention_fwd.restype = _i
lib.spa_kcache_append.argtypes = [_vp] * 4 + [_i] * 8 + [_vp]
lib.spa_kcache_append.restype = _i
lib.spa_attention_decode.argtypes = [_vp] * 6 + [_i] * 8 + [_vp]
lib.spa_attention_decode.restype = _i


class SpaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_str(status)}")


def status_str(status: int) -> str:
    return lib.spa_status_str(int(status)).decode()


def _check(status: int, where: str):
    if status != 0:
        raise SpaError(status, where)


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return SPA_BF16
    if t.dtype == torch.float32:
        return SPA_F32
    raise TypeError(f"unsupported dtype {t.dtype}: use torch.bfloat16 or torch.float32")


def _stream_ptr(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _shapes(q, k, v, P):
    B, H, N, d = q.shape
    dv = v.shape[-1]
    m = P.shape[-1]
    if tuple(k.shape) != (B, H, N, d) or tuple(v.shape) != (B, H, N, dv) or \
            tuple(P.shape) != (H, d, m):
        raise ValueError("shapes: q,k [B,H,N,d]; v [B,H,N,dv]; P [H,d,m]")
    for t in (q, k, v, P):
        if not t.is_contiguous():
            raise ValueError("all tensors must be contiguous")
    if len({t.dtype for t in (q, k, v, P)}) != 1:
        raise TypeError("q, k, v and P must share one dtype")
    return B, H, N, d, m, dv


def spa_project(x, P, out=None, stream=None):
    """x [B,H,N,d] @ P [H,d,m] -> fp32 [B,H,N,m] (device tensors)."""
    import torch
    B, H, N, d = x.shape
    m = P.shape[-1]
    if tuple(P.shape) != (H, d, m) or x.dtype != P.dtype:
        raise ValueError("P must be [H,d,m] with x's dtype")
    if out is None:
        out = torch.empty((B, H, N, m), dtype=torch.float32, device=x.device)
    _check(lib.spa_project(_ptr(x), _ptr(P), _ptr(out), B, H, N, d, m, _dtype_code(x),
                           _stream_ptr(stream)), "spa_project")
    return out


def spa_attention_fwd(q, k, v, P, causal=False, out=None, stream=None):
    """Forward on device tensors; returns fp32 [B,H,N,dv]."""
    import torch
    B, H, N, d, m, dv = _shapes(q, k, v, P)
    if out is None:
        out = torch.empty((B, H, N, dv), dtype=torch.float32, device=q.device)
    _check(lib.spa_attention_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(P), _ptr(out), B, H, N, d, m,
                                 dv, int(bool(causal)), _dtype_code(q), _stream_ptr(stream)),
           "spa_attention_fwd")
    return out


def spa_attention_workspace_size(B, H, N, d, m, dv, dtype_code) -> int:
    n = _sz(0)
    _check(lib.spa_attention_workspace_size(B, H, N, d, m, dv, dtype_code, ctypes.byref(n)),
           "spa_attention_workspace_size")
    return int(n.value)


def spa_attention_fwd_ws(q, k, v, P, workspace, causal=False, out=None, stream=None):
    """Forward with a caller-provided device workspace (uint8 tensor)."""
    import torch
    B, H, N, d, m, dv = _shapes(q, k, v, P)
    if out is None:
        out = torch.empty((B, H, N, dv), dtype=torch.float32, device=q.device)
    _check(lib.spa_attention_fwd_ws(_ptr(q), _ptr(k), _ptr(v), _ptr(P), _ptr(out), B, H, N, d, m,
                                    dv, int(bool(causal)), _dtype_code(q), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(),
                                    _stream_ptr(stream)), "spa_attention_fwd_ws")
    return out


def spa_attention_prepare(q, k, P, dv, workspace, stream=None):
    """Stage 1 of the forward: project q and k into `workspace` (uint8 device tensor)."""
    B, H, N, d = q.shape
    m = P.shape[-1]
    if tuple(k.shape) != (B, H, N, d) or tuple(P.shape) != (H, d, m):
        raise ValueError("shapes: q,k [B,H,N,d]; P [H,d,m]")
    _check(lib.spa_attention_prepare(_ptr(q), _ptr(k), _ptr(P), B, H, N, d, m, dv,
                                     _dtype_code(q), _ptr(workspace),
                                     workspace.numel() * workspace.element_size(),
                                     _stream_ptr(stream)), "spa_attention_prepare")


def spa_attention_apply(v, workspace, B, H, N, d, m, causal=False, out=None, stream=None,
                        dtype_code=None):
    """Stage 2 of the forward from a prepared workspace; returns fp32 [B,H,N,dv]."""
    import torch
    dv = v.shape[-1]
    if out is None:
        out = torch.empty((B, H, N, dv), dtype=torch.float32, device=v.device)
    code = _dtype_code(v) if dtype_code is None else dtype_code
    _check(lib.spa_attention_apply(_ptr(v), _ptr(out), B, H, N, d, m, dv, int(bool(causal)),
                                   code, _ptr(workspace),
                                   workspace.numel() * workspace.element_size(),
                                   _stream_ptr(stream)), "spa_attention_apply")
    return out


def spa_attention_fwd_host(q, k, v, P, causal=False, out=None, stream=None):
    """End-to-end form on host (CPU) tensors: copies in, computes, copies out."""
    import torch
    B, H, N, d, m, dv = _shapes(q, k, v, P)
    if out is None:
        out = torch.empty((B, H, N, dv), dtype=torch.float32)
    _check(lib.spa_attention_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(P), _ptr(out), B, H, N, d,
                                      m, dv, int(bool(causal)), _dtype_code(q),
                                      _stream_ptr(stream)), "spa_attention_fwd_host")
    return out


def spa_attention_bwd(q, k, v, P, out, dO, causal=False, stream=None):
    """Gradients (dq, dk, dv, dP) of spa_attention_fwd for the upstream gradient
    dO (same type as q), given the forward's fp32 output `out`."""
    import torch
    B, H, N, d, m, dv = _shapes(q, k, v, P)
    dev = q.device
    dq = torch.empty((B, H, N, d), dtype=torch.float32, device=dev)
    dk = torch.empty((B, H, N, d), dtype=torch.float32, device=dev)
    dvo = torch.empty((B, H, N, dv), dtype=torch.float32, device=dev)
    dP = torch.empty((H, d, m), dtype=torch.float32, device=dev)
    _check(lib.spa_attention_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(P), _ptr(out), _ptr(dO), _ptr(dq),
                                 _ptr(dk), _ptr(dvo), _ptr(dP), B, H, N, d, m, dv,
                                 int(bool(causal)), _dtype_code(q), _stream_ptr(stream)),
           "spa_attention_bwd")
    return dq, dk, dvo, dP


def spa_attention_fwd_lse(q, k, v, P, causal=False, out=None, lse=None, stream=None):
    """Forward that also returns the row log-sum-exp of the logits: (out, lse),
    out fp32 [B,H,N,dv], lse fp32 [B,H,N]."""
    import torch
    B, H, N, d, m, dv = _shapes(q, k, v, P)
    if out is None:
        out = torch.empty((B, H, N, dv), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    _check(lib.spa_attention_fwd_lse(_ptr(q), _ptr(k), _ptr(v), _ptr(P), _ptr(out), _ptr(lse), B,
                                     H, N, d, m, dv, int(bool(causal)), _dtype_code(q),
                                     _stream_ptr(stream)), "spa_attention_fwd_lse")
    return out, lse


def spa_attention_bwd_lse(q, k, v, P, out, lse, dO, causal=False, grads=None, stream=None):
    """Gradients (dq, dk, dv, dP) given the forward's output and row log-sum-exp
    (from spa_attention_fwd_lse).  `grads` may supply the four fp32 output tensors."""
    import torch
    B, H, N, d, m, dv = _shapes(q, k, v, P)
    dev = q.device
    if grads is None:
        grads = (torch.empty((B, H, N, d), dtype=torch.float32, device=dev),
                 torch.empty((B, H, N, d), dtype=torch.float32, device=dev),
                 torch.empty((B, H, N, dv), dtype=torch.float32, device=dev),
                 torch.empty((H, d, m), dtype=torch.float32, device=dev))
    dq, dk, dvo, dP = grads
    _check(lib.spa_attention_bwd_lse(_ptr(q), _ptr(k), _ptr(v), _ptr(P), _ptr(out), _ptr(lse),
                                     _ptr(dO), _ptr(dq), _ptr(dk), _ptr(dvo), _ptr(dP), B, H, N, d,
                                     m, dv, int(bool(causal)), _dtype_code(q),
                                     _stream_ptr(stream)), "spa_attention_bwd_lse")
    return dq, dk, dvo, dP


def spa_attention_bwd_workspace_size(B, H, N, d, m, dv, dtype_code) -> int:
    n = _sz(0)
    _check(lib.spa_attention_bwd_workspace_size(B, H, N, d, m, dv, dtype_code, ctypes.byref(n)),
           "spa_attention_bwd_workspace_size")
    return int(n.value)


def spa_attention_bwd_prepare(q, k, P, out, lse, dO, workspace, stream=None):
    """Fused backward stage 1 into `workspace` (uint8 device tensor)."""
    B, H, N, d = q.shape
    m, dv = P.shape[-1], dO.shape[-1]
    _check(lib.spa_attention_bwd_prepare(_ptr(q), _ptr(k), _ptr(P), _ptr(out), _ptr(lse), _ptr(dO),
                                         B, H, N, d, m, dv, _dtype_code(q), _ptr(workspace),
                                         workspace.numel() * workspace.element_size(),
                                         _stream_ptr(stream)), "spa_attention_bwd_prepare")


def spa_attention_bwd_apply(v, dO, dv_out, workspace, B, H, N, d, m, causal=False, stream=None):
    """Fused backward stage 2: the tensor-core kernel; writes dv_out (fp32)."""
    dv = v.shape[-1]
    _check(lib.spa_attention_bwd_apply(_ptr(v), _ptr(dO), _ptr(dv_out), B, H, N, d, m, dv,
                                       int(bool(causal)), _dtype_code(v), _ptr(workspace),
                                       workspace.numel() * workspace.element_size(),
                                       _stream_ptr(stream)), "spa_attention_bwd_apply")


def spa_attention_bwd_finish(q, k, P, dq, dk, dP, dv, workspace, stream=None):
    """Fused backward stage 3: dq, dk, dP (fp32) from the workspace; dv = d_v."""
    B, H, N, d = q.shape
    m = P.shape[-1]
    _check(lib.spa_attention_bwd_finish(_ptr(q), _ptr(k), _ptr(P), _ptr(dq), _ptr(dk), _ptr(dP), B,
                                        H, N, d, m, int(dv), _dtype_code(q), _ptr(workspace),
                                        workspace.numel() * workspace.element_size(),
                                        _stream_ptr(stream)), "spa_attention_bwd_finish")


def spa_topk_features(x, k, out=None, stream=None):
    """Row-wise Top-k over the last dimension of x (bf16 or fp32 CUDA tensor)."""
    import torch
    if out is None:
        out = torch.empty_like(x)
    d = x.shape[-1]
    rows = x.numel() // d if d else 0
    _check(lib.spa_topk_features(_ptr(x), _ptr(out), rows, d, int(k), _dtype_code(x),
                                 _stream_ptr(stream)), "spa_topk_features")
    return out


def spa_sfa_attention_fwd(q, k, v, topk, causal=False, out=None, stream=None):
    """softmax(Topk(q) Topk(k)^T / sqrt(d)) v; q, k [B,H,N,d], v [B,H,N,dv]."""
    import torch
    B, H, N, d = q.shape
    dv = v.shape[-1]
    if out is None:
        out = torch.empty((B, H, N, dv), dtype=torch.float32, device=q.device)
    _check(lib.spa_sfa_attention_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, H, N, d, dv,
                                     int(topk), int(bool(causal)), _dtype_code(q),
                                     _stream_ptr(stream)), "spa_sfa_attention_fwd")
    return out


def kcache_new(B, H, cap, m, device="cuda"):
    """Empty projected key cache: (kc [B,H,cap,m] int16 holding fp16 bits,
    kc_mul [B,H,cap] float32)."""
    import torch
    return (torch.zeros((B, H, cap, m), dtype=torch.int16, device=device),
            torch.zeros((B, H, cap), dtype=torch.float32, device=device))


def spa_kcache_append(k, P, kc, kc_mul, pos, stream=None):
    """Project k [B,H,T,d] (bf16) with P [H,d,m] into cache rows pos..pos+T-1."""
    B, H, T, d = k.shape
    m = P.shape[2]
    cap = kc.shape[2]
    _check(lib.spa_kcache_append(_ptr(k), _ptr(P), _ptr(kc), _ptr(kc_mul), B, H, T, d, m, pos,
                                 cap, _dtype_code(k), _stream_ptr(stream)), "spa_kcache_append")


def spa_attention_decode(q, P, kc, kc_mul, v, L, out=None, stream=None):
    """One query per (b, h): q [B,H,d] bf16 against cache rows 0..L-1 with the
    value cache v [B,H,cap,dv] bf16; returns out [B,H,dv] float32."""
    import torch
    B, H, d = q.shape
    m = P.shape[2]
    cap, dv = v.shape[2], v.shape[3]
    if out is None:
        out = torch.empty((B, H, dv), dtype=torch.float32, device=q.device)
    _check(lib.spa_attention_decode(_ptr(q), _ptr(P), _ptr(kc), _ptr(kc_mul), _ptr(v), _ptr(out),
                                    B, H, L, d, m, dv, cap, _dtype_code(q), _stream_ptr(stream)),
           "spa_attention_decode")
    return out


def selftest_wait_timeout(limit_ms: int = 50) -> int:
    """Run the failure-detection self-test; returns the spa_status code
    (SPA_ERR_TIMEOUT when the withheld barrier was detected, as expected)."""
    return int(lib.spa_selftest_wait_timeout(int(limit_ms)))


def selftest_bwd_wait_timeout(limit_ms: int = 50) -> int:
    """The same self-test for the fused backward kernel (returns the status code)."""
    return int(lib.spa_selftest_bwd_wait_timeout(int(limit_ms)))


def selftest_proj_wait_timeout(limit_ms: int = 50, m: int = 64) -> int:
    """The same self-test for the tensor-core projection kernels (m = 32: the
    per-CTA kernel, m = 64: the warp-specialised one); returns the status code."""
    return int(lib.spa_selftest_proj_wait_timeout(int(limit_ms), int(m)))


def selftest_copy_wait_timeout(limit_ms: int = 50, kernel: int = 0) -> int:
    """The same self-test for the kernels that wait on their own copies
    (kernel 0: the backward's statistics, 1: its finish, 2: the Top-k);
    returns the status code."""
    return int(lib.spa_selftest_copy_wait_timeout(int(limit_ms), int(kernel)))


def device_error() -> int:
    """Read and clear the device error word (0 or SPA_ERR_TIMEOUT)."""
    c = _i(0)
    _check(lib.spa_device_error(ctypes.byref(c)), "spa_device_error")
    return int(c.value)


def host_pool_trim() -> None:
    """Release the current device's unused memory kept by the library's pool."""
    _check(lib.spa_host_pool_trim(), "spa_host_pool_trim")
