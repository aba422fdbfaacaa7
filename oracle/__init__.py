"""fp64 CPU oracle for projected-feature softmax attention -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package.  The CUDA library never calls it
and shares no code with it.  The arithmetic lives in ``spa_oracle.c`` (plain
loops in double precision, one step per line of the method as the pages state
it); this module only compiles that file and marshals arrays.

Citations (page titles):
  * "Sparse Projection Attention: A Computationally Efficient Framework for
    Long Sequence Modeling" -- Sec. 3.1.2, Sec. 3.1.3, Algorithm 1.
  * "Projection-Decomposition Attention" (CSDN page) -- Algorithm 2.1 steps 1-3.

Parity status: ``project`` and ``attention`` are pinned by
tests/test_oracle_pins.py.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libspa_oracle.so")
_lock = threading.Lock()
_lib = None

F64, F32, BF16 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, OpenMP, no fast-math)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(path):
    lib = ctypes.CDLL(path)
    vp, dp, i, l = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_long
    lib.orc_project.argtypes = [vp, vp, i, dp, i, i, l, i, i]
    lib.orc_project.restype = i
    lib.orc_attention.argtypes = [vp, vp, vp, vp, i, dp, dp, i, i, l, i, i, i, i, vp, l]
    lib.orc_attention.restype = i
    lib.orc_num_threads.argtypes = []
    lib.orc_num_threads.restype = i
    lib.orc_attention_bwd.argtypes = [vp, vp, vp, vp, vp, i, dp, dp, dp, dp, i, i, l, i, i, i, i]
    lib.orc_attention_bwd.restype = i
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(build())
    return _lib


def num_threads() -> int:
    return int(_load().orc_num_threads())


def _as_raw(t, dt_code=None):
    """torch CPU tensor or numpy array -> (contiguous holder, pointer, type code)."""
    try:
        import torch
        if isinstance(t, torch.Tensor):
            t = t.detach().cpu().contiguous()
            if t.dtype == torch.bfloat16:
                holder = t.view(torch.int16).numpy()
                return holder, holder.ctypes.data, BF16
            if t.dtype == torch.float32:
                holder = t.numpy()
                return holder, holder.ctypes.data, F32
            if t.dtype == torch.float64:
                holder = t.numpy()
                return holder, holder.ctypes.data, F64
            raise TypeError(f"oracle: unsupported dtype {t.dtype}")
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(t)
    if a.dtype == np.float64:
        return a, a.ctypes.data, F64
    if a.dtype == np.float32:
        return a, a.ctypes.data, F32
    raise TypeError(f"oracle: unsupported dtype {a.dtype}")


def project(x, P, _lib=None) -> np.ndarray:
    """x [B,H,N,d], P [H,d,m] (same element type) -> x P_h in fp64, [B,H,N,m]."""
    B, H, N, d = x.shape
    Hp, dp_, m = P.shape
    assert Hp == H and dp_ == d
    hx, px, tx = _as_raw(x)
    hp, pp, tp = _as_raw(P)
    assert tx == tp, "x and P must share one element type"
    out = np.empty((B, H, N, m), dtype=np.float64)
    rc = (_lib or _load()).orc_project(px, pp, tx, out.ctypes.data, B, H, N, d, m)
    if rc:
        raise ValueError(f"orc_project failed ({rc})")
    return out


def attention(q, k, v, P, causal: bool = False, rows=None, return_lse: bool = False,
              _lib=None):
    """fp64 forward O = softmax((qP)(kP)^T / sqrt(m)) v.

    q, k [B,H,N,d]; v [B,H,N,dv]; P [H,d,m]; all of one element type.
    rows: optional 1-D sequence of query indices (applied to every head);
    the result then has shape [B,H,len(rows),dv].
    """
    B, H, N, d = q.shape
    assert tuple(k.shape) == (B, H, N, d)
    dv = v.shape[-1]
    assert tuple(v.shape) == (B, H, N, dv)
    m = P.shape[-1]
    assert tuple(P.shape) == (H, d, m)
    raws = [_as_raw(t) for t in (q, k, v, P)]
    codes = {r[2] for r in raws}
    assert len(codes) == 1, "q, k, v, P must share one element type"
    code = codes.pop()
    if rows is None:
        rows_arr, rows_ptr, nrows = None, None, N
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        rows_ptr, nrows = rows_arr.ctypes.data, int(rows_arr.size)
    out = np.empty((B, H, nrows, dv), dtype=np.float64)
    lse = np.empty((B, H, nrows), dtype=np.float64) if return_lse else None
    rc = (_lib or _load()).orc_attention(raws[0][1], raws[1][1], raws[2][1], raws[3][1], code,
                               out.ctypes.data, lse.ctypes.data if lse is not None else None,
                               B, H, N, d, m, dv, int(bool(causal)), rows_ptr, nrows)
    if rc:
        raise ValueError(f"orc_attention failed ({rc})")
    return (out, lse) if return_lse else out


def compile_variant(src_text: str, out_dir: str):
    """Compile a modified copy of the oracle source and bind it (mutation tests)."""
    os.makedirs(out_dir, exist_ok=True)
    src = os.path.join(out_dir, "variant.c")
    so = os.path.join(out_dir, "libvariant.so")
    with open(src, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", so, src,
                    "-lm"], check=True)
    return _bind(so)


def source() -> str:
    with open(_SRC) as f:
        return f.read()


def attention_bwd(q, k, v, P, dO, causal: bool = False, _lib=None):
    """fp64 gradients of O = softmax((qP)(kP)^T / sqrt(m)) v for the upstream
    gradient dO [B,H,N,dv] (same element type as the inputs).

    Returns (dq [B,H,N,d], dk [B,H,N,d], dv [B,H,N,dv], dP [H,d,m]) as float64.
    """
    B, H, N, d = q.shape
    dv = v.shape[-1]
    m = P.shape[-1]
    assert tuple(k.shape) == (B, H, N, d) and tuple(v.shape) == (B, H, N, dv)
    assert tuple(P.shape) == (H, d, m) and tuple(dO.shape) == (B, H, N, dv)
    raws = [_as_raw(t) for t in (q, k, v, P, dO)]
    codes = {r[2] for r in raws}
    assert len(codes) == 1, "q, k, v, P, dO must share one element type"
    code = codes.pop()
    dq = np.empty((B, H, N, d), dtype=np.float64)
    dk = np.empty((B, H, N, d), dtype=np.float64)
    dvo = np.empty((B, H, N, dv), dtype=np.float64)
    dP = np.empty((H, d, m), dtype=np.float64)
    rc = (_lib or _load()).orc_attention_bwd(
        raws[0][1], raws[1][1], raws[2][1], raws[3][1], raws[4][1], code, dq.ctypes.data,
        dk.ctypes.data, dvo.ctypes.data, dP.ctypes.data, B, H, N, d, m, dv, int(bool(causal)))
    if rc:
        raise ValueError(f"orc_attention_bwd failed ({rc})")
    return dq, dk, dvo, dP


def topk_features(x, k: int) -> np.ndarray:
    """Row-wise Top-k over the last axis ("Scaling Attention via Feature
    Sparsity" notes, Sec. 1): keep the k entries of largest magnitude, zero the
    rest.  Ties at the k-th magnitude keep the lowest indices (a stable sort on
    the negated exact magnitudes).  Returns float64 with exact copies of the
    kept values (signed zeros included)."""
    xs = np.asarray(x.double().numpy() if hasattr(x, "double") else x, dtype=np.float64)
    d = xs.shape[-1]
    flat = xs.reshape(-1, d)
    out = np.zeros_like(flat)
    for r in range(flat.shape[0]):
        order = np.argsort(-np.abs(flat[r]), kind="stable")[:k]
        out[r, order] = flat[r, order]
    return out.reshape(xs.shape)
