"""Seeded synthetic inputs for projected-feature softmax attention.

Shared by the oracle tests, the GPU parity tests, the smoke check and the
benchmark.  This module holds no arithmetic of the method itself: it only
draws Q, K, V and the per-head projection P (the random numbers the method
draws are inputs here), rescales rows where a workload asks for it, and casts.

Workloads (sizes as the method's target workloads state them):
  C1  B=1  H=1  N=256     d=64  m=16          dv=64  fp32  non-causal  Q,K iid N(0,1)
  C2  B=4  H=8  N=2048    d=64  m=32          dv=64  bf16  non-causal  Q,K rows norm sqrt(d)
  C3  B=2  H=16 N=8192    d=128 m=32          dv=128 bf16  causal      Q,K rows norm sqrt(d)
  C4  B=1  H=32 N=32768   d=128 m in 16/32/64 dv=128 bf16  non-causal  Q,K iid N(0,1)
  C5  B=1  H=8  N=131072  d=128 m=32          dv=128 bf16  causal      Q,K rows norm sqrt(d)
      plus a control run on the same inputs with m=d=128 and P=I (exact attention).
V is iid N(0,1) everywhere.  P_h has iid N(0, 1/m) entries, one matrix per
head, shared across the batch ("Projection-Decomposition Attention" page,
Algorithm 2.1 step 1; SPA paper, Theorem 1 proof step 1).

Recipe: a CPU torch.Generator seeded with 1000 + workload number draws Q, K, V
in float64 (in that order); rows are rescaled in float64 to L2 norm exactly
sqrt(d) where the workload says so (the "LayerNorm-style" reading of the PDA
page, Sec. 3.2); then everything is cast to the workload dtype.  P is drawn by
a second generator seeded with 2000 + 10 * workload number + index of m in the
workload's m list, as float64 N(0,1) scaled by 1/sqrt(m), then cast.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    number: int
    B: int
    H: int
    N: int
    d: int
    m: int
    dv: int
    dtype: str          # "f32" or "bf16"
    causal: bool
    qk: str             # "iid" or "norm"
    m_list: tuple = field(default=())
    identity_P: bool = False

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def m_index(self) -> int:
        ms = self.m_list or (self.m,)
        return ms.index(self.m) if self.m in ms else 0

    def with_m(self, m: int) -> "Workload":
        return replace(self, m=m)

    def scaled(self, **kw) -> "Workload":
        """Same recipe at other sizes (for parity tests at small shapes)."""
        return replace(self, **kw)


WORKLOADS = {
    "C1": Workload("C1", 1, 1, 1, 256, 64, 16, 64, "f32", False, "iid"),
    "C2": Workload("C2", 2, 4, 8, 2048, 64, 32, 64, "bf16", False, "norm"),
    "C3": Workload("C3", 3, 2, 16, 8192, 128, 32, 128, "bf16", True, "norm"),
    "C4": Workload("C4", 4, 1, 32, 32768, 128, 32, 128, "bf16", False, "iid",
                   m_list=(16, 32, 64)),
    "C5": Workload("C5", 5, 1, 8, 131072, 128, 32, 128, "bf16", True, "norm"),
}
# exact-attention control on the C5 inputs: m = d = 128 and P = I
WORKLOADS["C5ctl"] = replace(WORKLOADS["C5"], name="C5ctl", m=128, identity_P=True)
# decode with the projected key cache: one query per (batch, head) against N
# cached keys (the last causal row), C4-sized heads at batch 8
WORKLOADS["D1"] = Workload("D1", 6, 8, 32, 32768, 128, 32, 128, "bf16", True, "iid")


def _normalise_rows(x: torch.Tensor, target: float) -> torch.Tensor:
    n = torch.linalg.vector_norm(x, dim=-1, keepdim=True)
    return x * (target / n)


def make_qkv(w: Workload, seed: int | None = None, device="cpu"):
    """Q, K [B,H,N,d] and V [B,H,N,dv] in the workload dtype."""
    g = torch.Generator(device="cpu")
    g.manual_seed(1000 + w.number if seed is None else seed)
    shape_qk = (w.B, w.H, w.N, w.d)
    q = torch.randn(shape_qk, generator=g, dtype=torch.float64)
    k = torch.randn(shape_qk, generator=g, dtype=torch.float64)
    v = torch.randn((w.B, w.H, w.N, w.dv), generator=g, dtype=torch.float64)
    if w.qk == "norm":
        q = _normalise_rows(q, math.sqrt(w.d))
        k = _normalise_rows(k, math.sqrt(w.d))
    dt = w.torch_dtype
    return (q.to(dt).to(device), k.to(dt).to(device), v.to(dt).to(device))


def make_sparse_P(w: Workload, s: float, seed: int, device="cpu"):
    """Per-head projection drawn as the sparse random matrix of SPA Definition
    1 (Sec. 2.2): every entry is sqrt(s/m) times +1 with probability 1/(2s),
    -1 with probability 1/(2s), and 0 otherwise (s >= 1).  Drawn in fp64 from a
    seeded uniform, then cast to the workload dtype."""
    assert s >= 1
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    u = torch.rand((w.H, w.d, w.m), generator=g, dtype=torch.float64)
    sign = torch.zeros_like(u)
    sign[u < 0.5 / s] = 1.0
    sign[u >= 1.0 - 0.5 / s] = -1.0
    return (sign * math.sqrt(s / w.m)).to(w.torch_dtype).to(device)


def make_P(w: Workload, seed: int | None = None, device="cpu"):
    """Per-head projection P [H,d,m], entries N(0, 1/m), or the identity."""
    dt = w.torch_dtype
    if w.identity_P:
        assert w.m == w.d
        return torch.eye(w.d, dtype=dt).expand(w.H, w.d, w.d).contiguous().to(device)
    g = torch.Generator(device="cpu")
    g.manual_seed(2000 + 10 * w.number + w.m_index if seed is None else seed)
    P = torch.randn((w.H, w.d, w.m), generator=g, dtype=torch.float64) / math.sqrt(w.m)
    return P.to(dt).to(device)
