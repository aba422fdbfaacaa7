"""The entry points inside CUDA graphs: every call is stream-ordered (its
workspace from cudaMallocAsync or the caller, its launches on the given
stream), so a captured forward or backward replays with the same results as
the eager calls."""
import pytest
import torch

import spa_inputs as si
from helpers import spa

pytestmark = pytest.mark.gpu


def _inputs(B=2, H=4, N=640, d=128, m=32, dv=128, seed=11):
    w = si.WORKLOADS["C3"].scaled(B=B, H=H, N=N, d=d, m=m, dv=dv)
    q, k, v = (t.cuda() for t in si.make_qkv(w, seed=seed))
    P = si.make_P(w, seed=seed + 1).cuda()
    g = torch.Generator().manual_seed(seed + 2)
    dO = torch.randn((B, H, N, dv), generator=g).to(torch.bfloat16).cuda()
    return q, k, v, P, dO


def test_staged_forward_replays_in_a_graph():
    pkg = spa()
    q, k, v, P, _ = _inputs()
    B, H, N, d = q.shape
    m, dv = P.shape[-1], v.shape[-1]
    ws = torch.empty(pkg.spa_attention_workspace_size(B, H, N, d, m, dv, pkg.SPA_BF16),
                     dtype=torch.uint8, device="cuda")
    out = torch.empty((B, H, N, dv), device="cuda")
    ref = pkg.spa_attention_fwd(q, k, v, P, causal=True)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):  # warm-up outside the capture (function attributes)
        pkg.spa_attention_prepare(q, k, P, dv, ws)
        pkg.spa_attention_apply(v, ws, B, H, N, d, m, causal=True, out=out)
    torch.cuda.current_stream().wait_stream(s)
    out.zero_()
    with torch.cuda.graph(g):
        pkg.spa_attention_prepare(q, k, P, dv, ws)
        pkg.spa_attention_apply(v, ws, B, H, N, d, m, causal=True, out=out)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
    # new inputs in the same buffers: the graph reads them
    q.copy_(torch.flip(q, dims=[2]))
    ref2 = pkg.spa_attention_fwd(q, k, v, P, causal=True)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref2)


def test_allocating_forward_replays_in_a_graph():
    """spa_attention_fwd takes its workspace from the library's own memory
    pool with cudaMallocFromPoolAsync, which a graph records as allocation
    and free nodes on that pool."""
    pkg = spa()
    q, k, v, P, _ = _inputs(m=16)
    ref = pkg.spa_attention_fwd(q, k, v, P, causal=False)
    out = torch.empty_like(ref)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        pkg.spa_attention_fwd(q, k, v, P, causal=False, out=out)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref)


def test_staged_backward_replays_in_a_graph():
    pkg = spa()
    q, k, v, P, dO = _inputs(N=520, seed=21)
    B, H, N, d = q.shape
    m, dv = P.shape[-1], v.shape[-1]
    out, lse = pkg.spa_attention_fwd_lse(q, k, v, P, causal=True)
    ref = pkg.spa_attention_bwd_lse(q, k, v, P, out, lse, dO, causal=True)
    ws = torch.empty(pkg.spa_attention_bwd_workspace_size(B, H, N, d, m, dv, pkg.SPA_BF16),
                     dtype=torch.uint8, device="cuda")
    dq, dk, dvo = (torch.empty_like(t) for t in ref[:3])
    dP = torch.empty_like(ref[3])

    def step():
        pkg.spa_attention_bwd_prepare(q, k, P, out, lse, dO, ws)
        pkg.spa_attention_bwd_apply(v, dO, dvo, ws, B, H, N, d, m, causal=True)
        pkg.spa_attention_bwd_finish(q, k, P, dq, dk, dP, dv, ws)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for t in (dq, dk, dvo, dP):
        t.zero_()
    g.replay()
    torch.cuda.synchronize()
    # dk, dv bit for bit; dq, dP sum reduce-adds whose order may vary
    assert torch.equal(dk, ref[1]) and torch.equal(dvo, ref[2])
    for a, b in ((dq, ref[0]), (dP, ref[3])):
        assert torch.allclose(a, b, rtol=1e-4, atol=1e-5 * float(b.abs().max()))
