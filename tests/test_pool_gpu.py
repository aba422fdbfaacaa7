"""The library's own memory pool: the allocating entry points take their
workspaces from it, it keeps its reservation across synchronisations, and
spa_host_pool_trim hands the unused part back.  Repeated synchronised calls,
a trim in between, and the caller-workspace form all give the same bits."""
import pytest
import torch

import spa_inputs as si
from helpers import spa

pytestmark = pytest.mark.gpu


def test_synchronised_calls_and_trim_give_the_same_bits():
    pkg = spa()
    w = si.WORKLOADS["C3"].scaled(B=1, H=3, N=700)
    q, k, v = (t.cuda() for t in si.make_qkv(w, seed=71))
    P = si.make_P(w, seed=72).cuda()
    ws = torch.empty(pkg.spa_attention_workspace_size(1, 3, 700, w.d, w.m, w.dv, pkg.SPA_BF16),
                     dtype=torch.uint8, device="cuda")
    want = pkg.spa_attention_fwd_ws(q, k, v, P, ws, causal=True)
    torch.cuda.synchronize()
    for i in range(4):
        got = pkg.spa_attention_fwd(q, k, v, P, causal=True)
        torch.cuda.synchronize()
        assert torch.equal(got, want), f"call {i}"
        if i == 1:
            pkg.host_pool_trim()
    out, lse = pkg.spa_attention_fwd_lse(q, k, v, P, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(out, want)
    pkg.host_pool_trim()
    assert pkg.device_error() == 0
