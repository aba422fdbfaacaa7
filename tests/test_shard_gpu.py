"""The partition of one problem across ranks on the GPU: every share of the
(batch, head) pairs run through spa_attention_fwd_shard, put side by side,
gives the whole problem's forward bit for bit (every pair is computed by the
same kernels on the same data, whichever share it lands in).  The ranks are
run one after the other on one GPU; they never wait on one another."""
import pytest
import torch

import spa_inputs as si
from helpers import spa
from projected_feature_efficient_gb300.shard import gather_pairs, spa_attention_fwd_shard

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("world", [2, 3])
def test_shares_of_one_problem_give_the_whole_forward(world):
    pkg = spa()
    w = si.WORKLOADS["C3"].scaled(B=2, H=3, N=700)
    q, k, v = (t.cuda() for t in si.make_qkv(w, seed=801))
    P = si.make_P(w, seed=802).cuda()
    whole = pkg.spa_attention_fwd(q, k, v, P, causal=True)
    shares = [spa_attention_fwd_shard(q, k, v, P, world, r, causal=True) for r in range(world)]
    torch.cuda.synchronize()
    assert torch.equal(gather_pairs(shares, w.B, w.H), whole)
    assert pkg.device_error() == 0
