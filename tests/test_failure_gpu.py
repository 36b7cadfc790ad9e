"""Bounded waits.  With STREAMKL_DEBUG_INJECT_STALL the first CTA of the main
kernel waits on a barrier that nothing arrives on; after the wait limit
(20 ms here) the kernel gives up, records the failure in the workspace's
device error word and returns -- no trap, no hang -- and the context stays
usable for the next call, whose results are checked against the oracle."""
import pytest
import torch

from attention_kl_divergence_gb300 import make_g, make_qk, streamkl
from oracle import oracle
from parity import assert_grad, assert_kl

pytestmark = pytest.mark.gpu
DEV = "cuda"
STALL = dict(wait_limit_ns=20_000_000, debug_flags=streamkl.DEBUG_INJECT_STALL)


@pytest.mark.parametrize("Nq,Nk,causal", [(700, 700, True), (4, 9000, False)])
def test_forward_wait_timeout_is_reported(Nq, Nk, causal):
    Q1, K1, Q2, K2 = make_qk(1, 2, Nq, Nk, 128, 0.3, seed=Nq, device=DEV)
    plan = streamkl.fwd_plan(Q1, K1, causal=causal)
    ws = streamkl.new_workspace(plan.workspace_bytes, DEV)
    streamkl.kl_fwd(Q1, K1, Q2, K2, causal=causal, workspace=ws, **STALL)
    torch.cuda.synchronize()
    assert streamkl.workspace_status(ws) != 0       # a wait gave up and said so
    assert streamkl.workspace_status(ws) == 0       # reading clears the word
    KL, _, _ = streamkl.kl_fwd(Q1, K1, Q2, K2, causal=causal, workspace=ws)
    torch.cuda.synchronize()
    assert streamkl.workspace_status(ws) == 0
    rKL, _, _ = oracle.fwd(Q1, K1, Q2, K2, causal=causal)
    assert_kl(KL, rKL)


@pytest.mark.parametrize("mode,Nq,Nk,causal", [
    (streamkl.BWD_FUSED, 600, 600, True),
    (streamkl.BWD_SPLIT, 600, 600, True),
    (streamkl.BWD_KEYSPLIT, 8, 5000, False),
])
def test_backward_wait_timeout_is_reported(mode, Nq, Nk, causal):
    Q1, K1, Q2, K2 = make_qk(1, 2, Nq, Nk, 128, 0.3, seed=11, device=DEV)
    g = make_g(1, 2, Nq, 1.0, device=DEV)
    KL, L1, L2 = streamkl.kl_fwd(Q1, K1, Q2, K2, causal=causal)
    ws = streamkl.new_workspace(256, DEV)
    streamkl.kl_bwd(1, g, Q1, K1, Q2, K2, KL, L1, L2, causal=causal, mode=mode, workspace=ws, **STALL)
    torch.cuda.synchronize()
    assert streamkl.workspace_status(ws) != 0
    dQ, dK = streamkl.kl_bwd(1, g, Q1, K1, Q2, K2, KL, L1, L2, causal=causal, mode=mode, workspace=ws)
    torch.cuda.synchronize()
    assert streamkl.workspace_status(ws) == 0
    rdQ, rdK = oracle.bwd(1, g, Q1, K1, Q2, K2, causal=causal)
    assert_grad(dQ, rdQ, "dQ after a timed-out call")
    assert_grad(dK, rdK, "dK after a timed-out call")
