"""A training step captured in a CUDA graph: the forward, both backward
settings and the joint backward through the C ABI, with preallocated
outputs and workspaces, captured once on a side stream and replayed.  Every
entry point only launches asynchronous work on the caller's stream (no
synchronisation, no allocation), so the replays must give what eager calls
give: bitwise for the forward and the deterministic joint backward, within
the parity tolerance for the fused backward (its dQ is added in no fixed
order)."""
import pytest
import torch

from attention_kl_divergence_gb300 import make_g, make_qk, streamkl
from parity import grad_report

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("causal", [True, False])
def test_step_replays_from_a_cuda_graph(causal):
    B, H, N, d = 1, 4, 1000, 128
    Q1, K1, Q2, K2 = make_qk(B, H, N, N, d, 0.3, seed=13, device=DEV)
    g = make_g(B, H, N, 1.0 / (H * N), device=DEV)
    f32 = dict(dtype=torch.float32, device=DEV)
    fwd = tuple(torch.empty((B, H, N), **f32) for _ in range(3))
    g1 = (torch.empty((B, H, N, d), **f32), torch.empty((B, H, N, d), **f32))
    g2 = (torch.empty((B, H, N, d), **f32), torch.empty((B, H, N, d), **f32))
    jo = tuple(torch.empty((B, H, N, d), **f32) for _ in range(4))
    nbytes = max(streamkl.fwd_plan(Q1, K1, causal=causal).workspace_bytes,
                 streamkl.bwd_plan(Q1, K1, 1, causal=causal).workspace_bytes,
                 streamkl.bwd_plan(Q1, K1, 2, causal=causal).workspace_bytes)
    ws = streamkl.new_workspace(nbytes, DEV)

    def step():
        streamkl.kl_fwd(Q1, K1, Q2, K2, causal=causal, workspace=ws, out=fwd)
        streamkl.kl_bwd(1, g, Q1, K1, Q2, K2, *fwd, causal=causal, workspace=ws, out=g1)
        streamkl.kl_bwd(2, g, Q1, K1, Q2, K2, *fwd, causal=causal, workspace=ws, out=g2)
        streamkl.kl_bwd_joint(g, Q1, K1, Q2, K2, *fwd, causal=causal, workspace=ws, out=jo)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # eager, on the stream the graph is captured on
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = [t.clone() for t in (*fwd, *g1, *g2, *jo)]
    for t in (*fwd, *g1, *g2, *jo):
        t.fill_(float("nan"))

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        step()
    for _ in range(2):
        for t in (*fwd, *g1, *g2, *jo):
            t.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert streamkl.workspace_status(ws) == 0
        got = [*fwd, *g1, *g2, *jo]
        for k in range(3):
            assert torch.equal(got[k], eager[k]), "forward output differs on replay"
        for k in range(7, 11):
            assert torch.equal(got[k], eager[k]), "joint backward output differs on replay"
        for k in range(3, 7):
            cos, rel = grad_report(got[k], eager[k])
            assert cos > 0.99999 and rel < 1e-2, (k, cos, rel)
