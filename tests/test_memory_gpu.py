"""Extra HBM is O(N_Q): the forward needs its three [B, H, N_Q] outputs plus a
workspace of 256 bytes (plus 20 bytes per row and key split when the key
range is split); the backward needs only dQ and dK, and the joint backward
only the four gradients of both sides.  Nothing of size
N_Q x N_K is ever allocated (the pages' ~512 GB at 64K, 32 heads)."""
import pytest
import torch

from attention_kl_divergence_gb300 import make_g, make_qk, streamkl

pytestmark = pytest.mark.gpu
DEV = "cuda"
SLACK = 2 << 20  # caching-allocator rounding


def peak_extra(fn):
    torch.cuda.synchronize()
    base = torch.cuda.memory_allocated()
    torch.cuda.reset_peak_memory_stats()
    out = fn()
    torch.cuda.synchronize()
    return torch.cuda.max_memory_allocated() - base, out


@pytest.mark.parametrize("N", [4096, 16384, 65536, 524288])
def test_extra_memory_is_linear(N):
    B, H, d = 1, 4, 128
    Q1, K1, Q2, K2 = make_qk(B, H, N, N, d, 0.3, seed=1, device=DEV)
    g = make_g(B, H, N, 1.0 / (H * N), device=DEV)
    plan = streamkl.fwd_plan(Q1, K1, causal=True)
    extra_fwd, (KL, L1, L2) = peak_extra(lambda: streamkl.kl_fwd(Q1, K1, Q2, K2, causal=True))
    assert extra_fwd <= 3 * B * H * N * 4 + plan.workspace_bytes + SLACK
    extra_bwd, _ = peak_extra(lambda: streamkl.kl_bwd(1, g, Q1, K1, Q2, K2, KL, L1, L2, causal=True))
    grads = B * H * N * d * 4 * 2
    assert extra_bwd <= grads + 256 + SLACK
    extra_joint, _ = peak_extra(lambda: streamkl.kl_bwd_joint(g, Q1, K1, Q2, K2, KL, L1, L2, causal=True))
    assert extra_joint <= 2 * grads + 256 + SLACK
    # what materialising both distributions in bf16 would need
    assert 2 * B * H * N * N * 2 > 10 * (extra_fwd + extra_bwd) or N < 16384
