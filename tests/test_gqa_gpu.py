"""Keys shared by groups of query heads (K1, K2 with H_kv < H heads): query
head h attends to key head h // (H / H_kv).  The oracle sees the same problem
with every key head repeated for each query head of its group, and the shared
key's gradient is the sum over the group of the per-head gradients."""
import pytest
import torch

from attention_kl_divergence_gb300 import make_qk, streamkl
from oracle import oracle
from parity import assert_grad, assert_kl, assert_lse

pytestmark = pytest.mark.gpu
DEV = "cuda"


def gqa_inputs(B, H, H_kv, Nq, Nk, d, seed):
    Q1, _, Q2, _ = make_qk(B, H, Nq, Nk, d, 0.3, seed=seed, device=DEV)
    _, K1, _, K2 = make_qk(B, H_kv, Nq, Nk, d, 0.3, seed=seed + 1, device=DEV)
    return Q1, K1, Q2, K2


def expand(K, H):
    return K.repeat_interleave(H // K.shape[1], dim=1)


@pytest.mark.parametrize("B,H,H_kv,Nq,Nk,causal", [
    (1, 4, 1, 300, 300, True),      # tile kernel, one key head for all
    (2, 8, 2, 200, 333, False),
    (2, 8, 2, 1, 3000, False),      # decode: the group's 4 heads share one CTA (4 columns)
    (1, 6, 3, 16, 2000, True),      # causal decode, one head per CTA
    (1, 16, 2, 2, 1500, True),      # decode, 8 heads x 2 rows fill the 16 columns, causal
    (2, 8, 2, 3, 777, True),        # decode, 4 heads x 3 rows, ragged key tail
    (1, 8, 2, 5, 1000, False),      # decode, 2 of 4 heads per CTA (10 columns)
    (1, 12, 1, 1, 5000, False),     # decode, 12 heads on one key head
])
@pytest.mark.parametrize("d", [128, 64])
def test_forward_shared_keys(B, H, H_kv, Nq, Nk, causal, d):
    Q1, K1, Q2, K2 = gqa_inputs(B, H, H_kv, Nq, Nk, d, seed=Nq + Nk)
    if Nq <= 16:
        plan = streamkl.fwd_plan(Q1, K1, causal=causal)
        assert plan.path == streamkl.PATH_DECODE
    KL, L1, L2 = streamkl.kl_fwd(Q1, K1, Q2, K2, causal=causal)
    torch.cuda.synchronize()
    rKL, rL1, rL2 = oracle.fwd(Q1, expand(K1, H), Q2, expand(K2, H), causal=causal)
    assert_lse(L1, rL1, "LSE1")
    assert_lse(L2, rL2, "LSE2")
    assert_kl(KL, rKL)


@pytest.mark.parametrize("mode", [streamkl.BWD_FUSED, streamkl.BWD_SPLIT])
@pytest.mark.parametrize("setting", [1, 2])
@pytest.mark.parametrize("B,H,H_kv,N,causal", [(1, 4, 2, 260, True), (2, 6, 1, 130, False)])
def test_backward_shared_keys(B, H, H_kv, N, causal, setting, mode):
    Q1, K1, Q2, K2 = gqa_inputs(B, H, H_kv, N, N, 128, seed=N + H)
    g = torch.rand((B, H, N), device=DEV) + 0.5
    KL, L1, L2 = streamkl.kl_fwd(Q1, K1, Q2, K2, causal=causal)
    dQ, dK = streamkl.kl_bwd(setting, g, Q1, K1, Q2, K2, KL, L1, L2, causal=causal, mode=mode)
    torch.cuda.synchronize()
    assert dK.shape == (B, H_kv, N, 128)
    rdQ, rdK = oracle.bwd(setting, g, Q1, expand(K1, H), Q2, expand(K2, H), causal=causal)
    rdK = torch.as_tensor(rdK).reshape(B, H_kv, H // H_kv, N, 128).sum(2).numpy()
    assert_grad(dQ, rdQ, "dQ (shared keys)")
    assert_grad(dK, rdK, "dK (shared keys)")


def test_decode_shared_keys_strided_views():
    """[B, N, H, d] storage seen as [B, H, N, d] views: a box of several heads
    then spans non-adjacent rows of memory."""
    B, H, H_kv, Nq, Nk, d = 2, 8, 2, 2, 1200, 128
    g = torch.Generator(device="cpu").manual_seed(11)

    def t(h, n):
        return (torch.randn((B, n, h, d), generator=g) * 0.3).to(torch.bfloat16).to(DEV).transpose(1, 2)

    Q1, Q2, K1, K2 = t(H, Nq), t(H, Nq), t(H_kv, Nk), t(H_kv, Nk)
    KL, L1, L2 = streamkl.kl_fwd(Q1, K1, Q2, K2, causal=False)
    torch.cuda.synchronize()
    rKL, rL1, rL2 = oracle.fwd(Q1, expand(K1, H), Q2, expand(K2, H), causal=False)
    assert_lse(L1, rL1, "LSE1")
    assert_lse(L2, rL2, "LSE2")
    assert_kl(KL, rKL)


@pytest.mark.parametrize("splits", [1, 3])
def test_decode_shared_keys_split_counts(splits):
    Q1, K1, Q2, K2 = gqa_inputs(1, 8, 2, 4, 2500, 128, seed=5)
    KL, L1, L2 = streamkl.kl_fwd(Q1, K1, Q2, K2, causal=True, num_splits=splits)
    torch.cuda.synchronize()
    rKL, rL1, rL2 = oracle.fwd(Q1, expand(K1, 8), Q2, expand(K2, 8), causal=True)
    assert_lse(L1, rL1, "LSE1")
    assert_lse(L2, rL2, "LSE2")
    assert_kl(KL, rKL)
