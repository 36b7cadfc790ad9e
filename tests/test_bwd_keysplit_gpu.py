"""Key-split backward (at most 16 query rows per key head, the decode shape):
every CTA streams a range of 128-key tiles with the query heads of one key head
packed into 16 columns, writes dK for its keys and adds its share of dQ.
Checked against the float64 oracle on every element, both settings."""
import pytest
import torch

from attention_kl_divergence_gb300 import make_qk, streamkl
from oracle import oracle
from parity import assert_grad

pytestmark = pytest.mark.gpu
DEV = "cuda"
KEYSPLIT = streamkl.BWD_KEYSPLIT


def grouped_inputs(B, H, H_kv, Nq, Nk, d, seed):
    Q1, _, Q2, _ = make_qk(B, H, Nq, Nk, d, 0.4, seed=seed, device=DEV)
    _, K1, _, K2 = make_qk(B, H_kv, Nq, Nk, d, 0.4, seed=seed + 1, device=DEV)
    return Q1, K1, Q2, K2


def oracle_grads(setting, g, Q1, K1, Q2, K2, causal):
    """Keys shared by groups of query heads: the oracle sees every key head
    repeated per query head, and a shared key's gradient sums its group."""
    H, H_kv = Q1.shape[1], K1.shape[1]
    rep = H // H_kv
    rdQ, rdK = oracle.bwd(setting, g, Q1, K1.repeat_interleave(rep, 1), Q2, K2.repeat_interleave(rep, 1),
                          causal=causal)
    B, _, Nk, d = K1.shape
    return rdQ, torch.as_tensor(rdK).reshape(B, H_kv, rep, Nk, d).sum(2).numpy()


@pytest.mark.parametrize("setting", [1, 2])
@pytest.mark.parametrize("B,H,H_kv,Nq,Nk,causal,d", [
    (1, 2, 2, 1, 700, False, 128),    # one query row, ragged last key tile
    (2, 4, 4, 16, 3000, False, 128),  # 16 rows fill the columns
    (1, 2, 2, 5, 1000, True, 128),    # causal, bottom-right
    (1, 8, 2, 4, 2500, False, 128),   # 4 query heads share a key head: 16 packed columns
    (1, 4, 1, 3, 999, True, 64),      # d = 64, 4 heads x 3 rows, causal
    (1, 2, 2, 16, 128, False, 128),   # a single key tile
    (2, 2, 2, 7, 130, True, 64),      # two key tiles, the second holds 2 keys
])
def test_keysplit_backward(B, H, H_kv, Nq, Nk, causal, d, setting):
    Q1, K1, Q2, K2 = grouped_inputs(B, H, H_kv, Nq, Nk, d, seed=Nq + Nk + d)
    g = torch.rand((B, H, Nq), device=DEV) + 0.5
    plan = streamkl.bwd_plan(Q1, K1, setting, causal)
    assert plan.path == streamkl.PATH_BWD_KEYSPLIT, "the automatic choice for this shape"
    KL, L1, L2 = streamkl.kl_fwd(Q1, K1, Q2, K2, causal=causal)
    dQ, dK = streamkl.kl_bwd(setting, g, Q1, K1, Q2, K2, KL, L1, L2, causal=causal)
    torch.cuda.synchronize()
    assert dK.shape == K1.shape
    rdQ, rdK = oracle_grads(setting, g, Q1, K1, Q2, K2, causal)
    assert_grad(dQ, rdQ, f"dQ (setting {setting})")
    assert_grad(dK, rdK, f"dK (setting {setting})")


@pytest.mark.parametrize("setting", [1, 2])
def test_keysplit_matches_fused(setting):
    """The key-split and the fused kernels compute the same gradients."""
    Q1, K1, Q2, K2 = grouped_inputs(1, 4, 4, 8, 4096, 128, seed=3)
    g = torch.rand((1, 4, 8), device=DEV) + 0.5
    KL, L1, L2 = streamkl.kl_fwd(Q1, K1, Q2, K2)
    a = streamkl.kl_bwd(setting, g, Q1, K1, Q2, K2, KL, L1, L2, mode=KEYSPLIT)
    b = streamkl.kl_bwd(setting, g, Q1, K1, Q2, K2, KL, L1, L2, mode=streamkl.BWD_FUSED)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        torch.testing.assert_close(x, y, rtol=2e-3, atol=1e-6 * float(y.abs().max()))


@pytest.mark.parametrize("setting", [1, 2])
def test_keysplit_bf16_outputs(setting):
    Q1, K1, Q2, K2 = grouped_inputs(1, 2, 2, 16, 2000, 128, seed=9)
    g = torch.rand((1, 2, 16), device=DEV) + 0.5
    KL, L1, L2 = streamkl.kl_fwd(Q1, K1, Q2, K2)
    plan = streamkl.bwd_plan(Q1, K1, setting, False, grad_dtype=torch.bfloat16)
    assert plan.path == streamkl.PATH_BWD_KEYSPLIT and plan.launches == 3
    dQ, dK = streamkl.kl_bwd(setting, g, Q1, K1, Q2, K2, KL, L1, L2, grad_dtype=torch.bfloat16)
    f32 = streamkl.kl_bwd(setting, g, Q1, K1, Q2, K2, KL, L1, L2)
    torch.cuda.synchronize()
    assert dQ.dtype == torch.bfloat16 and dK.dtype == torch.bfloat16
    rdQ, rdK = oracle_grads(setting, g, Q1, K1, Q2, K2, False)
    assert_grad(dQ.float(), rdQ, "dQ (bf16 output)")
    assert_grad(dK.float(), rdK, "dK (bf16 output)")
    # dK rows have one writer: bit-exact rounding of the float32 result.  dQ adds one share per
    # CTA in no fixed order, so allow one bf16 ulp there.
    torch.testing.assert_close(dK, f32[1].to(torch.bfloat16), rtol=0, atol=0)
    torch.testing.assert_close(dQ.float(), f32[0].to(torch.bfloat16).float(), rtol=2.0 ** -7, atol=1e-30)


def test_keysplit_needs_sixteen_columns():
    """Explicit key-split mode on a shape whose query rows do not fit: UNSUPPORTED."""
    Q1, K1, Q2, K2 = grouped_inputs(1, 2, 2, 17, 500, 128, seed=1)
    with pytest.raises(RuntimeError, match="unsupported"):
        streamkl.bwd_plan(Q1, K1, 1, False, KEYSPLIT)
