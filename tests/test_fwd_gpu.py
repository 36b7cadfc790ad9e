"""Forward parity: libstreamkl (CUDA, through the C ABI) vs the float64 oracle."""
import math

import numpy as np
import pytest
import torch

from attention_kl_divergence_gb300 import WORKLOADS, make_qk, make_workload, streamkl
from oracle import oracle
from parity import assert_kl, assert_lse, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


def run_and_check(Q1, K1, Q2, K2, causal, splits=0):
    KL, L1, L2 = streamkl.kl_fwd(Q1, K1, Q2, K2, causal=causal, num_splits=splits)
    torch.cuda.synchronize()
    rKL, rL1, rL2 = oracle.fwd(Q1, K1, Q2, K2, causal=causal)
    assert_lse(L1, rL1, "LSE1")
    assert_lse(L2, rL2, "LSE2")
    assert_kl(KL, rKL)
    return KL


def test_tiny_workload_full():
    w = WORKLOADS["tiny"]
    Q1, K1, Q2, K2 = make_workload(w, device=DEV)
    KL = run_and_check(Q1, K1, Q2, K2, w.causal)
    assert float(KL.min()) >= -1e-4


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal,splits", [
    (1, 1, 1, 1, 64, False, 0),
    (1, 2, 7, 7, 64, True, 0),
    (2, 3, 129, 129, 128, True, 0),
    (1, 2, 255, 257, 64, False, 0),
    (1, 1, 257, 1000, 128, True, 0),
    (1, 2, 1000, 1000, 128, False, 1),
    (1, 2, 1000, 1000, 128, True, 3),
    (1, 1, 300, 5000, 64, True, 0),
    (2, 1, 513, 700, 128, False, 5),
    (1, 4, 384, 384, 128, True, 1),
    (1, 2, 700, 130, 128, False, 0),  # more query rows than keys
    (1, 1, 300, 1, 64, False, 0),     # a single key: KL = 0, LSE = the one score
])
def test_tile_forward_shapes(B, H, Nq, Nk, d, causal, splits):
    Q1, K1, Q2, K2 = make_qk(B, H, Nq, Nk, d, 0.5, seed=Nq + Nk, device=DEV)
    run_and_check(Q1, K1, Q2, K2, causal, splits)


@pytest.mark.parametrize("B,H,Nq,Nk,d,splits,causal", [
    (1, 2, 1, 1000, 64, 0, False),
    (2, 2, 5, 4099, 128, 0, False),
    (1, 3, 16, 2048, 128, 1, False),
    (4, 2, 16, 130, 64, 7, False),
    (1, 1, 3, 1, 128, 0, False),
    # causal (bottom-right): decode steps and chunked prefill
    (1, 2, 1, 1000, 64, 0, True),
    (2, 2, 5, 4099, 128, 0, True),
    (1, 3, 16, 2048, 128, 1, True),
    (4, 2, 16, 130, 64, 7, True),
    (1, 1, 16, 16, 128, 0, True),     # square: row i sees keys 0..i
    (1, 2, 13, 300, 128, 3, True),
])
def test_decode_forward_shapes(B, H, Nq, Nk, d, splits, causal):
    Q1, K1, Q2, K2 = make_qk(B, H, Nq, Nk, d, 0.3, seed=Nq * 7 + Nk, device=DEV)
    plan = streamkl.fwd_plan(Q1, K1, causal=causal, num_splits=splits)
    assert plan.path == streamkl.PATH_DECODE
    run_and_check(Q1, K1, Q2, K2, causal, splits)


@pytest.mark.parametrize("Nq,Nk,causal", [(300, 300, True), (7, 5000, True), (200, 333, False)])
def test_bnhd_layout_views(Nq, Nk, causal):
    """[B, N, H, d] storage passed as permuted [B, H, N, d] views (strides only)."""
    B, H, d = 2, 3, 128
    base = make_qk(B, H, Nq, Nk, d, 0.4, seed=Nq + Nk, device=DEV)
    views = [t.permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3) for t in base]  # same values, B N H d memory
    assert views[0].stride() == (Nq * H * d, d, H * d, 1)
    KL, L1, L2 = streamkl.kl_fwd(*views, causal=causal)
    torch.cuda.synchronize()
    rKL, rL1, rL2 = oracle.fwd(*base, causal=causal)
    assert_lse(L1, rL1, "LSE1")
    assert_lse(L2, rL2, "LSE2")
    assert_kl(KL, rKL)


def test_identical_inputs_give_zero_kl():
    Q, K, _, _ = make_qk(1, 2, 300, 300, 128, 0.3, seed=5, device=DEV)
    for causal in (False, True):
        KL, L1, L2 = streamkl.kl_fwd(Q, K, Q, K, causal=causal)
        assert float(KL.abs().max()) <= 1e-4
        assert torch.equal(L1, L2)


def test_zero_queries_uniform_rows():
    _, K1, _, K2 = make_qk(1, 1, 260, 260, 64, 0.3, seed=6, device=DEV)
    Z = torch.zeros((1, 1, 260, 64), dtype=torch.bfloat16, device=DEV)
    KL, L1, _ = streamkl.kl_fwd(Z, K1, Z, K2, causal=True)
    n = torch.arange(1, 261, device=DEV, dtype=torch.float64)
    assert float((L1[0, 0].double() - n.log()).abs().max()) <= 1e-5
    assert float(KL.abs().max()) <= 1e-5


def test_large_scores_do_not_overflow():
    """Peaked rows (scores in the hundreds) stay finite and match the oracle."""
    Q1, K1, Q2, K2 = make_qk(1, 1, 200, 600, 64, 0.3, teacher_scale=4.0, seed=9, device=DEV)
    run_and_check(Q1 * 3, K1, Q2 * 3, K2, False)


@pytest.mark.parametrize("causal,splits", [(False, 1), (True, 1), (False, 3)])
def test_scores_rising_along_the_keys(causal, splits):
    """Key norms grow with the key index, so a row's maximum keeps rising far
    above the reference the update holds: unmasked pieces well after a row's
    first must raise it again (and pieces that stay below it must be kept)."""
    Q1, K1, Q2, K2 = make_qk(1, 2, 520, 1500, 128, 0.3, teacher_scale=1.5, seed=21, device=DEV)
    ramp = torch.linspace(0.2, 6.0, 1500, device=DEV).view(1, 1, -1, 1)
    K1 = (K1.float() * ramp).to(torch.bfloat16)
    K2 = (K2.float() * ramp).to(torch.bfloat16)
    run_and_check(Q1, K1, Q2, K2, causal, splits)


def test_plan_uses_splits_when_the_grid_is_small():
    Q1, K1, _, _ = make_qk(1, 1, 256, 32768, 128, 0.3, seed=1, device=DEV)
    assert streamkl.fwd_plan(Q1, K1).num_splits > 1
    Q1, K1, _, _ = make_qk(1, 32, 8192, 8192, 128, 0.3, seed=1, device=DEV)
    assert streamkl.fwd_plan(Q1, K1, causal=True).num_splits == 1


def sample_rows(B, H, Nq, n, seed):
    rng = np.random.default_rng(seed)
    rows = set(rng.integers(0, B * H * Nq, size=n).tolist())
    for bh in (0, B * H - 1):
        for i in (0, 1, 127, 128, Nq - 1):  # first rows, tile edges, last row
            if i < Nq:
                rows.add(bh * Nq + i)
    return np.array(sorted(rows), dtype=np.int64)


def check_sampled(w, rows_n=512):
    Q1, K1, Q2, K2 = make_workload(w, device=DEV)
    KL, L1, L2 = streamkl.kl_fwd(Q1, K1, Q2, K2, causal=w.causal)
    torch.cuda.synchronize()
    rows = sample_rows(w.B, w.H, w.Nq, rows_n, w.seed)
    rKL, rL1, rL2 = oracle.fwd_rows(Q1, K1, Q2, K2, rows, causal=w.causal)
    assert_lse(L1.reshape(-1)[torch.as_tensor(rows, device=DEV)], rL1, "LSE1")
    assert_lse(L2.reshape(-1)[torch.as_tensor(rows, device=DEV)], rL2, "LSE2")
    assert_kl(KL.reshape(-1)[torch.as_tensor(rows, device=DEV)], rKL)
    k = KL.double()
    assert torch.isfinite(k).all() and float(k.min()) >= -1e-3
    return KL


def test_8k_causal_sampled():
    check_sampled(WORKLOADS["8k_causal"])
