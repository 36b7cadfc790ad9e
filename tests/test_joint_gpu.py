"""Joint backward (streamkl_bwd_joint): the gradients of both sides from one
recompute of the scores per kernel, through the C ABI, against the float64
oracle -- the teacher's dQ1, dK1 as in setting 2 and the student's dQ2, dK2
as in setting 1 (Methodology 2, the two settings)."""
import numpy as np
import pytest
import torch

from attention_kl_divergence_gb300 import WORKLOADS, make_g, make_qk, make_workload, streamkl
from oracle import oracle
from parity import assert_grad, grad_report

pytestmark = pytest.mark.gpu
DEV = "cuda"


def joint(Q1, K1, Q2, K2, g, causal, **kw):
    KL, L1, L2 = streamkl.kl_fwd(Q1, K1, Q2, K2, causal=causal)
    out = streamkl.kl_bwd_joint(g, Q1, K1, Q2, K2, KL, L1, L2, causal=causal, **kw)
    torch.cuda.synchronize()
    return out


def check_against_oracle(Q1, K1, Q2, K2, g, causal, grads, what=""):
    dQ1, dK1, dQ2, dK2 = grads
    r2 = oracle.bwd(2, g, Q1, K1, Q2, K2, causal=causal)
    r1 = oracle.bwd(1, g, Q1, K1, Q2, K2, causal=causal)
    assert_grad(dQ1, r2[0], f"dQ1 (teacher){what}")
    assert_grad(dK1, r2[1], f"dK1 (teacher){what}")
    assert_grad(dQ2, r1[0], f"dQ2 (student){what}")
    assert_grad(dK2, r1[1], f"dK2 (student){what}")


@pytest.mark.parametrize("d", [128, 64])
@pytest.mark.parametrize("B,H,Nq,Nk,causal", [
    (1, 2, 256, 256, True),
    (1, 1, 200, 333, False),
    (2, 1, 130, 130, True),
    (1, 2, 257, 1000, True),
    (1, 1, 1, 700, False),
    (1, 1, 64, 64, False),
    (1, 2, 700, 130, False),  # more query rows than keys
    (1, 1, 7, 7, True),
])
def test_joint_matches_oracle(B, H, Nq, Nk, d, causal):
    Q1, K1, Q2, K2 = make_qk(B, H, Nq, Nk, d, 0.4, seed=Nq * 7 + Nk + d, device=DEV)
    g = torch.rand((B, H, Nq), device=DEV) + 0.5
    check_against_oracle(Q1, K1, Q2, K2, g, causal, joint(Q1, K1, Q2, K2, g, causal))


def test_joint_tiny_workload():
    w = WORKLOADS["tiny"]
    Q1, K1, Q2, K2 = make_workload(w, device=DEV)
    g = make_g(w.B, w.H, w.Nq, w.g_value, device=DEV)
    check_against_oracle(Q1, K1, Q2, K2, g, w.causal, joint(Q1, K1, Q2, K2, g, w.causal))


@pytest.mark.parametrize("causal", [True, False])
def test_joint_shared_keys(causal):
    """6 query heads on 2 key heads: dK1 and dK2 sum the gradients of each
    key head's 3 query heads."""
    Q1, K1, Q2, K2 = make_qk(1, 6, 300, 300, 128, 0.3, seed=21, device=DEV, H_kv=2)
    g = torch.rand((1, 6, 300), device=DEV) + 0.5
    grads = joint(Q1, K1, Q2, K2, g, causal)
    assert grads[1].shape == (1, 2, 300, 128) and grads[3].shape == (1, 2, 300, 128)
    rep = [t.repeat_interleave(3, dim=1) for t in (K1, K2)]
    r2 = oracle.bwd(2, g, Q1, rep[0], Q2, rep[1], causal=causal)
    r1 = oracle.bwd(1, g, Q1, rep[0], Q2, rep[1], causal=causal)
    assert_grad(grads[0], r2[0], "dQ1, shared keys")
    assert_grad(grads[2], r1[0], "dQ2, shared keys")
    assert_grad(grads[1], r2[1].reshape(1, 2, 3, 300, 128).sum(2), "dK1, shared keys")
    assert_grad(grads[3], r1[1].reshape(1, 2, 3, 300, 128).sum(2), "dK2, shared keys")


def test_joint_strided_layout_and_bf16_outputs():
    """[B, N, H, d] views (strided heads) and bf16 gradients."""
    B, H, N, d = 1, 3, 200, 128
    base = [t.transpose(1, 2).contiguous().transpose(1, 2) for t in make_qk(B, H, N, N, d, 0.3, seed=3, device=DEV)]
    assert not base[0].is_contiguous()
    g = torch.rand((B, H, N), device=DEV) + 0.5
    grads = joint(*base, g, True, grad_dtype=torch.bfloat16)
    assert all(t.dtype == torch.bfloat16 for t in grads)
    check_against_oracle(*base, g, True, grads, " (bf16 outputs)")


def test_joint_equals_the_single_setting_paths_and_is_deterministic():
    """8K causal, 4 heads: the joint pass gives what the fused single-setting
    passes give, and two joint calls are bitwise equal (no atomics)."""
    Q1, K1, Q2, K2 = make_qk(1, 4, 8192, 8192, 128, 0.3, seed=1, device=DEV)
    g = make_g(1, 4, 8192, 1.0 / (32 * 8192), device=DEV)
    KL, L1, L2 = streamkl.kl_fwd(Q1, K1, Q2, K2, causal=True)
    a = streamkl.kl_bwd_joint(g, Q1, K1, Q2, K2, KL, L1, L2, causal=True)
    b = streamkl.kl_bwd_joint(g, Q1, K1, Q2, K2, KL, L1, L2, causal=True)
    s2 = streamkl.kl_bwd(2, g, Q1, K1, Q2, K2, KL, L1, L2, causal=True)
    s1 = streamkl.kl_bwd(1, g, Q1, K1, Q2, K2, KL, L1, L2, causal=True)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    for x, y in zip(a, (s2[0], s2[1], s1[0], s1[1])):
        cos, rel = grad_report(x, y)
        assert cos > 0.99999 and rel < 1e-2, (cos, rel)
    rows = np.array([0, 1, 127, 128, 4095, 8191], dtype=np.int64)
    hq = [t[0, 2][None, None] for t in (Q1, K1, Q2, K2)]
    hg = g[0, 2][None, None]
    idx = torch.as_tensor(rows, device=DEV)
    assert_grad(a[0][0, 2][idx], oracle.bwd_dq_rows(2, hg, *hq, rows, causal=True), "dQ1 rows at 8K")
    assert_grad(a[2][0, 2][idx], oracle.bwd_dq_rows(1, hg, *hq, rows, causal=True), "dQ2 rows at 8K")


def test_joint_64k_causal_sampled():
    """The headline workload: sampled rows of dQ1, dQ2 and the last keys' dK1,
    dK2 of two heads against the oracle."""
    w = WORKLOADS["64k_causal"]
    inputs = make_workload(w, device=DEV)
    g = make_g(w.B, w.H, w.Nq, w.g_value, device=DEV)
    KL, L1, L2 = streamkl.kl_fwd(*inputs, causal=True)
    dQ1, dK1, dQ2, dK2 = streamkl.kl_bwd_joint(g, *inputs, KL, L1, L2, causal=True)
    torch.cuda.synchronize()
    rng = np.random.default_rng(3)
    for bh in (5, 30):
        hq = [t[0, bh][None, None] for t in inputs]
        hg = g[0, bh][None, None]
        rows = np.array(sorted(set(rng.integers(0, w.Nq, 12).tolist()) | {0, 65535}), dtype=np.int64)
        keys = np.array(sorted(set(rng.integers(w.Nk - 1024, w.Nk, 12).tolist()) | {w.Nk - 1}), dtype=np.int64)
        ri, ki = torch.as_tensor(rows, device=DEV), torch.as_tensor(keys, device=DEV)
        for setting, dQ, dK in ((2, dQ1, dK1), (1, dQ2, dK2)):
            assert_grad(dQ[0, bh][ri], oracle.bwd_dq_rows(setting, hg, *hq, rows, causal=True),
                        f"dQ rows head {bh} (setting {setting})")
            assert_grad(dK[0, bh][ki], oracle.bwd_dk_keys(setting, hg, *hq, keys, causal=True),
                        f"dK keys head {bh} (setting {setting})")


def test_joint_wait_timeout_is_reported():
    Q1, K1, Q2, K2 = make_qk(1, 2, 600, 600, 128, 0.3, seed=11, device=DEV)
    g = make_g(1, 2, 600, 1.0, device=DEV)
    KL, L1, L2 = streamkl.kl_fwd(Q1, K1, Q2, K2, causal=True)
    ws = streamkl.new_workspace(256, DEV)
    streamkl.kl_bwd_joint(g, Q1, K1, Q2, K2, KL, L1, L2, causal=True, workspace=ws, wait_limit_ns=20_000_000,
                          debug_flags=streamkl.DEBUG_INJECT_STALL)
    torch.cuda.synchronize()
    assert streamkl.workspace_status(ws) != 0
    grads = streamkl.kl_bwd_joint(g, Q1, K1, Q2, K2, KL, L1, L2, causal=True, workspace=ws)
    torch.cuda.synchronize()
    assert streamkl.workspace_status(ws) == 0
    check_against_oracle(Q1, K1, Q2, K2, g, True, grads, " after a timed-out call")


def test_joint_64k_noncausal_sampled():
    """64K non-causal: sampled rows of dQ1 and dQ2 against the oracle on two
    heads; every head's dK1 and dK2 sum to zero over the keys and agree with
    the fused single-setting passes on those heads."""
    w = WORKLOADS["64k"]
    inputs = make_workload(w, device=DEV)
    g = make_g(w.B, w.H, w.Nq, w.g_value, device=DEV)
    KL, L1, L2 = streamkl.kl_fwd(*inputs, causal=False)
    dQ1, dK1, dQ2, dK2 = streamkl.kl_bwd_joint(g, *inputs, KL, L1, L2, causal=False)
    torch.cuda.synchronize()
    rng = np.random.default_rng(4)
    for bh in (3, 28):
        hq = [t[0, bh][None, None] for t in inputs]
        hg = g[0, bh][None, None]
        rows = np.array(sorted(set(rng.integers(0, w.Nq, 10).tolist()) | {0, 65535}), dtype=np.int64)
        ri = torch.as_tensor(rows, device=DEV)
        assert_grad(dQ1[0, bh][ri], oracle.bwd_dq_rows(2, hg, *hq, rows, causal=False), f"dQ1 rows head {bh}")
        assert_grad(dQ2[0, bh][ri], oracle.bwd_dq_rows(1, hg, *hq, rows, causal=False), f"dQ2 rows head {bh}")
    for dK in (dK1, dK2):
        s = dK.double().sum(dim=2).abs().max()
        assert float(s) <= 2e-3 * float(dK.double().abs().sum(dim=2).max())
        assert torch.isfinite(dK).all()
    f2 = streamkl.kl_bwd(2, g, *inputs, KL, L1, L2, causal=False)
    f1 = streamkl.kl_bwd(1, g, *inputs, KL, L1, L2, causal=False)
    torch.cuda.synchronize()
    for x, y in ((dK1, f2[1]), (dK2, f1[1]), (dQ1, f2[0]), (dQ2, f1[0])):
        cos, rel = grad_report(x[0, 3:5], y[0, 3:5])
        assert cos > 0.99999 and rel < 1e-2, (cos, rel)


@pytest.mark.parametrize("scale", [0.05, 0.3])
def test_joint_explicit_scale_and_signed_g(scale):
    """A softmax scale other than d^-1/2 and an upstream gradient of both
    signs (and some zeros)."""
    Q1, K1, Q2, K2 = make_qk(1, 2, 300, 420, 128, 0.4, seed=31, device=DEV)
    g = torch.randn((1, 2, 300), device=DEV)
    g[0, 0, ::7] = 0.0
    KL, L1, L2 = streamkl.kl_fwd(Q1, K1, Q2, K2, causal=True, scale=scale)
    grads = streamkl.kl_bwd_joint(g, Q1, K1, Q2, K2, KL, L1, L2, causal=True, scale=scale)
    torch.cuda.synchronize()
    r2 = oracle.bwd(2, g, Q1, K1, Q2, K2, causal=True, scale=scale)
    r1 = oracle.bwd(1, g, Q1, K1, Q2, K2, causal=True, scale=scale)
    for got, want, what in zip(grads, (r2[0], r2[1], r1[0], r1[1]), ("dQ1", "dK1", "dQ2", "dK2")):
        assert_grad(got, want, f"{what} (scale {scale}, signed g)")
