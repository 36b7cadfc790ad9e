"""Backward parity: libstreamkl (CUDA, through the C ABI) vs the float64 oracle,
both settings, fused (atomic dQ) and split (separate dQ / dK kernels) modes."""
import numpy as np
import pytest
import torch

from attention_kl_divergence_gb300 import WORKLOADS, make_g, make_qk, make_workload, streamkl
from oracle import oracle
from parity import assert_grad, assert_kl, assert_lse, grad_report

pytestmark = pytest.mark.gpu
DEV = "cuda"
FUSED, SPLIT = streamkl.BWD_FUSED, streamkl.BWD_SPLIT


def gpu_grads(setting, Q1, K1, Q2, K2, g, causal, mode):
    KL, L1, L2 = streamkl.kl_fwd(Q1, K1, Q2, K2, causal=causal)
    dQ, dK = streamkl.kl_bwd(setting, g, Q1, K1, Q2, K2, KL, L1, L2, causal=causal, mode=mode)
    torch.cuda.synchronize()
    return dQ, dK


def check_full(setting, Q1, K1, Q2, K2, g, causal, mode):
    dQ, dK = gpu_grads(setting, Q1, K1, Q2, K2, g, causal, mode)
    rdQ, rdK = oracle.bwd(setting, g, Q1, K1, Q2, K2, causal=causal)
    assert_grad(dQ, rdQ, f"dQ (setting {setting})")
    assert_grad(dK, rdK, f"dK (setting {setting})")
    return dQ, dK


@pytest.mark.parametrize("setting", [1, 2])
def test_tiny_workload(setting):
    w = WORKLOADS["tiny"]
    Q1, K1, Q2, K2 = make_workload(w, device=DEV)
    g = make_g(w.B, w.H, w.Nq, w.g_value, device=DEV)
    check_full(setting, Q1, K1, Q2, K2, g, w.causal, streamkl.BWD_AUTO)


@pytest.mark.parametrize("mode", [FUSED, SPLIT])
@pytest.mark.parametrize("setting", [1, 2])
@pytest.mark.parametrize("B,H,Nq,Nk,causal", [
    (1, 2, 256, 256, True),
    (1, 1, 200, 333, False),
    (2, 1, 130, 130, True),
    (1, 2, 257, 1000, True),
    (1, 1, 1, 700, False),
    (1, 1, 64, 64, False),
    (1, 2, 700, 130, False),  # more query rows than keys
])
def test_shapes_d128(B, H, Nq, Nk, causal, setting, mode):
    Q1, K1, Q2, K2 = make_qk(B, H, Nq, Nk, 128, 0.4, seed=Nq * 3 + Nk, device=DEV)
    g = torch.rand((B, H, Nq), device=DEV) + 0.5
    check_full(setting, Q1, K1, Q2, K2, g, causal, mode)


@pytest.mark.parametrize("mode", [FUSED, SPLIT])
@pytest.mark.parametrize("setting", [1, 2])
@pytest.mark.parametrize("B,H,Nq,Nk,causal", [(1, 2, 190, 190, True), (2, 1, 100, 300, False), (1, 1, 1, 500, False)])
def test_shapes_d64(B, H, Nq, Nk, causal, setting, mode):
    """d = 64: the fused kernel pads its dQ^T MMA to 128 features with a zero atom."""
    Q1, K1, Q2, K2 = make_qk(B, H, Nq, Nk, 64, 0.5, seed=Nq + 11 * Nk, device=DEV)
    g = torch.rand((B, H, Nq), device=DEV) + 0.5
    expect = streamkl.PATH_BWD_FUSED if mode == FUSED else streamkl.PATH_BWD_SPLIT
    assert streamkl.bwd_plan(Q1, K1, setting, causal, mode).path == expect
    check_full(setting, Q1, K1, Q2, K2, g, causal, mode)


def test_fused_and_split_agree():
    Q1, K1, Q2, K2 = make_qk(1, 4, 384, 384, 128, 0.3, seed=3, device=DEV)
    g = torch.full((1, 4, 384), 1.0 / 1536, device=DEV)
    for setting in (1, 2):
        a = gpu_grads(setting, Q1, K1, Q2, K2, g, True, FUSED)
        b = gpu_grads(setting, Q1, K1, Q2, K2, g, True, SPLIT)
        for x, y in zip(a, b):
            cos, rel = grad_report(x, y)
            assert cos > 0.99999 and rel < 1e-3


@pytest.mark.parametrize("setting", [1, 2])
def test_key_gradient_sums_to_zero(setting):
    """sum_j dS[i, j] = 0 in both settings, so dK summed over keys vanishes."""
    Q1, K1, Q2, K2 = make_qk(1, 2, 512, 512, 128, 0.3, seed=8, device=DEV)
    g = torch.ones((1, 2, 512), device=DEV)
    dQ, dK = gpu_grads(setting, Q1, K1, Q2, K2, g, True, streamkl.BWD_AUTO)
    s = dK.double().sum(dim=2).abs().max()
    assert float(s) <= 2e-3 * float(dK.double().abs().sum(dim=2).max())


def test_identical_inputs_give_zero_gradients():
    Q, K, _, _ = make_qk(1, 1, 300, 300, 128, 0.3, seed=4, device=DEV)
    g = torch.ones((1, 1, 300), device=DEV)
    for setting in (1, 2):
        dQ, dK = gpu_grads(setting, Q, K, Q, K, g, True, streamkl.BWD_AUTO)
        # P1 == P2 exactly in exact arithmetic; what remains is rounding
        assert float(dQ.abs().max()) < 1e-3 and float(dK.abs().max()) < 1e-3


def test_autograd_function():
    Q1, K1, Q2, K2 = make_qk(1, 2, 200, 200, 128, 0.5, seed=2, device=DEV)
    Q2.requires_grad_(True)
    K2.requires_grad_(True)
    KL = streamkl.AttentionKL.apply(Q1, K1, Q2, K2, True, None)
    KL.sum().backward()
    rdQ, rdK = oracle.bwd(1, np.ones((1, 2, 200)), Q1, K1, Q2.detach(), K2.detach(), causal=True)
    assert_grad(Q2.grad.float(), rdQ, "dQ2 (autograd)")
    assert_grad(K2.grad.float(), rdK, "dK2 (autograd)")


def sample_keys(B, H, Nk, seed, n=64):
    rng = np.random.default_rng(seed)
    heads = [0, B * H - 1]
    keys = []
    for bh in heads:
        js = set(rng.integers(Nk - 1024, Nk, size=n // 2).tolist()) | {0, 1, 127, 128, Nk // 2, Nk - 1}
        keys += [bh * Nk + j for j in sorted(js)]
    return np.array(keys, dtype=np.int64)


def sample_rows(B, H, Nq, seed, n=256):
    rng = np.random.default_rng(seed + 1)
    rows = set(rng.integers(0, B * H * Nq, size=n).tolist()) | {0, 127, 128, Nq - 1, B * H * Nq - 1}
    return np.array(sorted(rows), dtype=np.int64)


def check_sampled_grads(w, setting, mode=streamkl.BWD_AUTO):
    Q1, K1, Q2, K2 = make_workload(w, device=DEV)
    g = make_g(w.B, w.H, w.Nq, w.g_value, device=DEV)
    dQ, dK = gpu_grads(setting, Q1, K1, Q2, K2, g, w.causal, mode)
    rows = sample_rows(w.B, w.H, w.Nq, w.seed)
    keys = sample_keys(w.B, w.H, w.Nk, w.seed)
    rdQ = oracle.bwd_dq_rows(setting, g, Q1, K1, Q2, K2, rows, causal=w.causal)
    rdK = oracle.bwd_dk_keys(setting, g, Q1, K1, Q2, K2, keys, causal=w.causal)
    gdQ = dQ.reshape(-1, w.d)[torch.as_tensor(rows, device=DEV)]
    gdK = dK.reshape(-1, w.d)[torch.as_tensor(keys, device=DEV)]
    assert_grad(gdQ, rdQ, f"dQ rows (setting {setting})")
    assert_grad(gdK, rdK, f"dK keys (setting {setting})")
    assert torch.isfinite(dQ).all() and torch.isfinite(dK).all()


def test_8k_causal_setting1_sampled():
    check_sampled_grads(WORKLOADS["8k_causal"], 1)


def test_8k_causal_setting2_sampled():
    check_sampled_grads(WORKLOADS["8k_causal"], 2)


@pytest.mark.parametrize("setting", [1, 2])
@pytest.mark.parametrize("mode", [FUSED, SPLIT])
def test_bnhd_layout_views_backward(setting, mode):
    """Strided [B, N, H, d] inputs give the same gradients (outputs stay [B, H, N, d])."""
    B, H, N, d = 1, 2, 260, 128
    base = make_qk(B, H, N, N, d, 0.4, seed=17, device=DEV)
    views = [t.permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3) for t in base]
    g = torch.rand((B, H, N), device=DEV) + 0.5
    dQ, dK = gpu_grads(setting, *views, g, True, mode)
    rdQ, rdK = oracle.bwd(setting, g, *base, causal=True)
    assert_grad(dQ, rdQ, "dQ (B N H d views)")
    assert_grad(dK, rdK, "dK (B N H d views)")


@pytest.mark.parametrize("setting", [1, 2])
@pytest.mark.parametrize("mode", [FUSED, SPLIT])
def test_bf16_gradient_outputs(setting, mode):
    """grad_dtype=bf16: the same gradients, rounded once to bf16 on output."""
    Q1, K1, Q2, K2 = make_qk(1, 2, 300, 300, 128, 0.4, seed=23, device=DEV)
    g = torch.rand((1, 2, 300), device=DEV) + 0.5
    KL, L1, L2 = streamkl.kl_fwd(Q1, K1, Q2, K2, causal=True)
    plan = streamkl.bwd_plan(Q1, K1, setting, True, mode, grad_dtype=torch.bfloat16)
    dQ, dK = streamkl.kl_bwd(setting, g, Q1, K1, Q2, K2, KL, L1, L2, causal=True, mode=mode,
                             grad_dtype=torch.bfloat16)
    f32 = streamkl.kl_bwd(setting, g, Q1, K1, Q2, K2, KL, L1, L2, causal=True, mode=mode)
    torch.cuda.synchronize()
    assert dQ.dtype == torch.bfloat16 and dK.dtype == torch.bfloat16
    assert plan.launches == (3 if mode == FUSED else 2)
    rdQ, rdK = oracle.bwd(setting, g, Q1, K1, Q2, K2, causal=True)
    assert_grad(dQ.float(), rdQ, "dQ (bf16 output)")
    assert_grad(dK.float(), rdK, "dK (bf16 output)")
    # bf16 output = float32 output rounded to nearest even.  The fused mode adds dQ tiles in
    # no fixed order, so two runs may differ in the last float32 bits: allow one bf16 ulp there.
    torch.testing.assert_close(dK, f32[1].to(torch.bfloat16), rtol=0, atol=0)
    if mode == FUSED:
        torch.testing.assert_close(dQ.float(), f32[0].to(torch.bfloat16).float(), rtol=2.0 ** -7, atol=1e-30)
    else:
        torch.testing.assert_close(dQ, f32[0].to(torch.bfloat16), rtol=0, atol=0)


@pytest.mark.parametrize("mode", [FUSED, SPLIT, streamkl.BWD_KEYSPLIT])
def test_outputs_aligned_to_16_bytes_only(mode):
    """Gradient buffers that start 16 bytes past a 32-byte boundary (the ABI
    asks for 16): rows are written with 16-byte stores there."""
    Nq = 8 if mode == streamkl.BWD_KEYSPLIT else 200
    Q1, K1, Q2, K2 = make_qk(1, 2, Nq, 700, 128, 0.4, seed=31, device=DEV)
    g = torch.rand((1, 2, Nq), device=DEV) + 0.5
    KL, L1, L2 = streamkl.kl_fwd(Q1, K1, Q2, K2)

    def offset_empty(shape):
        n = int(np.prod(shape))
        buf = torch.empty(n + 4, dtype=torch.float32, device=DEV)
        view = buf[4:].view(shape)
        assert view.data_ptr() % 32 == 16
        return view

    out = (offset_empty(Q1.shape), offset_empty(K1.shape))
    dQ, dK = streamkl.kl_bwd(1, g, Q1, K1, Q2, K2, KL, L1, L2, mode=mode, out=out)
    ref = streamkl.kl_bwd(1, g, Q1, K1, Q2, K2, KL, L1, L2, mode=mode)
    torch.cuda.synchronize()
    rdQ, rdK = oracle.bwd(1, g, Q1, K1, Q2, K2, causal=False)
    assert_grad(dQ, rdQ, "dQ (16-byte aligned output)")
    assert_grad(dK, rdK, "dK (16-byte aligned output)")
    torch.testing.assert_close(dK, ref[1], rtol=0, atol=0)


MODES = {"fused": FUSED, "split": SPLIT, "keysplit": streamkl.BWD_KEYSPLIT}


@pytest.mark.parametrize("mode", sorted(MODES))
@pytest.mark.parametrize("setting", [1, 2])
def test_signed_and_zero_upstream_gradient(setting, mode):
    """g is any real per-row weight: mixed signs and exact zeros (rows that
    contribute nothing) in every backward path."""
    Nq, Nk, causal = (16, 900, False) if mode == "keysplit" else (200, 333, True)
    Q1, K1, Q2, K2 = make_qk(1, 2, Nq, Nk, 128, 0.4, seed=5 * Nq + setting, device=DEV)
    gen = torch.Generator(device="cpu").manual_seed(17 + setting)
    g = torch.randn((1, 2, Nq), generator=gen)
    g[:, :, ::5] = 0.0
    g = g.to(DEV)
    assert streamkl.bwd_plan(Q1, K1, setting, causal, MODES[mode]).path == {
        "fused": streamkl.PATH_BWD_FUSED, "split": streamkl.PATH_BWD_SPLIT,
        "keysplit": streamkl.PATH_BWD_KEYSPLIT}[mode]
    check_full(setting, Q1, K1, Q2, K2, g, causal, MODES[mode])


@pytest.mark.parametrize("mode", sorted(MODES))
@pytest.mark.parametrize("scale", [0.05, 0.3])
def test_softmax_scale_other_than_the_default(scale, mode):
    """An explicit softmax scale (not d^-1/2) reaches the forward and both
    gradients, which carry it through S = scale Q K^T."""
    Nq, Nk, causal = (16, 700, False) if mode == "keysplit" else (150, 300, True)
    Q1, K1, Q2, K2 = make_qk(1, 2, Nq, Nk, 64, 0.5, seed=int(scale * 100) + Nq, device=DEV)
    KL, L1, L2 = streamkl.kl_fwd(Q1, K1, Q2, K2, causal=causal, scale=scale)
    torch.cuda.synchronize()
    rKL, rL1, rL2 = oracle.fwd(Q1, K1, Q2, K2, causal=causal, scale=scale)
    assert_lse(L1, rL1, "LSE1")
    assert_lse(L2, rL2, "LSE2")
    assert_kl(KL, rKL)
    g = torch.rand((1, 2, Nq), device=DEV) + 0.5
    for setting in (1, 2):
        dQ, dK = streamkl.kl_bwd(setting, g, Q1, K1, Q2, K2, KL, L1, L2, causal=causal, scale=scale,
                                 mode=MODES[mode])
        torch.cuda.synchronize()
        rdQ, rdK = oracle.bwd(setting, g, Q1, K1, Q2, K2, causal=causal, scale=scale)
        assert_grad(dQ, rdQ, f"dQ (setting {setting}, scale {scale})")
        assert_grad(dK, rdK, f"dK (setting {setting}, scale {scale})")


def test_binding_rejects_mis_shaped_buffers():
    """Outputs, per-row inputs and the workspace are checked against the
    problem's shapes before anything launches (a short buffer would be written
    past its end)."""
    Q1, K1, Q2, K2 = make_qk(1, 4, 130, 200, 64, 0.4, seed=3, device=DEV, H_kv=2)
    KL, L1, L2 = streamkl.kl_fwd(Q1, K1, Q2, K2)
    g = torch.ones((1, 4, 130), device=DEV)
    f32 = dict(dtype=torch.float32, device=DEV)
    with pytest.raises(ValueError):
        streamkl.kl_fwd(Q1, K1, Q2, K2, out=(torch.empty((1, 4, 129), **f32), L1, L2))
    with pytest.raises(ValueError):
        streamkl.kl_fwd(Q1, K1, Q2, K2, out=(KL, L1, torch.empty((1, 4, 130), dtype=torch.float16, device=DEV)))
    with pytest.raises(ValueError):
        streamkl.kl_fwd(Q1, K1, Q2, K2, workspace=torch.zeros(1 << 20, dtype=torch.float32, device=DEV))
    with pytest.raises(ValueError):  # smaller than the plan asks for
        streamkl.kl_fwd(Q1, K1, Q2, K2, workspace=torch.zeros(16, dtype=torch.uint8, device=DEV))
    with pytest.raises(ValueError):  # dK has the key heads (2), not the query heads (4)
        streamkl.kl_bwd(1, g, Q1, K1, Q2, K2, KL, L1, L2,
                        out=(torch.empty((1, 4, 130, 64), **f32), torch.empty((1, 1, 200, 64), **f32)))
    with pytest.raises(ValueError):
        streamkl.kl_bwd(1, g[:, :, :100], Q1, K1, Q2, K2, KL, L1, L2)
    with pytest.raises(ValueError):
        streamkl.kl_bwd(1, g.cpu(), Q1, K1, Q2, K2, KL, L1, L2)
    dQ, dK = streamkl.kl_bwd(1, g, Q1, K1, Q2, K2, KL, L1, L2,
                             out=(torch.empty((1, 4, 130, 64), **f32), torch.empty((1, 2, 200, 64), **f32)))
    torch.cuda.synchronize()
    assert torch.isfinite(dQ).all() and torch.isfinite(dK).all()


def test_autograd_teacher_side():
    Q1, K1, Q2, K2 = make_qk(1, 2, 200, 330, 128, 0.5, seed=3, device=DEV)
    Q1.requires_grad_(True)
    K1.requires_grad_(True)
    KL = streamkl.AttentionKL.apply(Q1, K1, Q2, K2, True, None)
    KL.sum().backward()
    assert Q2.grad is None and K2.grad is None
    rdQ, rdK = oracle.bwd(2, np.ones((1, 2, 200)), Q1.detach(), K1.detach(), Q2, K2, causal=True)
    assert_grad(Q1.grad.float(), rdQ, "dQ1 (autograd)")
    assert_grad(K1.grad.float(), rdK, "dK1 (autograd)")


def test_autograd_both_sides():
    """Teacher and student both require grad: the joint backward gives each
    side its own setting's gradient (setting 1 holds P1 fixed, setting 2 holds
    P2 fixed) from one recompute per kernel."""
    Q1, K1, Q2, K2 = make_qk(1, 2, 180, 250, 64, 0.5, seed=4, device=DEV)
    for t in (Q1, K1, Q2, K2):
        t.requires_grad_(True)
    KL = streamkl.AttentionKL.apply(Q1, K1, Q2, K2, False, None)
    g = torch.rand((1, 2, 180), device=DEV) + 0.5
    (KL * g).sum().backward()
    det = [t.detach() for t in (Q1, K1, Q2, K2)]
    r1 = oracle.bwd(1, g, *det, causal=False)
    r2 = oracle.bwd(2, g, *det, causal=False)
    assert_grad(Q2.grad.float(), r1[0], "dQ2 (both sides)")
    assert_grad(K2.grad.float(), r1[1], "dK2 (both sides)")
    assert_grad(Q1.grad.float(), r2[0], "dQ1 (both sides)")
    assert_grad(K1.grad.float(), r2[1], "dK1 (both sides)")


def test_autograd_both_sides_decode_shape():
    """Both sides trainable with 8 query rows against 3000 keys: the two
    key-split passes serve it (the joint pass is for the fused shapes)."""
    Q1, K1, Q2, K2 = make_qk(1, 2, 8, 3000, 128, 0.5, seed=6, device=DEV)
    assert streamkl.bwd_plan(Q1, K1, 1).path == streamkl.PATH_BWD_KEYSPLIT
    for t in (Q1, K1, Q2, K2):
        t.requires_grad_(True)
    KL = streamkl.AttentionKL.apply(Q1, K1, Q2, K2, False, None)
    g = torch.rand((1, 2, 8), device=DEV) + 0.5
    (KL * g).sum().backward()
    det = [t.detach() for t in (Q1, K1, Q2, K2)]
    r1 = oracle.bwd(1, g, *det, causal=False)
    r2 = oracle.bwd(2, g, *det, causal=False)
    assert_grad(Q2.grad.float(), r1[0], "dQ2 (both sides, decode shape)")
    assert_grad(K2.grad.float(), r1[1], "dK2 (both sides, decode shape)")
    assert_grad(Q1.grad.float(), r2[0], "dQ1 (both sides, decode shape)")
    assert_grad(K1.grad.float(), r2[1], "dK1 (both sides, decode shape)")
