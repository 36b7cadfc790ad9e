"""Parity at the full workload sizes, in the launch configuration the
benchmark times: outputs the oracle can compute one row (or one key) at a
time are sampled -- first/last rows, tile edges, random rows -- from a few
heads; the oracle gets exact float64 copies of those heads only.

Workloads (seeded synthetic inputs, see attention_kl_divergence_gb300.inputs):
  decode-shaped backward, B4 H32 N_Q=16 N_K=128K d128, both settings;
  64K causal and non-causal, B1 H32 d128; decode Split-K, B4 H32 d128,
  N_Q in {1, 16}, N_K in {128K, 512K}; 512K causal, B1 H8 d128, teacher x1.5.
A key's dK needs every query row that sees it: dK is sampled among the last
keys of a causal sequence (few rows see them), and for keys spread over one
whole head of 64K causal and 64K non-causal, where the oracle computes the
statistics of all 65536 rows of that head once per call.
"""
import numpy as np
import pytest
import torch

from attention_kl_divergence_gb300 import WORKLOADS, make_g, make_workload, streamkl
from oracle import oracle
from parity import assert_grad, assert_kl, assert_lse, grad_report

pytestmark = pytest.mark.gpu
DEV = "cuda"


def head(t, bh):
    """[1, 1, N, d] view of flat head bh of a [B, H, N, d] tensor."""
    B, H = t.shape[:2]
    return t[bh // H, bh % H][None, None]


def rows_for_head(Nq, n, rng):
    rows = set(rng.integers(0, Nq, size=n).tolist()) | {0, 1, 127, 128, Nq - 129, Nq - 1}
    return np.array(sorted(r for r in rows if 0 <= r < Nq), dtype=np.int64)


KEYS_ACROSS_64K = np.array([0, 1, 127, 128, 129, 4095, 16384, 32767, 32768, 49151, 65536 - 129, 65535],
                           dtype=np.int64)


def check_forward(w, KL, L1, L2, inputs, heads, rows_per_head, seed):
    rng = np.random.default_rng(seed)
    for bh in heads:
        rows = rows_for_head(w.Nq, rows_per_head, rng)
        hq = [head(t, bh) for t in inputs]
        rKL, rL1, rL2 = oracle.fwd_rows(*hq, rows, causal=w.causal)
        idx = torch.as_tensor(rows, device=DEV)
        assert_lse(L1.reshape(-1, w.Nq)[bh][idx], rL1, f"LSE1 head {bh}")
        assert_lse(L2.reshape(-1, w.Nq)[bh][idx], rL2, f"LSE2 head {bh}")
        assert_kl(KL.reshape(-1, w.Nq)[bh][idx], rKL, f"KL head {bh}")


def check_backward(w, setting, dQ, dK, inputs, g, heads, rows_per_head, key_tail, keys_per_head, seed):
    rng = np.random.default_rng(seed + setting)
    gq, rq, gk, rk = [], [], [], []
    for bh in heads:
        hq = [head(t, bh) for t in inputs]
        hg = g.reshape(-1, w.Nq)[bh][None, None]
        rows = rows_for_head(w.Nq, rows_per_head, rng)
        rq.append(oracle.bwd_dq_rows(setting, hg, *hq, rows, causal=w.causal))
        gq.append(dQ.reshape(-1, w.Nq, w.d)[bh][torch.as_tensor(rows, device=DEV)])
        if key_tail:
            keys = np.array(sorted(set(rng.integers(w.Nk - key_tail, w.Nk, size=keys_per_head).tolist())
                                   | {w.Nk - key_tail, w.Nk - 1}), dtype=np.int64)
            rk.append(oracle.bwd_dk_keys(setting, hg, *hq, keys, causal=w.causal))
            gk.append(dK.reshape(-1, w.Nk, w.d)[bh][torch.as_tensor(keys, device=DEV)])
    assert_grad(torch.cat(gq), np.concatenate(rq), f"dQ rows (setting {setting})")
    if gk:
        assert_grad(torch.cat(gk), np.concatenate(rk), f"dK keys (setting {setting})")
    # sum over keys of dK vanishes in both settings (sum_j dS_ij = 0)
    s = dK.double().sum(dim=2).abs().max()
    assert float(s) <= 2e-3 * float(dK.double().abs().sum(dim=2).max())
    assert torch.isfinite(dQ).all() and torch.isfinite(dK).all()


def run_workload(name, settings, heads, rows_per_head=48, key_tail=0, keys_per_head=24):
    w = WORKLOADS[name]
    inputs = make_workload(w, device=DEV)
    KL, L1, L2 = streamkl.kl_fwd(*inputs, causal=w.causal)
    torch.cuda.synchronize()
    assert float(KL.min()) >= -1e-3 and torch.isfinite(KL).all()
    check_forward(w, KL, L1, L2, inputs, heads, rows_per_head, w.seed)
    g = make_g(w.B, w.H, w.Nq, w.g_value, device=DEV)
    for setting in settings:
        dQ, dK = streamkl.kl_bwd(setting, g, *inputs, KL, L1, L2, causal=w.causal)
        torch.cuda.synchronize()
        check_backward(w, setting, dQ, dK, inputs, g, heads, rows_per_head // 2, key_tail, keys_per_head, w.seed)
        del dQ, dK
    return inputs, KL, L1, L2, g


def test_64k_causal_forward_and_both_settings():
    run_workload("64k_causal", (1, 2), heads=(0, 13, 31), key_tail=1024)


def test_64k_causal_dk_of_keys_across_the_sequence():
    """dK of keys spread over one whole 64K causal head, the first keys
    included: their gradient sums over every query row of the sequence, the
    longest accumulation the fused kernel keeps in tensor memory.  The oracle
    computes the statistics of all 65536 rows of the head once (~1e12 flops)."""
    w = WORKLOADS["64k_causal"]
    inputs = make_workload(w, device=DEV)
    KL, L1, L2 = streamkl.kl_fwd(*inputs, causal=w.causal)
    g = make_g(w.B, w.H, w.Nq, w.g_value, device=DEV)
    dQ, dK = streamkl.kl_bwd(1, g, *inputs, KL, L1, L2, causal=w.causal)
    torch.cuda.synchronize()
    bh = 13
    keys = KEYS_ACROSS_64K
    rk = oracle.bwd_dk_keys(1, g.reshape(-1, w.Nq)[bh][None, None], *[head(t, bh) for t in inputs], keys,
                            causal=w.causal)
    gk = dK.reshape(-1, w.Nk, w.d)[bh][torch.as_tensor(keys, device=DEV)]
    assert_grad(gk, rk, "dK of keys across a 64K causal head (setting 1)")


def test_64k_noncausal_dk_of_keys_across_the_sequence_both_settings():
    """dK of keys spread over one whole 64K non-causal head, first and last
    keys included, in both settings: every key's gradient sums over all 65536
    query rows (the longest accumulation the fused kernel keeps in tensor
    memory, with every query tile of the head visiting the key's CTA)."""
    w = WORKLOADS["64k"]
    inputs = make_workload(w, device=DEV)
    KL, L1, L2 = streamkl.kl_fwd(*inputs, causal=w.causal)
    g = make_g(w.B, w.H, w.Nq, w.g_value, device=DEV)
    bh = 21
    hq = [head(t, bh) for t in inputs]
    hg = g.reshape(-1, w.Nq)[bh][None, None]
    keys = torch.as_tensor(KEYS_ACROSS_64K, device=DEV)
    for setting in (1, 2):
        dQ, dK = streamkl.kl_bwd(setting, g, *inputs, KL, L1, L2, causal=w.causal)
        torch.cuda.synchronize()
        gk = dK.reshape(-1, w.Nk, w.d)[bh][keys].cpu()
        del dQ, dK
        rk = oracle.bwd_dk_keys(setting, hg, *hq, KEYS_ACROSS_64K, causal=w.causal)
        assert_grad(gk, rk, f"dK of keys across a 64K non-causal head (setting {setting})")


def test_64k_noncausal_forward_and_both_settings():
    inputs, KL, L1, L2, g = run_workload("64k", (1, 2), heads=(0, 31), rows_per_head=24)
    # fused and split backward agree at full size (the split recomputes independently)
    w = WORKLOADS["64k"]
    a = streamkl.kl_bwd(1, g, *inputs, KL, L1, L2, causal=False, mode=streamkl.BWD_FUSED)
    b = streamkl.kl_bwd(1, g, *inputs, KL, L1, L2, causal=False, mode=streamkl.BWD_SPLIT)
    for x, y in zip(a, b):
        cos, rel = grad_report(x[0, :2], y[0, :2])
        assert cos > 0.99999 and rel < 1e-2, (cos, rel)


@pytest.mark.parametrize("splits", [0, 13])
@pytest.mark.parametrize("name", ["decode_q1_k128k", "decode_q16_k128k", "decode_q1_k512k", "decode_q16_k512k",
                                  "decode_causal_q16_k128k", "decode_gqa_q1_k128k", "decode_q1_k128k_b1"])
def test_decode_split_k_all_rows_of_sampled_heads(name, splits):
    """Automatic splits (one CTA per head once there are enough heads to keep
    HBM busy) and 13 forced splits with the combine step."""
    w = WORKLOADS[name]
    inputs = make_workload(w, device=DEV)
    plan = streamkl.fwd_plan(inputs[0], inputs[1], causal=w.causal, num_splits=splits)
    assert plan.path == streamkl.PATH_DECODE
    if splits:
        assert plan.num_splits == splits and plan.launches == 2
    KL, L1, L2 = streamkl.kl_fwd(*inputs, causal=w.causal, num_splits=splits)
    torch.cuda.synchronize()
    group = w.H // (w.H_kv or w.H)
    nbh = w.B * w.H
    for bh in sorted({0, 37 % nbh, 64 % nbh, nbh - 1}):
        b, h = divmod(bh, w.H)
        q1, k1, q2, k2 = inputs
        hq = [head(q1, bh), k1[b, h // group][None, None], head(q2, bh), k2[b, h // group][None, None]]
        rKL, rL1, rL2 = oracle.fwd(*hq, causal=w.causal)
        assert_lse(L1.reshape(-1, w.Nq)[bh], rL1, f"LSE1 head {bh}")
        assert_lse(L2.reshape(-1, w.Nq)[bh], rL2, f"LSE2 head {bh}")
        assert_kl(KL.reshape(-1, w.Nq)[bh], rKL, f"KL head {bh}")
    assert torch.isfinite(KL).all() and float(KL.min()) >= -1e-3


def test_512k_causal_forward_and_setting2():
    run_workload("512k_causal", (2,), heads=(0, 7), rows_per_head=24, key_tail=256, keys_per_head=12)


def test_64k_causal_d64_forward_and_setting1():
    run_workload("64k_causal_d64", (1,), heads=(0, 31), rows_per_head=32, key_tail=512, keys_per_head=16)


def test_decode_shaped_backward_both_settings():
    """16 query rows against 128K keys: every key tile is its own CTA, and all
    of them add into the same 16 rows of dQ.  dQ is checked on all rows of the
    sampled heads, dK on keys drawn from the whole key range."""
    w = WORKLOADS["decode_bwd_q16_k128k"]
    run_workload(w.name, (1, 2), heads=(0, 77, w.B * w.H - 1), rows_per_head=2 * w.Nq, key_tail=w.Nk,
                 keys_per_head=32)


def test_64k_causal_shared_keys_forward_and_both_settings():
    """64K causal, 32 query heads on 8 key heads: sampled rows of KL, LSE and
    dQ of query heads, and dK of the last keys of a key head, which sums the
    gradients of its 4 query heads -- for both settings."""
    w = WORKLOADS["64k_causal_gqa"]
    inputs = make_workload(w, device=DEV)
    Q1, K1, Q2, K2 = inputs
    group = w.H // w.H_kv
    KL, L1, L2 = streamkl.kl_fwd(*inputs, causal=w.causal)
    torch.cuda.synchronize()

    def views(h):  # query head h with the key head it shares
        return [Q1[0, h][None, None], K1[0, h // group][None, None], Q2[0, h][None, None],
                K2[0, h // group][None, None]]

    rng = np.random.default_rng(w.seed)
    for h in (0, 13, 31):
        rows = rows_for_head(w.Nq, 32, rng)
        rKL, rL1, rL2 = oracle.fwd_rows(*views(h), rows, causal=w.causal)
        idx = torch.as_tensor(rows, device=DEV)
        assert_lse(L1[0, h][idx], rL1, f"LSE1 head {h}")
        assert_lse(L2[0, h][idx], rL2, f"LSE2 head {h}")
        assert_kl(KL[0, h][idx], rKL, f"KL head {h}")
    g = make_g(w.B, w.H, w.Nq, w.g_value, device=DEV)
    for setting, hk in ((1, 3), (2, 6)):
        dQ, dK = streamkl.kl_bwd(setting, g, *inputs, KL, L1, L2, causal=w.causal)
        torch.cuda.synchronize()
        assert dK.shape[1] == w.H_kv
        gq, rq = [], []
        for h in (0, 13, 31):
            rows = rows_for_head(w.Nq, 16, rng)
            rq.append(oracle.bwd_dq_rows(setting, g[0, h][None, None], *views(h), rows, causal=w.causal))
            gq.append(dQ[0, h][torch.as_tensor(rows, device=DEV)])
        assert_grad(torch.cat(gq), np.concatenate(rq), f"dQ rows, shared keys (setting {setting})")
        keys = np.array(sorted(set(rng.integers(w.Nk - 512, w.Nk, size=16).tolist()) | {w.Nk - 512, w.Nk - 1}),
                        dtype=np.int64)
        rk = sum(oracle.bwd_dk_keys(setting, g[0, h][None, None], *views(h), keys, causal=w.causal)
                 for h in range(hk * group, (hk + 1) * group))
        assert_grad(dK[0, hk][torch.as_tensor(keys, device=DEV)], rk,
                    f"dK keys of a shared key head (setting {setting})")
        del dQ, dK
