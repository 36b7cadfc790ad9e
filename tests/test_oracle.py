"""Pins for the float64 CPU oracle, checked against things other than itself.

Each test names what fixes the expected value: a closed form, an invariant of
the definition, a brute-force restatement written independently of the
oracle's C code, or central finite differences.  Source of the definitions:
"StreamKL: Fast and Memory-Efficient KL Divergence for Boosting Attention
Distillation" (gist.science/paper/2606.20005, technical summary: Problem
Statement; Methodology 1 and 2).
"""
import math
import os

import numpy as np
import pytest

from oracle import oracle

RNG = np.random.default_rng(12345)


def rand_qk(B, H, Nq, Nk, d, rng=RNG, scale=1.0):
    Q1 = rng.standard_normal((B, H, Nq, d)) * scale
    K1 = rng.standard_normal((B, H, Nk, d)) * scale
    Q2 = rng.standard_normal((B, H, Nq, d)) * scale
    K2 = rng.standard_normal((B, H, Nk, d)) * scale
    return Q1, K1, Q2, K2


# --------------------------------------------------------------------------
# Brute force: every score an explicit dot product, softmax normalised by a
# direct sum (no max shift), sums exactly rounded (math.fsum), KL written as
# sum p1 * log(p1 / p2).  Pure Python; independent of the C oracle.
# --------------------------------------------------------------------------

def brute_force(Q1, K1, Q2, K2, causal, scale):
    B, H, Nq, d = Q1.shape
    Nk = K1.shape[2]
    KL = np.zeros((B, H, Nq))
    L1 = np.zeros((B, H, Nq))
    L2 = np.zeros((B, H, Nq))
    for b in range(B):
        for h in range(H):
            for i in range(Nq):
                keys = [j for j in range(Nk) if (not causal) or j - (Nk - Nq) <= i]
                s1 = [scale * math.fsum(Q1[b, h, i, k] * K1[b, h, j, k] for k in range(d)) for j in keys]
                s2 = [scale * math.fsum(Q2[b, h, i, k] * K2[b, h, j, k] for k in range(d)) for j in keys]
                z1 = math.fsum(math.exp(x) for x in s1)
                z2 = math.fsum(math.exp(x) for x in s2)
                p1 = [math.exp(x) / z1 for x in s1]
                p2 = [math.exp(x) / z2 for x in s2]
                KL[b, h, i] = math.fsum(a * math.log(a / c) for a, c in zip(p1, p2))
                L1[b, h, i] = math.log(z1)
                L2[b, h, i] = math.log(z2)
    return KL, L1, L2


@pytest.mark.parametrize("shape,causal", [
    ((1, 1, 5, 5, 3), False),
    ((1, 2, 6, 6, 4), True),
    ((2, 1, 3, 7, 8), True),     # Nq < Nk: bottom-right causal alignment
    ((1, 1, 7, 4, 2), False),    # Nq > Nk is fine without a mask
    ((1, 1, 1, 9, 5), True),     # one query row sees every key
])
def test_oracle_matches_brute_force(shape, causal):
    B, H, Nq, Nk, d = shape
    Q1, K1, Q2, K2 = rand_qk(B, H, Nq, Nk, d)
    scale = 0.7
    got = oracle.fwd(Q1, K1, Q2, K2, causal=causal, scale=scale)
    want = brute_force(Q1, K1, Q2, K2, causal, scale)
    for g, w in zip(got, want):
        np.testing.assert_allclose(g, w, rtol=1e-11, atol=1e-13)


def test_default_scale_is_inverse_sqrt_d():
    Q1, K1, Q2, K2 = rand_qk(1, 1, 4, 6, 9)
    got = oracle.fwd(Q1, K1, Q2, K2)
    want = brute_force(Q1, K1, Q2, K2, False, 1.0 / 3.0)
    for g, w in zip(got, want):
        np.testing.assert_allclose(g, w, rtol=1e-11, atol=1e-13)


# --------------------------------------------------------------------------
# Closed forms
# --------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
def test_zero_queries_give_uniform_rows(causal):
    """Q = 0 -> every score is 0 -> LSE = ln |visible keys|, KL = 0."""
    B, H, N, d = 1, 2, 9, 4
    _, K1, _, K2 = rand_qk(B, H, N, N, d)
    Z = np.zeros((B, H, N, d))
    KL, L1, L2 = oracle.fwd(Z, K1, Z, K2, causal=causal)
    n = np.arange(1, N + 1) if causal else np.full(N, N)
    np.testing.assert_allclose(L1[0, 0], np.log(n), rtol=0, atol=1e-14)
    np.testing.assert_allclose(L2[0, 1], np.log(n), rtol=0, atol=1e-14)
    np.testing.assert_allclose(KL, 0.0, atol=1e-15)


@pytest.mark.parametrize("causal", [False, True])
def test_identical_teacher_and_student(causal):
    Q, K, _, _ = rand_qk(2, 2, 11, 11, 6)
    KL, L1, L2 = oracle.fwd(Q, K, Q, K, causal=causal)
    np.testing.assert_allclose(KL, 0.0, atol=1e-14)
    np.testing.assert_array_equal(L1, L2)


def test_single_key():
    """One key: LSE equals the single score, KL = 0."""
    Q1, K1, Q2, K2 = rand_qk(1, 1, 3, 1, 5)
    KL, L1, L2 = oracle.fwd(Q1, K1, Q2, K2, scale=0.5)
    np.testing.assert_allclose(L1[0, 0], 0.5 * Q1[0, 0] @ K1[0, 0, 0], rtol=1e-14)
    np.testing.assert_allclose(L2[0, 0], 0.5 * Q2[0, 0] @ K2[0, 0, 0], rtol=1e-14)
    np.testing.assert_allclose(KL, 0.0, atol=1e-15)


def test_uniform_teacher_closed_form():
    """Q1 = 0: KL(U || P2) = LSE2 - mean_j S2[j] - ln n."""
    B, H, Nq, Nk, d = 1, 1, 5, 13, 4
    _, K1, Q2, K2 = rand_qk(B, H, Nq, Nk, d)
    Q1 = np.zeros((B, H, Nq, d))
    s = 0.8
    KL, L1, L2 = oracle.fwd(Q1, K1, Q2, K2, scale=s)
    S2 = s * np.einsum("id,jd->ij", Q2[0, 0], K2[0, 0])
    want = L2[0, 0] - S2.mean(axis=1) - math.log(Nk)
    np.testing.assert_allclose(KL[0, 0], want, rtol=1e-12, atol=1e-14)
    # and LSE2 itself against numpy's log-sum-exp of the same scores
    m = S2.max(axis=1)
    np.testing.assert_allclose(L2[0, 0], m + np.log(np.exp(S2 - m[:, None]).sum(axis=1)), rtol=1e-13)


def test_two_keys_bernoulli():
    """Two keys: the rows are Bernoulli(p) vs Bernoulli(q) with
    p = sigmoid(S1[0] - S1[1]); KL = p ln(p/q) + (1-p) ln((1-p)/(1-q))."""
    Q1, K1, Q2, K2 = rand_qk(1, 1, 6, 2, 3)
    s = 1.3
    KL, _, _ = oracle.fwd(Q1, K1, Q2, K2, scale=s)
    for i in range(6):
        a = s * (Q1[0, 0, i] @ (K1[0, 0, 0] - K1[0, 0, 1]))
        b = s * (Q2[0, 0, i] @ (K2[0, 0, 0] - K2[0, 0, 1]))
        p, pc = 1.0 / (1.0 + math.exp(-a)), 1.0 / (1.0 + math.exp(a))  # p and 1 - p
        q, qc = 1.0 / (1.0 + math.exp(-b)), 1.0 / (1.0 + math.exp(b))
        want = p * math.log(p / q) + pc * math.log(pc / qc)
        assert abs(KL[0, 0, i] - want) <= 1e-13 + 1e-12 * abs(want)


# --------------------------------------------------------------------------
# Invariants of the definition
# --------------------------------------------------------------------------

def test_gibbs_nonnegative():
    for causal in (False, True):
        Q1, K1, Q2, K2 = rand_qk(2, 3, 17, 17, 8, scale=2.0)
        KL, _, _ = oracle.fwd(Q1, K1, Q2, K2, causal=causal)
        assert KL.min() >= -1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_common_key_shift(causal):
    """K_t[j] += c for every j shifts S_t[i, :] by scale * <Q_t[i], c>:
    KL unchanged, LSE_t shifted by the same amount."""
    B, H, N, d = 1, 2, 10, 5
    Q1, K1, Q2, K2 = rand_qk(B, H, N, N, d)
    c1, c2 = RNG.standard_normal(d), RNG.standard_normal(d)
    s = 0.6
    KL, L1, L2 = oracle.fwd(Q1, K1, Q2, K2, causal=causal, scale=s)
    KLs, L1s, L2s = oracle.fwd(Q1, K1 + c1, Q2, K2 + c2, causal=causal, scale=s)
    np.testing.assert_allclose(KLs, KL, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(L1s - L1, s * Q1 @ c1, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(L2s - L2, s * Q2 @ c2, rtol=1e-10, atol=1e-12)


def test_key_permutation_noncausal():
    Q1, K1, Q2, K2 = rand_qk(1, 2, 7, 12, 4)
    perm = RNG.permutation(12)
    a = oracle.fwd(Q1, K1, Q2, K2)
    b = oracle.fwd(Q1, K1[:, :, perm], Q2, K2[:, :, perm])
    for x, y in zip(a, b):
        np.testing.assert_allclose(x, y, rtol=1e-12, atol=1e-14)


def test_causal_row_sees_only_its_prefix():
    """Changing key j may only change rows i >= j (Nq == Nk)."""
    Q1, K1, Q2, K2 = rand_qk(1, 1, 12, 12, 4)
    a = oracle.fwd(Q1, K1, Q2, K2, causal=True)
    K2b = K2.copy()
    K2b[0, 0, 7] += 3.0
    b = oracle.fwd(Q1, K1, Q2, K2b, causal=True)
    np.testing.assert_array_equal(a[0][0, 0, :7], b[0][0, 0, :7])
    assert np.all(np.abs(a[0][0, 0, 7:] - b[0][0, 0, 7:]) > 0)


# --------------------------------------------------------------------------
# The online recurrence (Methodology 1) reproduces the definition
# --------------------------------------------------------------------------

@pytest.mark.parametrize("bk", [1, 7, 64, 1000])
@pytest.mark.parametrize("causal", [False, True])
def test_online_recurrence_equals_definition(bk, causal):
    Q1, K1, Q2, K2 = rand_qk(1, 2, 70, 70, 8, scale=1.5)
    a = oracle.fwd(Q1, K1, Q2, K2, causal=causal)
    b = oracle.online_fwd(Q1, K1, Q2, K2, bk, causal=causal)
    for x, y in zip(a, b):
        np.testing.assert_allclose(y, x, rtol=1e-12, atol=1e-13)


def test_row_and_key_selections_match_full():
    Q1, K1, Q2, K2 = rand_qk(2, 2, 9, 11, 4)
    g = RNG.standard_normal((2, 2, 9))
    for causal in (False, True):
        full = oracle.fwd(Q1, K1, Q2, K2, causal=causal)
        rows = np.array([0, 5, 17, 35, 20])
        part = oracle.fwd_rows(Q1, K1, Q2, K2, rows, causal=causal)
        for x, y in zip(full, part):
            np.testing.assert_array_equal(x.reshape(-1)[rows], y)
        for setting in (1, 2):
            dQ, dK = oracle.bwd(setting, g, Q1, K1, Q2, K2, causal=causal)
            np.testing.assert_allclose(oracle.bwd_dq_rows(setting, g, Q1, K1, Q2, K2, rows, causal=causal),
                                       dQ.reshape(-1, 4)[rows], rtol=1e-14, atol=1e-16)
            keys = np.array([0, 10, 11, 43, 30])
            np.testing.assert_allclose(oracle.bwd_dk_keys(setting, g, Q1, K1, Q2, K2, keys, causal=causal),
                                       dK.reshape(-1, 4)[keys], rtol=1e-14, atol=1e-16)


def test_rejects_bad_arguments():
    Q1, K1, Q2, K2 = rand_qk(1, 1, 8, 4, 2)
    with pytest.raises(ValueError):
        oracle.fwd(Q1, K1, Q2, K2, causal=True)  # Nq > Nk with a causal mask
    with pytest.raises(ValueError):
        oracle.bwd(3, np.ones((1, 1, 8)), Q1, K1, Q2, K2)


# --------------------------------------------------------------------------
# Gradients: central finite differences of L = sum_i g[i] KL[i]
# --------------------------------------------------------------------------

def _fd_grad(f, X, h=1e-6):
    G = np.zeros_like(X)
    it = np.nditer(X, flags=["multi_index"])
    for _ in it:
        idx = it.multi_index
        old = X[idx]
        X[idx] = old + h
        fp = f()
        X[idx] = old - h
        fm = f()
        X[idx] = old
        G[idx] = (fp - fm) / (2 * h)
    return G


@pytest.mark.parametrize("setting", [1, 2])
@pytest.mark.parametrize("causal,shape", [(False, (1, 2, 5, 7, 3)), (True, (1, 1, 6, 6, 4)), (True, (2, 1, 3, 5, 2))])
def test_gradients_match_finite_differences(setting, causal, shape):
    """Setting 1 differentiates w.r.t. the student (Q2, K2); KL depends on
    them only through P2, so the finite difference is exactly that gradient.
    Setting 2 does the same for the teacher (Q1, K1) through P1."""
    B, H, Nq, Nk, d = shape
    Q1, K1, Q2, K2 = rand_qk(B, H, Nq, Nk, d)
    g = RNG.uniform(0.5, 2.0, (B, H, Nq))
    s = 0.9

    def loss():
        KL, _, _ = oracle.fwd(Q1, K1, Q2, K2, causal=causal, scale=s)
        return float((g * KL).sum())

    dQ, dK = oracle.bwd(setting, g, Q1, K1, Q2, K2, causal=causal, scale=s)
    Qt, Kt = (Q2, K2) if setting == 1 else (Q1, K1)
    fdQ = _fd_grad(loss, Qt)
    fdK = _fd_grad(loss, Kt)
    np.testing.assert_allclose(dQ, fdQ, rtol=0, atol=1e-6 * np.abs(fdQ).max() + 1e-9)
    np.testing.assert_allclose(dK, fdK, rtol=0, atol=1e-6 * np.abs(fdK).max() + 1e-9)
    assert np.abs(dQ).max() > 1e-3  # not trivially zero


@pytest.mark.parametrize("setting", [1, 2])
@pytest.mark.parametrize("causal", [False, True])
def test_gradient_invariants(setting, causal):
    B, H, N, d = 2, 2, 13, 5
    Q1, K1, Q2, K2 = rand_qk(B, H, N, N, d)
    g = RNG.uniform(0.5, 2.0, (B, H, N))
    # sum_j dS[i, j] = 0 in both settings -> sum over keys of dK vanishes
    _, dK = oracle.bwd(setting, g, Q1, K1, Q2, K2, causal=causal)
    np.testing.assert_allclose(dK.sum(axis=2), 0.0, atol=1e-13)
    # identical teacher and student -> every gradient vanishes
    dQ0, dK0 = oracle.bwd(setting, g, Q1, K1, Q1, K1, causal=causal)
    np.testing.assert_allclose(dQ0, 0.0, atol=1e-15)
    np.testing.assert_allclose(dK0, 0.0, atol=1e-15)
    # all keys equal -> uniform rows of the trainable side's scores -> dQ = 0
    Kc1 = np.broadcast_to(K1[:, :, :1], K1.shape).copy()
    Kc2 = np.broadcast_to(K2[:, :, :1], K2.shape).copy()
    dQc, _ = oracle.bwd(setting, g, Q1, Kc1, Q2, Kc2, causal=causal)
    np.testing.assert_allclose(dQc, 0.0, atol=1e-14)


def test_gradient_scales_linearly_with_g():
    Q1, K1, Q2, K2 = rand_qk(1, 1, 6, 6, 3)
    for setting in (1, 2):
        a = oracle.bwd(setting, np.ones((1, 1, 6)), Q1, K1, Q2, K2, causal=True)
        b = oracle.bwd(setting, 2.5 * np.ones((1, 1, 6)), Q1, K1, Q2, K2, causal=True)
        for x, y in zip(a, b):
            np.testing.assert_allclose(y, 2.5 * x, rtol=1e-13, atol=1e-16)


# --------------------------------------------------------------------------
# The one number the pages print: materialising both distributions at 64K
# context, 32 heads, BF16 takes ~512 GB (Problem Statement).
# --------------------------------------------------------------------------

def test_materialisation_estimate_golden():
    path = os.path.join(os.path.dirname(__file__), "golden", "materialisation_estimate.txt")
    vals = {}
    for line in open(path):
        line = line.split("#", 1)[0].strip()
        if line:
            k, v = line.split("=")
            vals[k.strip()] = float(v)
    n, heads, bytes_per = int(vals["context"]), int(vals["heads"]), int(vals["bytes_per_element"])
    total = 2 * heads * n * n * bytes_per  # two N x N distributions per head
    assert total / 2**30 == vals["expected_gib"]
    assert abs(total / 1e9 - vals["pages_gb_approx"]) / vals["pages_gb_approx"] < 0.08
