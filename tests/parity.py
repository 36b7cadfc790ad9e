"""Tolerances of the CUDA path against the float64 oracle.

KL: |err| <= 1e-3 + 1e-2 |KL| per row; LSE: |err| <= 2e-3 per row.
Gradients: cosine similarity >= 0.999 and max relative error <= 3e-2 over the
elements whose magnitude exceeds 1e-3 of the tensor's largest.
"""
import numpy as np

KL_ATOL, KL_RTOL, LSE_ATOL = 1e-3, 1e-2, 2e-3
GRAD_COS, GRAD_REL, GRAD_FLOOR = 0.999, 3e-2, 1e-3


def to_np(t):
    if hasattr(t, "detach"):
        return t.detach().double().cpu().numpy()
    return np.asarray(t, dtype=np.float64)


def assert_kl(got, want, what="KL"):
    got, want = to_np(got).ravel(), to_np(want).ravel()
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    err = np.abs(got - want)
    bound = KL_ATOL + KL_RTOL * np.abs(want)
    bad = np.flatnonzero(err > bound)
    assert bad.size == 0, (f"{what}: {bad.size}/{got.size} rows out of tolerance; worst row {bad[np.argmax(err[bad])]}"
                           f" got {got[bad[0]]} want {want[bad[0]]} max err {err.max():.3e}")


def assert_lse(got, want, what="LSE"):
    got, want = to_np(got).ravel(), to_np(want).ravel()
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    err = np.abs(got - want)
    assert err.max() <= LSE_ATOL, f"{what}: max |err| {err.max():.3e} at {int(np.argmax(err))}"


def grad_report(got, want):
    got, want = to_np(got).ravel(), to_np(want).ravel()
    cos = float(got @ want / (np.linalg.norm(got) * np.linalg.norm(want) + 1e-300))
    mask = np.abs(want) > GRAD_FLOOR * np.abs(want).max()
    rel = float((np.abs(got - want)[mask] / np.abs(want[mask])).max()) if mask.any() else 0.0
    return cos, rel


def assert_grad(got, want, what="grad"):
    g = to_np(got)
    assert np.all(np.isfinite(g)), f"{what}: non-finite values"
    cos, rel = grad_report(got, want)
    assert cos >= GRAD_COS and rel <= GRAD_REL, f"{what}: cosine {cos:.6f}, max rel err {rel:.3e}"
