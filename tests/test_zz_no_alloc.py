"""The allocation-free forward (streamkl_fwd_noalloc) through the C ABI.

Some callers cannot allocate device memory at all -- a host program or
plugin that only receives tensor pointers from a runtime owning all device
memory, or a caller whose memory plan is frozen.  For them the library keeps
its forward scratch in a fixed device array of its own.  These tests check,
on two calls in a row, that this entry point gives what the float64 oracle
gives and what the workspace-based streamkl_fwd gives (within the parity
tolerances); that a shape needing more scratch than the fixed array holds is
refused; and that a bounded wait that gives up inside it is reported by
streamkl_noalloc_status.  The file sorts last so that a stop-at-first-failure
run has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from attention_kl_divergence_gb300 import make_qk, streamkl
from oracle import oracle
from parity import assert_kl, assert_lse

pytestmark = pytest.mark.gpu
DEV = "cuda"


def noalloc_fwd(Q1, K1, Q2, K2, causal, out, num_splits=0, wait_limit_ns=0, debug_flags=0):
    lib = streamkl.load()
    shape = streamkl.make_shape(Q1, K1)
    opts = streamkl.Options(num_splits, 0, wait_limit_ns, debug_flags, 0)
    P = ctypes.c_void_p
    KL, L1, L2 = out
    return lib.streamkl_fwd_noalloc(ctypes.byref(shape), P(Q1.data_ptr()), P(K1.data_ptr()), P(Q2.data_ptr()),
                                    P(K2.data_ptr()), ctypes.c_float(0.0), int(causal), P(KL.data_ptr()),
                                    P(L1.data_ptr()), P(L2.data_ptr()), ctypes.byref(opts),
                                    P(torch.cuda.current_stream().cuda_stream))


def noalloc_status():
    """streamkl_noalloc_status through the C ABI: (status, error word)."""
    word = ctypes.c_uint32(0)
    rc = streamkl.load().streamkl_noalloc_status(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream),
                                                  ctypes.byref(word))
    return rc, int(word.value)


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal,splits", [
    (4, 8, 1, 20000, 128, False, 0),    # decode kernel, automatic key splits
    (2, 4, 16, 9000, 64, False, 0),     # decode kernel, 16 query rows
    (1, 2, 300, 5000, 128, True, 3),    # tile kernel with forced splits + combine
])
def test_noalloc_matches_oracle_and_workspace_forward_twice(B, H, Nq, Nk, d, causal, splits):
    Q1, K1, Q2, K2 = make_qk(B, H, Nq, Nk, d, 0.3, seed=Nq + Nk, device=DEV)
    plan = streamkl.fwd_plan(Q1, K1, causal=causal, num_splits=splits)
    assert plan.num_splits > 1  # the scratch really holds partial states here
    ref = streamkl.kl_fwd(Q1, K1, Q2, K2, causal=causal, num_splits=splits)
    rKL, rL1, rL2 = oracle.fwd(Q1, K1, Q2, K2, causal=causal)
    out = tuple(torch.empty((B, H, Nq), dtype=torch.float32, device=DEV) for _ in range(3))
    for _ in range(2):
        for t in out:
            t.fill_(float("nan"))
        assert noalloc_fwd(Q1, K1, Q2, K2, causal, out, splits) == streamkl.OK
        torch.cuda.synchronize()
        assert noalloc_status() == (streamkl.OK, 0)
        assert_kl(out[0], rKL, "KL (noalloc vs oracle)")
        assert_lse(out[1], rL1, "LSE1 (noalloc vs oracle)")
        assert_lse(out[2], rL2, "LSE2 (noalloc vs oracle)")
        assert_kl(out[0], ref[0], "KL (noalloc vs workspace entry point)")
        assert_lse(out[1], ref[1], "LSE1 (noalloc vs workspace entry point)")
        assert_lse(out[2], ref[2], "LSE2 (noalloc vs workspace entry point)")


def test_noalloc_refuses_shapes_beyond_its_scratch():
    # 8192 rows x 64 splits x 20 bytes > 8 MiB of built-in scratch
    Q1, K1, Q2, K2 = make_qk(1, 8, 1024, 8192, 128, 0.3, seed=1, device=DEV)
    plan = streamkl.fwd_plan(Q1, K1, num_splits=64)
    assert plan.workspace_bytes > (8 << 20)
    out = tuple(torch.full((1, 8, 1024), 7.0, device=DEV) for _ in range(3))
    assert noalloc_fwd(Q1, K1, Q2, K2, False, out, 64) == streamkl.ERR_WORKSPACE
    torch.cuda.synchronize()
    assert all(bool((t == 7.0).all()) for t in out)  # nothing was launched


def test_noalloc_wait_timeout_is_reported_by_its_status_query():
    """The first CTA's MMA issuer waits on a barrier nothing arrives on; after
    20 ms it gives up.  The call itself returns OK (it only covers validation
    and launch); streamkl_noalloc_status reports the timeout and clears the
    word; the stalled CTA's rows are NaN; the next call is correct again."""
    Q1, K1, Q2, K2 = make_qk(1, 2, 700, 700, 128, 0.3, seed=5, device=DEV)
    out = tuple(torch.zeros((1, 2, 700), dtype=torch.float32, device=DEV) for _ in range(3))
    rc = noalloc_fwd(Q1, K1, Q2, K2, True, out, wait_limit_ns=20_000_000,
                     debug_flags=streamkl.DEBUG_INJECT_STALL)
    assert rc == streamkl.OK
    st, word = noalloc_status()
    assert st == streamkl.ERR_TIMEOUT and word != 0
    assert noalloc_status() == (streamkl.OK, 0)  # reading cleared it
    assert bool(torch.isnan(out[0]).any())       # the rows of the CTA that gave up
    assert noalloc_fwd(Q1, K1, Q2, K2, True, out) == streamkl.OK
    torch.cuda.synchronize()
    assert noalloc_status() == (streamkl.OK, 0)
    rKL, rL1, _ = oracle.fwd(Q1, K1, Q2, K2, causal=True)
    assert_kl(out[0], rKL, "KL after a timed-out call")
    assert_lse(out[1], rL1, "LSE1 after a timed-out call")
    assert np.isfinite(out[2].cpu().numpy()).all()
