"""Python wrapper of the float64 CPU oracle (``streamkl_oracle.c``).

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``, the smoke check in
``__graft_entry__`` and the benchmark's CPU-baseline leg may import this
module.  It never imports the CUDA path, and the CUDA path never imports it.

The oracle follows "StreamKL: Fast and Memory-Efficient KL Divergence for
Boosting Attention Distillation" (gist.science/paper/2606.20005, technical
summary): Problem Statement (row-wise KL of two attention distributions),
Methodology 1 (online formulation), Methodology 2 (recompute backward, two
settings).  Inputs are float64 arrays in ``[B, H, N, d]`` layout; callers that
hold bf16 tensors widen them exactly to float64 first.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "streamkl_oracle.c")
_LIB = os.path.join(_HERE, "_build", "libstreamkl_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, OpenMP, IEEE arithmetic: no fast-math)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-fno-fast-math",
           "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            d = ctypes.POINTER(ctypes.c_double)
            i64p = ctypes.POINTER(ctypes.c_int64)
            I, L, D = ctypes.c_int, ctypes.c_int64, ctypes.c_double
            dims = [I, I, L, L, I]
            lib.oracle_fwd.argtypes = dims + [d, d, d, d, D, I, d, d, d, I]
            lib.oracle_fwd_rows.argtypes = dims + [d, d, d, d, D, I, L, i64p, d, d, d, I]
            lib.oracle_online_fwd.argtypes = dims + [d, d, d, d, D, I, L, d, d, d, I]
            lib.oracle_bwd.argtypes = [I] + dims + [d, d, d, d, d, D, I, d, d, I]
            lib.oracle_bwd_dq_rows.argtypes = [I] + dims + [d, d, d, d, d, D, I, L, i64p, d, I]
            lib.oracle_bwd_dk_keys.argtypes = [I] + dims + [d, d, d, d, d, D, I, L, i64p, d, I]
            for f in (lib.oracle_fwd, lib.oracle_fwd_rows, lib.oracle_online_fwd, lib.oracle_bwd,
                      lib.oracle_bwd_dq_rows, lib.oracle_bwd_dk_keys, lib.oracle_max_threads):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(x) -> np.ndarray:
    """Exact float64 copy of x (a numpy array or a torch tensor of any float dtype)."""
    if hasattr(x, "detach"):  # torch tensor: widen on its device, then copy to host
        import torch
        x = x.detach().to(torch.float64).cpu().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _iptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))


def _dims(Q1, K1):
    B, H, Nq, d = Q1.shape
    Nk = K1.shape[2]
    return B, H, Nq, Nk, d


def _scale(scale, d):
    return float(d) ** -0.5 if scale is None else float(scale)


def _check(rc, name):
    if rc != 0:
        raise ValueError(f"{name}: oracle rejected the arguments (code {rc})")


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def fwd(Q1, K1, Q2, K2, causal=False, scale=None, nthreads=0):
    """Per-row (KL, LSE1, LSE2), each float64 [B, H, Nq], by definition."""
    Q1, K1, Q2, K2 = map(_f64, (Q1, K1, Q2, K2))
    B, H, Nq, Nk, d = _dims(Q1, K1)
    KL, L1, L2 = (np.empty((B, H, Nq)) for _ in range(3))
    rc = _load().oracle_fwd(B, H, Nq, Nk, d, _ptr(Q1), _ptr(K1), _ptr(Q2), _ptr(K2), _scale(scale, d),
                            int(causal), _ptr(KL), _ptr(L1), _ptr(L2), nthreads)
    _check(rc, "fwd")
    return KL, L1, L2


def fwd_rows(Q1, K1, Q2, K2, rows, causal=False, scale=None, nthreads=0):
    """(KL, LSE1, LSE2) for the flat row indices ``rows`` (into [B, H, Nq])."""
    Q1, K1, Q2, K2 = map(_f64, (Q1, K1, Q2, K2))
    B, H, Nq, Nk, d = _dims(Q1, K1)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    KL, L1, L2 = (np.empty(len(rows)) for _ in range(3))
    rc = _load().oracle_fwd_rows(B, H, Nq, Nk, d, _ptr(Q1), _ptr(K1), _ptr(Q2), _ptr(K2), _scale(scale, d),
                                 int(causal), len(rows), _iptr(rows), _ptr(KL), _ptr(L1), _ptr(L2), nthreads)
    _check(rc, "fwd_rows")
    return KL, L1, L2


def online_fwd(Q1, K1, Q2, K2, block_k, causal=False, scale=None, nthreads=0):
    """The five-scalar online recurrence with key tiles of width ``block_k``."""
    Q1, K1, Q2, K2 = map(_f64, (Q1, K1, Q2, K2))
    B, H, Nq, Nk, d = _dims(Q1, K1)
    KL, L1, L2 = (np.empty((B, H, Nq)) for _ in range(3))
    rc = _load().oracle_online_fwd(B, H, Nq, Nk, d, _ptr(Q1), _ptr(K1), _ptr(Q2), _ptr(K2), _scale(scale, d),
                                   int(causal), int(block_k), _ptr(KL), _ptr(L1), _ptr(L2), nthreads)
    _check(rc, "online_fwd")
    return KL, L1, L2


def bwd(setting, g, Q1, K1, Q2, K2, causal=False, scale=None, nthreads=0):
    """(dQ, dK) of the trainable side: setting 1 -> (Q2, K2), setting 2 -> (Q1, K1)."""
    Q1, K1, Q2, K2, g = map(_f64, (Q1, K1, Q2, K2, g))
    B, H, Nq, Nk, d = _dims(Q1, K1)
    g = np.ascontiguousarray(np.broadcast_to(g, (B, H, Nq)))
    dQ = np.empty((B, H, Nq, d))
    dK = np.empty((B, H, Nk, d))
    rc = _load().oracle_bwd(int(setting), B, H, Nq, Nk, d, _ptr(g), _ptr(Q1), _ptr(K1), _ptr(Q2), _ptr(K2),
                            _scale(scale, d), int(causal), _ptr(dQ), _ptr(dK), nthreads)
    _check(rc, "bwd")
    return dQ, dK


def bwd_dq_rows(setting, g, Q1, K1, Q2, K2, rows, causal=False, scale=None, nthreads=0):
    """dQ of the trainable side for the flat query rows ``rows``; [len(rows), d]."""
    Q1, K1, Q2, K2, g = map(_f64, (Q1, K1, Q2, K2, g))
    B, H, Nq, Nk, d = _dims(Q1, K1)
    g = np.ascontiguousarray(np.broadcast_to(g, (B, H, Nq)))
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    out = np.empty((len(rows), d))
    rc = _load().oracle_bwd_dq_rows(int(setting), B, H, Nq, Nk, d, _ptr(g), _ptr(Q1), _ptr(K1), _ptr(Q2),
                                    _ptr(K2), _scale(scale, d), int(causal), len(rows), _iptr(rows), _ptr(out),
                                    nthreads)
    _check(rc, "bwd_dq_rows")
    return out


def bwd_dk_keys(setting, g, Q1, K1, Q2, K2, keys, causal=False, scale=None, nthreads=0):
    """dK of the trainable side for the flat key rows ``keys``; [len(keys), d]."""
    Q1, K1, Q2, K2, g = map(_f64, (Q1, K1, Q2, K2, g))
    B, H, Nq, Nk, d = _dims(Q1, K1)
    g = np.ascontiguousarray(np.broadcast_to(g, (B, H, Nq)))
    keys = np.ascontiguousarray(keys, dtype=np.int64)
    out = np.empty((len(keys), d))
    rc = _load().oracle_bwd_dk_keys(int(setting), B, H, Nq, Nk, d, _ptr(g), _ptr(Q1), _ptr(K1), _ptr(Q2),
                                    _ptr(K2), _scale(scale, d), int(causal), len(keys), _iptr(keys), _ptr(out),
                                    nthreads)
    _check(rc, "bwd_dk_keys")
    return out
