"""The C ABI loads, exports every symbol include/streamkl.h declares, and
rejects bad arguments before touching a device (no GPU needed)."""
import ctypes
import os
import re

import pytest

from attention_kl_divergence_gb300 import streamkl as sk

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    text = open(os.path.join(ROOT, "include", "streamkl.h")).read()
    return sorted(set(re.findall(r"STREAMKL_API\s+[\w\s\*]+?\b(streamkl_\w+)\s*\(", text)))


def test_header_declares_the_binding_symbols():
    assert declared_functions() == sorted(sk.EXPORTED)


def test_library_exports_every_declared_symbol():
    lib = sk.load()
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert lib.streamkl_version() >= 200


def test_status_strings():
    for code in range(6):
        assert sk.status_string(code)
    assert sk.status_string(99) == "unknown status"


def _shape(**kw):
    s = dict(B=1, H=2, Nq=256, Nk=256, d=64)
    s.update(kw)
    d, Nq, Nk, H = s["d"], s["Nq"], s["Nk"], s["H"]
    return sk.Shape(s["B"], H, Nq, Nk, d, H * Nq * d, Nq * d, d, H * Nk * d, Nk * d, d, s.get("H_kv", 0))


def _fwd(shape, ptrs=(256,) * 7, ws=256, ws_bytes=4096, causal=0):
    lib = sk.load()
    P = ctypes.c_void_p
    return lib.streamkl_fwd(ctypes.byref(shape) if shape is not None else None, *[P(p) for p in ptrs[:4]],
                            ctypes.c_float(0.0), causal, *[P(p) for p in ptrs[4:]], P(ws), ws_bytes, None, P(0))


def test_fwd_rejects_bad_shapes_without_device():
    assert _fwd(None) == sk.ERR_INVALID_ARG
    assert _fwd(_shape(B=0)) == sk.ERR_INVALID_ARG
    assert _fwd(_shape(Nk=0)) == sk.ERR_INVALID_ARG
    assert _fwd(_shape(d=96)) == sk.ERR_UNSUPPORTED
    assert _fwd(_shape(Nq=300, Nk=200), causal=1) == sk.ERR_INVALID_ARG
    bad = _shape()
    bad.q_stride_n = 60  # not a multiple of 8 elements
    assert _fwd(bad) == sk.ERR_INVALID_ARG
    assert _fwd(_shape(H=6, H_kv=4)) == sk.ERR_INVALID_ARG  # key heads must divide query heads
    assert _fwd(_shape(H=6, H_kv=-1)) == sk.ERR_INVALID_ARG


def test_fwd_rejects_bad_pointers_without_device():
    assert _fwd(_shape(), ptrs=(256, 0, 256, 256, 256, 256, 256)) == sk.ERR_INVALID_ARG
    assert _fwd(_shape(), ptrs=(256, 264, 256, 256, 256, 256, 256)) == sk.ERR_INVALID_ARG  # K1 not 16-B aligned
    assert _fwd(_shape(), ptrs=(256, 256, 256, 256, 258, 256, 256)) == sk.ERR_INVALID_ARG  # KL not 4-B aligned
    assert _fwd(_shape(), ws=0) == sk.ERR_WORKSPACE
    assert _fwd(_shape(), ws=8) == sk.ERR_WORKSPACE


def test_workspace_status_rejects_null():
    assert sk.load().streamkl_workspace_status(None, None, None) == sk.ERR_INVALID_ARG


def test_options_reject_unknown_debug_flags_without_device():
    lib = sk.load()
    P = ctypes.c_void_p
    bad = sk.Options(0, 0, 0, 8, 0)  # unknown debug flag
    rc = lib.streamkl_fwd(ctypes.byref(_shape()), *[P(256)] * 4, ctypes.c_float(0.0), 0, *[P(256)] * 3, P(256),
                          4096, ctypes.byref(bad), P(0))
    assert rc in (sk.ERR_INVALID_ARG, sk.ERR_CUDA)  # the option check needs no device but runs in the planner


def test_workspace_size_queries_reject_invalid_shapes_without_device():
    lib = sk.load()
    assert lib.streamkl_fwd_workspace_bytes(None, 0) == 0
    assert lib.streamkl_fwd_workspace_bytes(ctypes.byref(_shape(d=96)), 0) == 0
    assert lib.streamkl_fwd_workspace_bytes(ctypes.byref(_shape(Nq=300, Nk=200)), 1) == 0
    assert lib.streamkl_bwd_workspace_bytes(ctypes.byref(_shape()), 3, 0) == 0  # no setting 3
    assert lib.streamkl_bwd_workspace_bytes(ctypes.byref(_shape(B=0)), 1, 0) == 0


def test_joint_backward_rejects_bad_arguments_without_device():
    lib = sk.load()
    P = ctypes.c_void_p

    def call(shape, ptrs=(256,) * 12, ws=256, ws_bytes=4096, causal=0):
        # g, Q1, K1, Q2, K2, KL, LSE1, LSE2 | dQ1, dK1, dQ2, dK2
        return lib.streamkl_bwd_joint(ctypes.byref(shape) if shape is not None else None,
                                      *[P(p) for p in ptrs[:8]], ctypes.c_float(0.0), causal,
                                      *[P(p) for p in ptrs[8:]], P(ws), ws_bytes, None, P(0))

    assert call(None) == sk.ERR_INVALID_ARG
    assert call(_shape(d=96)) == sk.ERR_UNSUPPORTED
    assert call(_shape(Nq=300, Nk=200), causal=1) == sk.ERR_INVALID_ARG
    bad = list((256,) * 12)
    bad[11] = 0  # dK2 missing
    assert call(_shape(), ptrs=tuple(bad)) == sk.ERR_INVALID_ARG
    bad[11] = 264  # dK2 not 16-byte aligned
    assert call(_shape(), ptrs=tuple(bad)) == sk.ERR_INVALID_ARG
    bad = list((256,) * 12)
    bad[0] = 258  # g not 4-byte aligned
    assert call(_shape(), ptrs=tuple(bad)) == sk.ERR_INVALID_ARG
    assert call(_shape(), ws=0) == sk.ERR_WORKSPACE
