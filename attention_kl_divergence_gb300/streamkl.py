"""Python binding of libstreamkl (ctypes).  Argument marshalling only: every
step of the computation runs in the library's CUDA kernels.  PyTorch supplies
device memory and the current stream.

Functions mirror the C ABI in ``include/streamkl.h``:

    kl_fwd(Q1, K1, Q2, K2, causal=False, scale=None) -> (KL, LSE1, LSE2)
    kl_bwd(setting, g, Q1, K1, Q2, K2, KL, LSE1, LSE2, causal=False) -> (dQ, dK)
    kl_bwd_joint(g, Q1, K1, Q2, K2, KL, LSE1, LSE2, causal=False) -> (dQ1, dK1, dQ2, dK2)

plus ``fwd_plan`` / ``bwd_plan`` (what a call launches) and ``AttentionKL``,
an autograd Function.  There is no fallback: without the compiled library
every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA, ERR_TIMEOUT = range(6)
PATH_TILE, PATH_DECODE, PATH_BWD_FUSED, PATH_BWD_SPLIT, PATH_BWD_KEYSPLIT, PATH_BWD_JOINT = range(6)
BWD_AUTO, BWD_FUSED, BWD_SPLIT, BWD_KEYSPLIT = 0, 1, 2, 3


class Shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("H", ctypes.c_int32), ("Nq", ctypes.c_int32), ("Nk", ctypes.c_int32),
                ("d", ctypes.c_int32), ("q_stride_b", ctypes.c_int64), ("q_stride_h", ctypes.c_int64),
                ("q_stride_n", ctypes.c_int64), ("k_stride_b", ctypes.c_int64), ("k_stride_h", ctypes.c_int64),
                ("k_stride_n", ctypes.c_int64), ("H_kv", ctypes.c_int32)]


class Options(ctypes.Structure):
    _fields_ = [("num_splits", ctypes.c_int32), ("bwd_mode", ctypes.c_int32), ("wait_limit_ns", ctypes.c_int64),
                ("debug_flags", ctypes.c_int32), ("grad_bf16", ctypes.c_int32)]


DEBUG_INJECT_STALL = 1


class Plan(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int32), ("num_splits", ctypes.c_int32), ("num_ctas", ctypes.c_int32),
                ("launches", ctypes.c_int32), ("workspace_bytes", ctypes.c_size_t)]


class StreamKLError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} (status {code})")


EXPORTED = ("streamkl_fwd_plan", "streamkl_fwd", "streamkl_bwd_plan", "streamkl_bwd", "streamkl_workspace_status",
            "streamkl_status_string", "streamkl_version", "streamkl_fwd_noalloc", "streamkl_noalloc_status",
            "streamkl_fwd_workspace_bytes", "streamkl_bwd_workspace_bytes", "streamkl_bwd_joint_plan",
            "streamkl_bwd_joint")

_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def load(build_if_stale: bool = True):
    """Load libstreamkl.so (building it first when sources are newer)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if build_if_stale and _build.is_stale():
            _build.build()
        if not os.path.exists(_build.LIB):
            raise RuntimeError(f"libstreamkl.so is missing ({_build.LIB}); run __graft_entry__.build()")
        lib = ctypes.CDLL(_build.LIB)
        P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        sp, op, pp = ctypes.POINTER(Shape), ctypes.POINTER(Options), ctypes.POINTER(Plan)
        lib.streamkl_fwd_plan.argtypes = [sp, I, op, pp]
        lib.streamkl_fwd.argtypes = [sp, P, P, P, P, F, I, P, P, P, P, Z, op, P]
        lib.streamkl_bwd_plan.argtypes = [sp, I, I, op, pp]
        lib.streamkl_bwd.argtypes = [sp, I, P, P, P, P, P, P, P, P, F, I, P, P, P, Z, op, P]
        lib.streamkl_workspace_status.argtypes = [P, P, ctypes.POINTER(ctypes.c_uint32)]
        lib.streamkl_fwd_noalloc.argtypes = [sp, P, P, P, P, F, I, P, P, P, op, P]
        lib.streamkl_noalloc_status.argtypes = [P, ctypes.POINTER(ctypes.c_uint32)]
        lib.streamkl_bwd_joint_plan.argtypes = [sp, I, op, pp]
        lib.streamkl_bwd_joint.argtypes = [sp, P, P, P, P, P, P, P, P, F, I, P, P, P, P, P, Z, op, P]
        lib.streamkl_fwd_workspace_bytes.argtypes = [sp, I]
        lib.streamkl_bwd_workspace_bytes.argtypes = [sp, I, I]
        lib.streamkl_fwd_workspace_bytes.restype = Z
        lib.streamkl_bwd_workspace_bytes.restype = Z
        lib.streamkl_status_string.argtypes = [I]
        lib.streamkl_status_string.restype = ctypes.c_char_p
        for name in ("streamkl_fwd_plan", "streamkl_fwd", "streamkl_bwd_plan", "streamkl_bwd",
                     "streamkl_workspace_status", "streamkl_version", "streamkl_fwd_noalloc",
                     "streamkl_noalloc_status", "streamkl_bwd_joint_plan", "streamkl_bwd_joint"):
            getattr(lib, name).restype = ctypes.c_int
        _lib = lib
        return lib


def status_string(code: int) -> str:
    return load().streamkl_status_string(int(code)).decode()


def _raise(code, where):
    if code != OK:
        raise StreamKLError(code, where)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def make_shape(Q1, K1) -> Shape:
    """Shape/strides struct of [B, H, N, d] tensors (d must be contiguous)."""
    B, H, Nq, d = Q1.shape
    Nk = K1.shape[2]
    qs, ks = Q1.stride(), K1.stride()
    return Shape(B, H, Nq, Nk, d, qs[0], qs[1], qs[2], ks[0], ks[1], ks[2], K1.shape[1])


def _check_qk(Q1, K1, Q2, K2):
    for name, t in (("Q1", Q1), ("K1", K1), ("Q2", Q2), ("K2", K2)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if t.dtype != torch.bfloat16:
            raise ValueError(f"{name} must be bf16, got {t.dtype}")
        if t.dim() != 4 or t.stride(3) != 1:
            raise ValueError(f"{name} must be [B, H, N, d] with d contiguous")
    if Q1.shape != Q2.shape or K1.shape != K2.shape or Q1.stride() != Q2.stride() or K1.stride() != K2.stride():
        raise ValueError("teacher and student tensors must have equal shapes and strides")
    if Q1.shape[0] != K1.shape[0] or Q1.shape[3] != K1.shape[3]:
        raise ValueError("Q and K must share B and d")
    if Q1.shape[1] % K1.shape[1] != 0:
        raise ValueError("the key head count must divide the query head count")
    if any(t.device != Q1.device for t in (K1, Q2, K2)):
        raise ValueError("Q1, K1, Q2 and K2 must be on one device")


def _check_tensor(name, t, shape, dtype, device):
    """Outputs and per-row inputs are written or read as dense arrays of the
    given shape: anything else would send the kernels out of bounds."""
    if not isinstance(t, torch.Tensor) or t.device != device:
        raise ValueError(f"{name} must be a tensor on {device}")
    if t.dtype != dtype or not t.is_contiguous() or tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must be a contiguous {dtype} tensor of shape {tuple(shape)}, got "
                         f"{t.dtype} {tuple(t.shape)}{'' if t.is_contiguous() else ' (not contiguous)'}")


def _check_workspace(workspace, nbytes, device):
    """None allocates one; a caller's workspace must be a large enough
    contiguous uint8 tensor on the inputs' device (it is never replaced)."""
    if workspace is None:
        return new_workspace(nbytes, device)
    if not isinstance(workspace, torch.Tensor) or workspace.device != device or workspace.dtype != torch.uint8 \
            or not workspace.is_contiguous():
        raise ValueError(f"workspace must be a contiguous uint8 tensor on {device}")
    if workspace.numel() < nbytes:
        raise ValueError(f"workspace holds {workspace.numel()} bytes; this call needs {nbytes} (see fwd_plan / bwd_plan)")
    return workspace


def _opts(num_splits=0, bwd_mode=0, wait_limit_ns=0, debug_flags=0, grad_bf16=0):
    return Options(int(num_splits), int(bwd_mode), int(wait_limit_ns), int(debug_flags), int(grad_bf16))


def fwd_plan(Q1, K1, causal=False, num_splits=0) -> Plan:
    plan = Plan()
    _raise(load().streamkl_fwd_plan(ctypes.byref(make_shape(Q1, K1)), int(bool(causal)),
                                    ctypes.byref(_opts(num_splits)), ctypes.byref(plan)), "streamkl_fwd_plan")
    return plan


def bwd_plan(Q1, K1, setting, causal=False, mode=BWD_AUTO, grad_dtype=torch.float32, num_splits=0) -> Plan:
    plan = Plan()
    _raise(load().streamkl_bwd_plan(ctypes.byref(make_shape(Q1, K1)), int(setting), int(bool(causal)),
                                    ctypes.byref(_opts(num_splits, mode, grad_bf16=_grad_flag(grad_dtype))),
                                    ctypes.byref(plan)), "streamkl_bwd_plan")
    return plan


def fwd_workspace_bytes(Q1, K1, causal=False) -> int:
    """streamkl_fwd_workspace_bytes: the forward's workspace with default options (0 = invalid shape)."""
    return int(load().streamkl_fwd_workspace_bytes(ctypes.byref(make_shape(Q1, K1)), int(bool(causal))))


def bwd_workspace_bytes(Q1, K1, setting, causal=False) -> int:
    """streamkl_bwd_workspace_bytes: the backward's workspace with default options (0 = invalid)."""
    return int(load().streamkl_bwd_workspace_bytes(ctypes.byref(make_shape(Q1, K1)), int(setting),
                                                   int(bool(causal))))


def noalloc_status(device=None) -> int:
    """streamkl_noalloc_status: synchronise the current stream of ``device`` and
    return (and clear) the device error word of the allocation-free forward's
    built-in scratch (0 when no bounded wait gave up)."""
    word = ctypes.c_uint32(0)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    rc = load().streamkl_noalloc_status(_stream(dev), ctypes.byref(word))
    if rc not in (OK, ERR_TIMEOUT):
        _raise(rc, "streamkl_noalloc_status")
    return int(word.value)


def _grad_flag(grad_dtype):
    if grad_dtype == torch.float32:
        return 0
    if grad_dtype == torch.bfloat16:
        return 1
    raise ValueError(f"gradients are float32 or bfloat16, not {grad_dtype}")


def new_workspace(nbytes, device) -> torch.Tensor:
    """A zeroed workspace (the first 256 bytes hold the device error word)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def kl_fwd(Q1, K1, Q2, K2, causal=False, scale=None, num_splits=0, workspace=None, out=None,
           wait_limit_ns=0, debug_flags=0):
    """Per-row KL(P1 || P2), LSE1, LSE2 as float32 [B, H, Nq] tensors."""
    _check_qk(Q1, K1, Q2, K2)
    lib = load()
    shape = make_shape(Q1, K1)
    opts = _opts(num_splits, 0, wait_limit_ns, debug_flags)
    plan = Plan()
    _raise(lib.streamkl_fwd_plan(ctypes.byref(shape), int(bool(causal)), ctypes.byref(opts), ctypes.byref(plan)),
           "streamkl_fwd_plan")
    B, H, Nq, _ = Q1.shape
    if out is None:
        out = tuple(torch.empty((B, H, Nq), dtype=torch.float32, device=Q1.device) for _ in range(3))
    for name, t in zip(("KL", "LSE1", "LSE2"), out):
        _check_tensor(name, t, (B, H, Nq), torch.float32, Q1.device)
    workspace = _check_workspace(workspace, plan.workspace_bytes, Q1.device)
    KL, L1, L2 = out
    rc = lib.streamkl_fwd(ctypes.byref(shape), _ptr(Q1), _ptr(K1), _ptr(Q2), _ptr(K2),
                          ctypes.c_float(0.0 if scale is None else float(scale)), int(bool(causal)), _ptr(KL),
                          _ptr(L1), _ptr(L2), _ptr(workspace), workspace.numel(), ctypes.byref(opts),
                          _stream(Q1.device))
    _raise(rc, "streamkl_fwd")
    return KL, L1, L2


def kl_bwd(setting, g, Q1, K1, Q2, K2, KL, LSE1, LSE2, causal=False, scale=None, mode=BWD_AUTO, workspace=None,
           out=None, wait_limit_ns=0, debug_flags=0, grad_dtype=torch.float32, num_splits=0):
    """(dQ, dK) float32 of the trainable side: setting 1 -> (Q2, K2), 2 -> (Q1, K1).
    With keys shared by groups of query heads (K has fewer heads than Q), dK
    has K's head count and sums the gradients of each group.  num_splits sets
    the key-range splits of the key-split mode (0 = automatic)."""
    _check_qk(Q1, K1, Q2, K2)
    lib = load()
    shape = make_shape(Q1, K1)
    opts = _opts(num_splits, mode, wait_limit_ns, debug_flags, _grad_flag(grad_dtype))
    plan = Plan()
    _raise(lib.streamkl_bwd_plan(ctypes.byref(shape), int(setting), int(bool(causal)), ctypes.byref(opts),
                                 ctypes.byref(plan)), "streamkl_bwd_plan")
    B, H, Nq, d = Q1.shape
    Nk = K1.shape[2]
    for name, t in (("g", g), ("KL", KL), ("LSE1", LSE1), ("LSE2", LSE2)):
        _check_tensor(name, t, (B, H, Nq), torch.float32, Q1.device)
    if out is None:
        out = (torch.empty((B, H, Nq, d), dtype=grad_dtype, device=Q1.device),
               torch.empty((B, K1.shape[1], Nk, d), dtype=grad_dtype, device=Q1.device))
    _check_tensor("dQ", out[0], (B, H, Nq, d), grad_dtype, Q1.device)
    _check_tensor("dK", out[1], (B, K1.shape[1], Nk, d), grad_dtype, Q1.device)
    workspace = _check_workspace(workspace, plan.workspace_bytes, Q1.device)
    dQ, dK = out
    rc = lib.streamkl_bwd(ctypes.byref(shape), int(setting), _ptr(g), _ptr(Q1), _ptr(K1), _ptr(Q2), _ptr(K2),
                          _ptr(KL), _ptr(LSE1), _ptr(LSE2), ctypes.c_float(0.0 if scale is None else float(scale)),
                          int(bool(causal)), _ptr(dQ), _ptr(dK), _ptr(workspace), workspace.numel(),
                          ctypes.byref(opts), _stream(Q1.device))
    _raise(rc, "streamkl_bwd")
    return dQ, dK


def bwd_joint_plan(Q1, K1, causal=False, grad_dtype=torch.float32) -> Plan:
    plan = Plan()
    _raise(load().streamkl_bwd_joint_plan(ctypes.byref(make_shape(Q1, K1)), int(bool(causal)),
                                          ctypes.byref(_opts(grad_bf16=_grad_flag(grad_dtype))), ctypes.byref(plan)),
           "streamkl_bwd_joint_plan")
    return plan


def kl_bwd_joint(g, Q1, K1, Q2, K2, KL, LSE1, LSE2, causal=False, scale=None, workspace=None, out=None,
                 wait_limit_ns=0, debug_flags=0, grad_dtype=torch.float32):
    """(dQ1, dK1, dQ2, dK2): the gradients of both sides from one recompute of
    the scores per kernel -- the teacher's as in setting 2, the student's as
    in setting 1 (streamkl_bwd_joint)."""
    _check_qk(Q1, K1, Q2, K2)
    lib = load()
    shape = make_shape(Q1, K1)
    opts = _opts(0, 0, wait_limit_ns, debug_flags, _grad_flag(grad_dtype))
    plan = Plan()
    _raise(lib.streamkl_bwd_joint_plan(ctypes.byref(shape), int(bool(causal)), ctypes.byref(opts),
                                       ctypes.byref(plan)), "streamkl_bwd_joint_plan")
    B, H, Nq, d = Q1.shape
    Hk, Nk = K1.shape[1], K1.shape[2]
    for name, t in (("g", g), ("KL", KL), ("LSE1", LSE1), ("LSE2", LSE2)):
        _check_tensor(name, t, (B, H, Nq), torch.float32, Q1.device)
    if out is None:
        out = tuple(torch.empty(shp, dtype=grad_dtype, device=Q1.device)
                    for shp in ((B, H, Nq, d), (B, Hk, Nk, d), (B, H, Nq, d), (B, Hk, Nk, d)))
    for name, t, shp in zip(("dQ1", "dK1", "dQ2", "dK2"), out,
                            ((B, H, Nq, d), (B, Hk, Nk, d), (B, H, Nq, d), (B, Hk, Nk, d))):
        _check_tensor(name, t, shp, grad_dtype, Q1.device)
    workspace = _check_workspace(workspace, plan.workspace_bytes, Q1.device)
    dQ1, dK1, dQ2, dK2 = out
    rc = lib.streamkl_bwd_joint(ctypes.byref(shape), _ptr(g), _ptr(Q1), _ptr(K1), _ptr(Q2), _ptr(K2), _ptr(KL),
                                _ptr(LSE1), _ptr(LSE2), ctypes.c_float(0.0 if scale is None else float(scale)),
                                int(bool(causal)), _ptr(dQ1), _ptr(dK1), _ptr(dQ2), _ptr(dK2), _ptr(workspace),
                                workspace.numel(), ctypes.byref(opts), _stream(Q1.device))
    _raise(rc, "streamkl_bwd_joint")
    return dQ1, dK1, dQ2, dK2


def workspace_status(workspace) -> int:
    """Synchronise the current stream and return (and clear) the workspace's
    device error word; raises StreamKLError(ERR_TIMEOUT) when it was set."""
    word = ctypes.c_uint32(0)
    rc = load().streamkl_workspace_status(_ptr(workspace), _stream(workspace.device), ctypes.byref(word))
    if rc not in (OK, ERR_TIMEOUT):
        _raise(rc, "streamkl_workspace_status")
    return int(word.value)


class AttentionKL(torch.autograd.Function):
    """Per-row KL(softmax(Q1 K1^T s) || softmax(Q2 K2^T s)) with a recompute
    backward.  Gradients flow to the student (setting 1) or the teacher
    (setting 2), chosen by which inputs require grad; the other side gets
    None.  When both sides require grad, the joint backward forms the
    gradients of both from one recompute of the scores per kernel
    (streamkl_bwd_joint): measured on GB300 at 64K causal it takes as long as
    the two single-setting passes (145.7 vs 144.5 ms) and, adding no gradient
    through atomics, gives the same bits on every run.  For at most 16 query
    rows per key head (decode shapes) the two single-setting key-split passes
    run instead.  Together the two sides
    are the gradient of KL with respect to all four inputs: each setting
    differentiates through one side's distribution with the other side's held
    fixed.  Gradients come back in bf16, like the inputs."""

    @staticmethod
    def forward(ctx, Q1, K1, Q2, K2, causal=False, scale=None):
        KL, L1, L2 = kl_fwd(Q1, K1, Q2, K2, causal=causal, scale=scale)
        ctx.save_for_backward(Q1, K1, Q2, K2, KL, L1, L2)
        ctx.causal, ctx.scale = causal, scale
        return KL

    @staticmethod
    def backward(ctx, gKL):
        Q1, K1, Q2, K2, KL, L1, L2 = ctx.saved_tensors
        student = ctx.needs_input_grad[2] or ctx.needs_input_grad[3]
        teacher = ctx.needs_input_grad[0] or ctx.needs_input_grad[1]
        if not (student or teacher):
            return (None,) * 6
        g = gKL.float().contiguous()
        # the joint pass where the single-setting backward is the fused kernel; for at most 16 query
        # rows per key head the two key-split passes stream the keys far faster
        if student and teacher and bwd_plan(Q1, K1, 1, causal=ctx.causal).path == PATH_BWD_FUSED:
            dQ1, dK1, dQ2, dK2 = kl_bwd_joint(g, Q1, K1, Q2, K2, KL, L1, L2, causal=ctx.causal, scale=ctx.scale,
                                              grad_dtype=torch.bfloat16)
            return dQ1, dK1, dQ2, dK2, None, None
        grads = [None] * 6
        for setting, want, slot in ((1, student, 2), (2, teacher, 0)):
            if want:
                dQ, dK = kl_bwd(setting, g, Q1, K1, Q2, K2, KL, L1, L2, causal=ctx.causal, scale=ctx.scale,
                                grad_dtype=torch.bfloat16)
                grads[slot], grads[slot + 1] = dQ, dK
        return tuple(grads)
