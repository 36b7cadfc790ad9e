"""Benchmark of the fused attention KL divergence (libstreamkl) on GB300.

One step = the whole hot path on one batch: forward (KL, LSE1, LSE2) plus the
recompute backward in both settings (setting 1: gradients to the student
Q2/K2; setting 2: gradients to the teacher Q1/K1), on B=1, H=32,
N_Q=N_K=65536, d=128, bf16, causal -- the workload the headline metric is
quoted on.  Inputs are seeded synthetic tensors (teacher ~ N(0,1), student =
teacher + 0.3 N(0,1)), resident in HBM; at 2 GiB they exceed the 129 MB L2.

Printed (rank 0, one JSON line): the metric in TFLOP/s of algorithmic work
(forward 4 d per visible pair, each backward 8 d per visible pair), ms per
step and per pass, the roofline of the dominant kernel, the end-to-end rate
through the C ABI with host buffers, clocks, and the float64 CPU oracle timed
on a bounded sample of the same workload.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
Under torchrun the heads of the one problem are split across the ranks (heads
are independent problems, so there is no collective on the data path): strong
scaling, the value is the whole problem's work over the slowest rank's time.
After the headline step the same run times the N_Q=1, N_K=512K Split-K decode
forward (B=4, H=32, d=128), HBM-bound, with its own clock sample.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from attention_kl_divergence_gb300 import WORKLOADS, make_g, make_workload  # noqa: E402
from attention_kl_divergence_gb300.dist import (barrier, env as dist_env, head_range, init as init_dist,  # noqa: E402
                                                max_over_ranks)

WORKLOAD = "64k_causal"
DECODE_WORKLOAD = "decode_q1_k512k"
METRIC = "fwd/bwd TFLOP/s and ms at 64K causal, fraction of GB300 BF16 tensor peak"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# DRAM bytes (read + write) per launch of a kernel, from one ncu capture
# (dram__bytes_read.sum + dram__bytes_write.sum), with the hash of the kernel
# source files it was taken on: a table entry whose hash differs from the
# sources being run is stale and reported as null.
KERNEL_SOURCES = {
    "fwd": ("fwd.cu", "common.cuh", "ptx.cuh"),
    "bwd": ("bwd.cu", "bwd_common.cuh", "common.cuh", "ptx.cuh"),
}
TRAFFIC = {
    ("64k_causal", "fwd"): (2.164e9 + 0.039e9, "fwd", "908c094b14b22853"),
    ("64k_causal", "bwd_setting1"): (3.363e9 + 2.251e9, "bwd", "0db1caec739e066f"),
    ("64k_causal", "bwd_setting2"): (3.361e9 + 2.250e9, "bwd", "0db1caec739e066f"),
}


def source_hash(kind):
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kind]:
        with open(os.path.join(ROOT, "attention_kl_divergence_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_for(workload, which):
    """Measured DRAM bytes per launch, or None when there is no capture of the
    kernel as it is built now."""
    entry = TRAFFIC.get((workload, which))
    if entry is None:
        return None
    nbytes, kind, digest = entry
    return nbytes if source_hash(kind) == digest else None


BWD_MODE_NAMES = {2: "fused", 3: "split", 4: "keysplit"}  # plan paths of the backward


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(PEAKS_FALLBACK), "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    _count = 0

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        ClockSampler._count += 1  # one file per sampler: several may run in one process
        self.path = os.path.join("/tmp", f"streamkl_clocks_{os.getpid()}_{ClockSampler._count}.csv")

    def __enter__(self):
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.out,
                                         stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.out.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        loaded = [r for r in rows if r[2] > 300.0] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in loaded for k, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": max(r[1] for r in rows),
                "power_w_max": max(r[2] for r in rows), "samples": len(loaded), "reasons": reasons}


def gpu_id(dev):
    """nvidia-smi id of a torch device (its UUID, robust to CUDA_VISIBLE_DEVICES)."""
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return str(dev.index or 0)


L2_BYTES = 129 * 2**20  # GB300 L2


def input_bytes(w):
    """bf16 Q1, K1, Q2, K2 of the whole workload."""
    return 2 * 2 * w.d * w.B * (w.H * w.Nq + (w.H_kv or w.H) * w.Nk)


def config_for(w, world):
    return {"workload": f"{w.name}: B={w.B} H={w.H}{f' H_kv={w.H_kv}' if w.H_kv else ''} N_Q={w.Nq} N_K={w.Nk} d={w.d} "
                        f"{'causal' if w.causal else 'non-causal'}, "
                        + ("fwd only (Split-K decode) per step" if w.fwd_only else
                           "fwd + bwd setting 1 + bwd setting 2 per step"),
            "l2": "256 MB write between steps" + (" (inputs exceed L2 as well)" if input_bytes(w) > L2_BYTES else ""),
            "parallelism": f"heads split across {world} GPU(s), no collective on the data path"}


def rank_heads(w, rank, world):
    """[start, stop) of the flat key heads (b * H_kv + hk) this rank owns; the
    query heads of a key head's group go with it.  Shards differ by at most
    one key head and together cover every head exactly once."""
    units = w.B * (w.H_kv or w.H)
    if world > units:
        raise ValueError(f"{world} ranks for {units} heads")
    return head_range(units, rank, world)


def shard(t, start, stop, group=1):
    """Heads [start*group, stop*group) of a [B, H, N, ...] tensor as a
    contiguous [1, n, N, ...] view (B and H flattened)."""
    B, H = t.shape[:2]
    return t.reshape(B * H, *t.shape[2:])[start * group:stop * group].unsqueeze(0)


def flush_l2(buf):
    buf.add_(1)  # a write larger than L2 between timed steps


# ---------------------------------------------------------------------------
# CPU oracle leg (the float64 oracle as it stands, bounded sample)
# ---------------------------------------------------------------------------

def cpu_oracle_sample(w, budget_s=15.0):
    """Time the oracle's forward and both settings' dQ on sampled query rows of
    one head of the workload (each row sees up to 64K keys).  Rate in TFLOP/s
    of the same algorithmic work the GPU metric counts per pair."""
    from oracle import oracle
    from attention_kl_divergence_gb300 import make_qk
    g = make_g(1, 1, w.Nq, w.g_value)
    Q1, K1, Q2, K2 = make_qk(1, 1, w.Nq, w.Nk, w.d, w.sigma, w.teacher_scale, w.seed, device="cpu")
    rng = np.random.default_rng(0)
    cores = oracle.max_threads()
    n = cores * 2
    done_pairs, elapsed, nrows = 0, 0.0, 0
    Q1n, K1n, Q2n, K2n = (oracle._f64(t) for t in (Q1, K1, Q2, K2))
    gn = oracle._f64(g)
    while elapsed < budget_s and nrows < 4096:
        rows = rng.integers(0, w.Nq, size=n)
        t0 = time.perf_counter()
        oracle.fwd_rows(Q1n, K1n, Q2n, K2n, rows, causal=w.causal)
        if not w.fwd_only:
            oracle.bwd_dq_rows(1, gn, Q1n, K1n, Q2n, K2n, rows, causal=w.causal)
            oracle.bwd_dq_rows(2, gn, Q1n, K1n, Q2n, K2n, rows, causal=w.causal)
        elapsed += time.perf_counter() - t0
        off = w.Nk - w.Nq
        done_pairs += int(sum(min(w.Nk, int(i) + off + 1) if w.causal else w.Nk for i in rows))
        nrows += n
    # algorithmic flops the GPU metric credits for these pairs: 4d (fwd) + 2 x 8d (bwd)
    per_pair = 4 if w.fwd_only else 20
    flops = per_pair * w.d * done_pairs
    return {"value": flops / elapsed / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{nrows} random query rows of one head of {w.name} (N_Q={w.Nq} N_K={w.Nk} d={w.d}): "
                      f"{'forward' if w.fwd_only else 'forward + dQ of both settings'} per row, "
                      f"{elapsed:.1f} s, float64, {done_pairs} visible pairs; credited {per_pair}*d flops per pair",
            "seconds": elapsed}


# ---------------------------------------------------------------------------
# GPU leg
# ---------------------------------------------------------------------------

def run_gpu(args):
    from attention_kl_divergence_gb300 import streamkl

    ws_, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(ws_, "nccl")
    w = WORKLOADS[args.workload]
    peaks, peak_src = load_peaks()
    group = w.H // (w.H_kv or w.H)
    start, stop = rank_heads(w, rank, ws_)
    # the whole problem is drawn from its seed on every rank; each rank keeps its heads
    full = make_workload(w, device=dev)
    Q1, K1, Q2, K2 = (shard(t, start, stop, group if k % 2 == 0 else 1) for k, t in enumerate(full))
    Q1, K1, Q2, K2 = (t.clone() for t in (Q1, K1, Q2, K2))
    del full
    Hq, Hk = Q1.shape[1], K1.shape[1]
    g = make_g(1, Hq, w.Nq, w.g_value, device=dev)
    Nq, Nk, d = w.Nq, w.Nk, w.d
    f32 = dict(dtype=torch.float32, device=dev)
    with_bwd = not w.fwd_only

    def outputs():
        o = {"KL": torch.empty((1, Hq, Nq), **f32), "LSE1": torch.empty((1, Hq, Nq), **f32),
             "LSE2": torch.empty((1, Hq, Nq), **f32)}
        if with_bwd:  # setting 1 -> student gradients, setting 2 -> teacher gradients
            o.update(dQ2=torch.empty((1, Hq, Nq, d), **f32), dK2=torch.empty((1, Hk, Nk, d), **f32),
                     dQ1=torch.empty((1, Hq, Nq, d), **f32), dK1=torch.empty((1, Hk, Nk, d), **f32))
        return o

    out = outputs()
    fplan = streamkl.fwd_plan(Q1, K1, causal=w.causal)
    bplan1 = streamkl.bwd_plan(Q1, K1, 1, causal=w.causal)
    bplan2 = streamkl.bwd_plan(Q1, K1, 2, causal=w.causal)
    wsp = streamkl.new_workspace(max(fplan.workspace_bytes, bplan1.workspace_bytes, bplan2.workspace_bytes), dev)
    l2_flush = torch.empty(int(256e6) // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step_on(ins, o):
        q1, k1, q2, k2, gg = ins
        streamkl.kl_fwd(q1, k1, q2, k2, causal=w.causal, workspace=wsp, out=(o["KL"], o["LSE1"], o["LSE2"]))
        if with_bwd:
            streamkl.kl_bwd(1, gg, q1, k1, q2, k2, o["KL"], o["LSE1"], o["LSE2"], causal=w.causal, workspace=wsp,
                            out=(o["dQ2"], o["dK2"]))
            streamkl.kl_bwd(2, gg, q1, k1, q2, k2, o["KL"], o["LSE1"], o["LSE2"], causal=w.causal, workspace=wsp,
                            out=(o["dQ1"], o["dK1"]))

    ins = (Q1, K1, Q2, K2, g)
    launches_per_step = fplan.launches + ((bplan1.launches + bplan2.launches) if with_bwd else 0)
    adds_dq = (streamkl.PATH_BWD_FUSED, streamkl.PATH_BWD_KEYSPLIT)
    if with_bwd and bplan1.path in adds_dq:
        launches_per_step -= 1  # the dQ zero-fill is a memset, not one of our kernels
    if with_bwd and bplan2.path in adds_dq:
        launches_per_step -= 1

    for _ in range(args.warmup):
        step_on(ins, out)
    torch.cuda.synchronize()
    if streamkl.workspace_status(wsp):
        raise RuntimeError("device error word set during warm-up")

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    barrier(ws_)
    torch.cuda.synchronize()
    with ClockSampler(gpu_id(dev)) as clk:
        for k in range(args.steps):
            flush_l2(l2_flush)
            e = ev[k]
            e[0].record(stream)
            streamkl.kl_fwd(Q1, K1, Q2, K2, causal=w.causal, workspace=wsp, out=(out["KL"], out["LSE1"], out["LSE2"]))
            e[1].record(stream)
            if with_bwd:
                streamkl.kl_bwd(1, g, Q1, K1, Q2, K2, out["KL"], out["LSE1"], out["LSE2"], causal=w.causal,
                                workspace=wsp, out=(out["dQ2"], out["dK2"]))
            e[2].record(stream)
            if with_bwd:
                streamkl.kl_bwd(2, g, Q1, K1, Q2, K2, out["KL"], out["LSE1"], out["LSE2"], causal=w.causal,
                                workspace=wsp, out=(out["dQ1"], out["dK1"]))
            e[3].record(stream)
        torch.cuda.synchronize()
    barrier(ws_)
    step_clocks = clk.summary()
    status = streamkl.workspace_status(wsp)
    fwd_ms = statistics.median(e[0].elapsed_time(e[1]) for e in ev)
    b1_ms = statistics.median(e[1].elapsed_time(e[2]) for e in ev)
    b2_ms = statistics.median(e[2].elapsed_time(e[3]) for e in ev)
    step_ms = sum(e[0].elapsed_time(e[3]) for e in ev) / args.steps
    step_ms = max_over_ranks(step_ms, ws_, dev)

    # work of the whole problem (every rank's heads) and of this rank's share
    pairs_all = w.visible_pairs() * w.B * w.H
    pairs = w.visible_pairs() * Hq
    f_fwd, f_bwd = 4 * d * pairs, 8 * d * pairs
    step_flops_all = 4 * d * pairs_all + (2 * 8 * d * pairs_all if with_bwd else 0)
    value = step_flops_all / (step_ms * 1e-3) / 1e12
    peak_tf = peaks["bf16_tflops"]
    peak_sus = peaks.get("bf16_tflops_sustained", PEAKS_FALLBACK["bf16_tflops_sustained"])
    share = (stop - start) / (w.B * (w.H_kv or w.H))
    fwd_bytes, bwd_bytes = w.fwd_bytes() * share, w.bwd_bytes() * share
    kernels = {"fwd": {"ms": fwd_ms, "tflops": f_fwd / fwd_ms / 1e9, "frac_bf16_peak": f_fwd / fwd_ms / 1e9 / peak_tf,
                       "frac_bf16_sustained": f_fwd / fwd_ms / 1e9 / peak_sus,
                       "gbs": fwd_bytes / fwd_ms / 1e6, "frac_hbm_peak": fwd_bytes / fwd_ms / 1e6 / peaks["hbm_gbs"],
                       "path": "tile" if fplan.path == 0 else "decode", "splits": fplan.num_splits}}
    if with_bwd:
        for name, ms, plan in (("bwd_setting1", b1_ms, bplan1), ("bwd_setting2", b2_ms, bplan2)):
            kernels[name] = {"ms": ms, "tflops": f_bwd / ms / 1e9, "frac_bf16_peak": f_bwd / ms / 1e9 / peak_tf,
                             "frac_bf16_sustained": f_bwd / ms / 1e9 / peak_sus,
                             "gbs": bwd_bytes / ms / 1e6, "frac_hbm_peak": bwd_bytes / ms / 1e6 / peaks["hbm_gbs"],
                             "mode": BWD_MODE_NAMES[plan.path]}
    # Roofline of the dominant kernel (largest share of the step), timed live
    # with CUDA events around its call on the launching stream.  Forward call =
    # one fwd_tile_kernel launch (4*d flops per visible pair), or for decode one
    # fwd_decode_kernel + combine launch bounded by HBM (every Q/K byte once);
    # fused backward call = dQ zero-fill + one bwd_kv_kernel launch carrying the
    # whole backward (8*d flops per visible pair); split = bwd_q + bwd_kv;
    # key-split (at most 16 query rows per key head) = dQ zero-fill + one
    # bwd_decode_kernel launch, bounded by HBM like the decode forward.
    def bwd_name(plan, setting):
        if plan.path == streamkl.PATH_BWD_FUSED:
            return f"bwd_kv_kernel<setting {setting}, fused>"
        if plan.path == streamkl.PATH_BWD_KEYSPLIT:
            return f"bwd_decode_kernel<setting {setting}>"
        return f"bwd_q_kernel + bwd_kv_kernel (setting {setting})"

    names = {"fwd": "fwd_tile_kernel" if fplan.path == 0 else "fwd_decode_kernel + combine_kernel",
             "bwd_setting1": bwd_name(bplan1, 1), "bwd_setting2": bwd_name(bplan2, 2)}
    top = max(kernels, key=lambda k: kernels[k]["ms"])
    # traffic is per launch of the full problem on one GPU; a shard's launch moves its share
    traffic = traffic_for(w.name, top)
    traffic = traffic * share if traffic is not None else None
    # a decode-shaped problem (at most 16 query rows) moves ~1 (N_Q = 1) to ~16 flops per
    # byte in either direction, far below the ridge: HBM bounds its kernels
    if Nq <= 16:
        nbytes = fwd_bytes if top == "fwd" else bwd_bytes
        achieved = nbytes / kernels[top]["ms"] / 1e6
        roofline = {"kernel": names[top], "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                    "share_of_step": kernels[top]["ms"] / step_ms, "bytes_per_launch": nbytes,
                    "peak_source": f"hbm_gbs ({peak_src})"}
    else:
        flops_top = f_fwd if top == "fwd" else f_bwd
        achieved = flops_top / kernels[top]["ms"] / 1e9
        # frac: of the measured burst GEMM rate; the sustained (seconds-long, at the
        # power cap) rate is reported beside it
        roofline = {"kernel": names[top], "bound": "tensor", "achieved": achieved, "peak": peak_tf,
                    "unit": "TFLOP/s", "frac": achieved / peak_tf, "frac_sustained": achieved / peak_sus,
                    "peak_sustained": peak_sus, "traffic": traffic,
                    "traffic_kernel_hash": source_hash("fwd" if top == "fwd" else "bwd"),
                    "share_of_step": kernels[top]["ms"] / step_ms, "flops_per_launch": flops_top,
                    "peak_source": f"bf16_tflops ({peak_src}, burst)"}

    # ---------------- joint backward: both sides from one recompute per kernel,
    # timed on its own against the two single-setting passes of the step
    joint = None
    if with_bwd and not args.no_joint:
        jplan = streamkl.bwd_joint_plan(Q1, K1, causal=w.causal)
        jout = (out["dQ1"], out["dK1"], out["dQ2"], out["dK2"])

        def joint_call():
            streamkl.kl_bwd_joint(g, Q1, K1, Q2, K2, out["KL"], out["LSE1"], out["LSE2"], causal=w.causal,
                                  workspace=wsp, out=jout)

        for _ in range(2):
            joint_call()
        jt = []
        for _ in range(max(3, args.steps // 2)):
            flush_l2(l2_flush)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            joint_call()
            b.record(stream)
            torch.cuda.synchronize()
            jt.append(a.elapsed_time(b))
        jms = max_over_ranks(statistics.median(jt), ws_, dev)
        joint = {"ms": jms, "two_single_setting_passes_ms": b1_ms + b2_ms,
                 "tflops_12d": 12 * d * pairs / jms / 1e9, "frac_bf16_peak_12d": 12 * d * pairs / jms / 1e9 / peak_tf,
                 "kernels": "bwd_q_joint_kernel + bwd_kv_joint_kernel", "launches": jplan.launches,
                 "note": "12*d flops per visible pair: one recompute (4d) and four gradient GEMMs (8d)"}
        if streamkl.workspace_status(wsp):
            raise RuntimeError("device error word set by the joint backward")

    # ---------------- end to end through the C ABI with host buffers
    # Every step copies its inputs from pinned host memory and reads back all it
    # returns (KL, LSE1, LSE2 and, with the backward, dQ/dK of both settings).
    # Inputs and outputs are double-buffered on the device: step k+1's inputs
    # are copied in on one side stream and step k's outputs copied out on
    # another while the kernels run.  The timed region starts before the first
    # input copy and ends after the last output copy.
    host_in = tuple(t.cpu().pin_memory() for t in ins)
    host_out = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in out.items()}
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out.values())
    in_sets = [ins, tuple(torch.empty_like(t) for t in ins)]
    out_sets = [out, outputs()]
    h2d_stream, d2h_stream = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    copied, freed = [torch.cuda.Event(), torch.cuda.Event()], [torch.cuda.Event(), torch.cuda.Event()]
    computed, read_out = [torch.cuda.Event(), torch.cuda.Event()], [torch.cuda.Event(), torch.cuda.Event()]

    # per-step copy durations inside the loop, where they run beside the kernels
    copy_ev = {"h2d": [], "d2h": [], "compute": []}

    def timed_event():
        return torch.cuda.Event(enable_timing=True)

    def issue_copy_in(k, after=None):
        slot = k % 2
        with torch.cuda.stream(h2d_stream):
            if after is not None:
                h2d_stream.wait_event(after)
            if k >= 2:
                h2d_stream.wait_event(freed[slot])  # step k-2 is done with this input set
            t0 = timed_event()
            t0.record(h2d_stream)
            for dst, src in zip(in_sets[slot], host_in):
                dst.copy_(src, non_blocking=True)
            copied[slot].record(h2d_stream)
            t1 = timed_event()
            t1.record(h2d_stream)
            copy_ev["h2d"].append((t0, t1))

    def run_e2e(n, start_ev=None):
        for v in copy_ev.values():
            v.clear()
        issue_copy_in(0, after=start_ev)
        for k in range(n):
            slot = k % 2
            stream.wait_event(copied[slot])
            if k >= 2:
                stream.wait_event(read_out[slot])  # step k-2's outputs have been copied out
            c0 = timed_event()
            c0.record(stream)
            step_on(in_sets[slot], out_sets[slot])
            c1 = timed_event()
            c1.record(stream)
            copy_ev["compute"].append((c0, c1))
            freed[slot].record(stream)
            computed[slot].record(stream)
            with torch.cuda.stream(d2h_stream):
                d2h_stream.wait_event(computed[slot])
                t0 = timed_event()
                t0.record(d2h_stream)
                for key, t in out_sets[slot].items():
                    host_out[key].copy_(t, non_blocking=True)
                read_out[slot].record(d2h_stream)
                t1 = timed_event()
                t1.record(d2h_stream)
                copy_ev["d2h"].append((t0, t1))
            if k + 1 < n:
                issue_copy_in(k + 1)
        stream.wait_event(read_out[(n - 1) % 2])

    def copy_alone(fn, s):
        """One step's copies in one direction, timed alone on their stream."""
        ms = None
        for _ in range(2):  # the second, warm, copy is the one kept
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            a.record(s)
            with torch.cuda.stream(s):
                fn()
            b.record(s)
            torch.cuda.synchronize()
            ms = a.elapsed_time(b)
        return ms

    h2d_ms = copy_alone(lambda: [dst.copy_(src, non_blocking=True) for dst, src in zip(in_sets[1], host_in)],
                        h2d_stream)
    d2h_ms = copy_alone(lambda: [host_out[k].copy_(t, non_blocking=True) for k, t in out_sets[1].items()], d2h_stream)

    run_e2e(2)
    torch.cuda.synchronize()
    barrier(ws_)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(gpu_id(dev)) as e2e_clk:
        a.record(stream)
        run_e2e(args.steps, start_ev=a)
        b.record(stream)
        torch.cuda.synchronize()
    e2e_ms = max_over_ranks(a.elapsed_time(b) / args.steps, ws_, dev)
    in_loop = {d: statistics.median(x.elapsed_time(y) for x, y in copy_ev[d]) for d in ("h2d", "d2h", "compute")}
    e2e = {"value": step_flops_all / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": e2e_ms,
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "read_back": sorted(host_out), "clocks": e2e_clk.summary(),
           "copies_alone": {"h2d_ms": h2d_ms, "h2d_gbs": h2d / h2d_ms / 1e6, "d2h_ms": d2h_ms,
                            "d2h_gbs": d2h / d2h_ms / 1e6},
           "copies_in_loop": {"h2d_ms": in_loop["h2d"], "h2d_gbs": h2d / in_loop["h2d"] / 1e6,
                              "d2h_ms": in_loop["d2h"], "d2h_gbs": d2h / in_loop["d2h"] / 1e6},
           "kernels_in_loop_ms": in_loop["compute"]}
    kl_mean = float(host_out["KL"].double().mean())
    del in_sets, out_sets, host_in, host_out, out, ins, Q1, K1, Q2, K2, g
    torch.cuda.empty_cache()

    decode = run_decode_leg(args, dev, rank, ws_, peaks) if not args.no_decode else None

    result = None
    if rank == 0:
        result = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws_, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True,
            "scaling": "strong", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) teacher, student +0.3 N(0,1))",
            "config": config_for(w, ws_),
            "kernels": kernels, "roofline": roofline, "e2e": e2e, "gpu_launches": launches_per_step * args.steps,
            "device_error_word": status, "kl_mean": kl_mean,
            "peaks": {"bf16_tflops": peaks["bf16_tflops"], "bf16_tflops_sustained": peak_sus,
                      "hbm_gbs": peaks["hbm_gbs"], "source": peak_src},
        }
        if joint is not None:
            result["bwd_joint"] = joint
        if decode is not None:
            result.update(decode_ms=decode["ms"], decode_gbs=decode["gbs"], decode_frac_hbm=decode["frac_hbm"],
                          decode=decode)
        result["clocks"] = step_clocks
    return result, w


def run_decode_leg(args, dev, rank, world, peaks):
    """The N_Q=1 Split-K decode forward against 512K keys (B=4, H=32, d=128),
    timed after the headline step: every key byte is read once, so HBM bounds
    it.  Each rank takes its share of the 128 heads; GB/s counts the bytes of
    every rank over the slowest rank's median time."""
    from attention_kl_divergence_gb300 import streamkl
    w = WORKLOADS[DECODE_WORKLOAD]
    start, stop = rank_heads(w, rank, world)
    full = make_workload(w, device=dev)
    Q1, K1, Q2, K2 = (shard(t, start, stop).clone() for t in full)
    del full
    torch.cuda.empty_cache()
    plan = streamkl.fwd_plan(Q1, K1, causal=w.causal)
    wsp = streamkl.new_workspace(plan.workspace_bytes, dev)
    out = tuple(torch.empty((1, Q1.shape[1], w.Nq), dtype=torch.float32, device=dev) for _ in range(3))
    l2_flush = torch.empty(int(256e6) // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    reps = max(20, args.steps)
    for _ in range(max(3, args.warmup)):
        streamkl.kl_fwd(Q1, K1, Q2, K2, causal=w.causal, workspace=wsp, out=out)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    barrier(world)
    with ClockSampler(gpu_id(dev)) as clk:
        for a, b in ev:
            flush_l2(l2_flush)
            a.record(stream)
            streamkl.kl_fwd(Q1, K1, Q2, K2, causal=w.causal, workspace=wsp, out=out)
            b.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    ms = max_over_ranks(statistics.median(a.elapsed_time(b) for a, b in ev), world, dev)
    status = streamkl.workspace_status(wsp)
    gbs = w.fwd_bytes() / ms / 1e6
    del Q1, K1, Q2, K2, out, l2_flush
    torch.cuda.empty_cache()
    return {"workload": f"{w.name}: B={w.B} H={w.H} N_Q={w.Nq} N_K={w.Nk} d={w.d} non-causal, forward only",
            "ms": ms, "gbs": gbs, "frac_hbm": gbs / peaks["hbm_gbs"], "bytes_per_call": w.fwd_bytes(),
            "splits": plan.num_splits, "launches_per_call": plan.launches, "reps": reps,
            "kernel": "fwd_decode_kernel" + (" + combine_kernel" if plan.num_splits > 1 else ""),
            "device_error_word": status, "clocks": clk.summary(), "l2": "256 MB write between calls"}


def run_reference(args):
    """The float64 CPU oracle, as it stands, on the machine's host cores."""
    ws_, rank, _ = dist_env()
    if rank != 0:
        return None
    w = WORKLOADS[args.workload]
    for _ in range(args.warmup):
        cpu_oracle_sample(w, budget_s=0.5)
    vals = []
    for _ in range(args.steps):
        vals.append(cpu_oracle_sample(w, budget_s=max(2.0, 30.0 / max(1, args.steps))))
    v = statistics.median(x["value"] for x in vals)
    last = vals[-1]
    step_flops = (4 if w.fwd_only else 20) * w.d * w.visible_pairs() * w.B * w.H  # fwd 4d (+ 2 x 8d bwd)
    return {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": ws_, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_flops / (v * 1e12) * 1e3, "ms_per_step_kind": "extrapolated",
        "higher_is_better": True, "scaling": "strong", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded N(0,1) teacher, student +0.3 N(0,1))", "config": config_for(w, ws_),
        "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": last["cores"], "kind": "oracle",
                         "sample": last["sample"]},
        "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_ablations(args):
    """Design ablations, one JSON line each (not the benchmark contract line):
    the decode forward with its key range unsplit vs the automatic split, and
    the backward modes (fused, separate kernels, key-split) on the shapes each
    is meant for.  Medians of CUDA-event timings with L2 flushed before each."""
    from attention_kl_divergence_gb300 import streamkl

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    l2_flush = torch.empty(int(256e6) // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def timed(fn, reps):
        for _ in range(args.warmup):
            fn()
        ts = []
        for _ in range(reps):
            flush_l2(l2_flush)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        return statistics.median(ts)

    def emit(**kw):
        print(json.dumps(dict(ablation=True, **kw)), flush=True)

    # Split-K on the decode workloads: one CTA per head (splits = 1) vs the automatic choice
    for name in ("decode_q1_k128k", "decode_q16_k128k", "decode_q1_k512k", "decode_q16_k512k"):
        w = WORKLOADS[name]
        Q1, K1, Q2, K2 = make_workload(w, device=dev)
        out = tuple(torch.empty((w.B, w.H, w.Nq), dtype=torch.float32, device=dev) for _ in range(3))
        for splits in (1, 0):
            plan = streamkl.fwd_plan(Q1, K1, num_splits=splits)
            ms = timed(lambda: streamkl.kl_fwd(Q1, K1, Q2, K2, num_splits=splits, out=out), max(args.steps, 5))
            emit(what="decode split-K", workload=name, splits=plan.num_splits, ms=ms,
                 gbs=w.fwd_bytes() / ms / 1e6)
        del Q1, K1, Q2, K2
        torch.cuda.empty_cache()
    # backward modes
    modes = {"fused": streamkl.BWD_FUSED, "split": streamkl.BWD_SPLIT, "keysplit": streamkl.BWD_KEYSPLIT}
    for name, names in (("8k_causal", ("fused", "split")), ("64k_causal", ("fused", "split")),
                        ("decode_bwd_q16_k128k", ("keysplit", "fused", "split"))):
        w = WORKLOADS[name]
        Q1, K1, Q2, K2 = make_workload(w, device=dev)
        g = make_g(w.B, w.H, w.Nq, w.g_value, device=dev)
        KL, L1, L2 = streamkl.kl_fwd(Q1, K1, Q2, K2, causal=w.causal)
        grads = (torch.empty_like(Q1, dtype=torch.float32), torch.empty_like(K1, dtype=torch.float32))
        reps = 3 if w.Nq >= 65536 else max(args.steps, 5)
        if "fused" in names and w.Nq > 16:
            jo = tuple(torch.empty_like(t, dtype=torch.float32) for t in (Q1, K1, Q2, K2))
            ms = timed(lambda: streamkl.kl_bwd_joint(g, Q1, K1, Q2, K2, KL, L1, L2, causal=w.causal, out=jo), reps)
            emit(what="backward mode", workload=name, setting="both", mode="joint", ms=ms,
                 tflops_12d=12 * w.d * w.visible_pairs() * w.B * w.H / ms / 1e9)
            del jo
        for setting in (1, 2):
            for mname in names:
                ms = timed(lambda: streamkl.kl_bwd(setting, g, Q1, K1, Q2, K2, KL, L1, L2, causal=w.causal,
                                                   mode=modes[mname], out=grads), reps)
                emit(what="backward mode", workload=name, setting=setting, mode=mname, ms=ms,
                     tflops=8 * w.d * w.visible_pairs() * w.B * w.H / ms / 1e9, gbs=w.bwd_bytes() / ms / 1e6)
        del Q1, K1, Q2, K2, grads
        torch.cuda.empty_cache()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="streamkl", choices=["streamkl", "reference"])
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle leg")
    ap.add_argument("--no-decode", action="store_true", help="skip the N_Q=1 decode leg")
    ap.add_argument("--no-joint", action="store_true", help="skip timing the joint backward")
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(WORKLOADS),
                    help="another named workload (the headline metric is quoted on 64k_causal)")
    ap.add_argument("--ablate", action="store_true",
                    help="print the design ablations (split-K, backward modes) instead of the benchmark line")
    args = ap.parse_args()
    if args.ablate:
        run_ablations(args)
        return
    if args.warmup < 3 and args.impl != "reference":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        out = run_reference(args)
        if out is not None:
            print(json.dumps(out), flush=True)
        return
    # the oracle's thread pool starts before any CUDA call
    from oracle import oracle
    oracle.build()
    out, w = run_gpu(args)
    ws_, rank, _ = dist_env()
    if rank == 0:
        if ws_ == 1 and not args.no_cpu:
            out["cpu_baseline"] = cpu_oracle_sample(w)
        print(json.dumps(out), flush=True)
    if ws_ > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
