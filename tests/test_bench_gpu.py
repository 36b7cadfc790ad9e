"""The benchmark's JSON line: one short run of bench.py on the 8K causal
workload (in a subprocess, as the driver runs it) must print one line with
the contract's keys, a burst-peak roofline of the dominant kernel, an
end-to-end leg that copies inputs in and every output back, and the joint
backward's timing."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_line_on_8k_causal():
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "8k_causal", "--steps", "3", "--warmup", "3",
           "--no-cpu", "--no-decode"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches", "clocks", "kernels"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3 and d["scaling"] == "strong"
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["device_error_word"] == 0
    assert d["gpu_launches"] == 3 * 3  # forward, two fused backward launches per step
    roof = d["roofline"]
    assert roof["bound"] == "tensor" and roof["unit"] == "TFLOP/s" and roof["peak"] == d["peaks"]["bf16_tflops"]
    assert abs(roof["frac"] - roof["achieved"] / roof["peak"]) < 1e-9
    assert 0.0 < roof["frac"] < 1.2
    assert roof["traffic"] is None  # no capture is recorded for this workload
    e2e = d["e2e"]
    assert e2e["h2d_bytes_per_step"] == 4 * 32 * 8192 * 128 * 2 + 32 * 8192 * 4  # Q1, K1, Q2, K2, g
    assert e2e["d2h_bytes_per_step"] == 3 * 32 * 8192 * 4 + 4 * 32 * 8192 * 128 * 4  # KL, LSEs, four gradients
    assert e2e["value"] > 0 and e2e["value"] <= d["value"] * 1.05
    assert e2e["copies_alone"]["h2d_gbs"] > 0 and e2e["copies_alone"]["d2h_gbs"] > 0
    assert e2e["copies_in_loop"]["h2d_ms"] > 0 and e2e["copies_in_loop"]["d2h_ms"] > 0
    assert e2e["kernels_in_loop_ms"] > 0
    assert d["bwd_joint"]["ms"] > 0 and d["bwd_joint"]["launches"] == 2
    assert d["clocks"]["sm_mhz"] is None or d["clocks"]["sm_mhz"] > 0
