"""bench.py's JSON line on a GPU, for one small workload: the keys the benchmark contract asks for,
a roofline entry whose fraction follows from its own numbers, the e2e copies declared, and the
launch count the library reports."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_line_for_the_micro_workload():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "micro",
                          "--steps", "4", "--warmup", "3", "--no-cpu-baseline"],
                         capture_output=True, text=True, timeout=600, check=True, cwd=ROOT).stdout
    lines = [l for l in out.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "e2e", "gpu_launches", "graph", "clocks", "fp32_ffma_tflops"):
        assert key in d, key
    assert d["steps"] == 4 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["config"]["workload"] == "micro" and "l2" in d["config"]
    assert d["value"] == pytest.approx(256 / (d["ms_per_step"] * 1e-3), rel=1e-6)
    r = d["roofline"]
    assert r["bound"] == "alu" and r["unit"] == "TFLOP/s"
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"], rel=1e-9)
    assert 0 < r["frac"] < 1
    assert r["peak"] == pytest.approx(d["fp32_ffma_tflops"]["tflops"])
    e2e = d["e2e"]
    assert e2e["h2d_bytes_per_step"] == 256 * 128 * 4
    assert e2e["d2h_bytes_per_step"] == 256 * 128 * 4 + 4
    assert d["gpu_launches"] == 4 * 4   # four kernels per micro step
    assert d["clocks"]["samples"] >= 0
    # the backward of the same f32 layer (recomputing its pre-activations on the CUDA cores)
    b = d["backward"]
    assert b["pre_activations"] == "recomputed"
    assert b["roofline"]["bound"] in ("alu", "hbm") and 0 < b["roofline"]["frac"] < 1
    assert b["value"] == pytest.approx(256 / (b["ms_per_step"] * 1e-3), rel=1e-6)
    assert b["launches_per_step"] == 16 and b["gpu_launches"] == 16 * 4
    assert b["train_step"]["ms_per_step"] > 0
