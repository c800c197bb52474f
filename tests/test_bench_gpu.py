"""The bench line on a GPU: one short run of the default op and of the
attention op, checked against the JSON contract (every key, the roofline
object with a traffic figure from a committed profile of the same source, the
CPU baseline, the end-to-end figure, launches and clocks)."""
import json
import os
import subprocess
import sys

import pytest

import bench

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = ["metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
        "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks"]


def bench_line(*args):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


def check_common(line, steps):
    missing = [k for k in KEYS if k not in line]
    assert not missing, missing
    assert line["n_gpus"] == 1 and line["steps"] == steps and line["warmup"] == 3
    assert line["value"] > 0 and line["ms_per_step"] > 0 and line["higher_is_better"] is True
    assert line["scaling"] == "weak" and line["vs_baseline"] is None and line["data"] == "synthetic"
    assert "workload" in line["config"]
    rf = line["roofline"]
    for k in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert k in rf, k
    assert 0 < rf["frac"] < 1.2 and abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-9
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] > 0 and cb["sample"]
    e2e = line["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert line["gpu_launches"] >= steps
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(line["clocks"])


def test_default_bench_line():
    line = bench_line("--steps", "200", "--warmup", "3", "--cpu-budget", "0.2")
    check_common(line, 200)
    assert line["config"]["workload"] == "bf16_16384x4096"
    assert line["unit"] == "GB/s" and line["roofline"]["bound"] == "hbm"
    # the committed profile matches this source, so the DRAM bytes are reported
    traffic, _ = bench.profile_traffic("bf16_16384x4096", "softmax")
    assert line["roofline"]["traffic"] == traffic
    assert line["gpu_launches"] == 200


def test_attention_bench_line():
    line = bench_line("--op", "attention", "--steps", "5", "--warmup", "3", "--cpu-budget", "0.2")
    check_common(line, 5)
    assert line["unit"] == "TFLOP/s" and line["roofline"]["bound"] == "tensor"
    traffic, _ = bench.profile_traffic("attn_bf16_4x32x4096x128", "attention")
    assert line["roofline"]["traffic"] == traffic
