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
    # the timed output against the reference, all rows
    assert line["parity"]["within_tolerance"] and line["parity"]["rows"] == 16384
    assert line["parity"]["max_ulp"] <= 1 and line["parity"]["masked_zero_ok"]
    # every other workload of the bandwidth target, same steps, with its parity
    per = {e["workload"]: e for e in line["per_config"]}
    assert set(per) == {"f32_64x1000", "f16_32768x1024_len", "f32_64x1048576_rise"}
    for name, e in per.items():
        w = bench.wl.WORKLOADS[name]
        assert e["value"] > 0 and e["ms_per_step"] > 0 and 0 < e["roofline"]["frac"] < 1.2
        assert e["parity"]["within_tolerance"], (name, e["parity"])
        assert e["parity"]["rows"] == w.rows
        assert "max_rel" in e["parity"] if w.out_dtype == "f32" else "max_ulp" in e["parity"]
    assert per["f32_64x1048576_rise"]["path"] == "stripe"
    assert per["f32_64x1048576_rise"]["kernels_per_step"] == 1


def test_clocks_sampled_inside_a_short_region():
    """A 20-step region lasts about a millisecond: the NVML sampler still sees it."""
    line = bench_line("--steps", "20", "--warmup", "3", "--cpu-budget", "0.2", "--per-config", "0",
                      "--cpu-all-cores", "0")
    c = line["clocks"]
    assert c["samples"] >= 5 and c["sm_mhz"] > 0 and c["source"].startswith("NVML")


def test_attention_bench_line():
    line = bench_line("--op", "attention", "--steps", "5", "--warmup", "3", "--cpu-budget", "0.2")
    check_common(line, 5)
    assert line["unit"] == "TFLOP/s" and line["roofline"]["bound"] == "tensor"
    traffic, _ = bench.profile_traffic("attn_bf16_4x32x4096x128", "attention")
    assert line["roofline"]["traffic"] == traffic
