"""Host-side logic of bench.py, on CPU: the whole-job aggregation, the
max-over-ranks timing with two gloo ranks, the L2 rotation, the reference
arm's JSON line (fp64 CPU reference only, no GPU), the clock sampler's
parsing and throttle reasons, the profile lookup's source-hash gate and the
measured-peak fallback."""
import json
import os
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_aggregate_is_whole_job():
    a = bench.aggregate(bytes_per_step=1000, rows_per_step=10, steps=4, world=2, seconds=2.0)
    assert a["gbs"] == 1000 * 4 * 2 / 2.0 / 1e9
    assert a["rows_per_s"] == 10 * 4 * 2 / 2.0


def test_rotation_covers_l2():
    for set_bytes in (512_000, 64 * 2**20, 268_435_456, 4 * 2**30):
        n = bench.rotation_sets(set_bytes)
        assert 2 <= n <= 16
        assert (n - 1) * set_bytes >= bench.L2_BYTES or n == 16


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        out[rank] = bench.max_over_ranks(1.5 + rank, world)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    import socket

    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == out[1] == 2.5


def test_reference_arm_json_line():
    env = dict(os.environ, RANK="0", WORLD_SIZE="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "f32_64x1000", "--steps", "3", "--warmup", "3",
                        "--ref-budget", "1"], capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "GB/s"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "f32_64x1000", "--steps", "3", "--warmup", "3"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_bench_rejects_too_few_warmups():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])


def test_attention_flops_count_valid_pairs():
    """4 head_dim FLOPs per valid (query, key) pair, the pairs counted by brute
    force over the mask the attention entry point documents."""
    from numerically_stable_online_gb300 import workloads as wl

    for sq, sk in [(1, 1), (3, 5), (5, 3), (7, 7), (4, 0)]:
        for causal in (False, True):
            brute = sum(1 for i in range(sq) for j in range(sk) if not causal or j <= i + sk - sq)
            assert wl.attention_pairs(sq, sk, causal) == brute
            assert wl.attention_flops(2, sq, sk, 64, causal) == 4.0 * 2 * 64 * brute


@pytest.mark.parametrize("op", ["softmax", "apply_stats", "backward", "cross_entropy"])
def test_cpu_reference_on_all_cores(op):
    """The all-cores CPU baseline: one contiguous slice of rows per core of the
    affinity, in spawned workers; every op's extra inputs are sliced with the rows."""
    from numerically_stable_online_gb300 import workloads as wl

    w = wl.WORKLOADS["f16_32768x1024_len"]
    x, vl = wl.host_input(w.name, rows=64)
    import dataclasses

    w = dataclasses.replace(w, rows=64)
    gbs, cores = bench.oracle_all_cores(x, vl, w, 48, op)
    assert gbs > 0 and 1 <= cores <= min(48, len(os.sched_getaffinity(0)))


class _FakeSmi:
    """Stands in for the nvidia-smi process: canned CSV samples."""

    def __init__(self, lines):
        self.lines = lines
        self.terminated = False

    def terminate(self):
        self.terminated = True

    def communicate(self, timeout=None):
        return "\n".join(self.lines) + "\n", None


def _sample(sm, reasons=("Not Active",) * 4):
    return ", ".join(["0", str(sm), "2070", "900.5", "0x0000000000000000", *reasons])


def test_clock_sampler_median_and_reasons():
    import time

    cs = bench.ClockSampler(0)
    cs.t0 = time.time() - 1.0
    lines = [_sample(2070), _sample(2055), _sample(1980, ("Not Active", "Not Active", "Not Active", "Active")),
             "garbage line", _sample(2070)]
    cs.proc = _FakeSmi(lines)
    rec = cs.stop(t_begin=cs.t0 - 1, t_end=time.time() + 1)
    assert cs.proc.terminated
    assert rec["sm_mhz"] == 2062.5 and rec["sm_max_mhz"] == 2070.0
    assert rec["reasons"] == ["sw_power_cap"] and rec["samples"] == 4
    cs = bench.ClockSampler(0)
    cs.t0 = time.time() - 1.0
    cs.proc = _FakeSmi([_sample(1500, ("Active", "Not Active", "Active", "Not Active"))])
    rec = cs.stop(cs.t0 - 1, time.time() + 1)
    assert rec["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]


def test_clock_sampler_without_nvidia_smi():
    cs = bench.ClockSampler(0)
    rec = cs.stop(0.0, 1.0)
    assert rec["sm_mhz"] is None and rec["reasons"] == ["nvidia-smi unavailable"]


def test_profile_traffic_follows_the_source_hash(monkeypatch, tmp_path):
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "softmax_wl_a.md").write_text(
        "# ncu\n\nkernel: k_rows_stream<bf16,bf16>\nsource_hash: 0123456789abcdef\n"
        "dram_bytes_per_launch: 212694912\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "source_hash", lambda files=None: "0123456789abcdef")
    assert bench.profile_traffic("wl_a", "softmax") == (212694912, "k_rows_stream<bf16,bf16>")
    monkeypatch.setattr(bench, "source_hash", lambda files=None: "fedcba9876543210")
    # taken on other sources: the kernel is named, the traffic is not reported
    assert bench.profile_traffic("wl_a", "softmax") == (None, "k_rows_stream<bf16,bf16>")
    assert bench.profile_traffic("no_such_workload", "softmax") == (None, None)


def test_measured_peak_and_fallback(monkeypatch, tmp_path):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_peak("hbm_gbs") == (6800.0, "fallback")
    assert bench.measured_peak("bf16_tflops") == (1900.0, "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6689.1, "bf16_tflops": 1939.3}))
    assert bench.measured_peak("hbm_gbs") == (6689.1, "measured")
    assert bench.measured_peak("bf16_tflops") == (1939.3, "measured")


# ---------------------------------------------------------------------------
# The bench line's parity statistics and in-region clock summary.
# ---------------------------------------------------------------------------

def _reference_rows(in_dtype, rows, cols, seed, masked=False):
    import numpy as np

    import oracle
    from numerically_stable_online_gb300 import workloads as wl

    oracle.build()
    rng = np.random.default_rng(seed)
    x = wl.to_storage(rng.normal(0, 5, rows * cols).astype(np.float32), in_dtype)
    vl = rng.integers(0, cols + 1, rows).astype(np.int32) if masked else None
    return x, vl, oracle.softmax_rows(x, in_dtype, rows, cols, vl)


def test_parity_stats_pass_the_reference_and_catch_planted_mistakes():
    import numpy as np

    import oracle

    rows, cols = 12, 64
    x, vl, p = _reference_rows("f32", rows, cols, 3, masked=True)
    y = p.astype(np.float32)
    st = bench.parity_stats(y, p, "f32", vl)
    assert st["within_tolerance"] and st["masked_zero_ok"] and st["max_rel"] <= 6e-8
    bad = y.copy()
    bad[0, 0] *= 1 + 4e-6  # one element 4e-6 off
    assert not bench.parity_stats(bad, p, "f32", vl)["within_tolerance"]
    bad = y.copy()
    L = np.clip(vl, 0, cols)
    r = int(np.argmax(L < cols))
    bad[r, cols - 1] = 1e-9  # a masked lane written
    st = bench.parity_stats(bad, p, "f32", vl)
    assert not st["masked_zero_ok"] and not st["within_tolerance"]
    # 16-bit outputs: correctly rounded bits pass, two units off fail
    x16, _, p16 = _reference_rows("bf16", rows, cols, 4)
    bits = oracle.round_to(p16, "bf16")
    st = bench.parity_stats(bits, p16, "bf16")
    assert st["within_tolerance"] and st["max_ulp"] == 0 and st["frac_exact"] == 1.0
    bits2 = bits.copy()
    bits2[3, 5] += 2
    st = bench.parity_stats(bits2, p16, "bf16")
    assert st["max_ulp"] == 2 and not st["within_tolerance"]


def test_clock_samples_summarised_inside_the_region_only():
    lines = ["100.000100 1980 2070 0", "100.000300 2070 2070 4", "100.000500 2070 2070 0",
             "100.000900 1200 2070 8", "garbage", "101.5 500 2070 40"]
    c = bench.summarize_clock_samples(lines, 100.0, 100.0006)
    assert c["samples"] == 3 and c["sm_mhz"] == 2070 and c["sm_max_mhz"] == 2070
    assert c["reasons"] == ["sw_power_cap"] and not c["rejected"]
    c = bench.summarize_clock_samples(lines, 100.0, 100.001)
    assert "hw_slowdown" in c["reasons"] and c["rejected"]
    assert bench.summarize_clock_samples(lines, 200.0, 201.0)["samples"] == 0
