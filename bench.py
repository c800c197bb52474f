"""Benchmark: row softmax throughput on GB300 (algorithmic GB/s and rows/s).

A step is one pass of the whole hot path (the row softmax) over one batch of
the synthetic workload; the default workload is bf16 16384 x 4096 (N(0, 8^2)
logits, no mask).  Inputs are resident in HBM when the timed region starts; to
keep every step's reads and writes coming from HBM rather than L2, steps rotate
over several input/output buffer sets whose combined size is far above L2.

Prints one JSON line on rank 0:
  value        algorithmic bytes (valid input read once + output written once
               + row lengths) of all ranks' steps / max-over-ranks timed region
  e2e          the same metric end to end from pinned host memory: the softmax
               through its host-buffer call (the kernel reads and writes the
               mapped pinned buffers in place over the host link), the other
               ops through the device call with the copies around it, every step
  roofline     the softmax kernel's achieved bandwidth (CUDA events around every
               launch in the timed region) against the measured HBM copy peak
  cpu_baseline the fp64 CPU reference timed on this host on a bounded sample
  parity       the timed output buffer against the fp64 reference, all rows:
               max relative error (fp32) or max ulp (fp16/bf16), max |1 - sum|,
               masked lanes +0, and whether the bars are met
  per_config   (softmax, one GPU) the same throughput, roofline and parity for
               every workload of the bandwidth target, each timed over the same
               --steps after the same --warmup
  clocks       SM clock and clock-event reasons sampled through NVML every
               100 us inside the timed region, from a child process

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                       [--workload NAME] [--op softmax|log_softmax|lse|apply_stats|
                                              backward|cross_entropy]
--op times another entry point on the same workload (default: the softmax);
its bytes are that operation's algorithmic bytes (workloads.op_bytes).
For N > 1 it runs under torch.distributed.run, one independent replica per GPU.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from numerically_stable_online_gb300 import workloads as wl  # noqa: E402

METRIC = "softmax GB/s (read+write) and rows/s on 1 GB300; % of HBM peak"
UNIT = "GB/s"
L2_BYTES = 129 * 10 ** 6
LAUNCH_SAMPLE = 8
PATHS = {"auto": 0, "regs": 1, "cluster": 2, "generic": 3, "stream": 4, "split": 5, "stripe": 6}
PATH_NAMES = {v: k for k, v in PATHS.items()}
KERNEL_SOURCES = ["smx_device.cuh", "smx_async.cuh", "row_core.cuh", "kernel_regs.cuh",
                  "kernel_stream.cuh", "kernel_cluster.cuh", "kernel_generic.cuh",
                  "kernel_backward.cuh", "kernel_split_fused.cuh", "kernel_stripe.cuh", "launch_impl.cuh",
                  "smx_api.cu"]
ATTN_SOURCES = ["smx_device.cuh", "smx_async.cuh", "kernel_attention.cuh", "kernel_attention_tc.cuh",
                "kernel_attention_tma.cuh", "inst_attention.cu", "smx_api.cu"]


def metric_of(op: str) -> str:
    if op == "softmax":
        return METRIC
    return f"{op} GB/s (algorithmic bytes read+write) and rows/s on 1 GB300; % of HBM peak"


# ---------------------------------------------------------------------------
# Helpers that need no GPU (covered by the CPU tests).
# ---------------------------------------------------------------------------

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def max_over_ranks(value: float, world: int) -> float:
    """Largest value over all ranks (the job is as slow as its slowest rank)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(bytes_per_step: int, rows_per_step: int, steps: int, world: int, seconds: float):
    """Whole-job throughput: every rank processes its own replica of the batch."""
    total_bytes = bytes_per_step * steps * world
    return {"gbs": total_bytes / seconds / 1e9, "rows_per_s": rows_per_step * steps * world / seconds}


def rotation_sets(bytes_per_set: int, l2_bytes: int = L2_BYTES) -> int:
    """Buffer sets to rotate over so a set is evicted from L2 before its reuse."""
    return max(2, min(16, -(-3 * l2_bytes // max(1, bytes_per_set)) + 1))


def source_hash(files=None) -> str:
    h = hashlib.sha256()
    for f in files or KERNEL_SOURCES:
        with open(os.path.join(ROOT, "numerically_stable_online_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profile_traffic(workload: str, op: str = "softmax"):
    """DRAM bytes per launch of the dominant kernel from the committed ncu summary,
    or None when there is none or the kernel sources changed since it was taken."""
    path = os.path.join(ROOT, "profiles", f"{op}_{workload}.md")
    if not os.path.exists(path):
        return None, None
    text = open(path).read()
    mh = re.search(r"source_hash:\s*([0-9a-f]+)", text)
    mt = re.search(r"dram_bytes_per_launch:\s*([0-9]+)", text)
    mk = re.search(r"kernel:\s*(\S+)", text)
    if not mh or not mt or mh.group(1) != source_hash(ATTN_SOURCES if op == "attention" else None):
        return None, mk.group(1) if mk else None
    return int(mt.group(1)), mk.group(1) if mk else None


def measured_peak(kind: str = "hbm_gbs"):
    """The measured peak (HBM copy GB/s, or bf16 TFLOP/s burst), else the fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            return float(json.load(fh)[kind]), "measured"
    return (6800.0 if kind == "hbm_gbs" else 1900.0), "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.t0 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        self.t0 = time.time()
        time.sleep(0.4)

    def stop(self, t_begin: float, t_end: float):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        lines = [ln for ln in out.splitlines() if ln.strip()]
        # samples arrive every ~100 ms from t0; attribute times by order
        n = len(lines)
        t_last = time.time()
        samples = []
        for i, ln in enumerate(lines):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            ts = self.t0 + (t_last - self.t0) * (i + 0.5) / max(n, 1)
            samples.append((ts, parts))
        inside = [p for ts, p in samples if t_begin - 0.15 <= ts <= t_end + 0.15] or \
            [p for _, p in samples]
        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(p[1]) for p in inside if num(p[1]) is not None]
        smax = [num(p[2]) for p in inside if num(p[2]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for p in inside:
            for name, v in zip(names, p[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(inside)}


# NVML clock-event reason bits (read only; nvmlDeviceGetCurrentClocksEventReasons)
NVML_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}
REJECT_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


def nvml_sampler_main(device: str, path: str) -> int:
    """Child process: poll the GPU's SM clock and clock-event reasons through
    NVML (read-only queries) into `path`, one line per sample ("wall_time
    sm_mhz max_mhz reasons_hex"): every 100 us after the parent writes "f" to
    stdin (a timed region starts), every 20 ms after "s", until stdin closes.
    A process of its own, so the polling never takes the launching thread's
    interpreter lock."""
    import ctypes
    import select

    try:
        nv = ctypes.CDLL("libnvidia-ml.so.1")
    except OSError:
        print("error no-nvml", flush=True)
        return 0
    if nv.nvmlInit_v2() != 0:
        print("error init", flush=True)
        return 0
    h = ctypes.c_void_p()
    if device.startswith("GPU-"):
        rc = nv.nvmlDeviceGetHandleByUUID(device.encode(), ctypes.byref(h))
    else:
        rc = nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(int(device)), ctypes.byref(h))
    if rc != 0:
        print("error handle", flush=True)
        return 0
    reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
        getattr(nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
    mhz, mx, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
    nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))
    interval = 0.02
    with open(path, "w") as out:
        print("ready", flush=True)
        t_next = 0.0
        while True:
            # slow mode blocks on stdin until the next sample is due, so a
            # switch to fast mode is seen at once; fast mode only peeks
            wait = 0.0 if interval < 1e-3 else max(0.0, t_next - time.time())
            if select.select([sys.stdin], [], [], wait)[0]:
                c = sys.stdin.read(1)
                if not c:
                    break
                interval = 1e-4 if c == "f" else 0.02
                t_next = 0.0
            t = time.time()
            if t < t_next:
                continue
            t_next = t + interval
            nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(mhz))
            reasons_fn(h, ctypes.byref(rs))
            out.write(f"{t:.6f} {mhz.value} {mx.value} {rs.value:x}\n")
    nv.nvmlShutdown()
    return 0


def summarize_clock_samples(lines, t_begin: float, t_end: float):
    """Clock summary of the samples taken inside [t_begin, t_end] (wall time)."""
    sm, smax, reasons = [], [], set()
    for ln in lines:
        parts = ln.split()
        if len(parts) != 4:
            continue
        try:
            t, mhz, mx, bits = float(parts[0]), float(parts[1]), float(parts[2]), int(parts[3], 16)
        except ValueError:
            continue
        if not t_begin <= t <= t_end:
            continue
        sm.append(mhz)
        smax.append(mx)
        for bit, name in NVML_REASONS.items():
            if bits & bit:
                reasons.add(name)
    return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
            "reasons": sorted(reasons), "samples": len(sm), "source": "NVML, polled in a child process",
            "rejected": bool(reasons & set(REJECT_REASONS))}


class NvmlSampler:
    """Clocks sampled through NVML in a child process for the whole GPU leg,
    every 100 us between fast() and slow(); window() summarises the samples
    inside one timed region."""

    def __init__(self, device: str):
        import tempfile

        self.device = device
        self.proc = None
        self.lines = None
        fd, self.path = tempfile.mkstemp(prefix="smx_clocks_", suffix=".txt")
        os.close(fd)

    def start(self):
        try:
            self.proc = subprocess.Popen([sys.executable, os.path.abspath(__file__), "--nvml-sampler",
                                          self.device, self.path],
                                         stdin=subprocess.PIPE, stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            first = self.proc.stdout.readline().strip()
        except OSError:
            first = "error spawn"
        if first != "ready":
            if self.proc is not None:
                self.proc.kill()
                self.proc.wait()
            self.proc = None
        return self.proc is not None

    def _send(self, c: str):
        if self.proc is not None:
            self.proc.stdin.write(c)
            self.proc.stdin.flush()

    def fast(self):
        self._send("f")
        time.sleep(0.002)  # the child has switched before the region starts

    def slow(self):
        self._send("s")

    def stop(self):
        if self.proc is not None:
            self.proc.communicate(timeout=30)
            self.proc = None
        try:
            with open(self.path) as fh:
                self.lines = fh.read().splitlines()
            os.unlink(self.path)
        except OSError:
            self.lines = self.lines or []

    def window(self, t_begin: float, t_end: float):
        return summarize_clock_samples(self.lines or [], t_begin, t_end)


def nvml_device_id(torch, dev) -> str:
    """NVML's name for the torch device: its UUID when torch reports one."""
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        if u and not u.startswith("GPU-"):
            u = "GPU-" + u
        return u
    except Exception:  # noqa: BLE001 - older torch: fall back to the index
        return str(dev.index or 0)


# ---------------------------------------------------------------------------
# Parity of a timed output with the fp64 reference (for the bench line).
# ---------------------------------------------------------------------------
F32_REL_TOL, F32_TINY, SUM_TOL, ULP_TOL = 2e-6, 1e-30, 1e-5, 1


def parity_stats(y, p, out_dtype, valid_len=None):
    """Error statistics of one softmax output against the fp64 reference p
    [n, cols]: max relative error (fp32, where p >= 1e-30), max distance in
    units in the last place from the correctly rounded value (fp16/bf16), max
    |1 - sum(y)| over rows with a valid lane, and whether masked and
    zero-probability lanes are +0 bit for bit and NaN rows NaN.
    `within_tolerance` applies the bars: fp32 2e-6 relative and 1e-5 on the
    sum, fp16/bf16 1 ulp."""
    import oracle

    n, cols = p.shape
    L = np.full(n, cols, np.int64) if valid_len is None else np.clip(np.asarray(valid_len, np.int64), 0, cols)
    masked = np.arange(cols)[None, :] >= L[:, None]
    nan_rows = np.isnan(p).any(axis=1)
    ok_lanes = ~nan_rows[:, None] & ~masked
    zero_lanes = ok_lanes & (p == 0)
    st = {"rows": int(n)}
    if out_dtype == "f32":
        y = np.asarray(y, np.float32).reshape(n, cols)
        bits = y.view(np.uint32)
        yv = y.astype(np.float64)
        big = ok_lanes & (p >= F32_TINY)
        rel = np.abs(yv[big] - p[big]) / p[big]
        st["max_rel"] = float(rel.max()) if rel.size else 0.0
        st["masked_zero_ok"] = bool(np.all(bits[masked] == 0) and np.all(bits[zero_lanes] == 0))
        st["nan_rows_ok"] = bool(np.all(np.isnan(yv[nan_rows[:, None] & ~masked])))
        small = ok_lanes & (p < F32_TINY)
        tiny_ok = bool(np.all((yv[small] >= 0) & (yv[small] <= 2 * F32_TINY)))
        normal = ~nan_rows & (L > 0) & (p.sum(axis=1) > 0)
        s = np.where(masked, 0.0, yv)[normal].sum(axis=1)
        st["max_sum_err"] = float(np.abs(s - 1.0).max()) if s.size else 0.0
        st["within_tolerance"] = bool(st["max_rel"] <= F32_REL_TOL and st["max_sum_err"] <= SUM_TOL and tiny_ok
                                      and st["masked_zero_ok"] and st["nan_rows_ok"]
                                      and np.all(bits[ok_lanes] >> 31 == 0))
    else:
        yb = np.asarray(y).view(np.uint16).reshape(n, cols).astype(np.int64)
        r = oracle.round_to(np.where(ok_lanes, p, 0.0), out_dtype).astype(np.int64)
        diff = np.abs(yb - r)[ok_lanes]
        st["max_ulp"] = int(diff.max()) if diff.size else 0
        st["frac_exact"] = float((diff == 0).mean()) if diff.size else 1.0
        st["masked_zero_ok"] = bool(np.all(yb[masked] == 0) and np.all(yb[zero_lanes] == 0))
        exp_all = 0x7C00 if out_dtype == "f16" else 0x7F80
        isnan = ((yb & exp_all) == exp_all) & ((yb & ~exp_all & 0x7FFF) != 0)
        st["nan_rows_ok"] = bool(np.all(isnan[nan_rows[:, None] & ~masked]))
        yv = oracle.decode(yb.astype(np.uint16), out_dtype).reshape(n, cols)
        normal = ~nan_rows & (L > 0) & (p.sum(axis=1) > 0)
        s = np.where(masked, 0.0, yv)[normal].sum(axis=1)
        st["max_sum_err"] = float(np.abs(s - 1.0).max()) if s.size else 0.0
        st["within_tolerance"] = bool(st["max_ulp"] <= ULP_TOL and st["masked_zero_ok"] and st["nan_rows_ok"]
                                      and np.all(yb[ok_lanes] >> 15 == 0))
    return st


def parity_of_output(y_store, x_host, w, vl):
    """parity_stats over all rows of the workload, in blocks of about 8M
    elements; the statistics are the worst over the blocks."""
    import oracle

    block_rows = max(1, (8 << 20) // w.cols)
    agg = {}
    for r0 in range(0, w.rows, block_rows):
        sel = np.arange(r0, min(w.rows, r0 + block_rows))
        p = oracle.softmax_rows(x_host, w.in_dtype, w.rows, w.cols, vl, rows_sel=sel)
        yb = y_store.reshape(w.rows, w.cols)[sel]
        st = parity_stats(yb, p, w.out_dtype, None if vl is None else vl[sel])
        for k, v in st.items():
            if k == "rows":
                agg[k] = agg.get(k, 0) + v
            elif isinstance(v, bool):
                agg[k] = agg.get(k, True) and v
            elif k == "frac_exact":
                agg[k] = min(agg.get(k, 1.0), v)
            else:
                agg[k] = max(agg.get(k, v), v)
    return agg


# ---------------------------------------------------------------------------
# CPU reference leg.
# ---------------------------------------------------------------------------

def oracle_inputs(op: str, w, x_host, vl):
    """Host-side inputs the op's reference needs beyond x (seeded, like the GPU leg's)."""
    rows = w.rows
    extra = {}
    if op == "apply_stats":
        import oracle

        m, d = oracle.row_stats(x_host, w.in_dtype, rows, w.cols, vl)
        extra["m"], extra["d"] = m.astype(np.float32).astype(np.float64), d.astype(np.float32).astype(np.float64)
    if op == "cross_entropy":
        extra["target"] = op_targets(rows, w.cols)
    if op == "backward":
        extra["g"] = wl.to_storage(np.random.default_rng(77).normal(0, 1, rows * w.cols).astype(np.float32),
                                   w.in_dtype)
    return extra


def op_targets(rows: int, cols: int) -> np.ndarray:
    return np.random.default_rng(78).integers(0, cols, rows).astype(np.int64)


def oracle_call(op: str, w, x_host, vl, extra, sel):
    """The op's fp64 reference on the rows `sel` (for backward, x_host stands in for p)."""
    import oracle

    if op == "softmax":
        oracle.softmax_rows(x_host, w.in_dtype, w.rows, w.cols, vl, rows_sel=sel)
    elif op == "log_softmax":
        oracle.log_softmax_rows(x_host, w.in_dtype, w.rows, w.cols, vl, rows_sel=sel)
    elif op == "lse":
        oracle.row_stats(x_host, w.in_dtype, w.rows, w.cols, vl, rows_sel=sel)
    elif op == "apply_stats":
        oracle.apply_stats(x_host, w.in_dtype, w.rows, w.cols, extra["m"], extra["d"], vl, rows_sel=sel)
    elif op == "backward":
        oracle.softmax_backward(x_host, extra["g"], w.in_dtype, w.rows, w.cols, vl, rows_sel=sel)
    elif op == "cross_entropy":
        oracle.cross_entropy(x_host, w.in_dtype, w.rows, w.cols, extra["target"], vl, rows_sel=sel)
    else:
        raise ValueError(op)


def sample_bytes(op: str, w, vl, sel) -> int:
    in_size = 4 if w.in_dtype == "f32" else 2
    out_size = 4 if w.out_dtype == "f32" else 2
    return wl.op_bytes(op, sel.size, w.cols, in_size, out_size, None if vl is None else vl[sel])


def oracle_throughput(x_host, vl, w, budget_s: float, min_rows: int = 1, op: str = "softmax"):
    """Time the fp64 reference on a bounded sample of the workload's rows."""
    extra = oracle_inputs(op, w, x_host, vl)
    rows = w.rows
    t0 = time.perf_counter()
    oracle_call(op, w, x_host, vl, extra, np.arange(min(rows, 16)))
    per_row = (time.perf_counter() - t0) / min(rows, 16)
    n = int(max(min_rows, min(rows, budget_s / max(per_row, 1e-9))))
    sel = np.arange(n)
    t0 = time.perf_counter()
    oracle_call(op, w, x_host, vl, extra, sel)
    dt = time.perf_counter() - t0
    return sample_bytes(op, w, vl, sel) / dt / 1e9, n, dt, n / dt


def _oracle_slice(job):
    """Process-pool worker: the reference on one contiguous slice of rows;
    returns its compute time (the slice's data arrives before the clock starts)."""
    import dataclasses

    op, w, x_part, vl_part, extra_part, n = job
    ws = dataclasses.replace(w, rows=n)
    t0 = time.perf_counter()
    oracle_call(op, ws, x_part, vl_part, extra_part, np.arange(n))
    return time.perf_counter() - t0


def oracle_all_cores(x_host, vl, w, n: int, op: str = "softmax"):
    """The same reference on the first n rows, split into one contiguous slice
    per core of this process's CPU affinity (a spawn-context process pool: no
    state of this process, GPU or otherwise, is inherited).  Returns
    (GB/s over the slowest worker's compute time, cores)."""
    import multiprocessing as mp

    cores = max(1, len(os.sched_getaffinity(0)))
    extra = oracle_inputs(op, w, x_host, vl)
    bounds = np.linspace(0, n, min(cores, n) + 1).astype(np.int64)
    jobs = []
    for r0, r1 in zip(bounds[:-1], bounds[1:]):
        r0, r1 = int(r0), int(r1)
        part = {k: (v[r0:r1] if isinstance(v, np.ndarray) and v.shape[:1] == (w.rows,)
                    else v[r0 * w.cols:r1 * w.cols] if isinstance(v, np.ndarray) else v)
                for k, v in extra.items()}
        jobs.append((op, w, x_host[r0 * w.cols:r1 * w.cols], None if vl is None else vl[r0:r1], part, r1 - r0))
    with mp.get_context("spawn").Pool(len(jobs)) as pool:
        pool.map(_oracle_slice, jobs[:1] * len(jobs), chunksize=1)  # start the workers, load the reference
        dt = max(pool.map(_oracle_slice, jobs, chunksize=1))
    return sample_bytes(op, w, vl, np.arange(n)) / dt / 1e9, len(jobs)


def run_reference(args, w):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    x_host, vl = wl.host_input(w.name)
    import oracle

    oracle.build()
    op = args.op
    extra = oracle_inputs(op, w, x_host, vl)
    # size each step's sample so warm-up + timed steps take about a minute
    t0 = time.perf_counter()
    oracle_call(op, w, x_host, vl, extra, np.arange(4))
    per_row = (time.perf_counter() - t0) / 4
    per_step_rows = int(max(1, min(w.rows, args.ref_budget / max(1, args.steps + args.warmup)
                                   / per_row)))
    sel_all = np.arange(w.rows)
    for s in range(args.warmup):
        sel = sel_all[(s * per_step_rows) % w.rows:][:per_step_rows]
        oracle_call(op, w, x_host, vl, extra, sel)
    tot_bytes, tot_rows = 0, 0
    t0 = time.perf_counter()
    for s in range(args.steps):
        start = (s * per_step_rows) % w.rows
        sel = sel_all[start:start + per_step_rows]
        oracle_call(op, w, x_host, vl, extra, sel)
        tot_bytes += sample_bytes(op, w, vl, sel)
        tot_rows += sel.size
    dt = time.perf_counter() - t0
    value = tot_bytes / dt / 1e9
    line = {
        "impl": "reference", "metric": metric_of(op), "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config_of(w, None, op),
        "rows_per_s": tot_rows / dt,
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"{per_step_rows} rows of {w.rows} per step (fp64 C reference, "
                                   f"one thread)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def config_of(w, nsets, op="softmax"):
    c = {"workload": w.name, "rows": w.rows, "cols": w.cols, "in_dtype": w.in_dtype,
         "out_dtype": w.out_dtype, "mask": "valid_len" if w.masked else None,
         "description": w.description}
    if op != "softmax":
        c["op"] = op
    if nsets is not None:
        c["l2"] = f"rotating {nsets} input/output buffer sets, larger than L2 together"
    return c


# ---------------------------------------------------------------------------
# GPU leg.
# ---------------------------------------------------------------------------

class GpuOp:
    """Device buffers of one operation over `nsets` rotating sets, its launch
    through the raw C ABI (the timed steps) and its end-to-end step through the
    public Python call with host copies both ways."""

    def __init__(self, op, w, x_host, vl_host, dev, torch, smx, stream):
        self.op, self.w, self.torch, self.smx = op, w, torch, smx
        self.lib = smx.library()
        self.sptr = stream.cuda_stream
        in_size = 4 if w.in_dtype == "f32" else 2
        out_size = 4 if w.out_dtype == "f32" else 2
        rows, cols = w.rows, w.cols
        self.bytes_step = wl.op_bytes(op, rows, cols, in_size, out_size, vl_host)
        dense_out = op != "lse"
        set_bytes = rows * cols * (in_size * (2 if op == "backward" else 1) + (out_size if dense_out else 0))
        self.nsets = rotation_sets(set_bytes)
        out_dt = wl.torch_dtype(w.out_dtype)
        self.x_cpu = wl.storage_to_torch(x_host, w.in_dtype).reshape(rows, cols)
        self.vl_host = vl_host
        self.vl = None if vl_host is None else torch.from_numpy(vl_host).to(dev)
        x0 = self.x_cpu.to(dev)
        if op == "backward":
            # p: the softmax of the workload (what a forward pass stored); g: N(0, 1)
            p0 = smx.softmax_rows(x0, valid_len=self.vl)
            self.g_cpu = wl.storage_to_torch(
                wl.to_storage(np.random.default_rng(77).normal(0, 1, rows * cols).astype(np.float32),
                              w.in_dtype), w.in_dtype).reshape(rows, cols)
            self.xs = [p0.clone() for _ in range(self.nsets)]
            self.gs = [self.g_cpu.to(dev) for _ in range(self.nsets)]
            self.x_cpu = p0.cpu()
        else:
            self.xs = [x0.clone() for _ in range(self.nsets)]
        self.ys = ([torch.empty((rows, cols), dtype=out_dt, device=dev) for _ in range(self.nsets)]
                   if dense_out else [torch.empty(rows, dtype=torch.float32, device=dev)
                                      for _ in range(self.nsets)])
        if op == "apply_stats":
            self.m, self.d = smx.softmax_row_stats(x0, valid_len=self.vl)
        if op == "cross_entropy":
            self.t_cpu = torch.from_numpy(op_targets(rows, cols))
            self.t = self.t_cpu.to(dev)
            self.loss = [torch.empty(rows, dtype=torch.float32, device=dev) for _ in range(self.nsets)]
        del x0
        self.in_code = smx.DTYPES[self.xs[0].dtype]
        self.out_code = smx.DTYPES[out_dt]
        self.vl_ptr = None if self.vl is None else self.vl.data_ptr()

    def launch(self, i):
        k = i % self.nsets
        w, lib, x, y = self.w, self.lib, self.xs[k].data_ptr(), self.ys[k].data_ptr()
        op = self.op
        if op == "softmax":
            st = lib.smx_softmax_rows(x, y, w.rows, w.cols, self.vl_ptr, self.in_code, self.out_code, self.sptr)
        elif op == "log_softmax":
            st = lib.smx_log_softmax_rows(x, y, w.rows, w.cols, self.vl_ptr, self.in_code, self.out_code,
                                          self.sptr)
        elif op == "lse":
            st = lib.smx_softmax_lse(x, y, w.rows, w.cols, self.vl_ptr, self.in_code, self.sptr)
        elif op == "apply_stats":
            st = lib.smx_softmax_apply_stats(x, self.m.data_ptr(), self.d.data_ptr(), y, w.rows, w.cols,
                                             self.vl_ptr, self.in_code, self.out_code, self.sptr)
        elif op == "backward":
            st = lib.smx_softmax_backward(x, self.gs[k].data_ptr(), y, w.rows, w.cols, self.vl_ptr,
                                          self.in_code, self.out_code, self.sptr)
        else:
            st = lib.smx_cross_entropy(x, self.t.data_ptr(), self.loss[k].data_ptr(), y, w.rows, w.cols,
                                       self.vl_ptr, self.in_code, self.out_code, self.sptr)
        if st != 0:
            raise self.smx.SmxError(st, op)

    def e2e(self):
        """(step function, H2D bytes, D2H bytes) through the public call."""
        torch, smx, op = self.torch, self.smx, self.op
        x_pin = self.x_cpu.pin_memory()
        xd, yd = self.xs[0], self.ys[0]
        y_pin = torch.empty(yd.shape, dtype=yd.dtype).pin_memory()
        vl_pin = None if self.vl_host is None else torch.from_numpy(self.vl_host).pin_memory()
        vld = None if vl_pin is None else torch.empty_like(self.vl)
        extra_in = []  # (pinned host, device) pairs copied in every step
        if op == "backward":
            extra_in.append((self.g_cpu.pin_memory(), self.gs[0]))
        if op == "apply_stats":
            extra_in += [(self.m.cpu().pin_memory(), torch.empty_like(self.m)),
                         (self.d.cpu().pin_memory(), torch.empty_like(self.d))]
        if op == "cross_entropy":
            extra_in.append((self.t_cpu.pin_memory(), torch.empty_like(self.t)))
            loss_pin = torch.empty(self.w.rows, dtype=torch.float32).pin_memory()
        if op == "softmax":
            # the host-buffer entry point (pinned buffers: read and written in
            # place by the kernel over the host link)
            def host_step():
                smx.softmax_rows_host(x_pin, out=y_pin, valid_len=vl_pin, wait=False)
            h2d = x_pin.numel() * x_pin.element_size() + (0 if vl_pin is None else vl_pin.numel() * 4)
            return host_step, h2d, y_pin.numel() * y_pin.element_size()
        def step():
            xd.copy_(x_pin, non_blocking=True)
            if vld is not None:
                vld.copy_(vl_pin, non_blocking=True)
            for h, dv in extra_in:
                dv.copy_(h, non_blocking=True)
            if op == "softmax":
                smx.softmax_rows(xd, out=yd, valid_len=vld)
            elif op == "log_softmax":
                smx.log_softmax_rows(xd, out=yd, valid_len=vld)
            elif op == "lse":
                smx.softmax_lse(xd, valid_len=vld, out=yd)
            elif op == "apply_stats":
                smx.softmax_apply_stats(xd, extra_in[0][1], extra_in[1][1], out=yd, valid_len=vld)
            elif op == "backward":
                smx.softmax_backward(xd, extra_in[0][1], out=yd, valid_len=vld)
            else:
                smx.cross_entropy(xd, extra_in[0][1], valid_len=vld, grad=yd, loss=self.loss[0])
                loss_pin.copy_(self.loss[0], non_blocking=True)
            y_pin.copy_(yd, non_blocking=True)
        h2d = x_pin.numel() * x_pin.element_size() + (0 if vl_pin is None else vl_pin.numel() * 4)
        h2d += sum(h.numel() * h.element_size() for h, _ in extra_in)
        d2h = y_pin.numel() * y_pin.element_size() + (self.w.rows * 4 if op == "cross_entropy" else 0)
        return step, h2d, d2h


# the workloads the HBM-bandwidth target is stated for (per_config entries)
PER_CONFIG = ("f32_64x1000", "bf16_16384x4096", "f16_32768x1024_len", "f32_64x1048576_rise")


def time_op(g, steps, warmup, stream, torch, dev, sampler=None, world=1, sample_launches=True):
    """Warm up, then time `steps` launches of g between CUDA events on the
    launching stream (synchronised on both sides).  Returns the region's ms,
    sampled per-launch ms, the path and launches of a call, the wall-clock
    bounds of the region and the index of the last launch."""
    lib = g.lib
    for i in range(warmup):
        g.launch(i)
    used_path = lib.smx_debug_last_path()
    launches_per_call = lib.smx_debug_last_launches()
    torch.cuda.synchronize(dev)
    if g.smx.last_device_status() != 0:
        raise RuntimeError("device status set during warm-up")
    # per-launch durations from event pairs around every LAUNCH_SAMPLE-th step
    # (an event pair around every launch would add its own gaps to the steps),
    # starting half a period in: the first launch follows the region's start
    # with nothing recorded in between
    first = min(LAUNCH_SAMPLE // 2, steps - 1)
    sampled = set(range(first, steps, LAUNCH_SAMPLE)) if sample_launches else set()
    ev = {i: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for i in sampled}
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    if sampler is not None:
        sampler.fast()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    wall0 = time.time()
    t_start.record(stream)
    for i in range(steps):
        if i in sampled:
            ev[i][0].record(stream)
            g.launch(i)
            ev[i][1].record(stream)
        else:
            g.launch(i)
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    wall1 = time.time()
    if sampler is not None:
        sampler.slow()
    if world > 1:
        torch.distributed.barrier()
    status = g.smx.last_device_status()
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed region")
    return (t_start.elapsed_time(t_end), [a.elapsed_time(b) for a, b in ev.values()], used_path,
            launches_per_call, wall0, wall1, steps - 1)


def timed_output_parity(g, last, x_host, vl_host, w):
    """Parity statistics of the output buffer the last timed launch wrote."""
    y = g.ys[last % g.nsets]
    return parity_of_output(wl.torch_to_storage(y.cpu()).reshape(-1), x_host, w, vl_host)


def per_config_entry(name, args, torch, smx, dev, stream, sampler, peak):
    """The softmax on one workload: throughput over --steps after --warmup, the
    roofline fraction, the committed profile's traffic, and parity statistics
    of the timed output against the fp64 reference on all rows."""
    w = wl.WORKLOADS[name]
    x_host, vl_host = wl.host_input(name)
    g = GpuOp("softmax", w, x_host, vl_host, dev, torch, smx, stream)
    try:
        ms, _, path, launches, wall0, wall1, last = time_op(g, args.steps, args.warmup, stream, torch, dev,
                                                             sampler, sample_launches=False)
        step_ms = ms / args.steps
        achieved = g.bytes_step / (step_ms / 1e3) / 1e9
        traffic, kernel = profile_traffic(name)
        entry = {"workload": name, "value": achieved, "unit": UNIT, "ms_per_step": step_ms,
                 "rows_per_s": w.rows / (step_ms / 1e3), "bytes_per_step": g.bytes_step,
                 "path": PATH_NAMES.get(path, path), "kernels_per_step": launches,
                 "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "frac": achieved / peak,
                              "traffic": traffic, "kernel": kernel, "launch_timing": "timed region / steps"},
                 "clocks": sampler.window(wall0, wall1) if sampler is not None and sampler.lines else None,
                 "l2": f"rotating {g.nsets} input/output buffer sets, larger than L2 together"}
        entry["_wall"] = (wall0, wall1)
        entry["parity"] = timed_output_parity(g, last, x_host, vl_host, w)
        return entry
    finally:
        del g
        torch.cuda.empty_cache()


def run_ours(args, w):
    import torch

    import numerically_stable_online_gb300 as smx
    from numerically_stable_online_gb300 import build as smx_build

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group(backend="nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        smx_build.build()
    if world > 1:
        torch.distributed.barrier()
    smx.library()

    x_host, vl_host = wl.host_input(w.name)
    stream = torch.cuda.current_stream(dev)
    lib = smx.library()
    lib.smx_debug_force_path(PATHS[args.path])
    g = GpuOp(args.op, w, x_host, vl_host, dev, torch, smx, stream)
    bytes_step, nsets = g.bytes_step, g.nsets

    # clocks: NVML polled every 100 us inside each timed region (a child
    # process); nvidia-smi every 100 ms as the fallback
    sampler = NvmlSampler(nvml_device_id(torch, dev))
    if not sampler.start():
        sampler = None
    smi = None
    if sampler is None:
        smi = ClockSampler(local)
        smi.start()
    local_ms, launch_ms, used_path, launches_per_call, wall0, wall1, last = time_op(
        g, args.steps, args.warmup, stream, torch, dev, sampler, world)
    elapsed_ms = max_over_ranks(local_ms, world)
    agg = aggregate(bytes_step, w.rows, args.steps, world, elapsed_ms / 1e3)
    parity_main = timed_output_parity(g, last, x_host, vl_host, w) if args.op == "softmax" and rank == 0 else None

    # end to end through the public call: pinned host inputs in, outputs back
    e2e_step, h2d, d2h = g.e2e()
    e2e_steps = max(3, min(args.steps, 30))
    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
    e2e = aggregate(bytes_step, w.rows, e2e_steps, world, e2e_ms / 1e3)
    del g
    torch.cuda.empty_cache()

    peak, peak_kind = measured_peak()
    per_config = None
    if world == 1 and args.per_config and args.op == "softmax" and args.path == "auto":
        per_config = []
        for name in PER_CONFIG:
            if name == w.name:
                continue
            per_config.append(per_config_entry(name, args, torch, smx, dev, stream, sampler, peak))
    if sampler is not None:
        sampler.stop()
        clocks = sampler.window(wall0, wall1)
        for e in per_config or []:
            e["clocks"] = sampler.window(*e["_wall"])
    else:
        clocks = smi.stop(wall0, wall1)
    for e in per_config or []:
        e.pop("_wall", None)

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return 0

    # the kernel's average launch duration: when a step is one launch, this
    # rank's timed region (CUDA events on the launching stream) over its
    # launches; otherwise the step's sampled event pairs
    if launches_per_call == 1:
        mean_launch_ms, launch_timing = local_ms / args.steps, "timed region / launches"
    else:
        mean_launch_ms, launch_timing = statistics.fmean(launch_ms), "event pairs around sampled steps"
    achieved = bytes_step / (mean_launch_ms / 1e3) / 1e9
    traffic, kernel_name = profile_traffic(w.name, args.op)
    cpu_gbs, cpu_rows, cpu_s, cpu_rps = oracle_throughput(x_host, vl_host, w, args.cpu_budget,
                                                          op=args.op)
    cpu_all = oracle_all_cores(x_host, vl_host, w, cpu_rows, args.op) if args.cpu_all_cores else None
    line = {
        "metric": metric_of(args.op), "value": agg["gbs"], "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": dict(config_of(w, nsets, args.op), path=PATH_NAMES.get(used_path, used_path)),
        "rows_per_s": agg["rows_per_s"],
        "pct_of_hbm_peak": 100.0 * agg["gbs"] / world / peak,
        "bytes_per_step": bytes_step,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_source": f"{peak_kind} HBM copy bandwidth",
                     "kernel": kernel_name, "algorithmic_bytes_per_launch": bytes_step,
                     "mean_launch_us": mean_launch_ms * 1e3, "launch_timing": launch_timing,
                     "sampled_launches": len(launch_ms),
                     "sampled_median_launch_us": statistics.median(launch_ms) * 1e3},
        "cpu_baseline": dict({"value": cpu_gbs, "unit": UNIT, "cores": 1, "kind": "oracle",
                              "sample": f"first {cpu_rows} of {w.rows} rows, fp64 C reference, one "
                                        f"thread, {cpu_s:.1f} s"},
                             **({} if cpu_all is None else {
                                 "value_all_cores": cpu_all[0], "cores_all": cpu_all[1],
                                 "all_cores_sample": "the same rows in one contiguous slice per core of the "
                                                     "process's CPU affinity (spawned worker processes); "
                                                     "the slowest worker's compute time"})),
        "e2e": {"value": e2e["gbs"], "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "how": ("smx_softmax_rows_host on pinned host buffers: the kernel reads x and writes y "
                        "in place over the host link when they are mapped (else staged copies on two "
                        "streams)" if args.op == "softmax" else
                        "pinned host copies in, the device call, the outputs copied back, one stream")},
        "gpu_launches": args.steps * launches_per_call,
        "kernels_per_step": launches_per_call,
        "clocks": clocks,
    }
    if parity_main is not None:
        line["parity"] = parity_main
    if per_config is not None:
        line["per_config"] = per_config
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


ATTN_METRIC = ("attention forward TFLOP/s (4 head_dim FLOPs per valid query-key pair) on 1 GB300; "
               "% of bf16 tensor peak")


def attention_oracle_sample(name, q, k, v, budget_s, min_rows=4):
    """Time the fp64 reference attention on a bounded sample of rows of head 0."""
    import oracle

    heads, n, d, causal = wl.ATTN_WORKLOADS[name]
    qs = wl.torch_to_storage(q[:1].cpu()).reshape(-1)
    ks = wl.torch_to_storage(k[:1].cpu()).reshape(-1)
    vs = wl.torch_to_storage(v[:1].cpu()).reshape(-1)
    rows = np.arange(n - 4, n)  # the last rows see every key under either mask
    t0 = time.perf_counter()
    oracle.attention_rows(qs, ks, vs, "bf16", 1, n, n, d, d ** -0.5, causal, rows_sel=rows)
    per_row = (time.perf_counter() - t0) / rows.size
    m = int(max(min_rows, min(n, budget_s / max(per_row, 1e-9))))
    rows = np.arange(n - m, n)
    t0 = time.perf_counter()
    oracle.attention_rows(qs, ks, vs, "bf16", 1, n, n, d, d ** -0.5, causal, rows_sel=rows)
    dt = time.perf_counter() - t0
    flops = sum(4.0 * ((r + 1) if causal else n) * d for r in rows)
    return flops / dt / 1e12, m, dt


def run_attention(args):
    import torch

    import numerically_stable_online_gb300 as smx
    from numerically_stable_online_gb300 import build as smx_build

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group(backend="nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        smx_build.build()
    if world > 1:
        torch.distributed.barrier()
    lib = smx.library()
    name = args.workload
    heads, n, d, causal = wl.ATTN_WORKLOADS[name]
    q, k, v = wl.attention_inputs(name, dev)
    o = torch.empty_like(q)
    lse = torch.empty(heads, n, dtype=torch.float32, device=dev)
    flops = wl.attention_flops(heads, n, n, d, causal)
    stream = torch.cuda.current_stream(dev)
    sptr = stream.cuda_stream
    code = smx.DTYPES[q.dtype]

    def step():
        st = lib.smx_attention_forward(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                       heads, n, n, d, d ** -0.5, 1 if causal else 0, code, sptr)
        if st != 0:
            raise smx.SmxError(st, "smx_attention_forward")

    for _ in range(args.warmup):
        step()
    launches = lib.smx_debug_last_launches()
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(local)
    sampler.start()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    wall0 = time.time()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(args.steps):
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    t1.record(stream)
    torch.cuda.synchronize(dev)
    wall1 = time.time()
    clocks = sampler.stop(wall0, wall1)
    local_ms = t0.elapsed_time(t1)
    elapsed_ms = max_over_ranks(local_ms, world)
    value = flops * args.steps * world / (elapsed_ms / 1e3) / 1e12
    launch_ms = [a.elapsed_time(b) for a, b in ev]
    # end to end through the public call: q, k, v from pinned host memory, o and lse back
    qp, kp, vp = q.cpu().pin_memory(), k.cpu().pin_memory(), v.cpu().pin_memory()
    op = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    lp = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()

    def e2e_step():
        q.copy_(qp, non_blocking=True)
        k.copy_(kp, non_blocking=True)
        v.copy_(vp, non_blocking=True)
        smx.attention_forward(q, k, v, causal=causal, out=o, lse=lse)
        op.copy_(o, non_blocking=True)
        lp.copy_(lse, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize(dev)
    e2e_steps = max(3, min(args.steps, 10))
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return 0
    peak, peak_kind = measured_peak("bf16_tflops")
    # one launch per step: this rank's timed region over its launches
    mean_launch_ms = local_ms / args.steps if launches == 1 else statistics.fmean(launch_ms)
    achieved = flops / (mean_launch_ms / 1e3) / 1e12
    traffic, kernel_name = profile_traffic(name, "attention")
    cpu_tf, cpu_rows, cpu_s = attention_oracle_sample(name, q, k, v, args.cpu_budget)
    line = {
        "metric": ATTN_METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": name, "heads": heads, "seq": n, "head_dim": d, "causal": causal,
                   "op": "attention", "l2": "inputs 3 x 128 MiB, larger than L2"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_source": f"{peak_kind} cuBLAS bf16 GEMM throughput (burst)",
                     "kernel": kernel_name or ("k_attention_tma<bf16,128,2> (persistent, two query tiles, "
                                               "tcgen05.mma, TMEM accumulators)" if causal else
                                               "k_attention_tc<bf16,128> (tcgen05.mma, TMEM accumulators)"),
                     "flops_per_launch": flops, "mean_launch_us": mean_launch_ms * 1e3,
                     "median_launch_us": statistics.median(launch_ms) * 1e3},
        "cpu_baseline": {"value": cpu_tf, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
                         "sample": f"last {cpu_rows} query rows of head 0, fp64 C reference, one thread, "
                                   f"{cpu_s:.1f} s"},
        "e2e": {"value": flops * e2e_steps / (e2e_ms / 1e3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": 3 * q.numel() * 2, "d2h_bytes_per_step": o.numel() * 2 + lse.numel() * 4,
                "steps": e2e_steps,
                "how": "pinned host copies of q, k and v in, the device call, o and lse copied back, one stream"},
        "gpu_launches": args.steps * launches,
        "kernels_per_step": launches,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def run_attention_reference(args):
    rank, _, _ = dist_env()
    if rank != 0:
        return 0
    import torch

    import oracle

    oracle.build()
    name = args.workload
    heads, n, d, causal = wl.ATTN_WORKLOADS[name]
    q, k, v = wl.attention_inputs(name, "cpu")
    qs = wl.torch_to_storage(q[:1]).reshape(-1)
    ks = wl.torch_to_storage(k[:1]).reshape(-1)
    vs = wl.torch_to_storage(v[:1]).reshape(-1)
    t0 = time.perf_counter()
    oracle.attention_rows(qs, ks, vs, "bf16", 1, n, n, d, d ** -0.5, causal, rows_sel=np.arange(n - 2, n))
    per_row = (time.perf_counter() - t0) / 2
    per_step = int(max(1, min(n, args.ref_budget / max(1, args.steps + args.warmup) / per_row)))
    tot_flops = 0.0
    for s_ in range(args.warmup):
        oracle.attention_rows(qs, ks, vs, "bf16", 1, n, n, d, d ** -0.5, causal,
                              rows_sel=np.arange(n - per_step, n))
    t0 = time.perf_counter()
    for s_ in range(args.steps):
        rows = np.arange(n - per_step, n)
        oracle.attention_rows(qs, ks, vs, "bf16", 1, n, n, d, d ** -0.5, causal, rows_sel=rows)
        tot_flops += sum(4.0 * ((r + 1) if causal else n) * d for r in rows)
    dt = time.perf_counter() - t0
    value = tot_flops / dt / 1e12
    print(json.dumps({
        "impl": "reference", "metric": ATTN_METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": name, "op": "attention"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
                         "sample": f"{per_step} query rows of head 0 per step (fp64 C reference, one thread)"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)
    return 0


def main(argv=None):
    argv = sys.argv[1:] if argv is None else argv
    if argv[:1] == ["--nvml-sampler"]:
        return nvml_sampler_main(argv[1], argv[2])
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=None, choices=sorted(wl.WORKLOADS) + sorted(wl.ATTN_WORKLOADS))
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of CPU reference work for cpu_baseline")
    ap.add_argument("--cpu-all-cores", type=int, default=1,
                    help="also time the CPU reference on all cores of the affinity (1) or not (0)")
    ap.add_argument("--path", choices=sorted(PATHS), default="auto",
                    help="kernel family (diagnostics; the library chooses with auto)")
    ap.add_argument("--ref-budget", type=float, default=60.0,
                    help="seconds the reference arm spends over all its steps")
    ap.add_argument("--op", choices=list(wl.OPS), default="softmax",
                    help="entry point to time (default: the softmax)")
    ap.add_argument("--per-config", type=int, default=1,
                    help="softmax only, one GPU: also time every workload of the bandwidth target with "
                         "the same steps and report its parity against the reference (1) or not (0)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")
    if args.op == "attention":
        if args.workload is None:
            args.workload = "attn_bf16_4x32x4096x128"
        if args.workload not in wl.ATTN_WORKLOADS:
            ap.error("--op attention takes an attention workload")
        return run_attention_reference(args) if args.impl == "reference" else run_attention(args)
    if args.workload is None:
        args.workload = wl.BENCH_WORKLOAD
    if args.workload not in wl.WORKLOADS:
        ap.error("an attention workload needs --op attention")
    w = wl.WORKLOADS[args.workload]
    if w.name == "bf16_causal_8x32x4096x4096":
        ap.error("the causal batch is a parity case, not a benchmark workload")
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
