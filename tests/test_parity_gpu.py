"""Parity of the CUDA path (called through the C ABI) with the fp64 reference.

Every case runs the same seeded input through both and compares element by
element with the tolerances in tests/parity.py.  Sizes: the worked rows; each
workload at a reduced size that still spans several tiles and ragged tails; each
workload at full size in the launch configuration the benchmark times (all rows
against the reference, or whole sampled slices of the batched causal workload
plus properties of every row); and the edge cases of the declared policy.
"""
import math

import numpy as np
import pytest
import torch

import numerically_stable_online_gb300 as smx
import oracle
from numerically_stable_online_gb300 import workloads as wl
from tests import parity

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
PAIRS = [(a, b) for a in DT for b in DT]
PATH_REGS, PATH_CLUSTER, PATH_GENERIC, PATH_STREAM, PATH_SPLIT, PATH_STRIPE = 1, 2, 3, 4, 5, 6
ALL_PATHS = [PATH_REGS, PATH_CLUSTER, PATH_GENERIC, PATH_STREAM, PATH_SPLIT, PATH_STRIPE]


@pytest.fixture(scope="module", autouse=True)
def built():
    from numerically_stable_online_gb300 import build

    build.build()
    oracle.build()
    lib = smx.library()
    yield lib
    lib.smx_debug_force_path(0)
    lib.smx_debug_set_cluster(0, 0)
    lib.smx_debug_set_wait_limit(0)
    lib.smx_debug_set_regs_shape(0, 0)
    lib.smx_debug_set_stream_depth(0)


@pytest.fixture
def lib(built):
    yield built
    built.smx_debug_force_path(0)
    built.smx_debug_set_cluster(0, 0)
    built.smx_debug_set_wait_limit(0)
    built.smx_debug_set_regs_shape(0, 0)
    built.smx_debug_set_stream_depth(0)
    built.smx_debug_set_cluster_staging(0)
    built.smx_debug_set_split_slab(0)
    built.smx_debug_set_split_hints(-1, -1)
    built.smx_debug_set_stream_ctas(0)
    built.smx_debug_set_stream_warp(0)
    built.smx_debug_set_split_fused(0)
    built.smx_debug_set_count_probe(0)


DEV = "cuda:0"


def to_device(x_store, in_dtype, rows, cols, offset=0):
    t = wl.storage_to_torch(np.ascontiguousarray(x_store).reshape(-1), in_dtype)
    if offset == 0:
        return t.reshape(rows, cols).to(DEV)
    buf = torch.empty(rows * cols + offset, dtype=DT[in_dtype], device=DEV)
    v = buf[offset:]
    v.copy_(t.to(DEV))
    return v.view(rows, cols) if v.is_contiguous() else None


def run_and_compare(x_store, in_dtype, out_dtype, rows, cols, valid_len=None, offset=0,
                    block_rows=2048):
    x = to_device(x_store, in_dtype, rows, cols, offset)
    vl = None if valid_len is None else torch.from_numpy(np.asarray(valid_len, np.int32)).to(DEV)
    if offset:
        ybuf = torch.empty(rows * cols + offset, dtype=DT[out_dtype], device=DEV)
        y = ybuf[offset:].view(rows, cols)
        smx.softmax_rows(x, out=y, valid_len=vl)
    else:
        y = smx.softmax_rows(x, valid_len=vl, out_dtype=DT[out_dtype])
    assert smx.last_device_status() == 0
    y_host = wl.torch_to_storage(y.cpu())
    stats = {}
    for r0 in range(0, rows, block_rows):
        r1 = min(rows, r0 + block_rows)
        sel = np.arange(r0, r1)
        p = oracle.softmax_rows(x_store, in_dtype, rows, cols, valid_len, rows_sel=sel)
        s = parity.compare(y_host.reshape(rows, cols)[r0:r1], p, out_dtype, valid_len, rows_sel=sel)
        for k, v in s.items():
            stats[k] = max(stats.get(k, 0), v) if k != "frac_exact" else min(stats.get(k, 1), v)
    return stats


def stored(vals, dtype):
    return wl.to_storage(np.asarray(vals, dtype=np.float32), dtype)


# ---------------------------------------------------------------------------
# The pages' worked rows, every dtype pair, every path.
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("in_dtype,out_dtype", PAIRS)
@pytest.mark.parametrize("path", ALL_PATHS)
def test_worked_rows(lib, in_dtype, out_dtype, path):
    lib.smx_debug_force_path(path)
    for name, row in wl.WORKED_ROWS.items():
        # pad to a vector multiple with masked lanes so every path can take it
        cols = 8
        vals = np.zeros(cols, np.float32)
        vals[: len(row)] = row
        run_and_compare(stored(vals, in_dtype), in_dtype, out_dtype, 1, cols, [len(row)])
        # and unpadded (odd cols take the generic path)
        run_and_compare(stored(row, in_dtype), in_dtype, out_dtype, 1, len(row))


def test_worked_row_values_as_printed(lib):
    x = torch.tensor([[20.0, 18.0, 17.0, -5.0]], device=DEV)
    y = smx.softmax_rows(x).cpu().double().numpy()[0]
    assert np.all(np.abs(y[:3] - [0.84380, 0.11420, 0.04201]) <= 1e-5)
    x = torch.tensor([[1000.0, 999.0, 997.0]], device=DEV)
    y = smx.softmax_rows(x).cpu().double().numpy()[0]
    assert np.all(np.isfinite(y)) and abs(y.sum() - 1) < 1e-6
    for z, printed in [(0.5, 0.622), (2.5, 0.924)]:
        y = smx.softmax_rows(torch.tensor([[0.0, z]], device=DEV)).cpu().double().numpy()[0]
        assert round(y[1], 3) == printed and abs(y[1] - 1 / (1 + math.exp(-z))) < 2e-7


# ---------------------------------------------------------------------------
# Workloads at reduced size (several tiles, ragged tails) and at full size.
# ---------------------------------------------------------------------------

SMALL = [("f32_64x1000", 64), ("bf16_16384x4096", 96), ("f16_32768x1024_len", 777),
         ("f32_64x1048576_rise", 3)]


@pytest.mark.parametrize("name,rows", SMALL)
def test_workload_reduced(lib, name, rows):
    w = wl.WORKLOADS[name]
    x, vl = wl.host_input(name, rows=rows)
    st = run_and_compare(x, w.in_dtype, w.out_dtype, rows, w.cols, vl)
    print(name, rows, st)


@pytest.mark.parametrize("name,rows", SMALL)
@pytest.mark.parametrize("out_dtype", ["f32", "f16", "bf16"])
def test_workload_reduced_other_outputs(lib, name, rows, out_dtype):
    w = wl.WORKLOADS[name]
    x, vl = wl.host_input(name, rows=min(rows, 16))
    run_and_compare(x, w.in_dtype, out_dtype, min(rows, 16), w.cols, None if vl is None else vl)


@pytest.mark.parametrize("name", ["f32_64x1000", "bf16_16384x4096", "f16_32768x1024_len",
                                  "f32_64x1048576_rise"])
def test_workload_full_size(lib, name):
    """Full size, automatic kernel choice (what the benchmark times), all rows."""
    w = wl.WORKLOADS[name]
    x, vl = wl.host_input(name)
    st = run_and_compare(x, w.in_dtype, w.out_dtype, w.rows, w.cols, vl)
    print(name, "path", lib.smx_debug_last_path(), st)


def test_causal_batch_full_size(lib):
    """8 x 32 x 4096 x 4096 bf16 causal scores in one call: three whole 4096-row
    slices against the reference, masked lanes and row sums of every row on the
    device."""
    w = wl.WORKLOADS["bf16_causal_8x32x4096x4096"]
    S = wl.CAUSAL_SLICE_ROWS
    n_slices = w.rows // S
    x = torch.empty((w.rows, w.cols), dtype=torch.bfloat16, device=DEV)
    for s in range(n_slices):
        wl.device_causal_slice(s, x[s * S:(s + 1) * S])
    vl_host = wl.causal_valid_len(w.rows)
    vl = torch.from_numpy(vl_host).to(DEV)
    y = smx.softmax_rows(x, valid_len=vl)
    assert smx.last_device_status() == 0
    upper = torch.triu(torch.ones(S, S, dtype=torch.bool, device=DEV), diagonal=1)
    # every output within 1 ulp of RN(p_j), so |y_j - p_j| <= 1.5 ulp(p_j) <=
    # 1.5 * 2^-7 p_j, and |sum_j y_j - 1| <= 1.5 * 2^-7 (plus the fp32 sum's
    # own rounding, far below 2^-20)
    sum_tol = 1.5 * 2.0 ** -7 + 2.0 ** -20
    for s in range(n_slices):
        ys = y[s * S:(s + 1) * S]
        assert not torch.any(ys[upper] != 0)
        sums = ys.float().sum(dim=1)
        assert torch.all((sums - 1).abs() <= sum_tol)
    for s in (0, 137, n_slices - 1):
        xs = wl.torch_to_storage(x[s * S:(s + 1) * S].cpu())
        ys = wl.torch_to_storage(y[s * S:(s + 1) * S].cpu())
        for r0 in range(0, S, 1024):
            sel = np.arange(r0, r0 + 1024)
            p = oracle.softmax_rows(xs, "bf16", S, w.cols, vl_host[:S], rows_sel=sel)
            parity.compare(ys.reshape(S, w.cols)[r0:r0 + 1024], p, "bf16", vl_host[:S], rows_sel=sel)


# ---------------------------------------------------------------------------
# Edge cases: shapes, alignment, lengths, the policy rows, forced paths.
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("cols", [1, 3, 4, 7, 8, 16, 31, 33, 250, 1000, 4095, 4096, 4097, 8200,
                                  32768, 32776, 65544])
@pytest.mark.parametrize("in_dtype,out_dtype", [("f32", "f32"), ("bf16", "bf16"), ("f16", "f32")])
def test_shapes(lib, cols, in_dtype, out_dtype):
    rows = 5
    rng = np.random.default_rng(cols)
    x = stored(rng.normal(0, 6, size=rows * cols), in_dtype)
    vl = rng.integers(0, cols + 1, size=rows).astype(np.int32)
    vl[0] = cols
    run_and_compare(x, in_dtype, out_dtype, rows, cols, None)
    run_and_compare(x, in_dtype, out_dtype, rows, cols, vl)


@pytest.mark.parametrize("offset", [1, 2, 3])
def test_unaligned_pointers(lib, offset):
    rows, cols = 7, 1024
    x = stored(np.random.default_rng(offset).normal(0, 5, rows * cols), "f32")
    run_and_compare(x, "f32", "f32", rows, cols, offset=offset)
    assert lib.smx_debug_last_path() == PATH_GENERIC


def test_valid_lengths_clamped(lib):
    rows, cols = 6, 64
    x = stored(np.random.default_rng(1).normal(0, 3, rows * cols), "f32")
    vl = np.array([0, 1, 63, 64, 1000, -7], np.int32)
    for path in ALL_PATHS:
        lib.smx_debug_force_path(path)
        run_and_compare(x, "f32", "f32", rows, cols, vl)
        run_and_compare(stored(np.random.default_rng(2).normal(0, 3, rows * cols), "bf16"),
                        "bf16", "f16", rows, cols, vl)


POLICY_ROWS = [
    [1.0, 2.0, np.nan, 3.0, 0.0, 0.0, 0.0, 0.0],
    [1.0, np.inf, 2.0, -np.inf, 0.0, 0.0, 0.0, 0.0],
    [-np.inf] * 8,
    [-np.inf, 0.0, -np.inf, 0.0, -np.inf, -np.inf, -np.inf, -np.inf],
    [np.inf, np.inf, 1.0, 1.0, 1.0, 1.0, 1.0, 1.0],
    [np.nan, np.inf, -np.inf, 0.0, 1.0, 2.0, 3.0, 4.0],
    [5.0, -1e30, 1e30, -3e38, 3e38, 0.0, 0.0, 0.0],
    [-100.0, -200.0, -90.0, -105.0, 0.0, 0.0, 0.0, 0.0],
]


@pytest.mark.parametrize("in_dtype,out_dtype", PAIRS)
@pytest.mark.parametrize("path", ALL_PATHS)
def test_policy_rows(lib, in_dtype, out_dtype, path):
    lib.smx_debug_force_path(path)
    rows = np.array(POLICY_ROWS, np.float32)
    if in_dtype != "f32":
        rows = np.where(np.isfinite(rows), np.clip(rows, -60000, 60000), rows).astype(np.float32)
    x = stored(rows.reshape(-1), in_dtype)
    n = rows.shape[0]
    run_and_compare(x, in_dtype, out_dtype, n, 8)
    # a NaN / +inf in a masked lane must not matter
    run_and_compare(x, in_dtype, out_dtype, n, 8, np.array([2, 1, 8, 8, 2, 0, 1, 4], np.int32))


def test_subnormal_bf16_outputs(lib):
    """bf16 shares fp32's exponent range: probabilities below 2^-126 must come out
    as bf16 subnormals, not flushed."""
    row = np.array([0.0, -88.0, -90.0, -92.0, -95.0, -100.0, -87.5, -91.3], np.float32)
    for in_dtype in ("f32", "bf16"):
        for path in ALL_PATHS:
            lib.smx_debug_force_path(path)
            run_and_compare(stored(row, in_dtype), in_dtype, "bf16", 1, 8)


@pytest.mark.parametrize("in_dtype,out_dtype,cols", [("bf16", "bf16", 512), ("f16", "f16", 1024),
                                                     ("f32", "f32", 1000), ("bf16", "f32", 4096),
                                                     ("f32", "bf16", 8192), ("bf16", "bf16", 16384)])
@pytest.mark.parametrize("depth", [2, 3, 7])
def test_stream_ring_many_rows(lib, in_dtype, out_dtype, cols, depth):
    """Many rows per persistent CTA, so the ring of row slots wraps many times;
    lengths include 0, 1 and cols."""
    rows = max(600, 8_000_000 // cols)
    rng = np.random.default_rng(cols)
    x = stored(rng.normal(0, 7, rows * cols), in_dtype)
    vl = rng.integers(0, cols + 1, size=rows).astype(np.int32)
    vl[::97] = 0
    vl[1::89] = 1
    vl[2::83] = cols
    lib.smx_debug_force_path(PATH_STREAM)
    lib.smx_debug_set_stream_depth(depth)
    run_and_compare(x, in_dtype, out_dtype, rows, cols, vl)
    es = 4 if in_dtype == "f32" else 2
    # rows of a 16-byte multiple take path 4; others the scalar kernel
    assert lib.smx_debug_last_path() == (PATH_STREAM if cols * es % 16 == 0 else PATH_GENERIC)
    m, d = gpu_stats(x, in_dtype, rows, cols, vl)
    m_ref, d_ref = oracle.row_stats(x, in_dtype, rows, cols, vl)
    check_stats(m, d, m_ref, d_ref)


@pytest.mark.parametrize("staging", [1, 2])
@pytest.mark.parametrize("cap", [1, 2, 4, 8, 16])
def test_cluster_sizes_and_streamed_remainder(lib, cap, staging):
    """Cluster path with each cluster size and both ways of staging (bulk copies,
    per-thread cp.async), and with the staging area cut to 32 KiB so that part of
    each chunk is streamed from global memory twice."""
    lib.smx_debug_set_cluster_staging(staging)
    rows, cols = 3, 300000
    rng = np.random.default_rng(cap)
    x32 = (rng.normal(0, 1, rows * cols) + np.tile(np.linspace(0, 20, cols), rows)).astype(np.float32)
    vl = np.array([cols, 123457, 7], np.int32)
    lib.smx_debug_force_path(PATH_CLUSTER)
    lib.smx_debug_set_cluster(cap, 0)
    run_and_compare(x32, "f32", "f32", rows, cols, vl)
    lib.smx_debug_set_cluster(cap, 32768)
    run_and_compare(x32, "f32", "f32", rows, cols, vl)
    run_and_compare(stored(x32, "bf16"), "bf16", "bf16", rows, cols, vl)
    assert lib.smx_debug_last_path() == PATH_CLUSTER


@pytest.mark.parametrize("threads,vpt", [(32, 1), (32, 4), (64, 2), (128, 1), (256, 2), (1024, 1),
                                         (512, 4)])
def test_register_shapes(lib, threads, vpt):
    rows, cols = 9, 1024
    x = stored(np.random.default_rng(threads + vpt).normal(0, 8, rows * cols), "bf16")
    lib.smx_debug_set_regs_shape(threads, vpt)
    vl = np.array([1024, 0, 1, 511, 512, 513, 1000, 7, 1024], np.int32)
    run_and_compare(x, "bf16", "bf16", rows, cols, vl)
    run_and_compare(x, "bf16", "f32", rows, cols, vl)


# ---------------------------------------------------------------------------
# Row statistics and the merge.
# ---------------------------------------------------------------------------

def gpu_stats(x_store, in_dtype, rows, cols, valid_len=None):
    x = to_device(x_store, in_dtype, rows, cols)
    vl = None if valid_len is None else torch.from_numpy(np.asarray(valid_len, np.int32)).to(DEV)
    m, d = smx.softmax_row_stats(x, valid_len=vl)
    return m.cpu().double().numpy(), d.cpu().double().numpy()


def check_stats(m, d, m_ref, d_ref, rel=2e-6):
    same_nan = np.isnan(m) == np.isnan(m_ref)
    assert np.all(same_nan)
    ok = ~np.isnan(m_ref)
    assert np.array_equal(m[ok], m_ref[ok])
    assert np.all(np.isnan(d) == np.isnan(d_ref))
    fin = ~np.isnan(d_ref)
    assert np.all(np.abs(d[fin] - d_ref[fin]) <= rel * np.maximum(d_ref[fin], 1e-300))


@pytest.mark.parametrize("in_dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("path", ALL_PATHS)
def test_row_stats(lib, in_dtype, path):
    lib.smx_debug_force_path(path)
    rows, cols = 12, 4096
    rng = np.random.default_rng(5)
    x32 = rng.normal(0, 8, (rows, cols)).astype(np.float32)
    x32[3, 17] = np.nan
    x32[4, 100] = np.inf
    x32[5, :] = -np.inf
    x = stored(x32.reshape(-1), in_dtype)
    vl = np.array([4096, 0, 1, 4096, 4096, 4096, 4000, 13, 4096, 2048, 4095, 9], np.int32)
    for v in (None, vl):
        m, d = gpu_stats(x, in_dtype, rows, cols, v)
        m_ref, d_ref = oracle.row_stats(x, in_dtype, rows, cols, v)
        check_stats(m, d, m_ref, d_ref)


@pytest.mark.parametrize("in_dtype,out_dtype", [("f32", "f32"), ("bf16", "bf16"), ("f16", "f32"),
                                                ("f32", "f16")])
@pytest.mark.parametrize("slab", [0, 1 << 20])
def test_split_long_rows(lib, in_dtype, out_dtype, slab):
    """L2-slab path: chunk summaries then merge and normalise; ragged last chunks,
    varied lengths (0, 1, a chunk boundary, all), and slabs of one or many rows."""
    rows, cols = 9, 40000 + 8 * 7
    rng = np.random.default_rng(rows + slab)
    x32 = (rng.normal(0, 3, (rows, cols)) + np.linspace(-5, 25, cols)[None, :]).astype(np.float32)
    x32[6, 1234] = np.nan
    x32[7, 99] = np.inf
    x = stored(x32.reshape(-1), in_dtype)
    vl = np.array([cols, 0, 1, 4096, 8192, 39999, cols, 5000, cols], np.int32)
    lib.smx_debug_force_path(PATH_SPLIT)
    lib.smx_debug_set_split_slab(slab)
    run_and_compare(x, in_dtype, out_dtype, rows, cols, vl)
    assert lib.smx_debug_last_path() == PATH_SPLIT
    run_and_compare(x, in_dtype, out_dtype, rows, cols, None)
    m, d = gpu_stats(x, in_dtype, rows, cols, vl)
    m_ref, d_ref = oracle.row_stats(x, in_dtype, rows, cols, vl)
    check_stats(m, d, m_ref, d_ref)


@pytest.mark.parametrize("staging", [1, 2])
def test_row_stats_long_rows(lib, staging):
    lib.smx_debug_set_cluster_staging(staging)
    lib.smx_debug_force_path(PATH_CLUSTER)
    name = "f32_64x1048576_rise"
    x, _ = wl.host_input(name, rows=4)
    m, d = gpu_stats(x, "f32", 4, 1048576)
    m_ref, d_ref = oracle.row_stats(x, "f32", 4, 1048576)
    check_stats(m, d, m_ref, d_ref)
    assert lib.smx_debug_last_path() == PATH_CLUSTER


@pytest.mark.parametrize("staging", [1, 2])
def test_cluster_many_rows_per_cluster(lib, staging):
    """More rows than resident clusters, so every cluster walks several rows and
    refills its staged pieces from the next row; lengths vary per row."""
    lib.smx_debug_set_cluster_staging(staging)
    lib.smx_debug_force_path(PATH_CLUSTER)
    rows, cols = 41, 200000
    rng = np.random.default_rng(41)
    x32 = rng.normal(0, 4, rows * cols).astype(np.float32)
    vl = rng.integers(0, cols + 1, size=rows).astype(np.int32)
    vl[::5] = cols
    vl[3] = 0
    for out in ("f32", "bf16"):
        run_and_compare(x32, "f32", out, rows, cols, vl)
    run_and_compare(stored(x32, "f16"), "f16", "f16", rows, cols, vl)
    m, d = gpu_stats(x32, "f32", rows, cols, vl)
    m_ref, d_ref = oracle.row_stats(x32, "f32", rows, cols, vl)
    check_stats(m, d, m_ref, d_ref)


def test_merge_stats_against_reference(lib):
    rng = np.random.default_rng(6)
    n = 100000
    m_a = rng.normal(0, 20, n).astype(np.float32)
    m_b = rng.normal(0, 20, n).astype(np.float32)
    d_a = rng.uniform(1, 5000, n).astype(np.float32)
    d_b = rng.uniform(1, 5000, n).astype(np.float32)
    special = [(-np.inf, 0.0, 3.0, 2.0), (3.0, 2.0, -np.inf, 0.0), (-np.inf, 0.0, -np.inf, 0.0),
               (np.nan, np.nan, 1.0, 1.0), (1.0, 1.0, np.nan, 5.0), (np.inf, np.nan, 2.0, 1.0),
               (10.0, 1.8, 12.0, 1.3), (12.0, 1.3, 10.0, 1.8), (5.0, 1.0, 5.0, 2.0)]
    for i, (a, b, c, e) in enumerate(special):
        m_a[i], d_a[i], m_b[i], d_b[i] = a, b, c, e
    t = [torch.from_numpy(v).to(DEV) for v in (m_a, d_a, m_b, d_b)]
    m, d = smx.softmax_merge_stats(*t)
    m, d = m.cpu().double().numpy(), d.cpu().double().numpy()
    m_ref, d_ref = oracle.merge_stats(m_a, d_a, m_b, d_b)
    check_stats(m, d, m_ref, d_ref, rel=1e-6)
    assert abs(d[6] - 1.5436035) < 1e-6 and m[6] == 12.0
    # in place
    m2, d2 = smx.softmax_merge_stats(*t, m_out=t[0], d_out=t[1])
    assert np.array_equal(t[0].cpu().numpy(), m.astype(np.float32), equal_nan=True)


def test_split_row_through_stats_and_merge(lib):
    """A row split into blocks: per-block statistics merged in any order match the
    whole row's statistics ("Stable softmax...", third paragraph)."""
    rng = np.random.default_rng(7)
    cols, k = 8192, 8
    x32 = (rng.normal(0, 4, cols) + np.linspace(0, 30, cols)).astype(np.float32)
    blocks = torch.from_numpy(x32.reshape(k, cols // k)).to(DEV)
    m, d = smx.softmax_row_stats(blocks)
    order = rng.permutation(k)
    acc_m, acc_d = m[order[0]:order[0] + 1].clone(), d[order[0]:order[0] + 1].clone()
    for i in order[1:]:
        acc_m, acc_d = smx.softmax_merge_stats(acc_m, acc_d, m[i:i + 1].contiguous(),
                                               d[i:i + 1].contiguous())
    m_ref, d_ref = oracle.row_stats(x32, "f32", 1, cols)
    assert acc_m.item() == m_ref[0]
    assert abs(acc_d.item() - d_ref[0]) <= 2e-6 * d_ref[0]


# ---------------------------------------------------------------------------
# Device-side error path: a bounded staging wait that runs out.
# ---------------------------------------------------------------------------

def test_bounded_wait_reports_timeout(lib):
    """A bounded wait that runs out is reported through the status word, and the
    context stays usable: each CTA waits on a barrier nothing signals (a flag
    nothing sets) for 4 polls, then computes normally."""
    rows, cols = 2, 1 << 20
    x = torch.randn(rows, cols, device=DEV)
    x_host = x.cpu().numpy()
    lib.smx_debug_force_path(PATH_CLUSTER)
    assert smx.last_device_status() == 0
    lib.smx_debug_set_wait_limit(-4)
    y = smx.softmax_rows(x)
    st = smx.last_device_status()
    lib.smx_debug_set_wait_limit(0)
    assert st == 5, f"expected SMX_ERR_TIMEOUT, got {st}"
    assert smx.last_device_status() == 0  # cleared by the read
    p = oracle.softmax_rows(x_host.reshape(-1), "f32", rows, cols)
    parity.compare(y.cpu().numpy(), p, "f32")  # the probe did not disturb the result
    # a tiny (positive) limit on the real waits is harmless to the context
    lib.smx_debug_set_wait_limit(1)
    smx.softmax_rows(x)
    smx.last_device_status()
    lib.smx_debug_set_wait_limit(0)
    y = smx.softmax_rows(x)
    assert smx.last_device_status() == 0
    parity.compare(y.cpu().numpy(), p, "f32")


def test_bounded_wait_runs_out_while_walking_rows(lib):
    """More rows than resident clusters, so every cluster walks several rows,
    with one poll per staging wait: waits run out on whichever row of the walk
    they happen to, and the CTA stops refilling there.  Before it exits it must
    still let every copy it issued land (each piece's last issued phase, not
    the walk's last row).  The call's output is undefined; the next call on the
    same context must be correct and report nothing."""
    rows, cols = 48, 1 << 20
    g = torch.Generator(device=DEV).manual_seed(48)
    x = torch.randn(rows, cols, generator=g, device=DEV) * 3
    lib.smx_debug_force_path(PATH_CLUSTER)
    for staging in (1, 2):
        lib.smx_debug_set_cluster_staging(staging)
        lib.smx_debug_set_wait_limit(1)
        smx.softmax_rows(x)
        smx.last_device_status()  # a timeout may or may not have been recorded
        lib.smx_debug_set_wait_limit(0)
        y = smx.softmax_rows(x)
        assert lib.smx_debug_last_path() == PATH_CLUSTER
        assert smx.last_device_status() == 0
        sel = [0, 17, 47]
        xs = x[sel].cpu().numpy().reshape(-1)
        p = oracle.softmax_rows(xs, "f32", len(sel), cols)
        parity.compare(y[sel].cpu().numpy(), p, "f32")


@pytest.mark.parametrize("cols", [8, 100, 256, 1000, 1024, 2048])
@pytest.mark.parametrize("in_dtype,out_dtype", [("f32", "f32"), ("bf16", "bf16"), ("f16", "f16"),
                                                ("f16", "f32")])
@pytest.mark.parametrize("warp_off", [0, 1])
def test_stream_walkers(lib, cols, in_dtype, out_dtype, warp_off):
    """Path 4 with a row per warp (rows that fit one warp) and with a CTA per
    row, many rows per walker, lengths including 0, 1 and cols."""
    rows = 3000
    rng = np.random.default_rng(cols + 11)
    x = stored(rng.normal(0, 6, rows * cols), in_dtype)
    vl = rng.integers(0, cols + 1, size=rows).astype(np.int32)
    vl[::101] = 0
    vl[1::67] = 1
    vl[2::53] = cols
    lib.smx_debug_force_path(PATH_STREAM)
    lib.smx_debug_set_stream_warp(warp_off)
    run_and_compare(x, in_dtype, out_dtype, rows, cols, vl)
    es = 4 if in_dtype == "f32" else 2
    # rows of a 16-byte multiple take path 4; others the scalar kernel
    assert lib.smx_debug_last_path() == (PATH_STREAM if cols * es % 16 == 0 else PATH_GENERIC)
    m, d = gpu_stats(x, in_dtype, rows, cols, vl)
    m_ref, d_ref = oracle.row_stats(x, in_dtype, rows, cols, vl)
    check_stats(m, d, m_ref, d_ref)


@pytest.mark.parametrize("in_dtype,out_dtype,rows,cols,slab", [
    ("f32", "f32", 7, 300_000, 2 << 20), ("bf16", "bf16", 9, 150_000, 1 << 20),
    ("f16", "f32", 5, 40_000, 64 << 10), ("bf16", "f16", 33, 12_288, 96 << 10)])
@pytest.mark.parametrize("fused", [1, 0])
def test_long_rows_one_launch_and_two(lib, in_dtype, out_dtype, rows, cols, slab, fused):
    """Path 5 as one cooperative launch over all slabs (per-row completion
    counts) and as two launches per slab, with small slabs so that many slabs
    and chunk ranges that straddle rows occur; lengths include 0 and 1."""
    rng = np.random.default_rng(cols + rows)
    x = stored(rng.normal(0, 5, rows * cols), in_dtype)
    vl = rng.integers(0, cols + 1, size=rows).astype(np.int32)
    vl[0], vl[1] = 0, 1
    vl[-1] = cols
    lib.smx_debug_force_path(PATH_SPLIT)
    lib.smx_debug_set_split_slab(slab)
    lib.smx_debug_set_split_fused(fused)
    xt = to_device(x, in_dtype, rows, cols)
    smx.softmax_rows(xt, valid_len=torch.from_numpy(vl).to(DEV), out_dtype=DT[out_dtype])
    slab_rows = max(1, slab // (cols * (4 if in_dtype == "f32" else 2)))
    assert lib.smx_debug_last_path() == PATH_SPLIT
    assert lib.smx_debug_last_launches() == (1 if fused else 2 * -(-rows // slab_rows))
    assert smx.last_device_status() == 0
    run_and_compare(x, in_dtype, out_dtype, rows, cols, vl)
