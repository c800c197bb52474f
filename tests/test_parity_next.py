"""Parity of log_softmax, LSE and apply-statistics (CUDA path through the C ABI)
with the fp64 reference.

log_softmax and LSE are compared with the tolerances derived in tests/parity.py
(compare_log, compare_lse); the apply step with the softmax tolerances.  Cases:
the pages' worked rows on every dtype pair and every kernel that takes these
modes (streamed rows, long-row chunks, the scalar kernel), the policy rows, the
workloads at reduced size, the benchmark's workload at full size (sampled rows
against the reference, a property of every row), ragged and unaligned shapes,
and the column-split softmax that the apply step completes.
"""
import numpy as np
import pytest
import torch

import numerically_stable_online_gb300 as smx
import oracle
from numerically_stable_online_gb300 import workloads as wl
from tests import parity
from tests.test_parity_gpu import POLICY_ROWS, stored, to_device

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
PAIRS = [(a, b) for a in DT for b in DT]
PATH_GENERIC, PATH_STREAM, PATH_SPLIT = 3, 4, 5
PATHS = [PATH_GENERIC, PATH_STREAM, PATH_SPLIT]
LOG_PATHS = PATHS + [6]  # and the read-once long-row kernel
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def built():
    from numerically_stable_online_gb300 import build

    build.build()
    oracle.build()
    yield smx.library()


@pytest.fixture
def lib(built):
    yield built
    built.smx_debug_force_path(0)
    built.smx_debug_set_split_slab(0)
    built.smx_debug_set_stream_warp(0)


def lengths_t(valid_len):
    return None if valid_len is None else torch.from_numpy(np.asarray(valid_len, np.int32)).to(DEV)


def run_log(x_store, in_dtype, out_dtype, rows, cols, valid_len=None, offset=0, block_rows=2048):
    x = to_device(x_store, in_dtype, rows, cols, offset)
    vl = lengths_t(valid_len)
    if offset:
        ybuf = torch.empty(rows * cols + offset, dtype=DT[out_dtype], device=DEV)
        y = ybuf[offset:].view(rows, cols)
        smx.log_softmax_rows(x, out=y, valid_len=vl)
    else:
        y = smx.log_softmax_rows(x, valid_len=vl, out_dtype=DT[out_dtype])
    lse = smx.softmax_lse(x, valid_len=vl)
    y_host = wl.torch_to_storage(y.cpu())
    lse_host = lse.cpu().numpy()
    stats = {}
    for r0 in range(0, rows, block_rows):
        sel = np.arange(r0, min(rows, r0 + block_rows))
        ref, ref_lse = oracle.log_softmax_rows(x_store, in_dtype, rows, cols, valid_len, rows_sel=sel)
        _, d = oracle.row_stats(x_store, in_dtype, rows, cols, valid_len, rows_sel=sel)
        with np.errstate(divide="ignore", invalid="ignore"):
            log_d = np.where(d > 0, np.log(np.where(d > 0, d, 1.0)), 0.0)
        s = parity.compare_log(y_host.reshape(rows, cols)[sel], ref, log_d, out_dtype, valid_len,
                               rows_sel=sel)
        s.update(parity.compare_lse(lse_host[sel], ref_lse, log_d))
        for k, v in s.items():
            stats[k] = max(stats.get(k, 0.0), v)
    return stats


# ------------------------------------------------------------------ log space

@pytest.mark.parametrize("in_dtype,out_dtype", PAIRS)
@pytest.mark.parametrize("path", LOG_PATHS)
def test_log_worked_rows(lib, in_dtype, out_dtype, path):
    lib.smx_debug_force_path(path)
    for row in wl.WORKED_ROWS.values():
        vals = np.zeros(8, np.float32)
        vals[: len(row)] = row
        run_log(stored(vals, in_dtype), in_dtype, out_dtype, 1, 8, [len(row)])
        run_log(stored(row, in_dtype), in_dtype, out_dtype, 1, len(row))


def test_log_worked_row_printed_values(lib):
    y = smx.log_softmax_rows(torch.tensor([[20.0, 18.0, 17.0, -5.0]], device=DEV))
    p = torch.exp(y.double()).cpu().numpy()[0]
    assert np.all(np.abs(p[:3] - [0.84380, 0.11420, 0.04201]) <= 1e-5)
    lse = smx.softmax_lse(torch.tensor([[1000.0, 999.0, 997.0]], device=DEV)).item()
    assert np.isfinite(lse) and abs(lse - (1000 + np.log1p(np.exp(-1) + np.exp(-3)))) < 1e-4


@pytest.mark.parametrize("in_dtype,out_dtype", [("f32", "f32"), ("bf16", "bf16"), ("f16", "f32"),
                                                ("f32", "f16")])
@pytest.mark.parametrize("path", LOG_PATHS)
def test_log_policy_rows(lib, in_dtype, out_dtype, path):
    lib.smx_debug_force_path(path)
    rows = np.array(POLICY_ROWS, np.float32)
    if in_dtype != "f32":
        rows = np.where(np.isfinite(rows), np.clip(rows, -60000, 60000), rows).astype(np.float32)
    x = stored(rows.reshape(-1), in_dtype)
    n = rows.shape[0]
    run_log(x, in_dtype, out_dtype, n, 8)
    run_log(x, in_dtype, out_dtype, n, 8, np.array([2, 1, 8, 8, 2, 0, 1, 4], np.int32))


SMALL = [("f32_64x1000", 64), ("bf16_16384x4096", 96), ("f16_32768x1024_len", 777),
         ("f32_64x1048576_rise", 3)]


@pytest.mark.parametrize("name,rows", SMALL)
@pytest.mark.parametrize("out_dtype", [None, "f32"])
def test_log_workloads_reduced(lib, name, rows, out_dtype):
    w = wl.WORKLOADS[name]
    x, vl = wl.host_input(name, rows=rows)
    st = run_log(x, w.in_dtype, out_dtype or w.out_dtype, rows, w.cols, vl)
    print(name, rows, lib.smx_debug_last_path(), st)


@pytest.mark.parametrize("cols", [1, 3, 8, 33, 1000, 4096, 4100, 8200, 16384, 40000])
@pytest.mark.parametrize("in_dtype,out_dtype", [("f32", "f32"), ("bf16", "bf16"), ("f16", "f32")])
def test_log_shapes_and_lengths(lib, cols, in_dtype, out_dtype):
    rows = 7
    rng = np.random.default_rng(cols + 7)
    x = stored(rng.normal(0, 6, rows * cols), in_dtype)
    vl = rng.integers(0, cols + 2, size=rows).astype(np.int32)
    vl[0], vl[1] = 0, cols
    run_log(x, in_dtype, out_dtype, rows, cols, vl)
    run_log(x, in_dtype, out_dtype, rows, cols)


def test_log_unaligned(lib):
    rows, cols = 9, 1000
    rng = np.random.default_rng(3)
    x = stored(rng.normal(0, 4, rows * cols), "f32")
    run_log(x, "f32", "f32", rows, cols, rng.integers(0, cols, rows).astype(np.int32), offset=1)


def test_log_bench_workload_full_size(lib):
    """16384 x 4096 bf16 in the automatic configuration: 2048 sampled rows
    against the reference, and logsumexp(y) = 0 on every row."""
    name = "bf16_16384x4096"
    w = wl.WORKLOADS[name]
    x_host, _ = wl.host_input(name)
    x = to_device(x_host, w.in_dtype, w.rows, w.cols)
    y = smx.log_softmax_rows(x)
    lse = smx.softmax_lse(x)
    s = torch.logsumexp(y.float(), dim=1)
    assert float(s.abs().max()) <= 2e-2  # bf16 outputs: 1 unit of 2^-7 relative per lane
    rows_sel = np.random.default_rng(5).choice(w.rows, 2048, replace=False)
    ref, ref_lse = oracle.log_softmax_rows(x_host, w.in_dtype, w.rows, w.cols, rows_sel=rows_sel)
    _, d = oracle.row_stats(x_host, w.in_dtype, w.rows, w.cols, rows_sel=rows_sel)
    y_host = wl.torch_to_storage(y.cpu()).reshape(w.rows, w.cols)
    parity.compare_log(y_host[rows_sel], ref, np.log(d), "bf16")
    parity.compare_lse(lse.cpu().numpy()[rows_sel], ref_lse, np.log(d))


# ------------------------------------------------------------- apply stats

def run_apply(x_store, in_dtype, out_dtype, rows, cols, m, d, valid_len=None, offset=0):
    x = to_device(x_store, in_dtype, rows, cols, offset)
    vl = lengths_t(valid_len)
    mt = torch.from_numpy(np.asarray(m, np.float32)).to(DEV)
    dt = torch.from_numpy(np.asarray(d, np.float32)).to(DEV)
    if offset:
        ybuf = torch.empty(rows * cols + offset, dtype=DT[out_dtype], device=DEV)
        y = ybuf[offset:].view(rows, cols)
        smx.softmax_apply_stats(x, mt, dt, out=y, valid_len=vl)
    else:
        y = smx.softmax_apply_stats(x, mt, dt, valid_len=vl, out_dtype=DT[out_dtype])
    y_host = wl.torch_to_storage(y.cpu())
    p = oracle.apply_stats(x_store, in_dtype, rows, cols, np.asarray(m, np.float32).astype(np.float64),
                           np.asarray(d, np.float32).astype(np.float64), valid_len)
    return parity.compare(y_host, p, out_dtype, valid_len)


def own_stats(x_store, in_dtype, rows, cols, valid_len=None):
    m, d = oracle.row_stats(x_store, in_dtype, rows, cols, valid_len)
    return m.astype(np.float32), d.astype(np.float32)


@pytest.mark.parametrize("in_dtype,out_dtype", PAIRS)
@pytest.mark.parametrize("path", PATHS)
def test_apply_worked_rows(lib, in_dtype, out_dtype, path):
    lib.smx_debug_force_path(path)
    for row in wl.WORKED_ROWS.values():
        vals = np.zeros(8, np.float32)
        vals[: len(row)] = row
        xs = stored(vals, in_dtype)
        m, d = own_stats(xs, in_dtype, 1, 8, [len(row)])
        run_apply(xs, in_dtype, out_dtype, 1, 8, m, d, [len(row)])
        xs = stored(row, in_dtype)
        m, d = own_stats(xs, in_dtype, 1, len(row))
        run_apply(xs, in_dtype, out_dtype, 1, len(row), m, d)


@pytest.mark.parametrize("cols", [8, 1000, 4096, 8192, 300000])
@pytest.mark.parametrize("in_dtype,out_dtype", [("f32", "f32"), ("bf16", "bf16"), ("f16", "f16"),
                                                ("bf16", "f32")])
def test_apply_given_row_stats(lib, cols, in_dtype, out_dtype):
    rows = 6 if cols > 10000 else 37
    rng = np.random.default_rng(cols)
    x = stored(rng.normal(0, 5, rows * cols), in_dtype)
    vl = rng.integers(0, cols + 1, rows).astype(np.int32)
    vl[0] = cols
    m, d = own_stats(x, in_dtype, rows, cols, vl)
    st = run_apply(x, in_dtype, out_dtype, rows, cols, m, d, vl)
    print(cols, lib.smx_debug_last_path(), st)


@pytest.mark.parametrize("cols", [96, 512, 1000, 1024])
@pytest.mark.parametrize("in_dtype,out_dtype", [("f16", "f16"), ("bf16", "bf16"), ("f32", "bf16"), ("bf16", "f16")])
def test_apply_warp_walkers(lib, cols, in_dtype, out_dtype):
    """Rows that fit one warp with 16-bit outputs: a row per warp, many rows per
    walker, the given statistics per row (including the policy's special
    values: -inf m, NaN m or d, +inf m), lengths 0, 1 and cols."""
    rows = 3000
    rng = np.random.default_rng(cols + 17)
    x = stored(rng.normal(0, 4, rows * cols), in_dtype)
    vl = rng.integers(0, cols + 1, rows).astype(np.int32)
    vl[::97] = 0
    vl[1::89] = 1
    vl[2::83] = cols
    m, d = own_stats(x, in_dtype, rows, cols, vl)
    m[5], d[5] = -np.inf, 0.0
    m[6] = np.nan
    d[7] = np.nan
    m[8] = np.inf
    lib.smx_debug_force_path(PATH_STREAM)
    run_apply(x, in_dtype, out_dtype, rows, cols, m, d, vl)
    assert lib.smx_debug_last_path() == PATH_STREAM
    assert smx.last_device_status() == 0


def test_apply_unaligned_and_policy(lib):
    rows, cols = 5, 1001
    rng = np.random.default_rng(9)
    x = stored(rng.normal(0, 3, rows * cols), "f32")
    m, d = own_stats(x, "f32", rows, cols)
    run_apply(x, "f32", "f32", rows, cols, m, d, offset=1)
    # given -inf: zero row; NaN m or d, or +inf m: NaN valid lanes; masked +0
    m = np.array([-np.inf, np.nan, 1.0, np.inf, 0.0], np.float32)
    d = np.array([0.0, 1.0, np.nan, 1.0, 1.0], np.float32)
    xs = stored(np.tile(np.float32([0.5, -1.0, 0.25, 0.0, 0.0, 0.0, 0.0, 0.0]), rows), "f32")
    for path in PATHS:
        lib.smx_debug_force_path(path)
        run_apply(xs, "f32", "f32", rows, 8, m, d, np.array([3, 3, 2, 1, 0], np.int32))


@pytest.mark.parametrize("in_dtype,out_dtype,cols,cut", [("f32", "f32", 4000, 1536),
                                                         ("bf16", "bf16", 65536, 24576),
                                                         ("f16", "f32", 1000, 333),
                                                         ("f32", "f32", 2_000_000, 1_200_000)])
def test_column_split_softmax(lib, in_dtype, out_dtype, cols, cut):
    """Column blocks of a row in separate buffers: row_stats per block, merge,
    apply per block -- the concatenation is the softmax of the whole row."""
    rows = 3 if cols > 100000 else 24
    rng = np.random.default_rng(cols)
    x32 = rng.normal(0, 6, (rows, cols)).astype(np.float32)
    x32[1, cut + 5] = 40.0  # the maximum in the second block on one row
    xs = stored(x32.reshape(-1), in_dtype)
    xt = to_device(xs, in_dtype, rows, cols)
    a, b = xt[:, :cut].contiguous(), xt[:, cut:].contiguous()
    ma, da = smx.softmax_row_stats(a)
    mb, db = smx.softmax_row_stats(b)
    m, d = smx.softmax_merge_stats(ma, da, mb, db)
    ya = smx.softmax_apply_stats(a, m, d, out_dtype=DT[out_dtype])
    yb = smx.softmax_apply_stats(b, m, d, out_dtype=DT[out_dtype])
    y = torch.cat([ya, yb], dim=1)
    p = oracle.softmax_rows(xs, in_dtype, rows, cols)
    parity.compare(wl.torch_to_storage(y.cpu()), p, out_dtype)


@pytest.mark.parametrize("cols", [8, 256, 1000, 1024])
@pytest.mark.parametrize("in_dtype,out_dtype", [("f32", "f32"), ("bf16", "bf16"), ("f16", "f32")])
@pytest.mark.parametrize("warp_off", [0, 1])
def test_log_stream_walkers(lib, cols, in_dtype, out_dtype, warp_off):
    rows = 1500
    rng = np.random.default_rng(cols + 12)
    x = stored(rng.normal(0, 6, rows * cols), in_dtype)
    vl = rng.integers(0, cols + 1, size=rows).astype(np.int32)
    vl[::97] = 0
    lib.smx_debug_force_path(PATH_STREAM)
    lib.smx_debug_set_stream_warp(warp_off)
    run_log(x, in_dtype, out_dtype, rows, cols, vl)
