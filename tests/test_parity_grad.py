"""Parity of the softmax backward and the fused cross-entropy (CUDA path through
the C ABI) with the fp64 reference, with the tolerances derived in
tests/parity.py (compare_backward, compare_ce).

Cases: every dtype pair; each kernel that takes the op (whole rows streamed,
long rows in chunks, the scalar kernel for unaligned shapes); valid lengths
including 0 and cols; NaN rows; ignored targets; the loss alone; the pages'
worked rows and the "confidently wrong" row; the benchmark's workload shape at
full size on sampled rows.
"""
import math

import numpy as np
import pytest
import torch

import numerically_stable_online_gb300 as smx
import oracle
from numerically_stable_online_gb300 import workloads as wl
from tests import parity
from tests.test_parity_gpu import stored, to_device

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
PAIRS = [(a, b) for a in DT for b in DT]
PATH_GENERIC, PATH_STREAM, PATH_SPLIT = 3, 4, 5
PATHS = [PATH_GENERIC, PATH_STREAM, PATH_SPLIT]
CE_PATHS = PATHS + [6]  # and the read-once long-row kernel
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


# --------------------------------------------------------------- backward

def make_pg(rows, cols, dtype, seed, valid_len=None):
    """p: a stored softmax of random logits (0 in masked lanes); g: N(0, 1)."""
    rng = np.random.default_rng(seed)
    x = rng.normal(0, 3, (rows, cols)).astype(np.float32)
    L = parity.lengths(rows, cols, valid_len)
    p = np.zeros((rows, cols), np.float64)
    for r in range(rows):
        if L[r]:
            e = np.exp(x[r, :L[r]] - x[r, :L[r]].max())
            p[r, :L[r]] = e / e.sum()
    g = rng.normal(0, 1, (rows, cols))
    return stored(p.astype(np.float32).reshape(-1), dtype), stored(g.astype(np.float32).reshape(-1), dtype)


def run_backward(p_store, g_store, dtype, dx_dtype, rows, cols, valid_len=None, offset=0):
    p = to_device(p_store, dtype, rows, cols, offset)
    g = to_device(g_store, dtype, rows, cols, offset)
    vl = lengths_t(valid_len)
    if offset:
        buf = torch.empty(rows * cols + offset, dtype=DT[dx_dtype], device=DEV)
        dx = buf[offset:].view(rows, cols)
        smx.softmax_backward(p, g, out=dx, valid_len=vl)
    else:
        dx = smx.softmax_backward(p, g, valid_len=vl, out_dtype=DT[dx_dtype])
    ref = oracle.softmax_backward(p_store, g_store, dtype, rows, cols, valid_len)
    pv = oracle.decode(p_store, dtype).reshape(rows, cols)
    gv = oracle.decode(g_store, dtype).reshape(rows, cols)
    return parity.compare_backward(wl.torch_to_storage(dx.cpu()), ref, pv, gv, dx_dtype, valid_len)


@pytest.mark.parametrize("dtype,dx_dtype", PAIRS)
@pytest.mark.parametrize("path", PATHS)
def test_backward_pairs_and_paths(lib, dtype, dx_dtype, path):
    lib.smx_debug_force_path(path)
    rows, cols = 11, 1000
    vl = np.array([cols, 0, 1, 999, 500, 8, 7, cols, 3, 640, 2], np.int32)
    p, g = make_pg(rows, cols, dtype, 31, vl)
    run_backward(p, g, dtype, dx_dtype, rows, cols, vl)
    p, g = make_pg(rows, cols, dtype, 32)
    run_backward(p, g, dtype, dx_dtype, rows, cols)


@pytest.mark.parametrize("cols", [8, 24, 1000, 4096, 8192, 8200, 40000, 1_048_576])
@pytest.mark.parametrize("dtype,dx_dtype", [("f32", "f32"), ("bf16", "bf16"), ("f16", "f32")])
def test_backward_shapes(lib, cols, dtype, dx_dtype):
    rows = 2 if cols > 100000 else 9
    rng = np.random.default_rng(cols)
    vl = rng.integers(0, cols + 1, rows).astype(np.int32)
    vl[0] = cols
    p, g = make_pg(rows, cols, dtype, cols, vl)
    st = run_backward(p, g, dtype, dx_dtype, rows, cols, vl)
    print(cols, lib.smx_debug_last_path(), st)


def test_backward_unaligned_and_nan(lib):
    rows, cols = 6, 1001
    p, g = make_pg(rows, cols, "f32", 5)
    run_backward(p, g, "f32", "f32", rows, cols, offset=1)
    pv = np.array([[0.25, 0.75, 0.0, 0.0, 0, 0, 0, 0], [0.5, 0.5, 0, 0, 0, 0, 0, 0]], np.float32)
    gv = np.array([[1.0, 2.0, 9.0, 9.0, 0, 0, 0, 0], [np.nan, 1.0, 0, 0, 0, 0, 0, 0]], np.float32)
    for path in PATHS:
        lib.smx_debug_force_path(path)
        run_backward(stored(pv.reshape(-1), "f32"), stored(gv.reshape(-1), "f32"), "f32", "f32", 2, 8,
                     np.array([2, 2], np.int32))


def test_backward_bench_shape_full_size(lib):
    rows, cols = 16384, 4096
    gen = torch.Generator(device=DEV).manual_seed(41)
    x = torch.randn(rows, cols, generator=gen, device=DEV) * 8
    p = torch.softmax(x, dim=1).to(torch.bfloat16)
    g = torch.randn(rows, cols, generator=gen, device=DEV).to(torch.bfloat16)
    dx = smx.softmax_backward(p, g)
    sel = np.random.default_rng(6).choice(rows, 512, replace=False)
    ps = wl.torch_to_storage(p[sel].cpu()).reshape(-1)
    gs = wl.torch_to_storage(g[sel].cpu()).reshape(-1)
    ref = oracle.softmax_backward(ps, gs, "bf16", len(sel), cols)
    parity.compare_backward(wl.torch_to_storage(dx[sel].cpu()), ref,
                            oracle.decode(ps, "bf16").reshape(-1, cols),
                            oracle.decode(gs, "bf16").reshape(-1, cols), "bf16")


# ----------------------------------------------------------- cross-entropy

def run_ce(x_store, in_dtype, grad_dtype, rows, cols, target, valid_len=None, offset=0,
           with_grad=True):
    x = to_device(x_store, in_dtype, rows, cols, offset)
    vl = lengths_t(valid_len)
    t = torch.from_numpy(np.asarray(target, np.int64)).to(DEV)
    grad = None
    if with_grad:
        if offset:
            buf = torch.empty(rows * cols + offset, dtype=DT[grad_dtype], device=DEV)
            grad = buf[offset:].view(rows, cols)
        else:
            grad = torch.empty(rows, cols, dtype=DT[grad_dtype], device=DEV)
    loss, grad = smx.cross_entropy(x, t, valid_len=vl, with_grad=with_grad, grad=grad)
    ref_loss, ref_grad = oracle.cross_entropy(x_store, in_dtype, rows, cols, target, valid_len,
                                              want_grad=with_grad)
    _, d = oracle.row_stats(x_store, in_dtype, rows, cols, valid_len)
    with np.errstate(divide="ignore", invalid="ignore"):
        log_d = np.where(d > 0, np.log(np.where(d > 0, d, 1.0)), 0.0)
    g_host = None if grad is None else wl.torch_to_storage(grad.cpu())
    return parity.compare_ce(loss.cpu().numpy(), g_host, ref_loss, ref_grad, log_d, target,
                             grad_dtype, valid_len)


@pytest.mark.parametrize("in_dtype,grad_dtype", PAIRS)
@pytest.mark.parametrize("path", CE_PATHS)
def test_ce_worked_rows(lib, in_dtype, grad_dtype, path):
    lib.smx_debug_force_path(path)
    for row in list(wl.WORKED_ROWS.values()) + [[1000.0, 0.0]]:
        vals = np.zeros(8, np.float32)
        vals[: len(row)] = row
        for t in range(-1, len(row) + 1):
            run_ce(stored(vals, in_dtype), in_dtype, grad_dtype, 1, 8, [t], [len(row)])
            run_ce(stored(vals, in_dtype), in_dtype, grad_dtype, 1, 8, [t], [len(row)], with_grad=False)


def test_ce_confidently_wrong_is_finite(lib):
    x = torch.tensor([[1000.0, 0.0, 0.0, 0.0]], device=DEV)
    loss, grad = smx.cross_entropy(x, torch.tensor([1], device=DEV))
    assert math.isfinite(loss.item()) and abs(loss.item() - 1000.0) < 1e-3
    # p = (1, ~e^-1000 = 0, 0, 0) to within the gradient tolerance (6e-6 p + 2^-24)
    assert torch.all((grad.cpu() - torch.tensor([[1.0, -1.0, 0.0, 0.0]])).abs() <= 6.1e-6)


@pytest.mark.parametrize("path", CE_PATHS)
@pytest.mark.parametrize("with_grad", [True, False])
def test_ce_policy_rows(lib, path, with_grad):
    from tests.test_parity_gpu import POLICY_ROWS
    lib.smx_debug_force_path(path)
    rows = np.array(POLICY_ROWS, np.float32)
    n = rows.shape[0]
    x = stored(rows.reshape(-1), "f32")
    run_ce(x, "f32", "f32", n, 8, np.arange(n) % 8, with_grad=with_grad)
    run_ce(x, "f32", "f32", n, 8, np.array([1, 0, 7, 3, 1, 0, 0, 9]),
           np.array([2, 1, 8, 8, 2, 0, 1, 4], np.int32), with_grad=with_grad)


SMALL = [("f32_64x1000", 64), ("bf16_16384x4096", 96), ("f16_32768x1024_len", 777),
         ("f32_64x1048576_rise", 3)]


@pytest.mark.parametrize("name,rows", SMALL)
@pytest.mark.parametrize("with_grad", [True, False])
def test_ce_workloads_reduced(lib, name, rows, with_grad):
    w = wl.WORKLOADS[name]
    x, vl = wl.host_input(name, rows=rows)
    rng = np.random.default_rng(rows)
    t = rng.integers(0, w.cols, rows)
    t[::13] = -100  # ignored
    st = run_ce(x, w.in_dtype, w.out_dtype, rows, w.cols, t, vl, with_grad=with_grad)
    print(name, lib.smx_debug_last_path(), st)


@pytest.mark.parametrize("cols", [7, 8, 1000, 4096, 8200, 40000])
@pytest.mark.parametrize("in_dtype,grad_dtype", [("f32", "f32"), ("bf16", "bf16"), ("bf16", "f32")])
def test_ce_shapes(lib, cols, in_dtype, grad_dtype):
    rows = 9
    rng = np.random.default_rng(cols + 3)
    x = stored(rng.normal(0, 5, rows * cols), in_dtype)
    vl = rng.integers(0, cols + 1, rows).astype(np.int32)
    vl[0] = cols
    t = rng.integers(0, cols, rows)
    run_ce(x, in_dtype, grad_dtype, rows, cols, t, vl)
    run_ce(x, in_dtype, grad_dtype, rows, cols, t)


def test_ce_unaligned(lib):
    rows, cols = 5, 1000
    rng = np.random.default_rng(8)
    x = stored(rng.normal(0, 4, rows * cols), "f32")
    run_ce(x, "f32", "f32", rows, cols, rng.integers(0, cols, rows), offset=1)


def test_ce_bench_workload_full_size(lib):
    name = "bf16_16384x4096"
    w = wl.WORKLOADS[name]
    x_host, _ = wl.host_input(name)
    x = to_device(x_host, w.in_dtype, w.rows, w.cols)
    t = torch.from_numpy(np.random.default_rng(9).integers(0, w.cols, w.rows)).to(DEV)
    loss, grad = smx.cross_entropy(x, t)
    assert torch.all(grad.float().sum(dim=1).abs() <= 2e-2)
    sel = np.random.default_rng(10).choice(w.rows, 1024, replace=False)
    xs = x_host.reshape(w.rows, w.cols)[sel].reshape(-1)
    tt = t.cpu().numpy()[sel]
    ref_loss, ref_grad = oracle.cross_entropy(xs, "bf16", len(sel), w.cols, tt)
    _, d = oracle.row_stats(xs, "bf16", len(sel), w.cols)
    parity.compare_ce(loss.cpu().numpy()[sel], wl.torch_to_storage(grad[sel].cpu()), ref_loss,
                      ref_grad, np.log(d), tt, "bf16")


@pytest.mark.parametrize("cols", [8, 256, 1000, 1024])
@pytest.mark.parametrize("in_dtype,grad_dtype", [("f32", "f32"), ("bf16", "bf16"), ("f16", "f16")])
@pytest.mark.parametrize("warp_off", [0, 1])
@pytest.mark.parametrize("with_grad", [True, False])
def test_ce_stream_walkers(lib, cols, in_dtype, grad_dtype, warp_off, with_grad):
    rows = 1500
    rng = np.random.default_rng(cols + 13)
    x = stored(rng.normal(0, 6, rows * cols), in_dtype)
    vl = rng.integers(0, cols + 1, size=rows).astype(np.int32)
    vl[::97] = 0
    t = rng.integers(-1, cols + 1, rows)
    lib.smx_debug_force_path(PATH_STREAM)
    lib.smx_debug_set_stream_warp(warp_off)
    run_ce(x, in_dtype, grad_dtype, rows, cols, t, vl, with_grad=with_grad)
