"""Parity of the read-once long-row kernel (path 6: each row in column stripes
held in the shared memory of a cooperative grid) with the fp64 reference.

Cases: every input/output type pair on rows of one group of 152 stripes and
on many groups of a few stripes each; valid lengths 0, 1, cols and lengths
that end exactly on a stripe boundary or inside one; the policy rows (NaN and
+inf in one stripe, a stripe of -inf only, an all -inf row, an empty row);
log_softmax and the cross-entropy with its gradient (targets in any stripe,
ignored targets); the softmax backward (slots holding the stripes of p and
g, partial dots added across warps and stripes; NaN in one stripe, valid
lengths cut anywhere, rows of several groups); calls in a row with different
row counts and streams (the
kernel's per-row counters alternate between two arrays, and a call zeroes the
other one for the next); the error path of the per-row count waits; and that
the long-row workload takes this path by default in one launch.
"""
import numpy as np
import pytest
import torch

import numerically_stable_online_gb300 as smx
import oracle
from numerically_stable_online_gb300 import workloads as wl
from tests import parity
from tests.test_parity_gpu import run_and_compare, stored, to_device

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
PATH_SPLIT, PATH_STRIPE = 5, 6
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
    built.smx_debug_set_count_probe(0)
    built.smx_debug_set_split_fused(0)
    built.smx_debug_set_split_slab(0)


def lengths_t(valid_len):
    return None if valid_len is None else torch.from_numpy(np.asarray(valid_len, np.int32)).to(DEV)


def stripe_bounds(cols, in_dtype, q_count):
    """Column where each stripe starts, as the kernel cuts them (vector units)."""
    V = 4 if in_dtype == "f32" else 8
    nvec = cols // V
    return [q * nvec // q_count * V for q in range(q_count + 1)]


def rising_rows(rows, cols, seed, scale=3.0):
    rng = np.random.default_rng(seed)
    return (rng.normal(0, scale, (rows, cols)) + np.linspace(-4, 24, cols)[None, :]).astype(np.float32)


PAIRS = [("f32", "f32"), ("bf16", "bf16"), ("f16", "f16"), ("f16", "f32"), ("f32", "bf16"), ("bf16", "f16")]


@pytest.mark.parametrize("in_dtype,out_dtype", PAIRS)
@pytest.mark.parametrize("rows,cols", [(3, 1_048_576), (5, 300_000 + 8), (40, 65_536 + 24)])
def test_softmax_rows(lib, in_dtype, out_dtype, rows, cols):
    x32 = rising_rows(rows, cols, rows + cols)
    x = stored(x32.reshape(-1), in_dtype)
    b = stripe_bounds(cols, in_dtype, 152)
    vl = np.full(rows, cols, np.int32)
    vl[0] = cols
    if rows > 1:
        vl[1] = 0
    if rows > 2:
        vl[2] = b[37]  # ends exactly where a stripe (of a one-group grid) starts
    if rows > 3:
        vl[3] = 1
    if rows > 4:
        vl[4] = b[100] + 3  # ends inside a stripe
    lib.smx_debug_force_path(PATH_STRIPE)
    smx.softmax_rows(to_device(x, in_dtype, rows, cols), valid_len=lengths_t(vl), out_dtype=DT[out_dtype])
    assert lib.smx_debug_last_path() == PATH_STRIPE
    assert lib.smx_debug_last_launches() == 1
    assert smx.last_device_status() == 0
    run_and_compare(x, in_dtype, out_dtype, rows, cols, vl)
    assert lib.smx_debug_last_path() == PATH_STRIPE
    run_and_compare(x, in_dtype, out_dtype, rows, cols, None)
    assert lib.smx_debug_last_path() == PATH_STRIPE


@pytest.mark.parametrize("in_dtype,out_dtype", [("f32", "f32"), ("bf16", "bf16"), ("f16", "f32")])
def test_policy_long_rows(lib, in_dtype, out_dtype):
    rows, cols = 8, 400_000
    x32 = rising_rows(rows, cols, 7)
    b = stripe_bounds(cols, in_dtype, 152)
    x32[0, b[50] + 5] = np.nan                    # NaN in one stripe: the row is NaN
    x32[1, b[151] + 2] = np.inf                   # +inf in the last stripe: NaN row
    x32[2, b[10]:b[12]] = -np.inf                 # two stripes of -inf only: +0 there
    x32[3, :] = -np.inf                           # all -inf: the empty row's +0
    x32[4, 17] = -np.inf                          # one -inf lane: +0 there, the rest normal
    x32[5, b[80] + 1] = np.nan                    # NaN past the valid prefix: no effect
    x32[6, 0] = 80.0                              # one element dominates: others underflow
    vl = np.array([cols, cols, cols, cols, cols, b[80], 0, b[3] + 1], np.int32)
    x = stored(x32.reshape(-1), in_dtype)
    lib.smx_debug_force_path(PATH_STRIPE)
    run_and_compare(x, in_dtype, out_dtype, rows, cols, vl)
    assert lib.smx_debug_last_path() == PATH_STRIPE
    vl[6] = cols
    run_and_compare(x, in_dtype, out_dtype, rows, cols, vl)
    assert smx.last_device_status() == 0


@pytest.mark.parametrize("in_dtype,out_dtype", [("f32", "f32"), ("bf16", "bf16"), ("f16", "f32")])
@pytest.mark.parametrize("rows,cols", [(4, 1_048_576), (30, 100_000)])
def test_log_softmax(lib, in_dtype, out_dtype, rows, cols):
    x32 = rising_rows(rows, cols, 11 + rows)
    x32[1, 5000] = np.nan
    vl = np.full(rows, cols, np.int32)
    vl[2] = 0
    vl[3] = cols // 3
    x_store = stored(x32.reshape(-1), in_dtype)
    x = to_device(x_store, in_dtype, rows, cols)
    lib.smx_debug_force_path(PATH_STRIPE)
    y = smx.log_softmax_rows(x, valid_len=lengths_t(vl), out_dtype=DT[out_dtype])
    assert lib.smx_debug_last_path() == PATH_STRIPE
    assert smx.last_device_status() == 0
    ref, _ = oracle.log_softmax_rows(x_store, in_dtype, rows, cols, vl)
    _, d = oracle.row_stats(x_store, in_dtype, rows, cols, vl)
    with np.errstate(divide="ignore", invalid="ignore"):
        log_d = np.where(d > 0, np.log(np.where(d > 0, d, 1.0)), 0.0)
    parity.compare_log(wl.torch_to_storage(y.cpu()), ref, log_d, out_dtype, vl)


@pytest.mark.parametrize("in_dtype,grad_dtype", [("f32", "f32"), ("bf16", "bf16"), ("bf16", "f32"),
                                                 ("f32", "f16")])
def test_cross_entropy(lib, in_dtype, grad_dtype):
    rows, cols = 12, 500_000
    x32 = rising_rows(rows, cols, 5)
    x32[4, 123] = np.inf
    b = stripe_bounds(cols, in_dtype, 152)
    vl = np.full(rows, cols, np.int32)
    vl[5] = 0
    vl[6] = b[60]
    t = np.array([0, cols - 1, b[77], b[77] - 1, 10, 3, b[60], b[60] - 1, -1, cols, 250_001, b[151]])
    x_store = stored(x32.reshape(-1), in_dtype)
    x = to_device(x_store, in_dtype, rows, cols)
    lib.smx_debug_force_path(PATH_STRIPE)
    grad = torch.empty(rows, cols, dtype=DT[grad_dtype], device=DEV)
    loss, grad = smx.cross_entropy(x, torch.from_numpy(t).to(DEV), valid_len=lengths_t(vl), grad=grad)
    assert lib.smx_debug_last_path() == PATH_STRIPE
    assert smx.last_device_status() == 0
    ref_loss, ref_grad = oracle.cross_entropy(x_store, in_dtype, rows, cols, t, vl, want_grad=True)
    _, d = oracle.row_stats(x_store, in_dtype, rows, cols, vl)
    with np.errstate(divide="ignore", invalid="ignore"):
        log_d = np.where(d > 0, np.log(np.where(d > 0, d, 1.0)), 0.0)
    parity.compare_ce(loss.cpu().numpy(), wl.torch_to_storage(grad.cpu()), ref_loss, ref_grad, log_d, t,
                      grad_dtype, vl)


def test_calls_in_a_row_and_streams(lib):
    """The per-row counters alternate between two arrays from call to call; each
    call zeroes the array the next one counts in.  Row counts that grow (the
    counters are reallocated) and shrink, and a second stream, must all give
    the reference result."""
    cols = 262_144
    lib.smx_debug_force_path(PATH_STRIPE)
    side = torch.cuda.Stream()
    for k, rows in enumerate([3, 10, 2, 17, 17, 1, 33]):
        x32 = rising_rows(rows, cols, 100 + k)
        vl = np.random.default_rng(k).integers(0, cols + 1, rows).astype(np.int32)
        x = to_device(x32, "f32", rows, cols)
        if k % 3 == 2:
            with torch.cuda.stream(side):
                y = smx.softmax_rows(x, valid_len=lengths_t(vl))
            side.synchronize()
        else:
            y = smx.softmax_rows(x, valid_len=lengths_t(vl))
        assert lib.smx_debug_last_path() == PATH_STRIPE
        p = oracle.softmax_rows(x32.reshape(-1), "f32", rows, cols, vl)
        parity.compare(y.cpu().numpy(), p, "f32", vl)
    assert smx.last_device_status() == 0


@pytest.mark.parametrize("path,fused", [(PATH_STRIPE, 0), (PATH_SPLIT, 1)])
def test_count_wait_runs_out_and_context_stays_usable(lib, path, fused):
    """Each per-row count wait of the cooperative long-row kernels asks for one
    stripe (or chunk) more than the row has, gives up after 64 polls and
    records SMX_ERR_TIMEOUT; the next call on the same context is correct and
    reports nothing."""
    rows, cols = 6, 300_000
    x32 = rising_rows(rows, cols, 3)
    x = to_device(x32, "f32", rows, cols)
    lib.smx_debug_force_path(path)
    lib.smx_debug_set_split_fused(fused)
    assert smx.last_device_status() == 0
    lib.smx_debug_set_count_probe(64)
    smx.softmax_rows(x)
    st = smx.last_device_status()
    lib.smx_debug_set_count_probe(0)
    assert lib.smx_debug_last_path() == path
    assert st == 5, f"expected SMX_ERR_TIMEOUT, got {st}"
    y = smx.softmax_rows(x)
    assert smx.last_device_status() == 0
    p = oracle.softmax_rows(x32.reshape(-1), "f32", rows, cols)
    parity.compare(y.cpu().numpy(), p, "f32")


def test_long_row_workload_takes_the_read_once_path(lib):
    name = "f32_64x1048576_rise"
    w = wl.WORKLOADS[name]
    x_host, _ = wl.host_input(name, rows=8)
    x = to_device(x_host, "f32", 8, w.cols)
    y = smx.softmax_rows(x)
    assert lib.smx_debug_last_path() == PATH_STRIPE
    assert lib.smx_debug_last_launches() == 1
    assert smx.last_device_status() == 0
    p = oracle.softmax_rows(x_host, "f32", 8, w.cols)
    parity.compare(y.cpu().numpy(), p, "f32")


def test_fast_kept_exponentials_at_the_edge_of_their_range(lib):
    """fp32 rows whose warps hold values within 11 of their maximum take the
    plain exponential form; wider warps the compensated one.  Rows at the
    edge of that range (uniform over the 11 below the maximum), at large
    offsets (the row constant's rounding), with a few far values that send
    some warps back to the compensated form, all within the fp32 bar."""
    rows, cols = 6, 1_048_576
    rng = np.random.default_rng(611)
    x = np.empty((rows, cols), np.float32)
    x[0] = rng.normal(0, 1, cols)                       # narrow: every warp fast
    x[1] = rng.uniform(-10.999, 0, cols) + 5.0          # the whole range, small offset
    x[2] = rng.uniform(-10.999, 0, cols) + 1000.0       # the whole range, large offset
    x[3] = rng.uniform(-10.999, 0, cols) - 3000.0       # negative offset
    x[4] = rng.normal(0, 1, cols)
    x[4, ::9973] = -40.0                                # scattered far values: those warps compensated
    x[5] = rng.uniform(-11.5, 0, cols)                  # straddles the range: a mix
    lib.smx_debug_force_path(PATH_STRIPE)
    xd = to_device(x.reshape(-1), "f32", rows, cols)
    y = smx.softmax_rows(xd)
    assert lib.smx_debug_last_path() == PATH_STRIPE
    assert smx.last_device_status() == 0
    p = oracle.softmax_rows(x.reshape(-1), "f32", rows, cols)
    st = parity.compare(y.cpu().numpy(), p, "f32")
    print("fast kept exponentials:", st)


# ------------------------------------------------------------------ backward

def backward_inputs(rows, cols, dtype, seed, valid_len=None):
    """p: the stored softmax of rising logits (0 in masked lanes); g: N(0, 1)."""
    rng = np.random.default_rng(seed)
    x = rising_rows(rows, cols, seed).astype(np.float64)
    L = parity.lengths(rows, cols, valid_len)
    p = np.zeros((rows, cols), np.float64)
    for r in range(rows):
        if L[r]:
            e = np.exp(x[r, :L[r]] - x[r, :L[r]].max())
            p[r, :L[r]] = e / e.sum()
    g = rng.normal(0, 1, (rows, cols))
    return (stored(p.astype(np.float32).reshape(-1), dtype), stored(g.astype(np.float32).reshape(-1), dtype))


def backward_and_compare(p_store, g_store, dtype, dx_dtype, rows, cols, valid_len=None):
    p = to_device(p_store, dtype, rows, cols)
    g = to_device(g_store, dtype, rows, cols)
    dx = smx.softmax_backward(p, g, valid_len=lengths_t(valid_len), out_dtype=DT[dx_dtype])
    ref = oracle.softmax_backward(p_store, g_store, dtype, rows, cols, valid_len)
    pv = oracle.decode(p_store, dtype).reshape(rows, cols)
    gv = oracle.decode(g_store, dtype).reshape(rows, cols)
    return parity.compare_backward(wl.torch_to_storage(dx.cpu()), ref, pv, gv, dx_dtype, valid_len)


@pytest.mark.parametrize("dtype,dx_dtype", [("f32", "f32"), ("bf16", "bf16"), ("f16", "f32"), ("f32", "bf16")])
@pytest.mark.parametrize("rows,cols", [(3, 1_048_576), (6, 300_000 + 8), (40, 65_536 + 24)])
def test_backward_rows(lib, dtype, dx_dtype, rows, cols):
    """The backward read once: valid lengths 0, 1, cols, on a stripe boundary
    and inside a stripe; rows of one group of 152 stripes and of many groups."""
    b = stripe_bounds(cols, dtype, 152)
    vl = np.full(rows, cols, np.int32)
    if rows > 1:
        vl[1] = 0
    if rows > 2:
        vl[2] = b[37]
    if rows > 3:
        vl[3] = 1
    if rows > 4:
        vl[4] = b[100] + 3
    p, g = backward_inputs(rows, cols, dtype, rows + cols, vl)
    lib.smx_debug_force_path(PATH_STRIPE)
    backward_and_compare(p, g, dtype, dx_dtype, rows, cols, vl)
    assert lib.smx_debug_last_path() == PATH_STRIPE
    assert lib.smx_debug_last_launches() == 1
    assert smx.last_device_status() == 0
    p, g = backward_inputs(rows, cols, dtype, rows + cols + 1)
    backward_and_compare(p, g, dtype, dx_dtype, rows, cols)
    assert lib.smx_debug_last_path() == PATH_STRIPE


def test_backward_nan_and_default_path(lib):
    """NaN in g inside one stripe makes that row's dx NaN in its valid lanes
    (the dot is NaN), NaN past the valid prefix changes nothing; long rows take
    the read-once path by default, in one launch."""
    rows, cols = 5, 400_000
    b = stripe_bounds(cols, "f32", 152)
    vl = np.array([cols, cols, b[80], cols, 7], np.int32)
    p, g = backward_inputs(rows, cols, "f32", 99, vl)
    gv = g.view(np.float32).reshape(rows, cols) if g.dtype != np.float32 else g.reshape(rows, cols)
    gv[0, b[50] + 5] = np.nan
    gv[2, b[90]] = np.nan  # past the valid prefix
    backward_and_compare(p, g, "f32", "f32", rows, cols, vl)
    assert lib.smx_debug_last_path() == PATH_STRIPE
    assert lib.smx_debug_last_launches() == 1
    assert smx.last_device_status() == 0


def test_backward_workload_sampled(lib):
    """The long-row workload's shape (64 rows of 1M fp32) on the default path,
    checked on sampled rows against the reference."""
    rows, cols = 64, 1_048_576
    gen = torch.Generator(device=DEV).manual_seed(64)
    x = torch.randn(rows, cols, generator=gen, device=DEV) * 3
    pd = torch.softmax(x, dim=1)
    gd = torch.randn(rows, cols, generator=gen, device=DEV)
    dx = smx.softmax_backward(pd, gd)
    assert lib.smx_debug_last_path() == PATH_STRIPE
    assert smx.last_device_status() == 0
    sel = [0, 13, 63]
    ps = wl.torch_to_storage(pd[sel].cpu()).reshape(-1)
    gs = wl.torch_to_storage(gd[sel].cpu()).reshape(-1)
    ref = oracle.softmax_backward(ps, gs, "f32", len(sel), cols)
    parity.compare_backward(wl.torch_to_storage(dx[sel].cpu()), ref, oracle.decode(ps, "f32").reshape(-1, cols),
                            oracle.decode(gs, "f32").reshape(-1, cols), "f32")


def test_backward_count_wait_runs_out(lib):
    """The backward's per-row count waits share the error path: with the probe
    each asks for one stripe more than exists, gives up after 64 polls and
    records SMX_ERR_TIMEOUT; the next call is correct and reports nothing."""
    rows, cols = 6, 300_000
    p, g = backward_inputs(rows, cols, "f32", 5)
    lib.smx_debug_force_path(PATH_STRIPE)
    pd, gd = to_device(p, "f32", rows, cols), to_device(g, "f32", rows, cols)
    lib.smx_debug_set_count_probe(64)
    smx.softmax_backward(pd, gd)
    st = smx.last_device_status()
    lib.smx_debug_set_count_probe(0)
    assert lib.smx_debug_last_path() == PATH_STRIPE
    assert st == 5, f"expected SMX_ERR_TIMEOUT, got {st}"
    backward_and_compare(p, g, "f32", "f32", rows, cols)
    assert smx.last_device_status() == 0
