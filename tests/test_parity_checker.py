"""The parity checker (tests/parity.py) is itself checked on the CPU: the
reference's own results, rounded to each output type, pass; copies with one
planted mistake (an element a few units off, a masked or excluded lane
written, a -0, a NaN row with a finite lane, swapped lanes or rows, a row
not normalised, a log-space masked or excluded lane that is not -inf, a
dropped term of the backward, a wrong loss, a written ignored row) fail.  The GPU parity tests rest on these functions, so a checker
too lax to see such mistakes would make every parity claim empty.
"""
import numpy as np
import pytest

import oracle
from numerically_stable_online_gb300 import workloads as wl
from tests import parity

ROWS, COLS = 8, 16
VL = np.array([16, 9, 16, 16, 16, 0, 16, 12], np.int32)


@pytest.fixture(scope="module", autouse=True)
def built():
    oracle.build()


def logits():
    """Rows: 0 normal, 1 masked tail, 2 all -inf, 3 one -inf lane, 4 NaN row,
    5 empty, 6 a wide spread (probabilities below 1e-30), 7 normal with a tail."""
    rng = np.random.default_rng(3)
    x = rng.normal(0, 4, (ROWS, COLS)).astype(np.float32)
    x[2, :] = -np.inf
    x[3, 5] = -np.inf
    x[4, 7] = np.nan
    x[6, :] = np.linspace(0, -90, COLS, dtype=np.float32)
    return wl.to_storage(x.reshape(-1), "f32"), x


def must_fail(fn, *args, **kw):
    with pytest.raises(AssertionError):
        fn(*args, **kw)


# ------------------------------------------------------------------ softmax

@pytest.fixture(scope="module")
def softmax_ref():
    xs, _ = logits()
    return oracle.softmax_rows(xs, "f32", ROWS, COLS, VL)


def test_softmax_f32_exact_passes_and_mistakes_fail(softmax_ref):
    p = softmax_ref
    y0 = p.astype(np.float32)
    parity.compare(y0, p, "f32", VL)
    y = y0.copy()
    y[0] *= np.float32(1 + 1e-6)                  # inside 2e-6
    parity.compare(y, p, "f32", VL)

    def planted(r, c, v):
        y = y0.copy()
        y[r, c] = v
        return y

    must_fail(parity.compare, planted(0, 3, y0[0, 3] * np.float32(1 + 4e-6)), p, "f32", VL)
    must_fail(parity.compare, planted(1, 12, 1e-38), p, "f32", VL)       # masked lane
    must_fail(parity.compare, planted(2, 0, -0.0), p, "f32", VL)         # all -inf row
    must_fail(parity.compare, planted(2, 0, 1e-45), p, "f32", VL)
    must_fail(parity.compare, planted(3, 5, 1e-40), p, "f32", VL)        # excluded lane
    must_fail(parity.compare, planted(4, 2, 0.5), p, "f32", VL)          # NaN row lane finite
    must_fail(parity.compare, planted(0, 3, np.nan), p, "f32", VL)
    must_fail(parity.compare, planted(6, 15, -0.0), p, "f32", VL)        # tiny lane as -0
    must_fail(parity.compare, planted(6, 15, 3e-30), p, "f32", VL)       # tiny lane too big
    assert p[6, 15] < parity.F32_TINY and p[6, 15] > 0
    y = y0.copy()
    y[0, [1, 2]] = y[0, [2, 1]]                                           # swapped lanes
    assert p[0, 1] != p[0, 2]
    must_fail(parity.compare, y, p, "f32", VL)
    y = y0.copy()
    y[[0, 7]] = y[[7, 0]]                                                 # swapped rows
    must_fail(parity.compare, y, p, "f32", VL)
    y = y0.copy()
    y[7] *= np.float32(1 + 1e-4)                                          # not normalised
    must_fail(parity.compare, y, p, "f32", VL)


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
def test_softmax_16bit_exact_passes_and_mistakes_fail(softmax_ref, fmt):
    p = softmax_ref
    b0 = oracle.round_to(p, fmt)
    parity.compare(b0, p, fmt, VL)
    b = b0.copy()
    b[0, 3] += 1                                                          # one unit: allowed
    b[7, 0] -= 1
    parity.compare(b, p, fmt, VL)

    def planted(r, c, v):
        b = b0.copy()
        b[r, c] = v
        return b

    must_fail(parity.compare, planted(0, 3, b0[0, 3] + 2), p, fmt, VL)
    must_fail(parity.compare, planted(1, 12, 1), p, fmt, VL)             # masked lane
    must_fail(parity.compare, planted(3, 5, 1), p, fmt, VL)              # excluded lane
    must_fail(parity.compare, planted(2, 4, 0x8000), p, fmt, VL)         # -0 in an all -inf row
    must_fail(parity.compare, planted(0, 3, b0[0, 3] | 0x8000), p, fmt, VL)
    must_fail(parity.compare, planted(4, 2, b0[0, 3]), p, fmt, VL)       # NaN row lane finite
    b = b0.copy()
    b[[0, 7]] = b[[7, 0]]
    must_fail(parity.compare, b, p, fmt, VL)


# ------------------------------------------------------------------ log space

def log_case():
    xs, _ = logits()
    ref, lse = oracle.log_softmax_rows(xs, "f32", ROWS, COLS, VL)
    _, d = oracle.row_stats(xs, "f32", ROWS, COLS, VL)
    with np.errstate(divide="ignore", invalid="ignore"):
        log_d = np.where(d > 0, np.log(np.where(d > 0, d, 1.0)), 0.0)
    return ref, lse, log_d


def test_log_softmax_and_lse_checks():
    ref, lse, log_d = log_case()
    y0 = ref.astype(np.float32)
    parity.compare_log(y0, ref, log_d, "f32", VL)
    parity.compare_lse(lse.astype(np.float32), lse, log_d)
    y = y0.copy()
    y[1, 12] = 0.0                                                        # masked lane not -inf
    must_fail(parity.compare_log, y, ref, log_d, "f32", VL)
    y = y0.copy()
    y[0, 3] += np.float32(4 * (2.0 ** -22 * (abs(ref[0, 3]) + log_d[0]) + 2.0 ** -18))
    must_fail(parity.compare_log, y, ref, log_d, "f32", VL)
    y = y0.copy()
    y[3, 5] = np.float32(-200.0)                                          # excluded lane finite
    must_fail(parity.compare_log, y, ref, log_d, "f32", VL)
    b0 = oracle.round_to(ref, "bf16")
    parity.compare_log(b0, ref, log_d, "bf16", VL)
    lane = np.argmax(np.where(np.isfinite(ref[0]), np.abs(ref[0]), 0) > 0.5)
    b = b0.copy()
    b[0, lane] += 2
    must_fail(parity.compare_log, b, ref, log_d, "bf16", VL)
    bad = lse.copy()
    bad[0] += 1e-3
    must_fail(parity.compare_lse, bad, lse, log_d)
    bad = lse.copy()
    bad[5] = 0.0                                                          # empty row: -inf
    must_fail(parity.compare_lse, bad, lse, log_d)
    bad = lse.copy()
    bad[4] = 1.0                                                          # NaN row
    must_fail(parity.compare_lse, bad, lse, log_d)


# ------------------------------------------------------------------ backward

def test_backward_checks():
    rng = np.random.default_rng(9)
    _, x = logits()
    x = np.nan_to_num(x, nan=0.0, neginf=-50.0)
    p = np.exp(x - x.max(axis=1, keepdims=True))
    p = (p / p.sum(axis=1, keepdims=True)).astype(np.float32)
    g = rng.normal(0, 1, (ROWS, COLS)).astype(np.float32)
    ps, gs = wl.to_storage(p.reshape(-1), "f32"), wl.to_storage(g.reshape(-1), "f32")
    ref = oracle.softmax_backward(ps, gs, "f32", ROWS, COLS, VL)
    pv = oracle.decode(ps, "f32").reshape(ROWS, COLS)
    gv = oracle.decode(gs, "f32").reshape(ROWS, COLS)
    y0 = ref.astype(np.float32)
    parity.compare_backward(y0, ref, pv, gv, "f32", VL)
    y = y0.copy()
    y[1, 12] = 1e-30                                                      # masked lane
    must_fail(parity.compare_backward, y, ref, pv, gv, "f32", VL)
    # the bound is absolute in p (|g| + sum |g p|) (the fp32 sum's error enters
    # before the cancellation in g - sum g p): plant errors well beyond it
    y = y0.copy()
    y[0, 4] += np.float32(1e-3)
    must_fail(parity.compare_backward, y, ref, pv, gv, "f32", VL)
    dropped = np.where(np.arange(COLS)[None, :] < VL[:, None], pv * gv, 0.0).astype(np.float32)
    must_fail(parity.compare_backward, dropped, ref, pv, gv, "f32", VL)   # sum g p term dropped
    y = y0.copy()
    y[7] = -y[7]                                                          # sign of the product
    must_fail(parity.compare_backward, y, ref, pv, gv, "f32", VL)


# ------------------------------------------------------------------ cross-entropy

def test_cross_entropy_checks():
    xs, _ = logits()
    target = np.array([3, 10, 0, 2, 1, 0, 0, 5], np.int64)               # row 1: 10 >= 9, ignored
    loss, grad = oracle.cross_entropy(xs, "f32", ROWS, COLS, target, VL)
    _, d = oracle.row_stats(xs, "f32", ROWS, COLS, VL)
    with np.errstate(divide="ignore", invalid="ignore"):
        log_d = np.where(d > 0, np.log(np.where(d > 0, d, 1.0)), 0.0)
    l0, g0 = loss.astype(np.float32), grad.astype(np.float32)
    parity.compare_ce(l0, g0, loss, grad, log_d, target, "f32", VL)
    parity.compare_ce(l0, None, loss, None, log_d, target, "f32", VL)
    bad = l0.copy()
    bad[0] += np.float32(1e-3)
    must_fail(parity.compare_ce, bad, g0, loss, grad, log_d, target, "f32", VL)
    g = g0.copy()
    g[1, 0] = 0.25                                                        # ignored row written
    must_fail(parity.compare_ce, l0, g, loss, grad, log_d, target, "f32", VL)
    g = g0.copy()
    g[0, 3] += np.float32(1.0)                                            # onehot dropped twice
    must_fail(parity.compare_ce, l0, g, loss, grad, log_d, target, "f32", VL)
    g = g0.copy()
    g[7, 13] = 1e-20                                                      # masked lane
    must_fail(parity.compare_ce, l0, g, loss, grad, log_d, target, "f32", VL)
    gb = oracle.round_to(grad, "bf16")
    parity.compare_ce(l0, gb, loss, grad, log_d, target, "bf16", VL)
