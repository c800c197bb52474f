"""Pins of the oracle's log-space, apply-statistics, backward and cross-entropy parts.

Each function is checked against something other than itself, chosen so that a
dropped term, a wrong sign, a wrong index or a transposed operand fails:
values the pages print, closed forms evaluated with library routines
(``math.log1p``, ``math.fsum``), finite differences of the forward softmax, the
explicitly built Jacobian the pages say never to build, and the column-split
completion that the apply step exists for.

Sources (page title, section): "Softmax numerics architecture - max subtract,
fp32 accumulate, fusion, online" ("Log-sum-exp: log-probabilities without
probabilities"; "The Jacobian, and the backward pass that never divides";
"A worked example: naive fp16 versus the stable form"); "Online stable softmax"
("Derive the update for two blocks").
"""
import math

import numpy as np
import pytest

import oracle


def f32(v):
    return np.asarray(v, dtype=np.float32)


def softmax_np(x):
    """Forward softmax in fp64 from the definition (for finite differences)."""
    x = np.asarray(x, dtype=np.float64)
    e = np.array([math.exp(v - x.max()) for v in x])
    return e / math.fsum(e)


# ----------------------------------------------------------------- log space

def test_log_softmax_worked_row_matches_printed_probabilities():
    # the page prints 0.84380, 0.11420, 0.04201 for [20, 18, 17, -5]: within one
    # unit of the last printed digit
    out, lse = oracle.log_softmax_rows(f32([20, 18, 17, -5]), "f32", 1, 4)
    np.testing.assert_allclose(np.exp(out[0, :3]), [0.84380, 0.11420, 0.04201], rtol=0, atol=1e-5)
    # "the sum is at least 1 so the logarithm is defined and non-negative"
    assert 0.0 <= lse[0] - 20.0 <= math.log(4)


@pytest.mark.parametrize("t", [0.5, 2.5, -7.25, 30.0])
def test_log_softmax_two_lanes_is_log_sigmoid(t):
    out, lse = oracle.log_softmax_rows(f32([0.0, t]), "f32", 1, 2)
    t = float(np.float32(t))
    # x_i - LSE in fp64 is exact to a few units of LSE's last place
    tol = 8 * 2.0**-52 * max(1.0, abs(lse[0]))
    assert out[0, 0] == pytest.approx(-math.log1p(math.exp(t)), rel=0, abs=tol)
    assert out[0, 1] == pytest.approx(-math.log1p(math.exp(-t)), rel=0, abs=tol)
    assert lse[0] == pytest.approx(max(0.0, t) + math.log1p(math.exp(-abs(t))), rel=1e-14)


def test_lse_of_equal_lanes_and_brute_force_without_shift():
    out, lse = oracle.log_softmax_rows(np.full(7, 3.5, dtype=np.float32), "f32", 1, 7)
    assert lse[0] == pytest.approx(3.5 + math.log(7), rel=1e-15)
    np.testing.assert_allclose(out[0], -math.log(7), rtol=1e-15)
    rng = np.random.default_rng(11)
    x = f32(rng.normal(0, 3, 50))
    _, lse = oracle.log_softmax_rows(x, "f32", 1, 50)
    brute = math.log(math.fsum(math.exp(float(v)) for v in x))  # no shift: fine at this scale
    assert lse[0] == pytest.approx(brute, rel=1e-14)


def test_lse_shift_and_overflow_free_row():
    rng = np.random.default_rng(12)
    x = f32(np.round(rng.normal(0, 2, 33) * 64) / 64)  # x + 1024 stays exact in fp32
    o1, l1 = oracle.log_softmax_rows(x, "f32", 1, 33)
    o2, l2 = oracle.log_softmax_rows(x + np.float32(1024), "f32", 1, 33)
    assert l2[0] - l1[0] == pytest.approx(1024.0, abs=1e-12)
    np.testing.assert_allclose(o1, o2, atol=2e-12)
    # [1000, 999, 997]: finite, LSE = 1000 + log1p(e^-1 + e^-3)
    out, lse = oracle.log_softmax_rows(f32([1000, 999, 997]), "f32", 1, 3)
    assert lse[0] == pytest.approx(1000 + math.log1p(math.exp(-1) + math.exp(-3)), rel=1e-15)
    np.testing.assert_allclose(out[0], [1000 - lse[0], 999 - lse[0], 997 - lse[0]], rtol=1e-15)
    assert np.all(np.isfinite(out))


def test_log_softmax_policy_rows():
    x = f32([[1, 2, 3, 4], [1, np.nan, 3, 4], [-np.inf, -np.inf, 5, 6], [np.inf, 0, 1, 2]])
    vl = np.array([2, 4, 2, 4], dtype=np.int32)
    out, lse = oracle.log_softmax_rows(x.reshape(-1), "f32", 4, 4, vl)
    assert np.all(out[0, 2:] == -np.inf) and np.all(np.isfinite(out[0, :2]))
    assert np.all(np.isnan(out[1])) and np.isnan(lse[1])
    assert np.all(out[2] == -np.inf) and lse[2] == -np.inf  # all valid lanes -inf: log 0
    assert np.all(np.isnan(out[3])) and np.isnan(lse[3])


# ------------------------------------------------------------- apply stats

def test_apply_stats_completes_a_column_split_softmax():
    rng = np.random.default_rng(13)
    rows, cols, cut = 5, 40, 17
    x = f32(rng.normal(0, 4, (rows, cols)))
    a, b = np.ascontiguousarray(x[:, :cut]), np.ascontiguousarray(x[:, cut:])
    ma, da = oracle.row_stats(a.reshape(-1), "f32", rows, cut)
    mb, db = oracle.row_stats(b.reshape(-1), "f32", rows, cols - cut)
    m, d = oracle.merge_stats(ma, da, mb, db)
    pa = oracle.apply_stats(a.reshape(-1), "f32", rows, cut, m, d)
    pb = oracle.apply_stats(b.reshape(-1), "f32", rows, cols - cut, m, d)
    ref = np.array([softmax_np(r) for r in x])
    np.testing.assert_allclose(np.concatenate([pa, pb], axis=1), ref, rtol=1e-13)


def test_apply_stats_closed_forms_and_policy():
    x = f32([[0.5, -1.0, 2.0], [1.0, 2.0, 3.0], [1.0, 2.0, 3.0], [1.0, 2.0, 3.0]])
    m = np.array([0.0, -np.inf, np.nan, np.inf])
    d = np.array([1.0, 0.0, 1.0, 1.0])
    vl = np.array([2, 3, 3, 1], dtype=np.int32)
    p = oracle.apply_stats(x.reshape(-1), "f32", 4, 3, m, d, vl)
    np.testing.assert_array_equal(p[0], [math.exp(0.5), math.exp(-1.0), 0.0])
    np.testing.assert_array_equal(p[1], [0.0, 0.0, 0.0])
    assert np.all(np.isnan(p[2]))
    assert np.isnan(p[3, 0]) and np.all(p[3, 1:] == 0.0)


# --------------------------------------------------------------- backward

def test_backward_matches_finite_differences():
    rng = np.random.default_rng(14)
    n = 9
    x = rng.normal(0, 1.5, n)
    g = f32(rng.normal(0, 1, n))
    p = softmax_np(x)
    dx = oracle.softmax_backward(p.astype(np.float32), g, "f32", 1, n)[0]
    # the oracle used p rounded to fp32; differentiate the loss g . softmax(x)
    h = 1e-6
    fd = np.array([(np.dot(g, softmax_np(x + h * e)) - np.dot(g, softmax_np(x - h * e))) / (2 * h)
                   for e in np.eye(n)])
    np.testing.assert_allclose(dx, fd, rtol=2e-6, atol=1e-8)


def test_backward_is_the_jacobian_product():
    rng = np.random.default_rng(15)
    n = 12
    p32 = f32(softmax_np(rng.normal(0, 2, n)))
    g = f32(rng.normal(0, 1, n))
    pd = p32.astype(np.float64)
    J = np.diag(pd) - np.outer(pd, pd)  # dp_i/dx_j = p_i (delta_ij - p_j)
    dx = oracle.softmax_backward(p32, g, "f32", 1, n)[0]
    np.testing.assert_allclose(dx, J.T @ g.astype(np.float64), rtol=1e-12, atol=1e-15)
    # one-hot gradient picks one Jacobian column
    k = 4
    e = np.zeros(n, dtype=np.float32)
    e[k] = 1
    dx = oracle.softmax_backward(p32, e, "f32", 1, n)[0]
    np.testing.assert_allclose(dx, J[k], rtol=1e-13, atol=1e-18)
    # a constant gradient moves nothing (up to the rounding of p's sum)
    dx = oracle.softmax_backward(p32, np.full(n, 3.0, np.float32), "f32", 1, n)[0]
    assert np.all(np.abs(dx) <= 3 * 4 * n * 2.0**-24 * pd)


def test_backward_masked_lanes_and_nan():
    p = f32([[0.25, 0.75, 0.0, 0.0], [0.5, 0.5, 0.0, 0.0]])
    g = f32([[1.0, 2.0, 9.0, 9.0], [np.nan, 1.0, 0.0, 0.0]])
    vl = np.array([2, 2], dtype=np.int32)
    dx = oracle.softmax_backward(p.reshape(-1), g.reshape(-1), "f32", 2, 4, vl)
    s = 0.25 * 1 + 0.75 * 2
    np.testing.assert_array_equal(dx[0], [0.25 * (1 - s), 0.75 * (2 - s), 0.0, 0.0])
    assert np.all(np.isnan(dx[1, :2])) and np.all(dx[1, 2:] == 0.0)


# ----------------------------------------------------------- cross-entropy

def test_cross_entropy_is_negative_log_softmax_and_its_gradient():
    rng = np.random.default_rng(16)
    rows, cols = 6, 11
    x = f32(rng.normal(0, 3, (rows, cols)))
    t = rng.integers(0, cols, rows)
    loss, grad = oracle.cross_entropy(x.reshape(-1), "f32", rows, cols, t)
    out, _ = oracle.log_softmax_rows(x.reshape(-1), "f32", rows, cols)
    np.testing.assert_allclose(loss, -out[np.arange(rows), t], rtol=1e-14)
    # gradient by finite differences of LSE(x) - x_t
    for r in range(rows):
        xr = x[r].astype(np.float64)

        def ce(v):
            mv = v.max()
            return mv + math.log(math.fsum(math.exp(a - mv) for a in v)) - v[t[r]]

        h = 1e-6
        fd = np.array([(ce(xr + h * e) - ce(xr - h * e)) / (2 * h) for e in np.eye(cols)])
        np.testing.assert_allclose(grad[r], fd, rtol=1e-5, atol=1e-9)
        assert np.all(np.abs(grad[r]) <= 1.0) and abs(math.fsum(grad[r])) < 1e-14


def test_cross_entropy_confidently_wrong_and_softplus():
    # "a confidently wrong prediction yields a large finite loss"
    loss, grad = oracle.cross_entropy(f32([1000.0, 0.0]), "f32", 1, 2, np.array([1]))
    assert loss[0] == 1000.0 and np.isfinite(loss[0])
    np.testing.assert_array_equal(grad[0], [1.0, -1.0])
    for t in (0.5, -3.0, 12.0):
        loss, _ = oracle.cross_entropy(f32([0.0, t]), "f32", 1, 2, np.array([0]))
        tt = float(np.float32(t))
        assert loss[0] == pytest.approx(max(tt, 0) + math.log1p(math.exp(-abs(tt))), rel=1e-14)


def test_cross_entropy_ignored_targets_and_masks():
    x = f32([[1, 2, 3, 4], [1, 2, 3, 4], [1, 2, 3, 4]])
    vl = np.array([4, 2, 4], dtype=np.int32)
    t = np.array([-1, 3, 2])  # out of range; beyond the valid prefix; valid
    loss, grad = oracle.cross_entropy(x.reshape(-1), "f32", 3, 4, t, vl)
    assert loss[0] == 0.0 and np.all(grad[0] == 0.0)
    assert loss[1] == 0.0 and np.all(grad[1] == 0.0)
    p = softmax_np([1, 2, 3, 4])
    np.testing.assert_allclose(grad[2], p - np.eye(4)[2], rtol=1e-14, atol=1e-16)
