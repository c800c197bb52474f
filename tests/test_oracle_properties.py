"""Invariants of the oracle on random rows (hypothesis), beyond the pinned
worked values: what the mathematics of the max-shifted softmax fixes for any
input, so that a mistake in an index, a sign or a dropped term fails one of
them.

  permutation   softmax(x[perm]) = softmax(x)[perm] (the sum's rounding aside)
  monotonicity  x_i >= x_j  =>  p_i >= p_j
  masking       a valid prefix L gives the softmax of x[:L] followed by +0
  merge         the summaries of any two pieces of a row merge into the row's
                summary (m bit-equal, d within the sums' rounding)
  log space     log_softmax = log(softmax) where p is not subnormal, and
                LSE = m + log d
  backward      sum_j dx_j = 0, and a constant upstream gradient gives dx = 0
  cross-entropy loss = -log p_t >= 0; the gradient sums to 0, p_t - 1 at t
  attention     the keys (with their values) in any order give the same o and
                LSE; o lies in the box of the value rows; o is linear in V; the
                causal last query sees every key
"""
import math

import numpy as np
import pytest

import oracle
from numerically_stable_online_gb300 import workloads as wl

hyp = pytest.importorskip("hypothesis")
st = pytest.importorskip("hypothesis.strategies")
from hypothesis import given, settings  # noqa: E402

U = 2.0 ** -53
rows_f32 = st.lists(st.floats(min_value=-120.0, max_value=120.0, width=32, allow_nan=False),
                    min_size=1, max_size=64)
SETTINGS = settings(max_examples=60, deadline=None)


@pytest.fixture(scope="module", autouse=True)
def built():
    oracle.build()


def sm(row):
    x = np.asarray(row, np.float32)
    return oracle.softmax_rows(wl.to_storage(x, "f32"), "f32", 1, x.size)[0]


def stats(row):
    x = np.asarray(row, np.float32)
    m, d = oracle.row_stats(wl.to_storage(x, "f32"), "f32", 1, x.size)
    return m[0], d[0]


@SETTINGS
@given(rows_f32, st.randoms(use_true_random=False))
def test_permutation_equivariance(row, rnd):
    perm = list(range(len(row)))
    rnd.shuffle(perm)
    p = sm(row)
    q = sm([row[i] for i in perm])
    tol = 4 * len(row) * U * np.abs(p[perm]) + 1e-300
    assert np.all(np.abs(q - p[perm]) <= tol)


@SETTINGS
@given(rows_f32)
def test_monotone_in_the_logits(row):
    x = np.asarray(row, np.float32).astype(np.float64)
    p = sm(row)
    order = np.argsort(x, kind="stable")
    assert np.all(np.diff(p[order]) >= 0)
    assert abs(p.sum() - 1.0) <= 4 * len(row) * U


@SETTINGS
@given(rows_f32, st.integers(min_value=0, max_value=64))
def test_valid_prefix_is_truncation(row, L):
    x = np.asarray(row, np.float32)
    Lc = min(L, x.size)
    p = oracle.softmax_rows(wl.to_storage(x, "f32"), "f32", 1, x.size, [L])[0]
    assert np.all(p[Lc:] == 0) and not np.signbit(p[Lc:]).any()
    if Lc:
        assert np.array_equal(p[:Lc], sm(row[:Lc]))


@SETTINGS
@given(rows_f32, st.integers(min_value=0, max_value=64))
def test_merge_of_two_pieces(row, cut):
    cut = min(cut, len(row))
    m, d = stats(row)
    a = stats(row[:cut]) if cut else (-math.inf, 0.0)
    b = stats(row[cut:]) if cut < len(row) else (-math.inf, 0.0)
    mm, dd = oracle.merge_stats([a[0]], [a[1]], [b[0]], [b[1]])
    assert mm[0] == m
    assert abs(dd[0] - d) <= 4 * len(row) * U * d
    assert 1.0 <= d <= len(row) * (1 + 4 * len(row) * U)


@SETTINGS
@given(rows_f32)
def test_log_space_matches_log_of_softmax(row):
    x = np.asarray(row, np.float32)
    y, lse = oracle.log_softmax_rows(wl.to_storage(x, "f32"), "f32", 1, x.size)
    p = sm(row)
    m, d = stats(row)
    assert abs(lse[0] - (m + math.log(d))) <= 4 * U * (abs(m) + math.log(d)) + 1e-300
    ok = p > 1e-300
    assert np.all(np.abs(y[0][ok] - np.log(p[ok])) <= 1e-12 * (1 + np.abs(y[0][ok])))


# ------------------------------------------------------------------ gradients

@SETTINGS
@given(rows_f32, st.floats(min_value=-4.0, max_value=4.0, width=32), st.randoms(use_true_random=False))
def test_backward_sums_to_zero_and_ignores_constant_gradients(row, c, rnd):
    n = len(row)
    p = sm(row).astype(np.float32)
    g = np.asarray([rnd.uniform(-2, 2) for _ in range(n)], np.float32)
    ps, gs = wl.to_storage(p, "f32"), wl.to_storage(g, "f32")
    dx = oracle.softmax_backward(ps, gs, "f32", 1, n)[0]
    pv = p.astype(np.float64)
    # sum_j p_j (g_j - s) = s (1 - sum p): zero up to the stored p's rounding
    assert abs(dx.sum()) <= (abs(1 - pv.sum()) + 4 * n * U) * (np.abs(g).max() * 2 + 1)
    dc = oracle.softmax_backward(ps, wl.to_storage(np.full(n, c, np.float32), "f32"), "f32", 1, n)[0]
    assert np.all(np.abs(dc) <= abs(c) * (abs(1 - pv.sum()) + 4 * n * U) * pv + 1e-300)


@SETTINGS
@given(rows_f32, st.integers(min_value=0, max_value=63))
def test_cross_entropy_is_minus_log_p_and_its_gradient_sums_to_zero(row, t):
    n = len(row)
    t = min(t, n - 1)
    x = np.asarray(row, np.float32)
    loss, grad = oracle.cross_entropy(wl.to_storage(x, "f32"), "f32", 1, n, [t])
    p = sm(row)
    assert loss[0] >= 0.0
    if p[t] > 1e-300:
        assert abs(loss[0] + math.log(p[t])) <= 1e-12 * (1 + loss[0])
    assert abs(grad[0].sum()) <= 8 * n * U
    assert abs(grad[0][t] - (p[t] - 1.0)) <= 4 * n * U


# ------------------------------------------------------------------ attention

def att(q, k, v, causal=False, scale=0.25):
    h, sq, d = q.shape
    sk = k.shape[1]
    qs, ks, vs = (wl.to_storage(a.astype(np.float32).reshape(-1), "f32") for a in (q, k, v))
    return oracle.attention_rows(qs, ks, vs, "f32", h, sq, sk, d, scale, causal)[:2]


@settings(max_examples=30, deadline=None)
@given(st.integers(min_value=1, max_value=6), st.integers(min_value=1, max_value=9),
       st.integers(min_value=0, max_value=2 ** 31 - 1))
def test_attention_key_order_convexity_and_linearity(sq, sk, seed):
    rng = np.random.default_rng(seed)
    d = 4
    q = rng.normal(0, 2, (1, sq, d))
    k = rng.normal(0, 2, (1, sk, d))
    v = rng.normal(0, 1, (1, sk, d))
    o, lse = att(q, k, v)
    # the keys (with their values) in any order
    perm = rng.permutation(sk)
    o2, lse2 = att(q, k[:, perm], v[:, perm])
    assert np.allclose(o2, o, rtol=0, atol=1e-12) and np.allclose(lse2, lse, rtol=0, atol=1e-12)
    # each output is a convex combination of the value rows
    vv = v[0].astype(np.float32).astype(np.float64)
    assert np.all(o >= vv.min(axis=0) - 1e-12) and np.all(o <= vv.max(axis=0) + 1e-12)
    # linear in V (exact powers of two keep the stored values exact)
    o4, _ = att(q, k, 4.0 * v.astype(np.float32))
    assert np.allclose(o4, 4.0 * o, rtol=1e-12, atol=1e-12)
    # causal: query i sees keys j <= i + sk - sq; the last query sees every key
    oc, _ = att(q, k, v, causal=True)
    assert np.allclose(oc[sq - 1], o[sq - 1], rtol=0, atol=1e-12)
