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
