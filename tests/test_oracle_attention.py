"""Pins of the oracle's attention numerator ("Online stable softmax", sections
"Carry a weighted value numerator for attention" and "Reference summary";
"Softmax numerics architecture...", "From online softmax to tiled attention").

The direct oracle (per-row loops in C) is checked against: the matrix form
evaluated with numpy/scipy library routines on tiny inputs; closed forms
(constant values, one valid key, all-equal scores, the causal first row, the
empty row); LSE by brute force without the shift; and the pages' (m, l, o)
recurrence over key blocks of every size, with the pages' named error (the
numerator not rescaled) as a negative control.
"""
import math

import numpy as np
import pytest
import scipy.special

import oracle


def f32(a):
    return np.asarray(a, dtype=np.float32)


def rand(shape, seed, scale=1.0):
    return f32(np.random.default_rng(seed).normal(0, scale, shape))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("sq,sk", [(5, 5), (3, 7), (7, 4)])
def test_attention_matches_matrix_form(causal, sq, sk):
    H, D, scale = 3, 8, 0.35
    q, k, v = rand((H, sq, D), 1), rand((H, sk, D), 2), rand((H, sk, D), 3)
    o, lse, oabs, smax = oracle.attention_rows(q, k, v, "f32", H, sq, sk, D, scale, causal)
    for h in range(H):
        s = scale * q[h].astype(np.float64) @ k[h].astype(np.float64).T
        if causal:
            mask = np.arange(sk)[None, :] > np.arange(sq)[:, None] + (sk - sq)
            s = np.where(mask, -np.inf, s)
        for i in range(sq):
            n = h * sq + i
            if np.all(np.isneginf(s[i])):  # no valid key: the empty row
                assert np.all(o[n] == 0.0) and lse[n] == -np.inf
                continue
            p = scipy.special.softmax(s[i])
            np.testing.assert_allclose(o[n], p @ v[h].astype(np.float64), rtol=1e-12, atol=1e-14)
            assert lse[n] == pytest.approx(scipy.special.logsumexp(s[i]), rel=1e-13)
            np.testing.assert_allclose(oabs[n], p @ np.abs(v[h].astype(np.float64)), rtol=1e-12)


def test_attention_closed_forms():
    H, S, D = 1, 6, 4
    q, k = rand((H, S, D), 4), rand((H, S, D), 5)
    c = f32([0.5, -2.0, 3.25, 1.0])
    v = np.tile(c, (H, S, 1))
    o, _, _, _ = oracle.attention_rows(q, k, v, "f32", H, S, S, D, 0.7)
    np.testing.assert_allclose(o, np.tile(c, (S, 1)), rtol=1e-14)  # a convex combination of equal rows
    v = rand((H, S, D), 6)
    o, lse, _, _ = oracle.attention_rows(q, k, v, "f32", H, S, S, D, 0.7, causal=True)
    np.testing.assert_array_equal(o[0], v[0, 0].astype(np.float64))  # the first row sees one key
    assert lse[0] == pytest.approx(0.7 * float(np.dot(q[0, 0].astype(np.float64), k[0, 0])), rel=1e-14)
    kz = np.zeros((H, S, D), np.float32)
    o, lse, _, _ = oracle.attention_rows(q, kz, v, "f32", H, S, S, D, 0.7)
    np.testing.assert_allclose(o, np.tile(v[0].astype(np.float64).mean(axis=0), (S, 1)), rtol=1e-13)
    np.testing.assert_allclose(lse, math.log(S), rtol=1e-15)  # equal scores 0: log of the count


def test_attention_lse_brute_force_and_empty_rows():
    H, sq, sk, D = 2, 4, 9, 5
    q, k, v = rand((H, sq, D), 7), rand((H, sk, D), 8), rand((H, sk, D), 9)
    _, lse, _, _ = oracle.attention_rows(q, k, v, "f32", H, sq, sk, D, 0.3)
    for h in range(H):
        for i in range(sq):
            s = [0.3 * float(np.dot(q[h, i].astype(np.float64), k[h, j].astype(np.float64))) for j in range(sk)]
            assert lse[h * sq + i] == pytest.approx(math.log(math.fsum(math.exp(x) for x in s)), rel=1e-13)
    # causal with more queries than keys: the first sq - sk rows have no key
    o, lse, _, _ = oracle.attention_rows(k, q, q, "f32", H, sk, sq, D, 0.3, causal=True)
    empty = np.arange(sk) < sk - sq
    for h in range(H):
        assert np.all(lse[h * sk:(h + 1) * sk][empty] == -np.inf)
        assert np.all(o[h * sk:(h + 1) * sk][empty] == 0.0)


@pytest.mark.parametrize("block", [1, 2, 3, 5, 8, 64])
def test_running_state_over_blocks_equals_direct(block):
    # a rising score row: the maximum changes in many blocks
    n, D = 40, 6
    rng = np.random.default_rng(block)
    s = rng.normal(0, 2, n) + np.linspace(0, 12, n)
    v = rng.normal(0, 1, (n, D))
    o, m, l = oracle.attention_online(s, v, block)
    p = scipy.special.softmax(s)
    np.testing.assert_allclose(o, p @ v, rtol=1e-12, atol=1e-14)
    assert m == s.max() and l == pytest.approx(np.exp(s - s.max()).sum(), rel=1e-13)
    # the pages' named error: l rescaled, the numerator not
    o_bad, _, _ = oracle.attention_online(s, v, block, rescale_o=False)
    if block < n:
        assert np.max(np.abs(o_bad - p @ v)) > 1e-3
