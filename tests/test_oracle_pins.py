"""Pins for the fp64 CPU reference: values the pages print, closed forms,
invariants, library routines and brute force.  None of these re-types the
reference's own formula: each checks it against something independent of it,
and the negative controls show that the checks fail a plausible mistake.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                     "pages_worked_values.json")))


def f32(v):
    return np.asarray(v, dtype=np.float32)


def soft(row, dtype="f32", valid_len=None):
    a = f32(row) if dtype == "f32" else np.asarray(row)
    return oracle.softmax_rows(a, dtype, 1, a.size,
                               None if valid_len is None else [valid_len])[0]


def stats(row):
    m, d = oracle.row_stats(f32(row), "f32", 1, len(row))
    return m[0], d[0]


# ---------------------------------------------------------------------------
# Values the pages print.
# ---------------------------------------------------------------------------

def test_fp16_worked_example_stable():
    """'A worked example: naive fp16 versus the stable form': x = [20, 18, 17, -5]
    gives p = [0.84380, 0.11420, 0.04201, ~0], sum of shifted exps 1.185122, and
    the fourth term's true value 1.17e-11."""
    g = GOLDEN["fp16_example"]
    p = soft(g["x"])
    # printed values agree to within one unit of their last printed digit
    # (the page's 0.84380 is 0.8437947...)
    assert np.all(np.abs(p[:3] - g["p_printed"]) <= 1e-5)
    assert abs(p[3] - g["p4_true_printed"]) < 0.005e-11
    m, d = stats(g["x"])
    assert m == 20.0 and round(d, 6) == g["sum_printed"]
    assert abs(math.exp(-25.0) - g["exp4_printed_before_underflow"]) < 0.0005e-11


def test_fp16_worked_example_in_fp16_arithmetic():
    """The same example evaluated in fp16: shifted [0,-2,-3,-25], exps
    [1, 0.13534, 0.049787, 0] to fp16 precision (the fourth underflows)."""
    g = GOLDEN["fp16_example"]
    sh, e, p, s = oracle.stable_softmax_f16(g["x"])
    assert sh.tolist() == g["shifted"]
    u16 = 2.0 ** -11
    assert abs(u16 - GOLDEN["unit_roundoff_printed"]["fp16"]) < 0.05e-4
    for got, want in zip(e[:3], g["exp_printed"]):
        assert abs(got - want) <= 2 * u16 * want
    assert e[3] == 0.0
    assert abs(s - g["sum_printed"]) <= 2 * u16 * g["sum_printed"]
    assert np.all(np.isfinite(p))


def test_naive_fp16_negative_control_overflows():
    """Negative control: the unshifted softmax in fp16 overflows (exp(20) > 65504)
    and inf/inf gives NaN for the large terms, as the page shows."""
    p = oracle.naive_softmax_f16([20.0, 18.0, 17.0, -5.0])
    assert np.all(np.isnan(p[:3]))
    # The checks used on the product outputs reject it.
    ref = soft([20.0, 18.0, 17.0, -5.0])
    assert not np.allclose(p, ref, rtol=1e-3, equal_nan=False)


def test_large_logits_stay_finite():
    """'Online stable softmax': [1000, 999, 997] is computed from exp(0), exp(-1),
    exp(-3); closed form 1 / (1 + e^-1 + e^-3) for the first entry."""
    g = GOLDEN["large_logits"]
    p = soft(g["x"])
    assert np.all(np.isfinite(p))
    assert p.tolist() == soft(g["shifted"]).tolist()
    z = 1.0 + math.exp(-1.0) + math.exp(-3.0)
    want = [1.0 / z, math.exp(-1.0) / z, math.exp(-3.0) / z]
    assert np.allclose(p, want, rtol=1e-15, atol=0)
    assert np.round(p, 6).tolist() == [0.705385, 0.259496, 0.035119]


@pytest.mark.parametrize("case", GOLDEN["two_logit"]["cases"])
def test_two_logit_family(case):
    """'Stable softmax...' network lab: [0, z] gives p = sigma(z); sigma(0.5) ~ 0.622
    (x=1, w=1) and sigma(2.5) ~ 0.924 (x=1, w=3).  The complement is the zero logit."""
    z, printed = case["w"] * case["x"] - 0.5, case["p_printed"]
    p = soft([0.0, z])
    sigma = 1.0 / (1.0 + math.exp(-z))
    assert abs(p[1] - sigma) < 1e-15
    assert abs(p[0] - (1.0 - sigma)) < 1e-15
    assert round(p[1], 3) == printed


def test_merge_worked_example():
    """'Online stable softmax', worked merge: (10, 1.8) and (12, 1.3) combine to
    maximum 12 and sum 1.8 e^-2 + 1.3 ~ 0.244 + 1.3 = 1.544, not 3.1."""
    g = GOLDEN["merge_example"]
    (ma, da), (mb, db) = g["block_a"], g["block_b"]
    m, d = oracle.merge_stats(ma, da, mb, db)
    assert m[0] == g["m_printed"]
    assert round(da * math.exp(ma - mb), 3) == g["rescaled_a_printed"]
    assert round(d[0], 3) == g["d_printed"]
    assert da + db == g["direct_sum_printed"] and abs(d[0] - g["direct_sum_printed"]) > 1.0
    # m_b < m leaves the old sum unscaled; only the new block is scaled down.
    m2, d2 = oracle.merge_stats(12.0, 1.3, 10.0, 1.8)
    assert m2[0] == 12.0 and d2[0] == d[0]
    m3, d3 = oracle.merge_stats(12.0, 1.3, 12.0 - 1e9, 1.8)
    assert d3[0] == 1.3


def test_tile_trace_three_pass_vs_online():
    """'Kernel visualization: online softmax': the row [3,1,4,2,8,5,7,6] in tiles
    of 4.  Tile 0 gives m = 4, d = e^-1 + e^-3 + 1 + e^-2; at tile 1 the max moves
    to 8 and one multiply by e^(4-8) corrects d; the final d equals the three-pass
    denominator against m = 8."""
    x, B = GOLDEN["tile_row"]["x"], GOLDEN["tile_row"]["B"]
    m, corrected, d = oracle.online_tiled(x, B)
    d0 = math.exp(-1) + math.exp(-3) + 1 + math.exp(-2)
    assert m.tolist() == [4.0, 8.0]
    assert abs(d[0] - d0) < 1e-15 and round(d[0], 4) == 1.5530
    assert abs(corrected[1] - d0 * math.exp(-4)) < 1e-15 and round(corrected[1], 4) == 0.0284
    assert round(d[1], 4) == 1.5814
    m3, d3 = stats(x)
    assert m3 == 8.0 and abs(d3 - d[1]) < 1e-14
    p = soft(x)
    assert abs(p.max() - 1.0 / d3) < 1e-15 and round(p.max(), 6) == 0.632333


def test_element_trace_and_no_rescale_control():
    """'Online stable softmax' exercise: trace [1, 2, -3, 12, 11, 4] element by
    element.  The running (m, d) after each element is the three-pass statistic of
    that prefix (brute force); the variant that omits the rescale when 12 becomes
    the maximum is wrong (negative control)."""
    x = GOLDEN["element_trace_row"]["x"]
    m, d = oracle.online_elementwise(x)
    for i in range(len(x)):
        mi, di = stats(x[: i + 1])
        assert m[i] == mi
        assert abs(d[i] - di) <= 4 * (i + 1) * 2.0 ** -53 * di
    assert [round(v, 6) for v in d] == [1.0, 1.367879, 1.374617, 1.000062, 1.367942, 1.368277]
    m_bad, d_bad = oracle.online_elementwise(x, rescale=False)
    assert round(d_bad[-1], 6) == 3.374953
    assert abs(d_bad[-1] - d[-1]) > 1.0


# ---------------------------------------------------------------------------
# Invariants and closed forms.
# ---------------------------------------------------------------------------

def test_shift_invariance_bit_exact():
    """'The max-subtraction identity': softmax(x - c) = softmax(x).  With inputs
    on a 1/64 grid and an integer c every shifted value is exact, so the
    reference must give identical bits."""
    rng = np.random.default_rng(7)
    for _ in range(20):
        n = int(rng.integers(1, 300))
        x = (rng.integers(-2048, 2048, size=n) / 64.0).astype(np.float32)
        for c in (1.0, 1024.0, -4096.0):
            a = soft(x)
            b = soft((x + np.float32(c)).astype(np.float32))
            assert np.array_equal(a, b)


def test_normalisation_and_denominator_range():
    """Every p_i > 0 (unless underflowed), sum p = 1, and d lies in [1, L] because
    the argmax term contributes exactly 1 and every other term is at most 1."""
    rng = np.random.default_rng(8)
    for _ in range(50):
        n = int(rng.integers(1, 2000))
        scale = float(rng.choice([0.1, 3.0, 30.0]))
        x = (scale * rng.standard_normal(n)).astype(np.float32)
        p = soft(x)
        assert abs(p.sum() - 1.0) < 1e-13
        assert np.all(p >= 0)
        assert np.all(p[x > x.max() - 700] > 0)
        m, d = stats(x)
        assert m == x.max() and 1.0 <= d <= n


def test_matches_library_softmax_fp64():
    """Library routine: torch.softmax in fp64 on the same widened inputs."""
    rng = np.random.default_rng(9)
    for n in (1, 2, 7, 100, 1000, 4097):
        x = (10 * rng.standard_normal(n)).astype(np.float32)
        want = torch.softmax(torch.from_numpy(x).double(), dim=0).numpy()
        got = soft(x)
        assert np.allclose(got, want, rtol=1e-13, atol=1e-300)


def test_exercise_random_rows_with_large_logits():
    """'Online stable softmax' exercise: 1000 random rows with occasional logits in
    [50, 100].  The element-wise online recurrence's final (m, d) equals the
    three-pass statistics; the no-rescale variant's d does not."""
    rng = np.random.default_rng(10)
    wrong = 0
    for _ in range(1000):
        n = int(rng.integers(2, 64))
        x = rng.standard_normal(n)
        hot = rng.random(n) < 0.05
        x[hot] = rng.uniform(50, 100, size=hot.sum())
        x = x.astype(np.float32).astype(np.float64)
        m, d = oracle.online_elementwise(x)
        m3, d3 = stats(x)
        assert m[-1] == m3
        assert abs(d[-1] - d3) <= 4 * n * 2.0 ** -53 * d3
        _, d_bad = oracle.online_elementwise(x, rescale=False)
        if abs(d_bad[-1] - d3) > 1e-6 * d3:
            wrong += 1
    assert wrong > 100


def _compositions(n, max_parts):
    for k in range(1, max_parts + 1):
        for cuts in itertools.combinations(range(1, n), k - 1):
            yield [0, *cuts, n]


def _bracketings(leaves):
    """Every full binary bracketing of the sequence (Catalan many)."""
    if len(leaves) == 1:
        yield leaves[0]
        return
    for i in range(1, len(leaves)):
        for left in _bracketings(leaves[:i]):
            for right in _bracketings(leaves[i:]):
                yield ("merge", left, right)


def _eval_tree(node):
    if node[0] == "merge":
        a, b = _eval_tree(node[1]), _eval_tree(node[2])
        m, d = oracle.merge_stats(a[0], a[1], b[0], b[1])
        return float(m[0]), float(d[0])
    return node[1], node[2]


def test_merge_any_grouping_equals_three_pass():
    """'Stable softmax...' and 'Online stable softmax': block summaries merge
    associatively in real arithmetic.  Brute force: every split of a short row into
    up to 5 blocks and every bracketing of the merges gives the three-pass m
    exactly and d within 4 L u64."""
    rng = np.random.default_rng(11)
    count = 0
    for n in (1, 3, 6, 9):
        x = (5 * rng.standard_normal(n)).astype(np.float32)
        m3, d3 = stats(x)
        for cuts in _compositions(n, 5):
            leaves = []
            for a, b in zip(cuts[:-1], cuts[1:]):
                bm, bd = stats(x[a:b])
                leaves.append(("leaf", float(bm), float(bd)))
            for tree in _bracketings(leaves):
                m, d = _eval_tree(tree)
                assert m == m3
                assert abs(d - d3) <= 4 * n * 2.0 ** -53 * d3
                count += 1
    assert count > 1000


def test_merge_identity_and_masked_block():
    """The empty prefix (-inf, 0) is the identity of the merge, in either order,
    and merging it never evaluates -inf - (-inf)."""
    for m, d in [(3.0, 2.5), (-1e30, 1.0), (-math.inf, 0.0)]:
        a = oracle.merge_stats(-math.inf, 0.0, m, d)
        b = oracle.merge_stats(m, d, -math.inf, 0.0)
        assert (a[0][0], a[1][0]) == (m, d) == (b[0][0], b[1][0])


# ---------------------------------------------------------------------------
# The declared policy for masks, empty rows, -inf, +inf and NaN.
# ---------------------------------------------------------------------------

def test_policy_masks_and_empty_rows():
    x = f32([3.0, 1.0, 2.0, 100.0, np.nan])
    # valid prefix 3: masked lanes (even a huge value or a NaN there) do not count
    p = soft(x, valid_len=3)
    want = soft(x[:3])
    assert np.array_equal(p[:3], want) and np.all(p[3:] == 0)
    assert not np.any(np.signbit(p[3:]))
    # length 0, negative length (clamped to 0), and beyond cols (clamped to cols)
    for L, expect_zero in [(0, True), (-5, True)]:
        q = soft(x, valid_len=L)
        assert np.all(q == 0) and not np.any(np.signbit(q))
    y = f32([1.0, 2.0])
    assert np.array_equal(soft(y, valid_len=99), soft(y))
    m, d = oracle.row_stats(x, "f32", 1, 5, [0])
    assert m[0] == -math.inf and d[0] == 0.0


def test_policy_single_valid_element():
    p = soft(f32([-7.5, 9.0, 9.0]), valid_len=1)
    assert p.tolist() == [1.0, 0.0, 0.0]


def test_policy_negative_infinity():
    ninf = -np.inf
    p = soft(f32([ninf, 0.0, ninf, 0.0]))
    assert p.tolist() == [0.0, 0.5, 0.0, 0.5]
    q = soft(f32([ninf, ninf, ninf]))
    assert np.all(q == 0) and not np.any(np.signbit(q))
    m, d = stats([ninf, ninf])
    assert m == -math.inf and d == 0.0


def test_policy_nan_and_positive_infinity():
    p = soft(f32([1.0, np.nan, 2.0, 3.0]), valid_len=3)
    assert np.all(np.isnan(p[:3])) and p[3] == 0.0
    m, d = stats([1.0, np.nan])
    assert math.isnan(m) and math.isnan(d)
    q = soft(f32([1.0, np.inf, -np.inf, 2.0]))
    assert np.all(np.isnan(q))
    m, d = stats([1.0, np.inf])
    assert m == math.inf and math.isnan(d)
    # the merge agrees with the statistics of the concatenation
    for a, b in [([1.0, np.inf], [5.0]), ([np.nan], [2.0]), ([1.0], [np.inf, 3.0])]:
        ma, da = stats(a)
        mb, db = stats(b)
        mm, dm = oracle.merge_stats(ma, da, mb, db)
        mc, dc = stats(a + b)
        assert (math.isnan(mm[0]) and math.isnan(mc)) or mm[0] == mc
        assert math.isnan(dm[0]) and math.isnan(dc)
    # torch.softmax in fp64 gives NaN for the same rows (library reference behaviour)
    t = torch.softmax(torch.tensor([1.0, math.inf, -math.inf, 2.0], dtype=torch.float64), 0)
    assert torch.isnan(t).all()


def test_reference_inputs_of_all_storage_types():
    """The reference widens fp16/bf16 inputs exactly; the same values stored in
    each type give the same probabilities."""
    vals = f32([0.5, -2.0, 3.25, 8.0, -30.0])
    bits16 = vals.astype(np.float16).view(np.uint16)
    bitsbf = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    a = soft(vals)
    b = oracle.softmax_rows(bits16, "f16", 1, 5)[0]
    c = oracle.softmax_rows(bitsbf, "bf16", 1, 5)[0]
    assert np.array_equal(a, b) and np.array_equal(a, c)
