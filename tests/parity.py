"""Element-by-element comparison of a softmax output with the fp64 reference,
with the tolerances the library states:

  fp32 output:  |y - p| <= 2e-6 p where p >= 1e-30; 0 <= y <= 2e-30 below that;
                |1 - sum_j y_j| <= 1e-5 (summed in fp64) on every normal row.
  fp16 / bf16:  the output's bit pattern is within 1 of the correctly rounded
                fp64 result's (covers subnormals and binade edges).
  everywhere:   masked lanes, and valid lanes whose reference probability is
                exactly 0 (a -inf lane, every lane of an all -inf row, an
                exponential below the fp64 range), are +0 bit for bit; no
                output is -0; rows the policy makes NaN are NaN in every
                valid lane.

The error budget behind the fp32 bar, from the primitives' errors measured on
the GB300 (tests/test_math_error.py, against fp64):
  ex2.approx.ftz.f32            max relative error 1.44e-7 (2^-22.7) on [-126, 0)
  compensated e^(x - m)         1.80e-7 (2^-22.4) for x - m in [-87, 0]
  refined reciprocal 1/D        5.96e-8 (2^-24.0) on [1, 2^20)
  fast statistics-path term     2.06e-7 near the maximum, 3.85e-6 (2^-18) at
                                x - m = -87 (terms that small move d by less
                                than 2^-100 of its value)
An fp32 output e * (1/D) carries the exponential's 1.8e-7, the reciprocal's
6e-8, one product rounding 6e-8 and D's relative error (a sum of terms each
within 1.8e-7 plus about log2(cols) roundings of 6e-8: under 1.5e-6 for rows
of 2^20): well inside 2e-6.  The log-space, backward and cross-entropy bounds
below build on the same figures.
"""
import numpy as np

import oracle

F32_REL = 2e-6
F32_TINY = 1e-30
SUM_TOL = 1e-5


def lengths(rows, cols, valid_len):
    if valid_len is None:
        return np.full(rows, cols, dtype=np.int64)
    return np.clip(np.asarray(valid_len, dtype=np.int64), 0, cols)


def compare(y, p, out_dtype, valid_len=None, rows_sel=None):
    """y: output as stored (float32 array, or uint16 bits); p: fp64 reference [n, cols].

    Returns a dict of error statistics; raises AssertionError on any violation.
    """
    n, cols = p.shape
    L = lengths(n, cols, None if valid_len is None else
                (np.asarray(valid_len)[rows_sel] if rows_sel is not None else valid_len))
    j = np.arange(cols)[None, :]
    masked = j >= L[:, None]
    nan_rows = np.isnan(p).any(axis=1)
    stats = {}
    zero_lanes = ~nan_rows[:, None] & ~masked & (p == 0)
    if out_dtype == "f32":
        y = np.asarray(y, dtype=np.float32).reshape(n, cols)
        bits = y.view(np.uint32)
        assert np.all(bits[masked] == 0), "masked lanes must be +0"
        assert np.all(bits[zero_lanes] == 0), "lanes of probability 0 must be +0"
        yv = y.astype(np.float64)
        pv = p
        nn = ~nan_rows[:, None] & ~masked
        assert np.all(bits[nn] >> 31 == 0), "outputs must be non-negative (no -0)"
        assert np.all(np.isnan(yv[nan_rows[:, None] & ~masked])), "NaN rows must be NaN"
        big = nn & (pv >= F32_TINY)
        small = nn & (pv < F32_TINY)
        rel = np.abs(yv[big] - pv[big]) / pv[big] if big.any() else np.zeros(1)
        stats["max_rel"] = float(rel.max())
        assert stats["max_rel"] <= F32_REL, f"max relative error {stats['max_rel']:.3e}"
        assert np.all((yv[small] >= 0) & (yv[small] <= 2 * F32_TINY)), "tiny outputs out of range"
        normal = ~nan_rows & (p.sum(axis=1) > 0)
        if normal.any():
            s = np.where(masked, 0.0, yv)[normal].sum(axis=1)
            stats["max_sum_err"] = float(np.abs(s - 1.0).max())
            assert stats["max_sum_err"] <= SUM_TOL, f"row sum error {stats['max_sum_err']:.3e}"
    else:
        yb = np.asarray(y).view(np.uint16).reshape(n, cols).astype(np.int64)
        assert np.all(yb[masked] == 0), "masked lanes must be +0"
        assert np.all(yb[zero_lanes] == 0), "lanes of probability 0 must be +0"
        exp_all = 0x7C00 if out_dtype == "f16" else 0x7F80
        isnan = ((yb & exp_all) == exp_all) & ((yb & ~exp_all & 0x7FFF) != 0)
        nv = nan_rows[:, None] & ~masked
        assert np.all(isnan[nv]), "NaN rows must be NaN"
        ok = ~nan_rows[:, None] & ~masked
        r = oracle.round_to(np.where(ok, p, 0.0), out_dtype).astype(np.int64)
        assert np.all(yb[ok] >> 15 == 0), "outputs must be non-negative"
        diff = np.abs(yb - r)[ok]
        stats["max_ulp"] = int(diff.max()) if diff.size else 0
        stats["frac_exact"] = float((diff == 0).mean()) if diff.size else 1.0
        assert stats["max_ulp"] <= 1, f"max ulp difference {stats['max_ulp']}"
    return stats


# ---------------------------------------------------------------------------
# Log-space outputs.  The kernels form log_softmax as (x - m) - log d in fp32
# with d the fp32 sum: each subtraction rounds once (relative 2^-24 of |x - m|
# <= |y| + log d, and of |y|), log d comes from the correctly rounded-to-1-ulp
# logf of a sum whose relative error is at most 2^-18 (64 roundings or
# approximations of 2^-24 each along the summation tree and the exponentials),
# and an error e in d moves log d by e.  So
#     |y - ref| <= 2^-22 (|ref| + log d) + 2^-18
# for fp32 outputs, plus one unit of the format's spacing at |ref| for fp16 and
# bf16 outputs.  LSE = m + log d: |lse - ref| <= 2^-23 |ref| + 2^-22 log d + 2^-18.
# Masked lanes and the lanes of empty / all -inf rows are -inf bit for bit.
# ---------------------------------------------------------------------------
LOG_ABS = 2.0 ** -18
NEG_INF_BITS = {"f32": 0xFF800000, "f16": 0xFC00, "bf16": 0xFF80}
# magnitudes that round to infinity: the largest finite value plus half its spacing
OVERFLOW = {"f32": 2.0**128 - 2.0**103, "f16": 65520.0, "bf16": 2.0**128 - 2.0**119}


def format_spacing(v, fmt):
    """Spacing of the fp16 / bf16 grid at |v| (subnormal spacing at the bottom)."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 1e-300)))
    if fmt == "bf16":
        return 2.0 ** np.maximum(e - 7, -133)
    return 2.0 ** np.maximum(e - 10, -24)


def _decoded(y, out_dtype, n, cols):
    if out_dtype == "f32":
        y = np.asarray(y, dtype=np.float32).reshape(n, cols)
        return y.astype(np.float64), y.view(np.uint32).astype(np.int64)
    bits = np.asarray(y).view(np.uint16).reshape(n, cols)
    return oracle.decode(bits, out_dtype), bits.astype(np.int64)


def compare_log(y, ref, log_d, out_dtype, valid_len=None, rows_sel=None):
    """y: stored log_softmax output; ref: fp64 reference [n, cols]; log_d: fp64 [n]."""
    n, cols = ref.shape
    L = lengths(n, cols, None if valid_len is None else
                (np.asarray(valid_len)[rows_sel] if rows_sel is not None else valid_len))
    masked = np.arange(cols)[None, :] >= L[:, None]
    yv, bits = _decoded(y, out_dtype, n, cols)
    ninf = NEG_INF_BITS[out_dtype]
    assert np.all(bits[masked] == ninf), "masked lanes must be -inf"
    nan_rows = np.isnan(ref).any(axis=1)
    assert np.all(np.isnan(yv[nan_rows[:, None] & ~masked])), "NaN rows must be NaN"
    # probability 0, or a log-probability beyond the format's range (rounds to -inf)
    inf_lanes = ~nan_rows[:, None] & ~masked & (ref <= -OVERFLOW[out_dtype])
    assert np.all(bits[inf_lanes] == ninf), "lanes of probability 0 must be -inf"
    ok = ~nan_rows[:, None] & ~masked & np.isfinite(ref) & (ref > -OVERFLOW[out_dtype])
    ld = np.broadcast_to(np.asarray(log_d, dtype=np.float64)[:, None], ref.shape)
    tol = 2.0 ** -22 * (np.abs(ref) + ld) + LOG_ABS
    if out_dtype != "f32":
        tol = tol + format_spacing(ref, out_dtype)
    err = np.abs(yv[ok] - ref[ok])
    worst = float((err / tol[ok]).max()) if ok.any() else 0.0
    assert worst <= 1.0, f"log_softmax error {worst:.3f} x tolerance"
    return {"max_err_over_tol": worst, "max_abs": float(err.max()) if ok.any() else 0.0}


def compare_lse(lse, ref, log_d):
    lse = np.asarray(lse, dtype=np.float64)
    assert np.array_equal(np.isnan(lse), np.isnan(ref)), "NaN rows"
    assert np.array_equal(np.isneginf(lse), np.isneginf(ref)), "empty rows are -inf"
    ok = np.isfinite(ref)
    tol = 2.0 ** -23 * np.abs(ref[ok]) + 2.0 ** -22 * np.asarray(log_d)[ok] + LOG_ABS
    err = np.abs(lse[ok] - ref[ok])
    worst = float((err / tol).max()) if ok.any() else 0.0
    assert worst <= 1.0, f"LSE error {worst:.3f} x tolerance"
    return {"lse_err_over_tol": worst}


# ---------------------------------------------------------------------------
# Softmax backward: s = sum g p is an fp32 sum of FMAs whose error is at most
# 2^-18 of sum |g p| (as for d above); dx = RN(p RN(g - s)) adds a relative
# 2^-24 twice.  So |dx - ref| <= 2^-22 |ref| + |p| 2^-18 (|g| + sum |g p|), plus
# one unit of the format's spacing at |ref| for fp16 / bf16 outputs.
# Cross-entropy: loss = RN(RN(m - x_t) + log d) with m - x_t <= loss, so
# |loss - ref| <= 2^-22 (|ref| + log d) + 2^-18; the gradient p - onehot carries
# p's error, at most 2e-6 from the exponential and 2^-18 from d, relative to p:
# |grad - ref| <= 6e-6 p + 2^-24 (+ the format's spacing), p = ref + onehot.
# Masked lanes and ignored rows are +0 bit for bit.
# ---------------------------------------------------------------------------
def _check_zero_and_nan(bits, yv, masked, nan_lanes, zero_rows=None):
    zl = masked if zero_rows is None else (masked | zero_rows[:, None])
    assert np.all(bits[zl] == 0), "masked lanes / ignored rows must be +0"
    assert np.all(np.isnan(yv[nan_lanes])), "NaN lanes"


def compare_backward(dx, ref, p_vals, g_vals, out_dtype, valid_len=None):
    n, cols = ref.shape
    L = lengths(n, cols, valid_len)
    masked = np.arange(cols)[None, :] >= L[:, None]
    yv, bits = _decoded(dx, out_dtype, n, cols)
    nan_lanes = np.isnan(ref) & ~masked
    _check_zero_and_nan(bits, yv, masked, nan_lanes)
    ok = ~masked & ~np.isnan(ref)
    gp = np.where(masked, 0.0, np.abs(g_vals * p_vals)).sum(axis=1)[:, None]
    tol = 2.0 ** -22 * np.abs(ref) + np.abs(p_vals) * 2.0 ** -18 * (np.abs(g_vals) + gp)
    if out_dtype != "f32":
        tol = tol + format_spacing(ref, out_dtype)
    tol = tol + 1e-38  # exact zeros compare equal
    err = np.abs(yv[ok] - ref[ok])
    worst = float((err / tol[ok]).max()) if ok.any() else 0.0
    assert worst <= 1.0, f"backward error {worst:.3f} x tolerance"
    return {"bwd_err_over_tol": worst}


def compare_ce(loss, grad, ref_loss, ref_grad, log_d, target, out_dtype, valid_len=None):
    n = ref_loss.shape[0]
    loss = np.asarray(loss, dtype=np.float64)
    assert np.array_equal(np.isnan(loss), np.isnan(ref_loss)), "NaN losses"
    ok = ~np.isnan(ref_loss)
    assert np.all(np.isfinite(loss[ok]) == np.isfinite(ref_loss[ok]))
    fin = ok & np.isfinite(ref_loss)
    tol = 2.0 ** -22 * (np.abs(ref_loss[fin]) + np.asarray(log_d)[fin]) + LOG_ABS
    err = np.abs(loss[fin] - ref_loss[fin])
    stats = {"loss_err_over_tol": float((err / tol).max()) if fin.any() else 0.0}
    assert stats["loss_err_over_tol"] <= 1.0, f"loss error {stats['loss_err_over_tol']:.3f} x tol"
    if grad is None:
        return stats
    cols = ref_grad.shape[1]
    L = lengths(n, cols, valid_len)
    masked = np.arange(cols)[None, :] >= L[:, None]
    t = np.asarray(target, dtype=np.int64)
    ignored = (t < 0) | (t >= L)
    yv, bits = _decoded(grad, out_dtype, n, cols)
    nan_lanes = np.isnan(ref_grad) & ~masked
    _check_zero_and_nan(bits, yv, masked, nan_lanes, ignored)
    onehot = (np.arange(cols)[None, :] == t[:, None]) & ~ignored[:, None]
    pv = np.where(onehot, ref_grad + 1.0, ref_grad)
    gok = ~masked & ~ignored[:, None] & ~np.isnan(ref_grad)
    tol = 6e-6 * np.abs(pv) + 2.0 ** -24
    if out_dtype != "f32":
        tol = tol + format_spacing(ref_grad, out_dtype)
    err = np.abs(yv[gok] - ref_grad[gok])
    stats["grad_err_over_tol"] = float((err / tol[gok]).max()) if gok.any() else 0.0
    assert stats["grad_err_over_tol"] <= 1.0, f"grad error {stats['grad_err_over_tol']:.3f} x tol"
    return stats
