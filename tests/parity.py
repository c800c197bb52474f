"""Element-by-element comparison of a softmax output with the fp64 reference,
with the tolerances the library states:

  fp32 output:  |y - p| <= 2e-6 p where p >= 1e-30; 0 <= y <= 2e-30 below that;
                |1 - sum_j y_j| <= 1e-5 (summed in fp64) on every normal row.
  fp16 / bf16:  the output's bit pattern is within 1 of the correctly rounded
                fp64 result's (covers subnormals and binade edges).
  everywhere:   masked lanes and empty / all -inf rows are +0 bit for bit; rows
                the policy makes NaN are NaN in every valid lane.
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
    if out_dtype == "f32":
        y = np.asarray(y, dtype=np.float32).reshape(n, cols)
        bits = y.view(np.uint32)
        assert np.all(bits[masked] == 0), "masked lanes must be +0"
        yv = y.astype(np.float64)
        pv = p
        nn = ~nan_rows[:, None] & ~masked
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
