"""Reference (oracle) for row-wise numerically stable softmax: fp64, plain C, CPU.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline legs of ``bench.py`` may import this package.  The product path
(``numerically_stable_online_gb300``) never imports it, and the two share no
code: this package compiles ``softmax_ref.c`` with the host C compiler and calls
it through ctypes.

The arithmetic is in ``softmax_ref.c``; each function there cites the page
section it follows.  This module only marshals numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

F32, F16, BF16 = 0, 1, 2
_DTYPE_CODE = {"f32": F32, "f16": F16, "bf16": BF16}
_ITEMSIZE = {F32: 4, F16: 2, BF16: 2}

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "softmax_ref.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile softmax_ref.c into oracle/_build/liboracle.so (plain -O2, no fast-math)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P, I64, I32, D = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double
        lib.orc_decode_f16.argtypes = [ctypes.c_uint16]
        lib.orc_decode_f16.restype = D
        lib.orc_decode_bf16.argtypes = [ctypes.c_uint16]
        lib.orc_decode_bf16.restype = D
        lib.orc_round_f16.argtypes = [D]
        lib.orc_round_f16.restype = ctypes.c_uint16
        lib.orc_round_bf16.argtypes = [D]
        lib.orc_round_bf16.restype = ctypes.c_uint16
        lib.orc_round_array.argtypes = [P, I64, I32, P]
        lib.orc_decode_array.argtypes = [P, I64, I32, P]
        lib.orc_softmax_rows.argtypes = [P, I32, I64, P, P, I64, P]
        lib.orc_row_stats.argtypes = [P, I32, I64, P, P, I64, P, P]
        lib.orc_merge_stats.argtypes = [P, P, P, P, P, P, I64]
        lib.orc_online_elementwise.argtypes = [P, I64, I32, P, P]
        lib.orc_online_tiled.argtypes = [P, I64, I64, P, P, P]
        lib.orc_naive_softmax_f16.argtypes = [P, I64, P]
        lib.orc_stable_softmax_f16.argtypes = [P, I64, P, P, P, P]
        lib.orc_log_softmax_rows.argtypes = [P, I32, I64, P, P, I64, P, P]
        lib.orc_apply_stats.argtypes = [P, I32, I64, P, P, P, P, I64, P]
        lib.orc_softmax_backward.argtypes = [P, P, I32, I64, P, P, I64, P]
        lib.orc_cross_entropy.argtypes = [P, I32, I64, P, P, P, I64, P, P]
        lib.orc_attention_rows.argtypes = [P, P, P, I32, I64, I64, I64, D, I32, P, I64, P, P, P, P]
        lib.orc_attention_online.argtypes = [P, P, I64, I64, I64, I32, P, P, P]
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _code(dtype) -> int:
    if isinstance(dtype, int):
        return dtype
    return _DTYPE_CODE[dtype]


def _as_storage(x, dtype):
    """x as a C-contiguous array of the storage type's raw bits (or float32)."""
    code = _code(dtype)
    a = np.ascontiguousarray(x)
    if code == F32:
        if a.dtype != np.float32:
            raise TypeError("f32 input must be a float32 array")
    else:
        if a.dtype == np.float16 and code == F16:
            a = a.view(np.uint16)
        if a.dtype != np.uint16:
            raise TypeError("f16/bf16 input must be given as uint16 bit patterns")
    return a, code


def _lengths(valid_len, rows):
    if valid_len is None:
        return None
    v = np.ascontiguousarray(valid_len, dtype=np.int32)
    if v.shape != (rows,):
        raise ValueError("valid_len must have one entry per row")
    return v


def softmax_rows(x, dtype, rows: int, cols: int, valid_len=None, rows_sel=None) -> np.ndarray:
    """fp64 softmax of rows of the [rows, cols] input (stored bits), per the declared policy.

    rows_sel: optional list of row indices; the result then has len(rows_sel) rows.
    """
    lib = _load()
    a, code = _as_storage(x, dtype)
    if a.size != rows * cols:
        raise ValueError("x has the wrong number of elements")
    vl = _lengths(valid_len, rows)
    sel = None if rows_sel is None else np.ascontiguousarray(rows_sel, dtype=np.int64)
    n_sel = rows if sel is None else sel.size
    p = np.empty((n_sel, cols), dtype=np.float64)
    lib.orc_softmax_rows(_ptr(a), code, cols, _ptr(vl), _ptr(sel), n_sel, _ptr(p))
    return p


def row_stats(x, dtype, rows: int, cols: int, valid_len=None, rows_sel=None):
    """fp64 (m, d) per row: m = max of the valid prefix, d = sum exp(x - m)."""
    lib = _load()
    a, code = _as_storage(x, dtype)
    if a.size != rows * cols:
        raise ValueError("x has the wrong number of elements")
    vl = _lengths(valid_len, rows)
    sel = None if rows_sel is None else np.ascontiguousarray(rows_sel, dtype=np.int64)
    n_sel = rows if sel is None else sel.size
    m = np.empty(n_sel, dtype=np.float64)
    d = np.empty(n_sel, dtype=np.float64)
    lib.orc_row_stats(_ptr(a), code, cols, _ptr(vl), _ptr(sel), n_sel, _ptr(m), _ptr(d))
    return m, d


def merge_stats(m_a, d_a, m_b, d_b):
    """fp64 merge of two arrays of block summaries (empty block = (-inf, 0))."""
    lib = _load()
    arrs = [np.ascontiguousarray(np.atleast_1d(v), dtype=np.float64) for v in (m_a, d_a, m_b, d_b)]
    n = arrs[0].size
    if any(v.size != n for v in arrs):
        raise ValueError("summary arrays differ in length")
    m = np.empty(n, dtype=np.float64)
    d = np.empty(n, dtype=np.float64)
    lib.orc_merge_stats(*[_ptr(v) for v in arrs], _ptr(m), _ptr(d), n)
    return m, d


def round_to(p, dtype) -> np.ndarray:
    """Round doubles to the storage type, ties to even, straight from fp64.

    Returns uint16 bit patterns for f16/bf16 and uint32 bit patterns for f32.
    """
    lib = _load()
    code = _code(dtype)
    v = np.ascontiguousarray(p, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint32 if code == F32 else np.uint16)
    lib.orc_round_array(_ptr(v), v.size, code, _ptr(out))
    return out


def decode(bits, dtype) -> np.ndarray:
    """Widen stored values (float32 array, or uint16 bits for f16/bf16) to fp64."""
    lib = _load()
    a, code = _as_storage(bits, dtype)
    out = np.empty(a.shape, dtype=np.float64)
    lib.orc_decode_array(_ptr(a), a.size, code, _ptr(out))
    return out


def online_elementwise(x, rescale: bool = True):
    """Per-element online recurrence; returns the (m_i, d_i) trace after each element."""
    lib = _load()
    v = np.ascontiguousarray(x, dtype=np.float64)
    m = np.empty(v.size)
    d = np.empty(v.size)
    lib.orc_online_elementwise(_ptr(v), v.size, 1 if rescale else 0, _ptr(m), _ptr(d))
    return m, d


def online_tiled(x, B: int):
    """Tiled online update; returns per tile (m, corrected old d, d)."""
    lib = _load()
    v = np.ascontiguousarray(x, dtype=np.float64)
    nt = (v.size + B - 1) // B
    m, c, d = np.empty(nt), np.empty(nt), np.empty(nt)
    lib.orc_online_tiled(_ptr(v), v.size, B, _ptr(m), _ptr(c), _ptr(d))
    return m, c, d


def naive_softmax_f16(x) -> np.ndarray:
    """The unshifted softmax evaluated in fp16 arithmetic (negative control)."""
    lib = _load()
    v = np.ascontiguousarray(x, dtype=np.float64)
    p = np.empty(v.size)
    lib.orc_naive_softmax_f16(_ptr(v), v.size, _ptr(p))
    return p


def stable_softmax_f16(x):
    """The max-shifted softmax evaluated in fp16 arithmetic: (shifted, exp, p, sum)."""
    lib = _load()
    v = np.ascontiguousarray(x, dtype=np.float64)
    sh, e, p = np.empty(v.size), np.empty(v.size), np.empty(v.size)
    s = np.empty(1)
    lib.orc_stable_softmax_f16(_ptr(v), v.size, _ptr(sh), _ptr(e), _ptr(p), _ptr(s))
    return sh, e, p, float(s[0])


def _rows_args(x, dtype, rows, cols, valid_len, rows_sel):
    a, code = _as_storage(x, dtype)
    if a.size != rows * cols:
        raise ValueError("x has the wrong number of elements")
    vl = _lengths(valid_len, rows)
    sel = None if rows_sel is None else np.ascontiguousarray(rows_sel, dtype=np.int64)
    n_sel = rows if sel is None else sel.size
    return a, code, vl, sel, n_sel


def log_softmax_rows(x, dtype, rows: int, cols: int, valid_len=None, rows_sel=None):
    """fp64 (log_softmax [n, cols], LSE [n]) of the selected rows.

    log_softmax_j = x_j - LSE over the valid prefix, -inf in masked lanes;
    LSE = m + log d (-inf for an empty row, NaN for a NaN or +inf row).
    """
    lib = _load()
    a, code, vl, sel, n_sel = _rows_args(x, dtype, rows, cols, valid_len, rows_sel)
    out = np.empty((n_sel, cols), dtype=np.float64)
    lse = np.empty(n_sel, dtype=np.float64)
    lib.orc_log_softmax_rows(_ptr(a), code, cols, _ptr(vl), _ptr(sel), n_sel, _ptr(out), _ptr(lse))
    return out, lse


def apply_stats(x, dtype, rows: int, cols: int, m, d, valid_len=None, rows_sel=None):
    """fp64 exp(x - m_r) / d_r over each valid prefix (+0 beyond), with given per-row (m, d)."""
    lib = _load()
    a, code, vl, sel, n_sel = _rows_args(x, dtype, rows, cols, valid_len, rows_sel)
    mm = np.ascontiguousarray(m, dtype=np.float64)
    dd = np.ascontiguousarray(d, dtype=np.float64)
    if mm.shape != (rows,) or dd.shape != (rows,):
        raise ValueError("m and d must have one entry per row")
    p = np.empty((n_sel, cols), dtype=np.float64)
    lib.orc_apply_stats(_ptr(a), code, cols, _ptr(vl), _ptr(mm), _ptr(dd), _ptr(sel), n_sel, _ptr(p))
    return p


def softmax_backward(p, g, dtype, rows: int, cols: int, valid_len=None, rows_sel=None):
    """fp64 dx = p (g - sum(g p)) per row over the valid prefix (0 beyond).

    p and g are stored values of one type (float32, or uint16 bits).
    """
    lib = _load()
    a, code, vl, sel, n_sel = _rows_args(p, dtype, rows, cols, valid_len, rows_sel)
    b, code_g = _as_storage(g, dtype)
    if b.size != rows * cols:
        raise ValueError("g has the wrong number of elements")
    dx = np.empty((n_sel, cols), dtype=np.float64)
    lib.orc_softmax_backward(_ptr(a), _ptr(b), code, cols, _ptr(vl), _ptr(sel), n_sel, _ptr(dx))
    return dx


def cross_entropy(x, dtype, rows: int, cols: int, target, valid_len=None, rows_sel=None,
                  want_grad: bool = True):
    """fp64 (loss [n], grad [n, cols] or None) of cross-entropy with logits.

    loss = LSE - x_t, grad = softmax - onehot(t); a target outside the valid
    prefix is ignored (loss 0, gradient 0).
    """
    lib = _load()
    a, code, vl, sel, n_sel = _rows_args(x, dtype, rows, cols, valid_len, rows_sel)
    t = np.ascontiguousarray(target, dtype=np.int64)
    if t.shape != (rows,):
        raise ValueError("target must have one entry per row")
    loss = np.empty(n_sel, dtype=np.float64)
    grad = np.empty((n_sel, cols), dtype=np.float64) if want_grad else None
    lib.orc_cross_entropy(_ptr(a), code, cols, _ptr(vl), _ptr(t), _ptr(sel), n_sel, _ptr(loss),
                          _ptr(grad))
    return loss, grad


def attention_rows(q, k, v, dtype, heads: int, sq: int, sk: int, d: int, scale: float,
                   causal: bool = False, rows_sel=None):
    """fp64 attention of the selected (head, row) pairs, index head * sq + row.

    q: [heads, sq, d], k and v: [heads, sk, d] stored values of one type.
    Returns (o [n, d], lse [n], oabs [n, d] = sum p |v|, smax [n] = max scale |q|.|k|).
    """
    lib = _load()
    a, code = _as_storage(q, dtype)
    b, _ = _as_storage(k, dtype)
    c, _ = _as_storage(v, dtype)
    if a.size != heads * sq * d or b.size != heads * sk * d or c.size != heads * sk * d:
        raise ValueError("q, k, v have the wrong number of elements")
    sel = None if rows_sel is None else np.ascontiguousarray(rows_sel, dtype=np.int64)
    n = heads * sq if sel is None else sel.size
    o = np.empty((n, d), dtype=np.float64)
    lse = np.empty(n, dtype=np.float64)
    oabs = np.empty((n, d), dtype=np.float64)
    smax = np.empty(n, dtype=np.float64)
    lib.orc_attention_rows(_ptr(a), _ptr(b), _ptr(c), code, sq, sk, d, float(scale), 1 if causal else 0,
                           _ptr(sel), n, _ptr(o), _ptr(lse), _ptr(oabs), _ptr(smax))
    return o, lse, oabs, smax


def attention_online(s, v, block: int, rescale_o: bool = True):
    """The pages' (m, l, o) running state over blocks of scores s [n] and values v [n, d]."""
    lib = _load()
    sv = np.ascontiguousarray(s, dtype=np.float64)
    vv = np.ascontiguousarray(v, dtype=np.float64)
    n, d = vv.shape
    o = np.empty(d)
    m = np.empty(1)
    l = np.empty(1)
    lib.orc_attention_online(_ptr(sv), _ptr(vv), n, d, block, 1 if rescale_o else 0, _ptr(o), _ptr(m),
                             _ptr(l))
    return o, float(m[0]), float(l[0])
