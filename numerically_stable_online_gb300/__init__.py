"""Row-wise numerically stable softmax for GB300 (sm_103a).

Thin Python binding of the C ABI in ``include/smx.h``: each function marshals
torch tensors (device memory and the current CUDA stream) into pointers and
sizes and calls the same-named entry point of ``_build/libsmx.so``.  Every step
of the computation runs in the library's CUDA kernels; there is no fallback.
If the library has not been built (``python -m numerically_stable_online_gb300.build``)
or no sm_103 device is present, the calls raise.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = [
    "SmxError", "library", "softmax_rows", "softmax_rows_fixed_scratch", "softmax_rows_host", "softmax_row_stats",
    "softmax_merge_stats", "log_softmax_rows", "softmax_lse", "softmax_apply_stats",
    "softmax_backward", "cross_entropy", "attention_forward",
    "last_device_status", "status_string", "DTYPES",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libsmx.so")

SMX_F32, SMX_F16, SMX_BF16 = 0, 1, 2
DTYPES = {torch.float32: SMX_F32, torch.float16: SMX_F16, torch.bfloat16: SMX_BF16}
STATUS = {0: "SMX_OK", 1: "SMX_ERR_INVALID_ARG", 2: "SMX_ERR_UNSUPPORTED", 3: "SMX_ERR_ALIAS",
          4: "SMX_ERR_LAUNCH", 5: "SMX_ERR_TIMEOUT", 6: "SMX_ERR_DEVICE", 7: "SMX_ERR_TOO_LARGE"}

_lock = threading.Lock()
_lib = None


class SmxError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        lib = _lib
        text = lib.smx_status_string(status).decode() if lib is not None else STATUS.get(status, "?")
        cuda = lib.smx_last_cuda_error() if lib is not None else 0
        super().__init__(f"{where}: {STATUS.get(status, status)} ({text}); cuda error {cuda}")


def library() -> ctypes.CDLL:
    """The loaded C library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"CUDA library not built: {LIB_PATH} is missing "
                               "(run python -m numerically_stable_online_gb300.build)")
        lib = ctypes.CDLL(LIB_PATH)
        P, I64, I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        st = ctypes.c_int
        lib.smx_softmax_rows.argtypes = [P, P, I64, I64, P, I32, I32, P]
        lib.smx_softmax_rows.restype = st
        lib.smx_softmax_rows_host.argtypes = [P, P, I64, I64, P, I32, I32, P]
        lib.smx_softmax_rows_host.restype = st
        lib.smx_softmax_rows_fixed_scratch.argtypes = [P, P, I64, I64, P, I32, I32, P]
        lib.smx_softmax_rows_fixed_scratch.restype = st
        lib.smx_softmax_row_stats.argtypes = [P, P, P, I64, I64, P, I32, P]
        lib.smx_softmax_row_stats.restype = st
        lib.smx_softmax_merge_stats.argtypes = [P, P, P, P, P, P, I64, P]
        lib.smx_softmax_merge_stats.restype = st
        lib.smx_log_softmax_rows.argtypes = [P, P, I64, I64, P, I32, I32, P]
        lib.smx_log_softmax_rows.restype = st
        lib.smx_softmax_lse.argtypes = [P, P, I64, I64, P, I32, P]
        lib.smx_softmax_lse.restype = st
        lib.smx_softmax_apply_stats.argtypes = [P, P, P, P, I64, I64, P, I32, I32, P]
        lib.smx_softmax_apply_stats.restype = st
        lib.smx_softmax_backward.argtypes = [P, P, P, I64, I64, P, I32, I32, P]
        lib.smx_softmax_backward.restype = st
        lib.smx_cross_entropy.argtypes = [P, P, P, P, I64, I64, P, I32, I32, P]
        lib.smx_cross_entropy.restype = st
        lib.smx_attention_forward.argtypes = [P, P, P, P, P, I64, I64, I64, I32, ctypes.c_double, I32, I32, P]
        lib.smx_attention_forward.restype = st
        lib.smx_last_device_status.argtypes = [P]
        lib.smx_last_device_status.restype = st
        lib.smx_status_string.argtypes = [st]
        lib.smx_status_string.restype = ctypes.c_char_p
        lib.smx_last_cuda_error.argtypes = []
        lib.smx_last_cuda_error.restype = I32
        lib.smx_version.argtypes = []
        lib.smx_version.restype = I32
        lib.smx_debug_force_path.argtypes = [I32]
        lib.smx_debug_force_path.restype = None
        lib.smx_debug_set_cluster.argtypes = [I32, I64]
        lib.smx_debug_set_cluster.restype = None
        lib.smx_debug_set_wait_limit.argtypes = [I64]
        lib.smx_debug_set_wait_limit.restype = None
        lib.smx_debug_last_path.argtypes = []
        lib.smx_debug_last_path.restype = I32
        lib.smx_debug_last_launches.argtypes = []
        lib.smx_debug_last_launches.restype = I32
        lib.smx_debug_set_regs_shape.argtypes = [I32, I32]
        lib.smx_debug_set_regs_shape.restype = None
        lib.smx_debug_set_stream_depth.argtypes = [I32]
        lib.smx_debug_set_stream_depth.restype = None
        lib.smx_debug_set_stream_ctas.argtypes = [I32]
        lib.smx_debug_set_stream_ctas.restype = None
        lib.smx_debug_set_cluster_staging.argtypes = [I32]
        lib.smx_debug_set_cluster_staging.restype = None
        lib.smx_debug_set_split_slab.argtypes = [I64]
        lib.smx_debug_set_split_slab.restype = None
        lib.smx_debug_set_split_hints.argtypes = [I32, I32]
        lib.smx_debug_set_split_hints.restype = None
        lib.smx_debug_set_inflight.argtypes = [I64, I64]
        lib.smx_debug_set_inflight.restype = None
        lib.smx_debug_set_stream_warp.argtypes = [I32]
        lib.smx_debug_set_stream_warp.restype = None
        lib.smx_debug_set_split_fused.argtypes = [I32]
        lib.smx_debug_set_split_fused.restype = None
        lib.smx_debug_set_host_chunk.argtypes = [I64, I32, I32]
        lib.smx_debug_set_host_chunk.restype = None
        lib.smx_debug_set_attention_kernel.argtypes = [I32]
        lib.smx_debug_set_attention_kernel.restype = None
        lib.smx_debug_alloc_count.argtypes = []
        lib.smx_debug_alloc_count.restype = I64
        lib.smx_debug_set_count_probe.argtypes = [I64]
        lib.smx_debug_set_count_probe.restype = None
        lib.smx_debug_set_stripe_tuning.argtypes = [I32, I32, I32]
        lib.smx_debug_set_stripe_tuning.restype = None
        lib.smx_debug_probe_math.argtypes = [P, P, P, I64, I32, P]
        lib.smx_debug_probe_math.restype = st
        _lib = lib
        return lib


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dtype(t: torch.dtype) -> int:
    try:
        return DTYPES[t]
    except KeyError:
        raise TypeError(f"unsupported dtype {t}: use float32, float16 or bfloat16") from None


def _check_2d(x: torch.Tensor, name: str):
    if not x.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if x.dim() != 2 or not x.is_contiguous():
        raise ValueError(f"{name} must be a contiguous 2-D [rows, cols] tensor")


def _lengths(valid_len, rows, device):
    if valid_len is None:
        return None
    if not (valid_len.is_cuda and valid_len.dtype == torch.int32 and valid_len.is_contiguous()
            and valid_len.numel() == rows and valid_len.device == device):
        raise ValueError("valid_len must be a contiguous int32 CUDA tensor with one entry per row")
    return valid_len.data_ptr()


def softmax_rows(x: torch.Tensor, out: torch.Tensor | None = None, valid_len: torch.Tensor | None = None,
                 out_dtype: torch.dtype | None = None, stream=None) -> torch.Tensor:
    """y[r, j] = exp(x[r, j] - m_r) / d_r over the valid prefix of each row; +0 elsewhere."""
    _check_2d(x, "x")
    rows, cols = x.shape
    if out is None:
        out = torch.empty((rows, cols), dtype=out_dtype or x.dtype, device=x.device)
    _check_2d(out, "out")
    if out.shape != x.shape or out.device != x.device:
        raise ValueError("out must match x's shape and device")
    st = library().smx_softmax_rows(x.data_ptr(), out.data_ptr(), rows, cols,
                                    _lengths(valid_len, rows, x.device), _dtype(x.dtype),
                                    _dtype(out.dtype), _stream(stream))
    if st != 0:
        raise SmxError(st, "smx_softmax_rows")
    return out


def softmax_rows_host(x: torch.Tensor, out: torch.Tensor | None = None, valid_len: torch.Tensor | None = None,
                      out_dtype: torch.dtype | None = None, stream=None, wait: bool = True) -> torch.Tensor:
    """softmax_rows of a HOST matrix into a host matrix, through the current device.

    Pinned tensors (``x.pin_memory()``; ``out=None`` allocates a pinned output
    when ``x`` is pinned, and ``valid_len`` must be pinned too) are read and
    written in place by the kernel over the host link when the rows take the
    streamed or register-resident kernels (up to 32,768 elements, 16,384 for
    float32 outputs; 16-byte aligned rows).  Otherwise the library moves
    the rows through two device staging buffers in chunks, overlapping each
    chunk's copy in, softmax and copy back.  With ``wait`` the call returns
    after the stream has finished; otherwise ``out`` is ready once the stream
    reaches this point.
    """
    for t, name in ((x, "x"), (out, "out")):
        if t is not None and (t.is_cuda or t.dim() != 2 or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous 2-D [rows, cols] host tensor")
    rows, cols = x.shape
    if out is None:
        out = torch.empty((rows, cols), dtype=out_dtype or x.dtype, pin_memory=x.is_pinned())
    if out.shape != x.shape:
        raise ValueError("out must match x's shape")
    vl = None
    if valid_len is not None:
        if valid_len.is_cuda or valid_len.dtype != torch.int32 or not valid_len.is_contiguous() \
                or valid_len.numel() != rows:
            raise ValueError("valid_len must be a contiguous int32 host tensor with one entry per row")
        vl = valid_len.data_ptr()
    sp = _stream(stream)
    st = library().smx_softmax_rows_host(x.data_ptr(), out.data_ptr(), rows, cols, vl, _dtype(x.dtype),
                                         _dtype(out.dtype), sp)
    if st != 0:
        raise SmxError(st, "smx_softmax_rows_host")
    if wait:
        s = stream if hasattr(stream, "synchronize") else (
            torch.cuda.current_stream() if stream is None else torch.cuda.ExternalStream(sp))
        s.synchronize()
    return out


def softmax_rows_fixed_scratch(x: torch.Tensor, out: torch.Tensor | None = None,
                               valid_len: torch.Tensor | None = None,
                               out_dtype: torch.dtype | None = None, stream=None) -> torch.Tensor:
    """softmax_rows without any device allocation inside the library call.

    The long-row kernels keep their chunk summaries in one fixed per-device
    array (256 KiB); calls that can overlap on the device race on it, so issue
    them on one stream.  Rows longer than 134217728 elements raise
    SMX_ERR_TOO_LARGE.  (``out=None`` allocates the output here, in torch,
    before the call.)
    """
    _check_2d(x, "x")
    rows, cols = x.shape
    if out is None:
        out = torch.empty((rows, cols), dtype=out_dtype or x.dtype, device=x.device)
    _check_2d(out, "out")
    if out.shape != x.shape or out.device != x.device:
        raise ValueError("out must match x's shape and device")
    st = library().smx_softmax_rows_fixed_scratch(x.data_ptr(), out.data_ptr(), rows, cols,
                                                  _lengths(valid_len, rows, x.device),
                                                  _dtype(x.dtype), _dtype(out.dtype), _stream(stream))
    if st != 0:
        raise SmxError(st, "smx_softmax_rows_fixed_scratch")
    return out


def softmax_row_stats(x: torch.Tensor, valid_len: torch.Tensor | None = None, m_out=None, d_out=None,
                      stream=None):
    """Per-row block summary (m, d) in fp32: m = max, d = sum exp(x - m)."""
    _check_2d(x, "x")
    rows, cols = x.shape
    if m_out is None:
        m_out = torch.empty(rows, dtype=torch.float32, device=x.device)
    if d_out is None:
        d_out = torch.empty(rows, dtype=torch.float32, device=x.device)
    for t in (m_out, d_out):
        if not (t.is_cuda and t.dtype == torch.float32 and t.is_contiguous() and t.numel() == rows):
            raise ValueError("m_out/d_out must be contiguous float32 CUDA tensors of length rows")
    st = library().smx_softmax_row_stats(x.data_ptr(), m_out.data_ptr(), d_out.data_ptr(), rows, cols,
                                         _lengths(valid_len, rows, x.device), _dtype(x.dtype),
                                         _stream(stream))
    if st != 0:
        raise SmxError(st, "smx_softmax_row_stats")
    return m_out, d_out


def softmax_merge_stats(m_a, d_a, m_b, d_b, m_out=None, d_out=None, stream=None):
    """Element-wise merge of two arrays of (m, d) summaries (may run in place)."""
    n = m_a.numel()
    for t in (m_a, d_a, m_b, d_b):
        if not (t.is_cuda and t.dtype == torch.float32 and t.is_contiguous() and t.numel() == n):
            raise ValueError("summaries must be contiguous float32 CUDA tensors of one length")
    if m_out is None:
        m_out = torch.empty_like(m_a)
    if d_out is None:
        d_out = torch.empty_like(d_a)
    st = library().smx_softmax_merge_stats(m_a.data_ptr(), d_a.data_ptr(), m_b.data_ptr(),
                                           d_b.data_ptr(), m_out.data_ptr(), d_out.data_ptr(), n,
                                           _stream(stream))
    if st != 0:
        raise SmxError(st, "smx_softmax_merge_stats")
    return m_out, d_out


def _rows_vec(t, rows, device, name):
    if not (t.is_cuda and t.dtype == torch.float32 and t.is_contiguous() and t.numel() == rows
            and t.device == device):
        raise ValueError(f"{name} must be a contiguous float32 CUDA tensor of length rows")
    return t.data_ptr()


def log_softmax_rows(x: torch.Tensor, out: torch.Tensor | None = None,
                     valid_len: torch.Tensor | None = None, out_dtype: torch.dtype | None = None,
                     stream=None) -> torch.Tensor:
    """y[r, j] = (x[r, j] - m_r) - log d_r over the valid prefix; -inf elsewhere."""
    _check_2d(x, "x")
    rows, cols = x.shape
    if out is None:
        out = torch.empty((rows, cols), dtype=out_dtype or x.dtype, device=x.device)
    _check_2d(out, "out")
    if out.shape != x.shape or out.device != x.device:
        raise ValueError("out must match x's shape and device")
    st = library().smx_log_softmax_rows(x.data_ptr(), out.data_ptr(), rows, cols,
                                        _lengths(valid_len, rows, x.device), _dtype(x.dtype),
                                        _dtype(out.dtype), _stream(stream))
    if st != 0:
        raise SmxError(st, "smx_log_softmax_rows")
    return out


def softmax_lse(x: torch.Tensor, valid_len: torch.Tensor | None = None, out=None, stream=None):
    """Per-row log-sum-exp m + log d in fp32."""
    _check_2d(x, "x")
    rows, cols = x.shape
    if out is None:
        out = torch.empty(rows, dtype=torch.float32, device=x.device)
    st = library().smx_softmax_lse(x.data_ptr(), _rows_vec(out, rows, x.device, "out"), rows, cols,
                                   _lengths(valid_len, rows, x.device), _dtype(x.dtype),
                                   _stream(stream))
    if st != 0:
        raise SmxError(st, "smx_softmax_lse")
    return out


def softmax_apply_stats(x: torch.Tensor, m: torch.Tensor, d: torch.Tensor, out: torch.Tensor | None = None,
                        valid_len: torch.Tensor | None = None, out_dtype: torch.dtype | None = None,
                        stream=None) -> torch.Tensor:
    """y[r, j] = exp(x[r, j] - m[r]) / d[r] over the valid prefix, +0 elsewhere."""
    _check_2d(x, "x")
    rows, cols = x.shape
    if out is None:
        out = torch.empty((rows, cols), dtype=out_dtype or x.dtype, device=x.device)
    _check_2d(out, "out")
    if out.shape != x.shape or out.device != x.device:
        raise ValueError("out must match x's shape and device")
    st = library().smx_softmax_apply_stats(x.data_ptr(), _rows_vec(m, rows, x.device, "m"),
                                           _rows_vec(d, rows, x.device, "d"), out.data_ptr(), rows,
                                           cols, _lengths(valid_len, rows, x.device),
                                           _dtype(x.dtype), _dtype(out.dtype), _stream(stream))
    if st != 0:
        raise SmxError(st, "smx_softmax_apply_stats")
    return out


def softmax_backward(p: torch.Tensor, g: torch.Tensor, out: torch.Tensor | None = None,
                     valid_len: torch.Tensor | None = None, out_dtype: torch.dtype | None = None,
                     stream=None) -> torch.Tensor:
    """dx = p (g - sum(g p)) per row over the valid prefix (0 elsewhere)."""
    _check_2d(p, "p")
    _check_2d(g, "g")
    if g.shape != p.shape or g.dtype != p.dtype or g.device != p.device:
        raise ValueError("g must match p's shape, dtype and device")
    rows, cols = p.shape
    if out is None:
        out = torch.empty((rows, cols), dtype=out_dtype or p.dtype, device=p.device)
    _check_2d(out, "out")
    if out.shape != p.shape or out.device != p.device:
        raise ValueError("out must match p's shape and device")
    st = library().smx_softmax_backward(p.data_ptr(), g.data_ptr(), out.data_ptr(), rows, cols,
                                        _lengths(valid_len, rows, p.device), _dtype(p.dtype),
                                        _dtype(out.dtype), _stream(stream))
    if st != 0:
        raise SmxError(st, "smx_softmax_backward")
    return out


def cross_entropy(x: torch.Tensor, target: torch.Tensor, valid_len: torch.Tensor | None = None,
                  with_grad: bool = True, grad: torch.Tensor | None = None,
                  grad_dtype: torch.dtype | None = None, loss: torch.Tensor | None = None, stream=None):
    """(loss [rows] fp32, grad [rows, cols] or None): loss = LSE - x_t, grad = p - onehot(t)."""
    _check_2d(x, "x")
    rows, cols = x.shape
    if not (target.is_cuda and target.dtype == torch.int64 and target.is_contiguous()
            and target.numel() == rows and target.device == x.device):
        raise ValueError("target must be a contiguous int64 CUDA tensor with one entry per row")
    if loss is None:
        loss = torch.empty(rows, dtype=torch.float32, device=x.device)
    if with_grad and grad is None:
        grad = torch.empty((rows, cols), dtype=grad_dtype or x.dtype, device=x.device)
    if grad is not None:
        _check_2d(grad, "grad")
        if grad.shape != x.shape or grad.device != x.device:
            raise ValueError("grad must match x's shape and device")
    st = library().smx_cross_entropy(x.data_ptr(), target.data_ptr(),
                                     _rows_vec(loss, rows, x.device, "loss"),
                                     None if grad is None else grad.data_ptr(), rows, cols,
                                     _lengths(valid_len, rows, x.device), _dtype(x.dtype),
                                     _dtype(grad.dtype if grad is not None else x.dtype),
                                     _stream(stream))
    if st != 0:
        raise SmxError(st, "smx_cross_entropy")
    return loss, grad


def attention_forward(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: float | None = None,
                      causal: bool = False, out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                      with_lse: bool = True, stream=None):
    """(o, lse) of attention over [..., seq, head_dim] fp16/bf16 tensors (leading dims = heads)."""
    for t, name in ((q, "q"), (k, "k"), (v, "v")):
        if not t.is_cuda or not t.is_contiguous() or t.dim() < 2:
            raise ValueError(f"{name} must be a contiguous CUDA tensor [..., seq, head_dim]")
    if k.shape != v.shape or q.shape[:-2] != k.shape[:-2] or q.shape[-1] != k.shape[-1]:
        raise ValueError("q, k, v shapes do not match")
    if not (q.dtype == k.dtype == v.dtype):
        raise ValueError("q, k, v must share a dtype")
    d = q.shape[-1]
    heads = int(q.numel() // (q.shape[-2] * d)) if q.numel() else 0
    sq, sk = q.shape[-2], k.shape[-2]
    if scale is None:
        scale = d ** -0.5
    if out is None:
        out = torch.empty_like(q)
    if with_lse and lse is None:
        lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
    st = library().smx_attention_forward(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                         None if lse is None else lse.data_ptr(), heads, sq, sk, d,
                                         float(scale), 1 if causal else 0, _dtype(q.dtype), _stream(stream))
    if st != 0:
        raise SmxError(st, "smx_attention_forward")
    return out, lse


def last_device_status(stream=None) -> int:
    """Synchronise the stream; return and clear the device status word (0 = ok)."""
    return library().smx_last_device_status(_stream(stream))


def status_string(status: int) -> str:
    return library().smx_status_string(status).decode()
