"""Seeded synthetic inputs for the softmax workloads.

This module only draws inputs: it holds none of the softmax arithmetic, and it is
the one module that both the CUDA path's tests/benchmark and the CPU reference
read.  Every array is drawn on the host from numpy's PCG64 with a fixed seed per
workload (numpy's generator is platform independent), in fp32, then rounded to
the storage type with round-to-nearest-even (torch's CPU conversion).  The
batched causal workload is too large to draw on the host in test time; it is
drawn on the device slice by slice from torch's seeded CUDA generator, and the
rows a test checks are copied back to the host for the reference.

Workloads (sizes as named):
  f32_64x1000          fp32 in/out, 64 x 1000, x ~ N(0, 3^2), one element per row
                       set to +30.0 at a seeded position, no mask.
  bf16_16384x4096      bf16 in/out, 16384 x 4096, x ~ N(0, 8^2), no mask.
  f16_32768x1024_len   fp16 in/out, 32768 x 1024, x ~ U[-30, 30]; valid length per
                       row ~ U{0..1024}, and exactly 328 seeded rows (1%) of
                       length 0.
  f32_64x1048576_rise  fp32 in/out, 64 x 1,048,576, x_j = N(0,1) + 20 j / cols
                       (the running maximum keeps rising along the row).
  bf16_causal_8x32x4096x4096
                       bf16 in/out, 8*32*4096 = 1,048,576 rows x 4096, x ~ N(0,1);
                       row i of every 4096-row slice is valid for cols <= i.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

F32, F16, BF16 = "f32", "f16", "bf16"


@dataclass(frozen=True)
class Workload:
    name: str
    rows: int
    cols: int
    in_dtype: str
    out_dtype: str
    seed: int
    masked: bool
    description: str


WORKLOADS = {
    "f32_64x1000": Workload("f32_64x1000", 64, 1000, F32, F32, 1001, False,
                            "fp32 64x1000, N(0,3^2) with one +30.0 per row"),
    "bf16_16384x4096": Workload("bf16_16384x4096", 16384, 4096, BF16, BF16, 1002, False,
                                "bf16 16384x4096, N(0,8^2)"),
    "f16_32768x1024_len": Workload("f16_32768x1024_len", 32768, 1024, F16, F16, 1003, True,
                                   "fp16 32768x1024, U[-30,30], valid length U{0..1024}, 1% empty"),
    "f32_64x1048576_rise": Workload("f32_64x1048576_rise", 64, 1048576, F32, F32, 1004, False,
                                    "fp32 64x1048576, N(0,1) + 20 j/cols"),
    "bf16_causal_8x32x4096x4096": Workload("bf16_causal_8x32x4096x4096", 8 * 32 * 4096, 4096, BF16,
                                           BF16, 1005, True,
                                           "bf16 8x32x4096x4096 causal, N(0,1)"),
}

BENCH_WORKLOAD = "bf16_16384x4096"

# The worked rows the pages print, run as fixed cases.
WORKED_ROWS = {
    "fp16_example": [20.0, 18.0, 17.0, -5.0],
    "large_logits": [1000.0, 999.0, 997.0],
    "two_logit_z0.5": [0.0, 0.5],
    "two_logit_z2.5": [0.0, 2.5],
}


def to_storage(x32: np.ndarray, dtype: str) -> np.ndarray:
    """fp32 values -> stored array: float32 for f32, uint16 bit patterns for f16/bf16."""
    x32 = np.ascontiguousarray(x32, dtype=np.float32)
    if dtype == F32:
        return x32
    t = torch.from_numpy(x32).to(torch.float16 if dtype == F16 else torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def storage_to_torch(a: np.ndarray, dtype: str) -> torch.Tensor:
    """Stored array -> CPU torch tensor of the matching dtype (no copy of values)."""
    if dtype == F32:
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16))
    return t.view(torch.float16 if dtype == F16 else torch.bfloat16)


def torch_to_storage(t: torch.Tensor) -> np.ndarray:
    """CPU torch tensor -> stored numpy array (float32, or uint16 bits)."""
    t = t.contiguous()
    if t.dtype == torch.float32:
        return t.numpy()
    return t.view(torch.int16).numpy().view(np.uint16)


def torch_dtype(dtype: str) -> torch.dtype:
    return {F32: torch.float32, F16: torch.float16, BF16: torch.bfloat16}[dtype]


def host_input(name: str, rows: int | None = None):
    """Draw a host workload.  Returns (x stored array [rows*cols], valid_len int32 or None).

    rows: draw only the first `rows` rows' worth of the recipe (smaller cases of
    the same distribution, for tests); the draw is re-seeded so it is the same
    for a given (workload, rows).
    """
    w = WORKLOADS[name]
    if name == "bf16_causal_8x32x4096x4096" and rows is None:
        raise ValueError("the causal batch is drawn on the device: use device_causal_slice()")
    R = w.rows if rows is None else rows
    C = w.cols
    g = np.random.Generator(np.random.PCG64(w.seed))
    vl = None
    if name == "f32_64x1000":
        x = (3.0 * g.standard_normal((R, C), dtype=np.float32)).astype(np.float32)
        pos = g.integers(0, C, size=R)
        x[np.arange(R), pos] = 30.0
    elif name == "bf16_16384x4096":
        x = (8.0 * g.standard_normal((R, C), dtype=np.float32)).astype(np.float32)
    elif name == "f16_32768x1024_len":
        x = g.uniform(-30.0, 30.0, size=(R, C)).astype(np.float32)
        vl = g.integers(0, C + 1, size=R).astype(np.int32)
        n_empty = max(1, int(round(0.01 * R)))  # 328 rows at the full 32768
        empty = g.choice(R, size=n_empty, replace=False)
        vl[empty] = 0
    elif name == "f32_64x1048576_rise":
        x = g.standard_normal((R, C), dtype=np.float32)
        x += (20.0 * np.arange(C, dtype=np.float64) / C).astype(np.float32)[None, :]
    elif name == "bf16_causal_8x32x4096x4096":
        x = g.standard_normal((R, C), dtype=np.float32)
        vl = (np.arange(R) % 4096 + 1).astype(np.int32)
    else:
        raise KeyError(name)
    return to_storage(x.reshape(-1), w.in_dtype), vl


CAUSAL_SLICE_ROWS = 4096


def device_causal_slice(s: int, out: torch.Tensor) -> None:
    """Fill `out` (a [4096, 4096] bf16 CUDA tensor) with slice s of the causal batch."""
    g = torch.Generator(device=out.device)
    g.manual_seed(WORKLOADS["bf16_causal_8x32x4096x4096"].seed * 100003 + s)
    out.copy_(torch.randn(out.shape, generator=g, device=out.device, dtype=torch.float32))


def causal_valid_len(rows: int) -> np.ndarray:
    """Row i of each 4096-row slice is valid for cols <= i (length i + 1)."""
    return (np.arange(rows) % CAUSAL_SLICE_ROWS + 1).astype(np.int32)


OPS = ("softmax", "log_softmax", "lse", "apply_stats", "backward", "cross_entropy", "attention")

# Attention workloads (name -> heads, sequence length, head dim, causal): the
# pages' N = 4096 attention example ("Softmax numerics architecture...", "From
# online softmax to tiled attention") as 4 x 32 heads of head dim 128, bf16,
# q, k, v ~ N(0, 1) drawn on the device from one seeded generator.
ATTN_WORKLOADS = {
    "attn_bf16_4x32x4096x128": (128, 4096, 128, False),
    "attn_bf16_4x32x4096x128_causal": (128, 4096, 128, True),
}
ATTN_SEED = 1006


def attention_inputs(name: str, device):
    """(q, k, v) bf16 [heads, seq, d] on `device`, seeded."""
    heads, n, d, _ = ATTN_WORKLOADS[name]
    g = torch.Generator(device=device).manual_seed(ATTN_SEED)
    return tuple(torch.randn(heads, n, d, generator=g, device=device).to(torch.bfloat16) for _ in range(3))


def attention_pairs(sq: int, sk: int, causal: bool) -> int:
    """Valid (query, key) pairs of one head: all of them, or under the
    bottom-right aligned causal mask (key j valid for query i when
    j <= i + sk - sq) sum_i clamp(i + sk - sq + 1, 0, sk)."""
    if not causal:
        return sq * sk
    i = np.arange(sq, dtype=np.int64)
    return int(np.clip(i + sk - sq + 1, 0, sk).sum())


def attention_flops(heads: int, sq: int, sk: int, d: int, causal: bool) -> float:
    """Multiply-adds of the two products over the valid pairs, 2 flops each:
    4 d per pair."""
    return 4.0 * heads * d * attention_pairs(sq, sk, causal)


def op_bytes(op: str, rows: int, cols: int, in_size: int, out_size: int, valid_len=None) -> int:
    """Bytes an operation must move over a [rows, cols] batch: the valid inputs
    read once (the backward reads two arrays), each dense output written once,
    and the per-row values (lengths 4 B, statistics 8 B, LSE 4 B, targets 8 B +
    loss 4 B) once."""
    if valid_len is None:
        valid = rows * cols
        lens = 0
    else:
        valid = int(np.clip(np.asarray(valid_len, dtype=np.int64), 0, cols).sum())
        lens = rows * 4
    dense_out = rows * cols * out_size
    if op in ("softmax", "log_softmax"):
        return valid * in_size + dense_out + lens
    if op == "lse":
        return valid * in_size + rows * 4 + lens
    if op == "apply_stats":
        return valid * in_size + dense_out + rows * 8 + lens
    if op == "backward":
        return 2 * valid * in_size + dense_out + lens
    if op == "cross_entropy":
        return valid * in_size + dense_out + rows * 12 + lens
    raise ValueError(f"unknown op {op}")


def algorithmic_bytes(rows: int, cols: int, in_size: int, out_size: int, valid_len=None) -> int:
    """Bytes the method must move: the valid input read once, every output written
    once, and the row lengths read once when given."""
    if valid_len is None:
        read = rows * cols * in_size
    else:
        vl = np.clip(np.asarray(valid_len, dtype=np.int64), 0, cols)
        read = int(vl.sum()) * in_size + rows * 4
    return int(read + rows * cols * out_size)
