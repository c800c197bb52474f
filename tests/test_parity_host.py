"""Parity of the host-buffer softmax call (smx_softmax_rows_host) with the
fp64 reference.

The call moves host rows through two device staging slots in chunks of about
16 MiB of input, each chunk's copy in and softmax on the caller's stream and
its copy back on a second stream.  These cases span several chunks with a
ragged last one, rows longer than a chunk (one row a chunk, long-row kernels),
lengths, every output dtype, pinned and pageable host memory, and a caller
stream other than the default; every element is compared with the reference.
"""
import numpy as np
import pytest
import torch

import numerically_stable_online_gb300 as smx
import oracle
from numerically_stable_online_gb300 import workloads as wl
from tests import parity

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
ES = {"f32": 4, "f16": 2, "bf16": 2}
CHUNK_BYTES = 16 << 20


@pytest.fixture(scope="module", autouse=True)
def built():
    from numerically_stable_online_gb300 import build

    build.build()
    oracle.build()
    lib = smx.library()
    yield lib
    lib.smx_debug_set_host_chunk(0, 0, 0)


@pytest.fixture(autouse=True)
def default_host_path(built):
    """Every test starts and ends with the default chunk, slots and path."""
    built.smx_debug_set_host_chunk(0, 0, 0)
    yield
    built.smx_debug_set_host_chunk(0, 0, 0)


def host_tensor(x_store, in_dtype, rows, cols, pinned):
    t = wl.storage_to_torch(np.ascontiguousarray(x_store).reshape(-1), in_dtype).reshape(rows, cols)
    return t.pin_memory() if pinned else t.contiguous()


def compare_all(y, x_store, in_dtype, out_dtype, rows, cols, vl, block_rows=2048):
    y_host = wl.torch_to_storage(y).reshape(rows, cols)
    for r0 in range(0, rows, block_rows):
        sel = np.arange(r0, min(rows, r0 + block_rows))
        p = oracle.softmax_rows(x_store, in_dtype, rows, cols, vl, rows_sel=sel)
        parity.compare(y_host[r0:sel[-1] + 1], p, out_dtype, vl, rows_sel=sel)


def chunks(rows, cols, in_dtype):
    cr = max(1, min(rows, CHUNK_BYTES // (cols * ES[in_dtype])))
    return -(-rows // cr)


PATH_REGS, PATH_STREAM, PATH_SPLIT, PATH_STRIPE = 1, 4, 5, 6


@pytest.mark.parametrize("name,rows,out_dtype,pinned", [
    ("bf16_16384x4096", 3 * 2048 + 77, "bf16", True),     # 4 chunks staged, ragged last
    ("bf16_16384x4096", 2 * 2048 + 1, "f32", False),      # pageable, wider output
    ("f16_32768x1024_len", 2 * 8192 + 5, "f16", True),    # lengths from host memory
    ("f32_64x1000", 64, "bf16", True),                    # one chunk
    ("f32_64x1048576_rise", 7, "f32", True),              # 4 MiB rows, 4 a chunk; always staged
                                                          # (the read-once kernel's bulk copies stay in HBM)
])
@pytest.mark.parametrize("staged", [0, 1])
def test_host_call_workloads(built, name, rows, out_dtype, pinned, staged):
    """Page-locked buffers are read and written in place by the streamed
    kernel (one launch) unless staging is forced or the rows take the
    long-row kernels; pageable buffers always go through the staging slots."""
    built.smx_debug_set_host_chunk(0, 0, staged)
    w = wl.WORKLOADS[name]
    x_store, vl = wl.host_input(name, rows=rows)
    x = host_tensor(x_store, w.in_dtype, rows, w.cols, pinned)
    vlt = None if vl is None else torch.from_numpy(np.asarray(vl, np.int32))
    if pinned and vlt is not None:
        vlt = vlt.pin_memory()
    y = smx.softmax_rows_host(x, valid_len=vlt, out_dtype=DT[out_dtype])
    assert not y.is_cuda and y.is_pinned() == pinned and y.dtype == DT[out_dtype]
    in_place = pinned and not staged and built.smx_debug_last_path() not in (PATH_SPLIT, PATH_STRIPE)
    if in_place:
        assert built.smx_debug_last_launches() == 1
        assert built.smx_debug_last_path() in (PATH_REGS, PATH_STREAM)
    else:
        assert built.smx_debug_last_launches() >= chunks(rows, w.cols, w.in_dtype)
    assert smx.last_device_status() == 0
    compare_all(y, x_store, w.in_dtype, out_dtype, rows, w.cols, vl)
    if name == "f32_64x1048576_rise":
        assert built.smx_debug_last_path() == PATH_STRIPE


def test_lengths_in_pageable_memory_stage(built):
    """In place needs every buffer mapped: pinned rows with pageable lengths
    go through the staging slots."""
    name, rows = "f16_32768x1024_len", 8192 + 3
    w = wl.WORKLOADS[name]
    x_store, vl = wl.host_input(name, rows=rows)
    x = host_tensor(x_store, w.in_dtype, rows, w.cols, True)
    y = smx.softmax_rows_host(x, valid_len=torch.from_numpy(np.asarray(vl, np.int32)))
    assert built.smx_debug_last_launches() >= 2
    assert smx.last_device_status() == 0
    compare_all(y, x_store, w.in_dtype, w.out_dtype, rows, w.cols, vl)


def test_rows_longer_than_a_chunk(built):
    """8M-element fp32 rows (32 MiB each): one row a chunk, the long-row kernels."""
    rows, cols = 3, 1 << 23
    rng = np.random.default_rng(11)
    x_store = wl.to_storage(rng.normal(0, 4, rows * cols).astype(np.float32), "f32")
    x = host_tensor(x_store, "f32", rows, cols, True)
    y = smx.softmax_rows_host(x)
    assert smx.last_device_status() == 0
    compare_all(y, x_store, "f32", "f32", rows, cols, None, block_rows=1)


@pytest.mark.parametrize("staged", [0, 1])
def test_caller_stream_and_output_buffer(built, staged):
    """On a side stream, into a given output, in place and staged: the result
    is complete once that stream is synchronised, and repeated calls give the
    same bits."""
    built.smx_debug_set_host_chunk(0, 0, staged)
    name, rows = "bf16_16384x4096", 2048 + 513
    w = wl.WORKLOADS[name]
    x_store, _ = wl.host_input(name, rows=rows)
    x = host_tensor(x_store, w.in_dtype, rows, w.cols, True)
    out = torch.full((rows, w.cols), float("nan"), dtype=torch.bfloat16).pin_memory()
    s = torch.cuda.Stream()
    y = smx.softmax_rows_host(x, out=out, stream=s, wait=False)
    assert y is out
    s.synchronize()
    assert smx.last_device_status() == 0
    compare_all(y, x_store, w.in_dtype, w.out_dtype, rows, w.cols, None)
    # repeated calls reuse the library's copy stream and pool without leaking
    for _ in range(3):
        y2 = smx.softmax_rows_host(x, stream=s)
        assert torch.equal(y2.view(torch.int16), y.view(torch.int16))


def test_empty_and_policy_rows(built):
    assert smx.softmax_rows_host(torch.zeros(0, 16)).shape == (0, 16)
    assert smx.softmax_rows_host(torch.zeros(4, 0)).shape == (4, 0)
    x = torch.tensor([[-np.inf] * 8, [1.0, np.nan, 2.0, 0, 0, 0, 0, 0], [20.0, 18.0, 17.0, -5.0, 0, 0, 0, 0]])
    vl = torch.tensor([8, 8, 4], dtype=torch.int32)
    y = smx.softmax_rows_host(x, valid_len=vl).double().numpy()
    assert np.all(y[0] == 0) and not np.signbit(y[0]).any()
    assert np.isnan(y[1]).all()
    assert np.all(np.abs(y[2, :3] - [0.84380, 0.11420, 0.04201]) <= 1e-5) and np.all(y[2, 4:] == 0)


@pytest.mark.parametrize("chunk_bytes,slots,pinned", [(64 << 10, 2, True), (100000, 3, True),
                                                      (1 << 20, 4, False), (5000, 2, True)])
def test_many_chunks_and_slots(built, chunk_bytes, slots, pinned):
    """Small chunks (tens to hundreds of them, a ragged last one; 5000 bytes is
    less than one 8000-byte row, so one row a chunk) through 2, 3 and 4 staging
    slots, so every slot is reused many times while copies are in flight."""
    built.smx_debug_set_host_chunk(chunk_bytes, slots, 1)
    try:
        name, rows = "f16_32768x1024_len", 1000
        w = wl.WORKLOADS[name]
        x_store, vl = wl.host_input(name, rows=rows)
        x = host_tensor(x_store, w.in_dtype, rows, w.cols, pinned)
        y = smx.softmax_rows_host(x, valid_len=torch.from_numpy(np.asarray(vl, np.int32)))
        assert smx.last_device_status() == 0
        compare_all(y, x_store, w.in_dtype, w.out_dtype, rows, w.cols, vl)
        rows, cols = 300, 2000  # f32: 8000-byte rows, not a multiple of the chunk
        x_store = wl.to_storage(np.random.default_rng(5).normal(0, 6, rows * cols).astype(np.float32), "f32")
        x = host_tensor(x_store, "f32", rows, cols, pinned)
        y = smx.softmax_rows_host(x, out_dtype=torch.bfloat16)
        assert built.smx_debug_last_launches() >= -(-rows // max(1, chunk_bytes // (cols * 4)))
        assert smx.last_device_status() == 0
        compare_all(y, x_store, "f32", "bf16", rows, cols, None)
    finally:
        built.smx_debug_set_host_chunk(0, 0, 0)
