"""The C ABI library loads, exports every entry point include/smx.h declares, and
rejects bad arguments on the host before touching the GPU (runs without a GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from numerically_stable_online_gb300 import build

    build.build()
    import numerically_stable_online_gb300 as smx

    return smx.library()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "smx.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(smx_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("smx_softmax_rows", "smx_softmax_row_stats", "smx_softmax_merge_stats",
              "smx_last_device_status", "smx_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/smx.h but not exported"


def test_host_argument_checks_need_no_gpu(lib):
    P = ctypes.c_void_p
    fake_x, fake_y = P(0x10000000), P(0x20000000)
    # negative sizes and bad dtypes
    assert lib.smx_softmax_rows(fake_x, fake_y, -1, 4, None, 0, 0, None) == 1
    assert lib.smx_softmax_rows(fake_x, fake_y, 4, -1, None, 0, 0, None) == 1
    assert lib.smx_softmax_rows(fake_x, fake_y, 4, 4, None, 7, 0, None) == 1
    assert lib.smx_softmax_rows(fake_x, fake_y, 4, 4, None, 0, 3, None) == 1
    # null pointers with work to do
    assert lib.smx_softmax_rows(None, fake_y, 4, 4, None, 0, 0, None) == 1
    assert lib.smx_softmax_rows(fake_x, None, 4, 4, None, 0, 0, None) == 1
    # nothing to do is fine, even with null pointers
    assert lib.smx_softmax_rows(None, None, 0, 4, None, 0, 0, None) == 0
    assert lib.smx_softmax_rows(None, None, 4, 0, None, 0, 0, None) == 0
    # overlapping input and output
    assert lib.smx_softmax_rows(fake_x, P(0x10000000 + 8), 4, 4, None, 0, 0, None) == 3
    # an fp16 output ending right where the fp32 input starts does not overlap
    # (the call then needs a device: it reports that there is none)
    st = lib.smx_softmax_rows(P(0x10000000), P(0x10000000 - 32), 4, 4, None, 0, 1, None)
    assert st in (0, 2) and st != 3
    # row statistics
    assert lib.smx_softmax_row_stats(fake_x, None, fake_y, 4, 4, None, 0, None) == 1
    assert lib.smx_softmax_row_stats(fake_x, P(0x30000000), P(0x30000000 + 4), 4, 4, None, 0, None) == 3
    # merge: negative n, nulls, partial overlap (in place is allowed)
    a, b, c, d = (P(0x1000000 * k) for k in (1, 2, 3, 4))
    assert lib.smx_softmax_merge_stats(a, b, c, d, a, b, -1, None) == 1
    assert lib.smx_softmax_merge_stats(a, b, c, d, None, b, 4, None) == 1
    assert lib.smx_softmax_merge_stats(a, b, c, d, P(0x1000000 + 4), P(0x5000000), 4, None) == 3
    assert lib.smx_softmax_merge_stats(a, b, c, d, a, a, 4, None) == 3


def test_status_strings_and_version(lib):
    for s in range(7):
        assert lib.smx_status_string(s)
    assert lib.smx_version() >= 100


def test_binding_refuses_cpu_tensors():
    import torch

    import numerically_stable_online_gb300 as smx

    with pytest.raises(ValueError):
        smx.softmax_rows(torch.zeros(2, 4))


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """No fallback: with the CUDA library absent the binding raises instead of
    computing anything another way."""
    import numerically_stable_online_gb300 as smx

    monkeypatch.setattr(smx, "_lib", None)
    monkeypatch.setattr(smx, "LIB_PATH", str(tmp_path / "libsmx.so"))
    with pytest.raises(RuntimeError, match="not built"):
        smx.library()
    with pytest.raises(RuntimeError, match="not built"):
        smx.last_device_status()  # a public call that reaches the library without a GPU tensor


def test_host_buffer_call_checks_need_no_gpu(lib):
    """smx_softmax_rows_host validates like smx_softmax_rows, on host
    buffers, before it needs a device; with valid arguments and no device it
    reports SMX_ERR_UNSUPPORTED and enqueues nothing."""
    import numpy as np

    x = np.zeros((4, 8), np.float32)
    y = np.zeros((4, 8), np.float32)
    vl = np.full(4, 8, np.int32)
    px, py, pv = (ctypes.c_void_p(a.ctypes.data) for a in (x, y, vl))
    f = lib.smx_softmax_rows_host
    assert f(px, py, -1, 8, None, 0, 0, None) == 1
    assert f(px, py, 4, -1, None, 0, 0, None) == 1
    assert f(px, py, 4, 8, None, 5, 0, None) == 1
    assert f(None, py, 4, 8, None, 0, 0, None) == 1
    assert f(px, None, 4, 8, None, 0, 0, None) == 1
    assert f(None, None, 0, 8, None, 0, 0, None) == 0
    assert f(None, None, 4, 0, None, 0, 0, None) == 0
    assert f(px, ctypes.c_void_p(x.ctypes.data + 4), 4, 8, None, 0, 0, None) == 3
    assert f(px, py, 4, 8, ctypes.c_void_p(y.ctypes.data + 8), 0, 0, None) == 3
    st = f(px, py, 4, 8, pv, 0, 0, None)
    assert st in (0, 2)
    if st == 2:
        assert not y.any()  # nothing written without a device


def test_host_buffer_binding_checks_arguments():
    import torch

    import numerically_stable_online_gb300 as smx

    with pytest.raises(ValueError):
        smx.softmax_rows_host(torch.zeros(8))
    with pytest.raises(ValueError):
        smx.softmax_rows_host(torch.zeros(2, 8), out=torch.zeros(2, 8).t())
    with pytest.raises(ValueError):
        smx.softmax_rows_host(torch.zeros(2, 8), valid_len=torch.zeros(2, dtype=torch.int64))
    with pytest.raises(ValueError):
        smx.softmax_rows_host(torch.zeros(2, 8), out=torch.zeros(3, 8))
