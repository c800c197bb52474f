"""The seeded inputs follow their stated recipes, and the byte and FLOP counts
the measurements divide by are the ones the traffic account fixes.

Recipes (numerically_stable_online_gb300/workloads.py): shapes, distributions
(moments of a large sample), the one +30.0 per row, the 1% of empty rows and
the length range, the rising row, the causal lengths; the draw is
deterministic.  Counts: the algorithmic bytes of each workload (valid input
read once, every output written once, lengths once), checked against the
figures worked out from the shapes by hand, and the attention pair and FLOP
counts against brute force.
"""
import numpy as np
import pytest
import torch

from numerically_stable_online_gb300 import workloads as wl


def values(name, rows=None):
    x, vl = wl.host_input(name, rows=rows)
    w = wl.WORKLOADS[name]
    t = wl.storage_to_torch(x, w.in_dtype).to(torch.float64).numpy()
    return t.reshape(-1 if rows is None else rows, w.cols), vl


def test_draw_is_deterministic():
    for name in ("f32_64x1000", "f16_32768x1024_len"):
        a, va = wl.host_input(name, rows=300)
        b, vb = wl.host_input(name, rows=300)
        assert np.array_equal(a, b)
        assert (va is None and vb is None) or np.array_equal(va, vb)


def test_f32_64x1000_recipe():
    x, vl = values("f32_64x1000")
    assert x.shape == (64, 1000) and vl is None
    assert np.all((x == 30.0).sum(axis=1) == 1)
    assert np.all(x.max(axis=1) == 30.0)
    rest = x[x != 30.0]
    assert abs(rest.mean()) < 0.05 and 2.95 < rest.std() < 3.05


def test_bf16_16384x4096_recipe():
    x, vl = values("bf16_16384x4096", rows=512)
    assert vl is None and x.shape == (512, 4096)
    assert abs(x.mean()) < 0.05 and 7.95 < x.std() < 8.05
    # every value is a bf16: its low 16 float32 bits are zero
    assert np.all(x.astype(np.float32).view(np.uint32) & 0xFFFF == 0)


def test_f16_32768x1024_len_recipe():
    x, vl = wl.host_input("f16_32768x1024_len")
    assert vl.dtype == np.int32 and vl.shape == (32768,)
    assert vl.min() == 0 and vl.max() <= 1024
    # 328 rows forced empty, plus the few the uniform lengths make 0 themselves
    n0 = int((vl == 0).sum())
    assert 328 <= n0 <= 328 + 80
    nonempty = vl[vl > 0]
    assert abs(nonempty.mean() - 512.5) < 10
    v = wl.storage_to_torch(x[: 64 * 1024], "f16").to(torch.float64).numpy()
    assert v.min() >= -30.0 and v.max() <= 30.0 and abs(v.std() - 60 / 12 ** 0.5) < 0.2  # U[-30, 30]


def test_f32_rising_row_recipe():
    x, vl = values("f32_64x1048576_rise", rows=2)
    assert vl is None
    ramp = 20.0 * np.arange(x.shape[1]) / x.shape[1]
    noise = x - ramp[None, :]
    assert abs(noise.mean()) < 0.01 and 0.99 < noise.std() < 1.01
    # the running maximum keeps rising: the row's maximum sits in its last tenth
    assert np.all(x.argmax(axis=1) > 0.9 * x.shape[1])
    spread = (x - x.max(axis=1, keepdims=True)).min(axis=1)
    assert np.all((spread < -24.0) & (spread > -32.0))


def test_causal_lengths():
    vl = wl.causal_valid_len(3 * 4096)
    assert vl[0] == 1 and vl[4095] == 4096 and vl[4096] == 1 and vl[-1] == 4096
    assert int(vl[:4096].sum()) == 4096 * 4097 // 2


@pytest.mark.parametrize("name,expected", [
    ("f32_64x1000", 512_000),                        # 64 x 1000 x (4 + 4)
    ("bf16_16384x4096", 268_435_456),                # 16384 x 4096 x (2 + 2)
    ("f32_64x1048576_rise", 536_870_912),            # 64 x 2^20 x (4 + 4)
])
def test_algorithmic_bytes_of_the_dense_workloads(name, expected):
    w = wl.WORKLOADS[name]
    es = {"f32": 4, "f16": 2, "bf16": 2}
    assert wl.algorithmic_bytes(w.rows, w.cols, es[w.in_dtype], es[w.out_dtype]) == expected
    assert wl.op_bytes("softmax", w.rows, w.cols, es[w.in_dtype], es[w.out_dtype]) == expected


def test_algorithmic_bytes_with_lengths():
    _, vl = wl.host_input("f16_32768x1024_len")
    expected = 2 * int(vl.sum()) + 32768 * 1024 * 2 + 32768 * 4
    assert wl.algorithmic_bytes(32768, 1024, 2, 2, vl) == expected
    assert wl.op_bytes("softmax", 32768, 1024, 2, 2, vl) == expected
    assert 95e6 < expected < 106e6                   # about 100.5 MB
    # lengths past the row are clamped, negative ones count as 0
    assert wl.algorithmic_bytes(2, 8, 4, 4, [100, -3]) == 8 * 4 + 2 * 4 + 2 * 8 * 4
    # the causal batch: 256 slices of 4096 rows, row i valid for i + 1 columns
    vl = wl.causal_valid_len(1_048_576)
    b = wl.algorithmic_bytes(1_048_576, 4096, 2, 2, vl)
    assert b == 2 * 256 * (4096 * 4097 // 2) + 1_048_576 * 4096 * 2 + 1_048_576 * 4
    assert abs(b - 12.89e9) < 0.01e9


def test_op_bytes_of_the_other_operations():
    r, c = 16384, 4096
    dense = r * c * 2
    assert wl.op_bytes("log_softmax", r, c, 2, 2) == 2 * dense
    assert wl.op_bytes("lse", r, c, 2, 4) == dense + r * 4
    assert wl.op_bytes("apply_stats", r, c, 2, 2) == 2 * dense + r * 8
    assert wl.op_bytes("backward", r, c, 2, 2) == 3 * dense
    assert wl.op_bytes("cross_entropy", r, c, 2, 2) == 2 * dense + r * 12
    with pytest.raises(ValueError):
        wl.op_bytes("attention", r, c, 2, 2)


@pytest.mark.parametrize("sq,sk", [(5, 5), (3, 7), (7, 3), (1, 4), (4, 1), (0, 3)])
def test_attention_pairs_brute_force(sq, sk):
    full = sum(1 for i in range(sq) for j in range(sk))
    causal = sum(1 for i in range(sq) for j in range(sk) if j <= i + sk - sq)
    assert wl.attention_pairs(sq, sk, False) == full
    assert wl.attention_pairs(sq, sk, True) == causal


def test_attention_flops_of_the_workloads():
    assert wl.attention_flops(128, 4096, 4096, 128, False) == 4.0 * 128 * 128 * 4096 * 4096
    assert abs(wl.attention_flops(128, 4096, 4096, 128, False) - 1.0995e12) < 1e8
    assert wl.attention_flops(128, 4096, 4096, 128, True) == 4.0 * 128 * 128 * (4096 * 4097 // 2)
    assert abs(wl.attention_flops(128, 4096, 4096, 128, True) - 5.499e11) < 1e8
