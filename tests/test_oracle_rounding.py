"""Pins for the reference's decoding of stored fp16/bf16 values and its
correctly rounded fp64 -> fp16/bf16/fp32 conversion (IEEE 754 binary formats,
round to nearest, ties to even, subnormals kept).

Checked against library routines (numpy's float16, torch's bfloat16, numpy's
float32 cast, which all round straight from their source type) and against the
definition itself by brute force: the result must be a representable neighbour
of v that is at least as close as the codes on either side, with ties going to
the even code.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.filterwarnings("ignore:overflow encountered in cast")


def _random_doubles(rng, n):
    parts = [
        rng.standard_normal(n) * 10.0 ** rng.integers(-12, 6, size=n),
        rng.uniform(-70000, 70000, n),
        np.ldexp(rng.uniform(0.5, 1.0, n), rng.integers(-160, 130, size=n)),
        np.ldexp(rng.uniform(0.5, 1.0, n), rng.integers(-30, 18, size=n)),
    ]
    v = np.concatenate(parts)
    v[::3] *= -1
    return v


def test_decode_f16_every_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.decode(bits, "f16")
    want = bits.view(np.float16).astype(np.float64)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(want[ok]))


def test_decode_bf16_every_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.decode(bits, "bf16")
    want = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(want[ok]))


def test_round_f16_matches_numpy():
    rng = np.random.default_rng(1)
    v = _random_doubles(rng, 50000)
    # exact midpoints between neighbouring fp16 values, including subnormals
    h = rng.integers(0, 0x7BFF, size=20000).astype(np.uint16)
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).astype(np.uint16).view(np.float16).astype(np.float64)
    v = np.concatenate([v, (lo + hi) / 2, -(lo + hi) / 2, [0.0, -0.0, 65504.0, 65520.0,
                                                            65519.99, np.inf, -np.inf]])
    got = oracle.round_to(v, "f16")
    want = v.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, want)


def test_round_bf16_matches_torch_on_fp32_values():
    """torch rounds fp32 -> bf16 to nearest even; on values exactly representable
    in fp32 the reference's direct fp64 -> bf16 must agree."""
    rng = np.random.default_rng(2)
    v32 = _random_doubles(rng, 50000).astype(np.float32)
    b = rng.integers(0, 0x7F7F, size=20000).astype(np.uint16)
    mids = ((b.astype(np.uint32) << 16) | 0x8000).view(np.float32)  # exact midpoints
    v32 = np.concatenate([v32, mids, -mids])
    got = oracle.round_to(v32.astype(np.float64), "bf16")
    want = torch.from_numpy(v32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)


def test_round_f32_matches_numpy():
    rng = np.random.default_rng(3)
    v = _random_doubles(rng, 50000)
    v = np.concatenate([v, np.ldexp(rng.uniform(0.5, 1, 1000), rng.integers(-152, -120, 1000))])
    got = oracle.round_to(v, "f32")
    want = v.astype(np.float32).view(np.uint32)
    assert np.array_equal(got, want)


def _neighbour_check(v, dtype, max_finite_bits):
    r = oracle.round_to(v, dtype).astype(np.int64)
    sign = r & 0x8000
    mag = r & 0x7FFF
    dec = lambda m: oracle.decode(((m & 0x7FFF) | sign).astype(np.uint16), dtype)
    x = dec(mag)
    finite = mag <= max_finite_bits
    assert np.all(finite), "no overflow expected for these inputs"
    down = dec(np.maximum(mag - 1, 0))
    up = dec(np.minimum(mag + 1, max_finite_bits))
    e0 = np.abs(v - x)
    assert np.all(e0 <= np.abs(v - down))
    assert np.all(e0 <= np.abs(v - up))
    tie = (e0 == np.abs(v - down)) & (mag > 0) | (e0 == np.abs(v - up)) & (mag < max_finite_bits)
    tie &= e0 > 0
    assert np.all(mag[tie] % 2 == 0)


def test_round_is_nearest_even_by_brute_force():
    rng = np.random.default_rng(4)
    v16 = _random_doubles(rng, 20000)
    v16 = v16[np.abs(v16) < 65504.0]
    _neighbour_check(v16, "f16", 0x7BFF)
    vbf = _random_doubles(rng, 20000)
    vbf = vbf[np.abs(vbf) < 3.3e38]
    _neighbour_check(vbf, "bf16", 0x7F7F)
    # exact midpoints go to the even neighbour
    h = np.arange(0, 0x7BFF, dtype=np.uint16)
    mid = (h.view(np.float16).astype(np.float64) + (h + 1).astype(np.uint16).view(np.float16).astype(np.float64)) / 2
    r = oracle.round_to(mid, "f16").astype(np.int64)
    assert np.all(r % 2 == 0) and np.all((r == h) | (r == h + 1))
