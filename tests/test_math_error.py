"""Measured error of the exponential and reciprocal primitives the kernels use,
against fp64 on the host (numpy).

The pages warn that approximate exponential instructions carry an error of
their own ("Stable softmax: keep the normalizer consistent as tiles arrive",
first paragraph; "Online stable softmax", "Masks, empty rows, and precision"),
and the kernels evaluate e^z as 2^(z log2 e) ("Softmax numerics
architecture...", "On CPU, and the pitfalls worth naming").  Each primitive is
evaluated on the GPU through smx_debug_probe_math on dense and stratified
argument sets:

  ex2.approx.ftz.f32   every fp32 in [-1, -0.25) (two binades of the fraction,
                       which decides the error: 2^(k+f) = 2^k 2^f), and 65536
                       fractions in each unit interval of [-126, 0)
  ex2.approx.f32       65536 fractions in each unit interval of [-150, -126)
                       (subnormal results: absolute error in units of 2^-149)
  rcp.approx.ftz.f32   every fp32 in [1, 2), and 2^16 values in each binade up
  and the refined 1/D  to 2^20 (the normaliser D lies in [1, cols])
  compensated e^(x-m)  x - m dense in [-110, 0] for maxima m of either sign and
                       size up to 1e4
  statistics term      the same arguments, the fast form with its row offset

and each maximum error is asserted under a bound a little above the measured
value (printed with -s; the measured figures are the table in the design notes).
"""
import numpy as np
import pytest
import torch

import numerically_stable_online_gb300 as smx

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def lib():
    from numerically_stable_online_gb300 import build

    build.build()
    return smx.library()


def probe(lib, which, a, b=None):
    ta = torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(DEV)
    tb = None if b is None else torch.from_numpy(np.ascontiguousarray(b, np.float32)).to(DEV)
    out = torch.empty_like(ta)
    st = lib.smx_debug_probe_math(ta.data_ptr(), None if tb is None else tb.data_ptr(), out.data_ptr(),
                                  ta.numel(), which, torch.cuda.current_stream().cuda_stream)
    assert st == 0
    return out.cpu().numpy().astype(np.float64)


def floats_between(lo, hi):
    """Every fp32 value v with lo <= v < hi (lo, hi of one sign, |lo| > |hi| for negatives)."""
    a, b = np.float32(lo).view(np.int32), np.float32(hi).view(np.int32)
    lo_b, hi_b = (b + 1, a + 1) if lo < 0 else (a, b)
    return np.arange(min(lo_b, hi_b), max(lo_b, hi_b), dtype=np.int32).view(np.float32)


def stratified(k0, k1, n=65536):
    f = (np.arange(n, dtype=np.float64) + 0.5) / n
    return (np.arange(k0, k1, dtype=np.float64)[:, None] + f[None, :]).astype(np.float32).reshape(-1)


def rel_err(got, want):
    ok = want != 0
    return np.abs(got[ok] - want[ok]) / want[ok]


def report(name, err, unit="relative"):
    m = float(err.max())
    print(f"MATH {name}: max {unit} error {m:.3e} (2^{np.log2(m) if m > 0 else -np.inf:.2f}), "
          f"mean {float(err.mean()):.3e}, n={err.size}")
    return m


def test_ex2_ftz(lib):
    u = np.concatenate([floats_between(-1.0, -0.25), stratified(-126, 0)])
    got = probe(lib, 0, u)
    want = np.exp2(u.astype(np.float64))
    m = report("ex2.approx.ftz.f32 on [-126, 0)", rel_err(got, want))
    assert m <= 2.0 ** -22.5  # measured 1.44e-7 = 2^-22.73
    # flush to zero below 2^-126 (the .ftz form)
    assert np.all(probe(lib, 0, np.float32([-126.5, -130.0, -149.0, -200.0])) == 0)


def test_ex2_subnormal_results(lib):
    u = stratified(-150, -126)
    got = probe(lib, 1, u)
    want = np.exp2(u.astype(np.float64))
    m = report("ex2.approx.f32 on [-150, -126) (subnormal results)", np.abs(got - want) / 2.0 ** -149,
               "absolute (units of 2^-149)")
    # measured 2.21 units: negligible next to the bf16 subnormal spacing 2^-133 = 2^16 units
    assert m <= 3.0


def test_reciprocal(lib):
    d = np.concatenate([floats_between(1.0, 2.0),
                        (2.0 ** np.repeat(np.arange(1, 20), 65536) *
                         np.tile(1 + (np.arange(65536) + 0.5) / 65536, 19)).astype(np.float32)])
    want = 1.0 / d.astype(np.float64)
    m_raw = report("rcp.approx.ftz.f32 on [1, 2^20)", rel_err(probe(lib, 2, d), want))
    got = probe(lib, 3, d)
    m = report("refined reciprocal on [1, 2^20)", rel_err(got, want))
    assert m <= 2.0 ** -23.9  # measured 5.96e-8 = 2^-24.0: half an ulp after the Newton step
    assert m_raw <= 2.0 ** -23  # measured 9.83e-8 = 2^-23.28


def exp_arguments():
    rng = np.random.default_rng(5)
    m = np.concatenate([rng.normal(0, 3, 2000), rng.normal(0, 300, 2000), rng.uniform(-1e4, 1e4, 1000)])
    m = m.astype(np.float32)
    t = -np.linspace(0, 110, 2000)
    x = (m[:, None].astype(np.float64) + t[None, :]).astype(np.float32)
    mm = np.broadcast_to(m[:, None], x.shape)
    return x.reshape(-1), np.ascontiguousarray(mm).reshape(-1)


def test_compensated_exponential(lib):
    x, m = exp_arguments()
    got = probe(lib, 4, x, m)
    want = np.exp(x.astype(np.float64) - m.astype(np.float64))
    big = want >= 2.0 ** -126  # the .ftz exp2 flushes below
    mx = report("compensated e^(x - m), x - m in [-87, 0]", rel_err(got[big], want[big]))
    assert mx <= 2.0 ** -22  # measured 1.80e-7 = 2^-22.40
    assert np.all(got[want < 2.0 ** -126 * 0.5] <= 2.0 ** -125)


def test_statistics_term(lib):
    x, m = exp_arguments()
    d = x.astype(np.float64) - m.astype(np.float64)
    got = probe(lib, 5, x, m)
    want = np.exp(d)
    sel = want >= 2.0 ** -126
    err = rel_err(got[sel], want[sel])
    report("statistics-path term e^(x - m), x - m in [-87, 0]", err)
    # the error grows with |x - m| (the rounded exponent argument); near the
    # maximum, where the terms that make up d lie, it is that of ex2 itself
    near = np.abs(d[sel]) <= 1.0
    mn = report("statistics-path term, |x - m| <= 1", err[near])
    assert mn <= 2.0 ** -22  # measured 2.06e-7 = 2^-22.21
    assert float(err.max()) <= 2.0 ** -17.5  # measured 3.85e-6 = 2^-17.99 (at x - m near -87)
