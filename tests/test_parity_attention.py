"""Parity of the attention forward (CUDA path through the C ABI) with the fp64
reference of tests/test_oracle_attention.py.

Tolerance, from the arithmetic: scores are fp32 dot products of exact 16-bit
products (error at most 2^-16 of the largest |s| computed from |q|.|k|, the
reference's `smax`); the probabilities enter the second product rounded to the
input type (relative 2^-9 for bf16, 2^-12 for fp16), so an output element is
off by at most 2^-8 sum_j p_j |v_j| (the reference's `oabs`) plus the score
error carried through the same weights, plus the rounding of the output:
    |o - ref| <= (2^-8 + smax 2^-15) oabs + spacing(ref) + 2^-24.
LSE (fp32): |lse - ref| <= 2^-16 (|ref| + smax) + 2^-18.  Empty rows: o = +0 and
lse = -inf exactly.

Every case runs on both kernels (tcgen05/TMEM, and mma.sync).  Cases:
head_dim 64 and 128; bf16 and fp16; causal and not; query and key
counts that are not multiples of the 64-row blocks; more queries than keys
under the causal mask (empty rows); no keys at all; large scores; and the
4 x 32 heads x 4096 x 128 shape of the pages' attention example on sampled
rows.
"""
import numpy as np
import pytest
import torch

import numerically_stable_online_gb300 as smx
import oracle
from numerically_stable_online_gb300 import workloads as wl
from tests import parity

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
DT = {"bf16": torch.bfloat16, "f16": torch.float16}


@pytest.fixture(scope="module", autouse=True)
def built():
    from numerically_stable_online_gb300 import build

    build.build()
    oracle.build()
    yield smx.library()


KERNELS = {"auto": -1, "tile": 0, "tma": 1, "mma_sync": 2, "tma2": 3}


@pytest.fixture(autouse=True, params=list(KERNELS))
def kernel(request, built):
    """Every case on the default choice and on each of the four kernels:
    tcgen05 with operands copied by the row threads, tcgen05 with operands
    fetched by tensor-map copies in their own warps (persistent CTAs of one
    or two query tiles), and mma.sync."""
    built.smx_debug_set_attention_kernel(KERNELS[request.param])
    yield request.param
    built.smx_debug_set_attention_kernel(-1)
    assert smx.last_device_status() == 0


def check(o_dev, lse_dev, q, k, v, dt, heads, sq, sk, d, scale, causal, rows_sel=None):
    qs = wl.torch_to_storage(q.cpu()).reshape(-1)
    ks = wl.torch_to_storage(k.cpu()).reshape(-1)
    vs = wl.torch_to_storage(v.cpu()).reshape(-1)
    ref, ref_lse, oabs, smax = oracle.attention_rows(qs, ks, vs, dt, heads, sq, sk, d, scale, causal,
                                                     rows_sel=rows_sel)
    o_rows = o_dev.reshape(heads * sq, d)
    l_rows = lse_dev.reshape(heads * sq)
    if rows_sel is not None:
        sel = torch.from_numpy(np.asarray(rows_sel)).to(o_dev.device)
        o_rows, l_rows = o_rows[sel], l_rows[sel]
    ov = oracle.decode(wl.torch_to_storage(o_rows.cpu()).reshape(-1), dt).reshape(ref.shape)
    lv = l_rows.cpu().double().numpy()
    empty = np.isneginf(ref_lse)
    assert np.all(ov[empty] == 0.0) and np.all(np.isneginf(lv[empty])), "empty rows"
    ok = ~empty
    tol = (2.0 ** -8 + smax[:, None] * 2.0 ** -15) * oabs + parity.format_spacing(ref, dt) + 2.0 ** -24
    err = np.abs(ov - ref)[ok]
    worst = float((err / tol[ok]).max()) if ok.any() else 0.0
    assert worst <= 1.0, f"attention output error {worst:.3f} x tolerance"
    ltol = 2.0 ** -16 * (np.abs(ref_lse[ok]) + smax[ok]) + 2.0 ** -18
    lworst = float((np.abs(lv[ok] - ref_lse[ok]) / ltol).max()) if ok.any() else 0.0
    assert lworst <= 1.0, f"LSE error {lworst:.3f} x tolerance"
    return worst, lworst


def run(heads, sq, sk, d, causal, dt, seed, qscale=1.0):
    g = torch.Generator(device=DEV).manual_seed(seed)
    q = (torch.randn(heads, sq, d, generator=g, device=DEV) * qscale).to(DT[dt])
    k = torch.randn(heads, sk, d, generator=g, device=DEV).to(DT[dt])
    v = torch.randn(heads, sk, d, generator=g, device=DEV).to(DT[dt])
    scale = d ** -0.5
    o, lse = smx.attention_forward(q, k, v, scale=scale, causal=causal)
    assert smx.library().smx_debug_last_launches() == 1
    return check(o, lse, q, k, v, dt, heads, sq, sk, d, scale, causal)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("causal", [False, True])
# (300, 100) causal: the first 128-row tile sees no key while the second does;
# (257, 64): a CTA whose second tile is wholly past the queries; (520, 1000):
# more key blocks than stages, a ragged last block and a ragged last tile
@pytest.mark.parametrize("sq,sk", [(64, 64), (70, 70), (130, 200), (200, 130), (1, 1), (1, 300), (257, 64),
                                   (300, 100), (520, 1000)])
def test_attention_shapes(d, dt, causal, sq, sk):
    w = run(3, sq, sk, d, causal, dt, seed=sq * 1000 + sk)
    print(d, dt, causal, sq, sk, w)


@pytest.mark.parametrize("qscale", [8.0, 40.0])
def test_attention_large_scores(qscale):
    # scores of tens to hundreds: the exponent must be taken against the maximum
    run(2, 96, 160, 128, False, "bf16", seed=7, qscale=qscale)
    run(2, 96, 160, 64, True, "f16", seed=8, qscale=qscale)


def test_attention_no_keys():
    q = torch.randn(2, 10, 64, device=DEV).to(torch.bfloat16)
    e = torch.empty(2, 0, 64, device=DEV, dtype=torch.bfloat16)
    o, lse = smx.attention_forward(q, e, e)
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))


@pytest.mark.parametrize("causal", [False, True])
def test_attention_pages_shape_sampled(causal):
    """4 x 32 heads, 4096 queries and keys, head_dim 128 (the pages' N = 4096
    attention example), bf16; 3 heads x 48 rows against the reference."""
    heads, n, d = 128, 4096, 128
    g = torch.Generator(device=DEV).manual_seed(11 + causal)
    q = torch.randn(heads, n, d, generator=g, device=DEV).to(torch.bfloat16)
    k = torch.randn(heads, n, d, generator=g, device=DEV).to(torch.bfloat16)
    v = torch.randn(heads, n, d, generator=g, device=DEV).to(torch.bfloat16)
    o, lse = smx.attention_forward(q, k, v, causal=causal)
    rng = np.random.default_rng(12)
    hs = [0, 77, 127]
    rows = np.concatenate([h * n + np.sort(rng.choice(n, 48, replace=False)) for h in hs])
    rows = np.concatenate([rows, [0, n - 1, 64 * n + 63, 64 * n + 64]])
    # the reference over only the sampled heads
    sub = torch.tensor(sorted(set(hs + [64])), device=DEV)
    remap = {int(h): i for i, h in enumerate(sub.tolist())}
    sel = np.array([remap[int(r // n)] * n + int(r % n) for r in rows])
    check(o[sub], lse[sub], q[sub], k[sub], v[sub], "bf16", len(sub), n, n, d, d ** -0.5, causal,
          rows_sel=sel)


def test_attention_timeout_reported_and_context_usable(kernel):
    """The error path of the tcgen05 kernels: with a negative wait limit one
    thread per CTA waits on a barrier that nothing signals, the wait runs out
    and SMX_ERR_TIMEOUT is recorded; every other wait of the launch then stops
    early (its output is not meaningful), the kernel still lets its own
    products finish before it frees tensor memory, and the next call on the
    same context is correct and clean."""
    if kernel == "mma_sync":
        pytest.skip("the probe is in the tcgen05 kernels")
    lib = smx.library()
    g = torch.Generator(device=DEV).manual_seed(93)
    q, k, v = (torch.randn(4, n, 128, generator=g, device=DEV).to(torch.bfloat16) for n in (256, 320, 320))
    lib.smx_debug_set_wait_limit(-2000)
    try:
        smx.attention_forward(q, k, v, causal=True)
        torch.cuda.synchronize()
    finally:
        lib.smx_debug_set_wait_limit(0)
    assert smx.last_device_status() == 5  # SMX_ERR_TIMEOUT
    run(3, 200, 260, 128, True, "bf16", seed=94)
    assert smx.last_device_status() == 0
