"""The library allocates nothing per call in a steady loop.

Its scratch (long-row summaries and counters, the staged host call's device
slots) lives in per-device buffers that grow only when a call needs more than
any call before; the host call's events and copy stream are created once.
smx_debug_alloc_count() counts every device allocation, event and stream the
library creates.  After one warm-up call of each kind, 100 more rounds of the
same calls must leave it unchanged: the long-row workload's softmax (read
once), log_softmax and cross-entropy with a gradient, its LSE and row
statistics (chunk summaries), the backward of long rows (two passes over
chunks), the two-launch chunked path forced, and the host-buffer call staged
through device slots.  One more call with more rows than ever grows the
scratch (the count moves), and the loop after it is steady again.
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


@pytest.fixture(scope="module")
def lib():
    from numerically_stable_online_gb300 import build

    build.build()
    oracle.build()
    lib = smx.library()
    yield lib
    lib.smx_debug_force_path(0)


def test_steady_loop_allocates_nothing(lib):
    name = "f32_64x1048576_rise"
    w = wl.WORKLOADS[name]
    rows, cols = w.rows, w.cols
    x_host, _ = wl.host_input(name)
    x = torch.from_numpy(x_host.reshape(rows, cols)).to(DEV)
    y = torch.empty_like(x)
    g = torch.randn(8, cols, device=DEV)
    dx = torch.empty_like(g)
    t = torch.from_numpy(np.random.default_rng(4).integers(0, cols, rows)).to(DEV)
    loss = torch.empty(rows, device=DEV)
    lse = torch.empty(rows, device=DEV)
    m = torch.empty(rows, device=DEV)
    d = torch.empty(rows, device=DEV)
    hx = torch.randn(4, 262_144).pin_memory()
    hy = torch.empty_like(hx).pin_memory()
    lib.smx_debug_set_host_chunk(1 << 20, 0, 1)  # staged, several chunks a call

    def softmax_forced_split():
        lib.smx_debug_force_path(5)
        smx.softmax_rows(x[:8], out=y[:8])
        lib.smx_debug_force_path(0)

    calls = [
        lambda: smx.softmax_rows(x, out=y),
        lambda: smx.log_softmax_rows(x, out=y),
        lambda: smx.cross_entropy(x, t, grad=y, loss=loss),
        lambda: smx.softmax_lse(x, out=lse),
        lambda: smx.softmax_row_stats(x, m_out=m, d_out=d),
        lambda: smx.softmax_backward(y[:8], g, out=dx),
        softmax_forced_split,
        lambda: smx.softmax_rows_host(hx, out=hy, wait=False),
    ]
    try:
        for c in calls:
            c()
        torch.cuda.synchronize()
        before = lib.smx_debug_alloc_count()
        assert before > 0
        for _ in range(100):
            for c in calls:
                c()
        torch.cuda.synchronize()
        assert lib.smx_debug_alloc_count() == before
        assert smx.last_device_status() == 0
        # the results of the last round are still right
        smx.softmax_rows(x[:4], out=y[:4])
        p = oracle.softmax_rows(x_host[: 4 * cols], "f32", 4, cols)
        parity.compare(y[:4].cpu().numpy(), p, "f32")
        ph = oracle.softmax_rows(hx.numpy().reshape(-1), "f32", 4, 262_144)
        parity.compare(hy.numpy(), ph, "f32")
        # a call with more long rows than any before grows the scratch once
        # (160 rows of 4 MiB: 160 x 152 stripe summaries, more than any
        # buffer so far holds)
        x2 = torch.randn(160, cols, device=DEV)
        y2 = torch.empty_like(x2)
        smx.softmax_rows(x2, out=y2)
        torch.cuda.synchronize()
        grown = lib.smx_debug_alloc_count()
        assert grown > before
        for _ in range(20):
            smx.softmax_rows(x2, out=y2)
            smx.softmax_rows(x, out=y)
        torch.cuda.synchronize()
        assert lib.smx_debug_alloc_count() == grown
    finally:
        lib.smx_debug_set_host_chunk(0, 0, 0)
        lib.smx_debug_force_path(0)
