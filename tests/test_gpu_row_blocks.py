"""Row blocks: the multi-GPU partition, on one GPU (GPU).

Rows are independent, so several GPUs split a [rows][d] tensor into
contiguous row blocks, one per device, with no exchange (each device gets
the whole gamma/beta or w). These tests run the blocks two ranks would own
as two calls on one device, at the offsets the blocks have inside the whole
tensor, and require y, mean and rstd to equal those of one whole-tensor call
bit for bit: a row's result must not depend on which call, CTA or cluster
computed it, nor on how many rows shared the launch.
"""
import numpy as np
import pytest

import gpu_util as G
import workloads
from row_wise_normalization_gb300 import capi

pytestmark = pytest.mark.gpu

EPS = float(np.float32(1e-5))


def _run(op, variant, x, g, b, y, mean, rstd, rows, d, s):
    if op == "ln":
        return capi.ln_fwd_variant(variant, x, g, b, y, mean, rstd, rows, d, EPS, s)
    return capi.rms_fwd_variant(variant, x, g, y, rows, d, EPS, s)


@pytest.mark.parametrize("op", ["ln", "rms"])
@pytest.mark.parametrize("rows,d,split", [
    (4096, 768, 2048),      # warp per row, even halves
    (8192, 1024, 3001),     # warp per row, uneven blocks
    (1000, 4096, 500),      # CTA per row
    (300, 771, 149),        # unaligned width: rows at every 16-byte phase
    (2048, 32768, 1024),    # 1024-thread rows
    (96, 65536, 40),        # cluster-split rows
    (40, 200000, 17),       # cluster-split, 512-thread CTAs
])
def test_two_row_blocks_equal_the_whole_call(op, rows, d, split):
    torch = G.torch_cuda()
    wl = workloads.Workload(op, rows, d, seed=950, x_dist="offset", x_std=2.0)
    x = G.dev_copy(wl.x())
    ps = wl.params()
    g = G.dev_copy(ps[0])
    b = G.dev_copy(ps[1]) if op == "ln" else (None, 0)
    s = G.stream_handle()

    def outputs():
        return (torch.empty(rows * d, dtype=torch.float32, device="cuda"),
                torch.empty(rows, dtype=torch.float32, device="cuda"),
                torch.empty(rows, dtype=torch.float32, device="cuda"))

    whole = outputs()
    capi.check(_run(op, capi.RN_VARIANT_AUTO, x[1], g[1], b[1], whole[0].data_ptr(),
                    whole[1].data_ptr(), whole[2].data_ptr(), rows, d, s))
    parts = outputs()
    for r0, n in ((0, split), (split, rows - split)):
        capi.check(_run(op, capi.RN_VARIANT_AUTO, x[1] + 4 * r0 * d, g[1], b[1],
                        parts[0].data_ptr() + 4 * r0 * d, parts[1].data_ptr() + 4 * r0,
                        parts[2].data_ptr() + 4 * r0, n, d, s))
    torch.cuda.synchronize()
    names = ("y", "mean", "rstd") if op == "ln" else ("y",)
    for a, c, what in zip(whole, parts, names):
        au = a.cpu().numpy().view(np.uint32)
        cu = c.cpu().numpy().view(np.uint32)
        bad = np.flatnonzero(au != cu)
        assert bad.size == 0, f"{what}: {bad.size} elements differ, first at {bad[0]}"
