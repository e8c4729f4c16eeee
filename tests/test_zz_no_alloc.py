"""ln_bwd_noalloc on the GPU, through the C ABI.

ln_bwd_noalloc is the LayerNorm backward for callers that cannot allocate
device memory at the point where they run it -- a process whose caching
allocator already holds nearly all of HBM, a loop that cannot take
cudaFree's device-wide synchronisation, C code with no allocator -- so its
parameter-gradient partials live in one static device array of the library
instead of a caller-owned workspace.

Each case runs it, then ln_bwd (the entry point with a caller-owned
workspace) on the same inputs, and requires the two to agree within the
tolerances of the other backward tests; the results are also checked against
the float64 oracle directly, with the same tolerances. Two calls in a row
with different shapes check that the second call is not disturbed by what
the first left in the shared array. ln_bwd given a workspace of the array's
size runs the same grid, so those results must match bit for bit. The file
sorts last so that it also runs after every other GPU test; it passes alone
in a fresh process too (the first call there does the set-up for the
device's context).
"""
import numpy as np
import pytest

import gpu_util as G
import parity
import workloads
from oracle import reference
from row_wise_normalization_gb300 import capi

pytestmark = pytest.mark.gpu


def _inputs(rows, d, seed):
    wl = workloads.Workload("ln", rows, d, seed=seed, x_dist="offset", x_std=2.0)
    x = wl.x()
    dy = workloads.Workload("ln", rows, d, seed=seed + 1).x()
    g, _ = wl.params()
    _, mean, rstd = reference.layer_norm(x, g, np.zeros_like(g))
    return x, dy, g, mean.astype(np.float32), rstd.astype(np.float32)


def _outputs(rows, d):
    return G.Guarded(rows * d), G.Guarded(d), G.Guarded(d)


def _fetch(outs, rows, d):
    dx, dg, db = outs
    return dx.fetch("dx guard").reshape(rows, d), dg.fetch("dgamma guard"), db.fetch("dbeta guard")


def _call_pair(rows, d, seed):
    torch = G.torch_cuda()
    x, dy, g, m32, r32 = _inputs(rows, d, seed)
    bufs = [G.dev_copy(a) for a in (dy, x, g, m32, r32)]
    ins = [b[1] for b in bufs]
    s = G.stream_handle()

    mine = _outputs(rows, d)
    capi.check(capi.ln_bwd_noalloc(*ins, mine[0].ptr, mine[1].ptr, mine[2].ptr, rows, d, s))

    results = {}
    for name, nbytes in (("full", capi.bwd_workspace_size(capi.RN_OP_LN, rows, d)),
                         ("same_size", capi.RN_NOALLOC_SCRATCH_BYTES)):
        ws = torch.empty(nbytes // 4 + 4, dtype=torch.float32, device="cuda")
        outs = _outputs(rows, d)
        capi.check(capi.ln_bwd(*ins, outs[0].ptr, outs[1].ptr, outs[2].ptr, rows, d,
                               ws.data_ptr(), nbytes, s))
        results[name] = outs
    torch.cuda.synchronize()
    got = _fetch(mine, rows, d)
    full = _fetch(results["full"], rows, d)
    same = _fetch(results["same_size"], rows, d)

    # within the backward tests' tolerances of ln_bwd with its full workspace;
    # both column sums carry rounding, so the summation chain counts twice
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    one = max(4, -(-rows // sms)) + 16   # a row group's rows plus a CTA's groups
    parity.check_y(got[0], full[0], what="dx")
    xhat = (x.astype(np.float64) - m32[:, None]) * r32[:, None]
    terms_g = np.abs(dy * xhat).sum(axis=0)
    terms_b = np.abs(dy.astype(np.float64)).sum(axis=0)
    parity.check_colsum(got[1], full[1], terms_g, 2 * one, "dgamma")
    parity.check_colsum(got[2], full[2], terms_b, 2 * one, "dbeta")
    # and against the float64 oracle itself
    dxr, dgr, dbr = reference.layer_norm_backward(dy, x, g, m32, r32)
    parity.check_y(got[0], dxr, what="dx vs oracle")
    parity.check_colsum(got[1], dgr, terms_g, one, "dgamma vs oracle")
    parity.check_colsum(got[2], dbr, terms_b, one, "dbeta vs oracle")
    # and bit for bit with ln_bwd on a workspace of the static array's size
    for a, b, what in zip(got, same, ("dx", "dgamma", "dbeta")):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32)), what


def test_no_alloc_matches_ln_bwd_on_two_calls_in_a_row():
    _call_pair(3000, 768, seed=201)
    _call_pair(1000, capi.RN_NOALLOC_MAX_D, seed=203)


def test_no_alloc_rejects_rows_wider_than_its_limit():
    torch = G.torch_cuda()
    d = capi.RN_NOALLOC_MAX_D + 1
    rows = 2
    # dy, x, dx [rows][d]; gamma, dgamma, dbeta [d]; mean, rstd [rows]: disjoint
    sizes = [rows * d, rows * d, d, rows, rows, rows * d, d, d]
    buf = torch.zeros(sum(sizes) + 64, device="cuda")
    ptrs, off = [], 0
    for n in sizes:
        ptrs.append(buf.data_ptr() + 4 * off)
        off += -(-n // 4) * 4
    st = capi.ln_bwd_noalloc(*ptrs, rows, d, G.stream_handle())
    assert st == capi.RN_ERR_SCRATCH
    assert "4096" in capi.status_str(st)
    # without parameter gradients no partials are needed: any width runs
    dy, x, g, m32, r32 = _inputs(rows, d, seed=205)
    ins = [G.dev_copy(a) for a in (dy, x, g, m32, r32)]
    dx = G.Guarded(rows * d)
    capi.check(capi.ln_bwd_noalloc(*[b[1] for b in ins], dx.ptr, 0, 0, rows, d,
                                   G.stream_handle()))
    torch.cuda.synchronize()
    dxr, _, _ = reference.layer_norm_backward(dy, x, g, m32, r32)
    parity.check_y(dx.fetch("dx guard").reshape(rows, d), dxr, what="dx")
