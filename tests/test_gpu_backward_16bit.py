"""LayerNorm / RMSNorm backward with BF16 / FP16 storage against the oracle.

The oracle differentiates the same function on the widened (exact FP32)
values of the 16-bit inputs, from the same saved FP32 statistics. dx is
rounded once to the storage type, so it follows the 16-bit element rule of
tests/parity.py; the parameter gradients are FP32 sums over rows rounded
once at the end, so they follow the recursive-summation bound of
check_colsum plus one unit in the last place of the storage type.
"""
import numpy as np
import pytest

import gpu_util as G
import parity
import workloads
from oracle import reference
from row_wise_normalization_gb300 import capi

pytestmark = pytest.mark.gpu

LN, RMS = capi.RN_OP_LN, capi.RN_OP_RMS
CODE = {"bf16": capi.RN_DTYPE_BF16, "f16": capi.RN_DTYPE_F16}


def _ulp(v, dtype):
    mant = 7 if dtype == "bf16" else 10
    a = np.maximum(np.abs(np.asarray(v, np.float64)), 2.0 ** -14)
    return 2.0 ** (np.floor(np.log2(a)) - mant)


def _check_grad(got_bits, ref, abs_terms, chain, dtype, what):
    got = workloads.from_storage(got_bits, dtype).astype(np.float64)
    lim = ((chain + 4) * parity.U32 * np.asarray(abs_terms) + 1e-4 * np.abs(ref) + 1e-7
           + _ulp(ref, dtype))
    bad = ~(np.abs(got - ref) <= lim)
    if bad.any():
        i = int(np.nonzero(bad)[0][0])
        raise parity.ParityError(f"{what}: {int(bad.sum())} columns out of tolerance; first {i}: "
                                 f"got {got[i]!r}, want {ref[i]!r} (limit {lim[i]:.3e})")


def _inputs(rows, d, dtype, seed, dist):
    wl = workloads.Workload("ln", rows, d, seed=seed, x_dist=dist, x_std=2.0)
    xb, xw = workloads.to_storage(wl.x(), dtype)
    dyb, dyw = workloads.to_storage(workloads.Workload("ln", rows, d, seed=seed + 1).x(), dtype)
    g, b = wl.params()
    gb, gw = workloads.to_storage(g, dtype)
    _, bw = workloads.to_storage(b, dtype)
    return xb, xw, dyb, dyw, gb, gw, bw


def _run(op, dtype, xb, dyb, gb, m32, r32, off=0, ws_bytes=None, grads=True):
    torch = G.torch_cuda()
    rows, d = xb.shape
    bufs = [G.dev_copy16(a, off) for a in (dyb, xb, gb)]
    stats = [G.dev_copy(a) for a in (m32, r32)] if op == LN else None
    dx = G.Guarded16(rows * d, off)
    g0 = G.Guarded16(d) if grads else None
    g1 = G.Guarded16(d) if (grads and op == LN) else None
    need = capi.bwd_workspace_size(op, rows, d) if ws_bytes is None else ws_bytes
    ws = torch.empty(max(need // 4, 4), dtype=torch.float32, device="cuda")
    s = G.stream_handle()
    if op == LN:
        st = capi.ln_bwd_typed(CODE[dtype], bufs[0][1], bufs[1][1], bufs[2][1], stats[0][1],
                               stats[1][1], dx.ptr, g0.ptr if g0 else 0, g1.ptr if g1 else 0,
                               rows, d, ws.data_ptr() if grads else 0, need if grads else 0, s)
    else:
        st = capi.rms_bwd_typed(CODE[dtype], bufs[0][1], bufs[1][1], bufs[2][1], dx.ptr,
                                g0.ptr if g0 else 0, rows, d, float(np.float32(1e-5)),
                                ws.data_ptr() if grads else 0, need if grads else 0, s)
    capi.check(st)
    torch.cuda.synchronize()
    return (dx.fetch("dx guard").reshape(rows, d), g0.fetch("grad guard") if g0 else None,
            g1.fetch("grad guard") if g1 else None)


def _check(op, dtype, xw, dyw, gw, bw, out, chain):
    dx, g0, g1 = out
    if op == LN:
        _, mean, rstd = reference.layer_norm(xw, gw, bw)
        m32, r32 = mean.astype(np.float32), rstd.astype(np.float32)
        dxr, dgr, dbr = reference.layer_norm_backward(dyw, xw, gw, m32, r32)
        parity.check_y_storage(dx, dxr, dtype, what="dx")
        if g0 is not None:
            xhat = (xw.astype(np.float64) - m32[:, None]) * r32[:, None]
            _check_grad(g0, dgr, np.abs(dyw * xhat).sum(axis=0), chain, dtype, "dgamma")
            _check_grad(g1, dbr, np.abs(dyw.astype(np.float64)).sum(axis=0), chain, dtype,
                        "dbeta")
    else:
        dxr, dwr = reference.rms_norm_backward(dyw, xw, gw)
        parity.check_y_storage(dx, dxr, dtype, what="dx")
        if g0 is not None:
            _, r = reference.rms_norm(xw, gw)
            terms = np.abs(dyw.astype(np.float64) * xw * r[:, None]).sum(axis=0)
            _check_grad(g0, dwr, terms, chain, dtype, "dw")


def _stats(xw, gw, bw):
    _, mean, rstd = reference.layer_norm(xw, gw, bw)
    return mean.astype(np.float32), rstd.astype(np.float32)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("op", [LN, RMS])
@pytest.mark.parametrize("d,off", [(1, 0), (33, 1), (768, 0), (768, 1), (1000, 0), (1000, 3),
                                   (4096, 0), (8192, 2), (12288, 0), (16384, 0)])
def test_backward_16bit(dtype, op, d, off):
    rows = 300 if d <= 4096 else 61
    dist = "offset" if dtype == "bf16" else "normal"
    xb, xw, dyb, dyw, gb, gw, bw = _inputs(rows, d, dtype, 811, dist)
    m32, r32 = _stats(xw, gw, bw)
    out = _run(op, dtype, xb, dyb, gb, m32, r32, off=off)
    _check(op, dtype, xw, dyw, gw, bw, out, chain=max(4, -(-rows // 152)) + 16)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_backward_16bit_small_workspace_and_no_grads(dtype):
    rows, d = 700, 512
    xb, xw, dyb, dyw, gb, gw, bw = _inputs(rows, d, dtype, 813, "normal")
    m32, r32 = _stats(xw, gw, bw)
    out = _run(LN, dtype, xb, dyb, gb, m32, r32, ws_bytes=2 * d * 4)   # one partial row
    _check(LN, dtype, xw, dyw, gw, bw, out, chain=rows + 16)
    out = _run(RMS, dtype, xb, dyb, gb, m32, r32, grads=False)
    _check(RMS, dtype, xw, dyw, gw, bw, out, chain=0)


def test_backward_16bit_torch_binding_against_autograd():
    torch = G.torch_cuda()
    import row_wise_normalization_gb300 as rn

    rows, d = 400, 1024
    for dt in (torch.bfloat16, torch.float16):
        wl = workloads.Workload("ln", rows, d, seed=815)
        x = torch.from_numpy(wl.x()).to("cuda").to(dt)
        dy = torch.from_numpy(workloads.Workload("ln", rows, d, seed=816).x()).to("cuda").to(dt)
        g, b = (torch.from_numpy(p_).to("cuda").to(dt) for p_ in wl.params())
        _, mean, rstd = rn.ln_fwd(x, g, b)
        dx, dg, db = rn.ln_bwd(dy, x, g, mean, rstd)
        assert dx.dtype == dg.dtype == db.dtype == dt
        xr, gr, br = (t.double().requires_grad_() for t in (x, g, b))
        torch.nn.functional.layer_norm(xr, [d], gr, br, 1e-5).backward(dy.double())
        tol = 1e-2 if dt == torch.bfloat16 else 2e-3
        np.testing.assert_allclose(dx.double().cpu().numpy(), xr.grad.cpu().numpy(),
                                   rtol=tol, atol=tol)
        np.testing.assert_allclose(dg.double().cpu().numpy(), gr.grad.cpu().numpy(),
                                   rtol=tol, atol=tol * 10)
        np.testing.assert_allclose(db.double().cpu().numpy(), br.grad.cpu().numpy(),
                                   rtol=tol, atol=tol * 10)
        dxq, dwq = rn.rms_bwd(dy, x, g)
        xr, wr = (t.double().requires_grad_() for t in (x, g))
        torch.nn.functional.rms_norm(xr, [d], wr, 1e-5).backward(dy.double())
        np.testing.assert_allclose(dxq.double().cpu().numpy(), xr.grad.cpu().numpy(),
                                   rtol=tol, atol=tol)
        np.testing.assert_allclose(dwq.double().cpu().numpy(), wr.grad.cpu().numpy(),
                                   rtol=tol, atol=tol * 10)


def test_backward_16bit_rejects_unknown_type_and_misalignment():
    torch = G.torch_cuda()
    buf = torch.zeros(4096, dtype=torch.int16, device="cuda")
    p = buf.data_ptr()
    stats = torch.zeros(64, device="cuda").data_ptr()
    assert capi.ln_bwd_typed(5, p, p + 1024, p + 2048, stats, stats + 64, p + 4096, 0, 0, 4, 8,
                             0, 0, 0) == capi.RN_ERR_DTYPE
    assert capi.ln_bwd_typed(capi.RN_DTYPE_BF16, p + 1, p + 1024, p + 2048, stats, stats + 64,
                             p + 4096, 0, 0, 4, 8, 0, 0, 0) == capi.RN_ERR_ALIGN


# Rows of 256 or 512 threads on the vector layout run the staged backward
# (x and dy rows brought into a shared-memory ring by bulk copies). Widths on
# both thread counts, single rows, ragged row counts, and a one-CTA grid
# (workspace of one partial row) whose ring wraps hundreds of times.
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("op", [LN, RMS])
@pytest.mark.parametrize("d", [2056, 4096, 4104, 8192])
@pytest.mark.parametrize("rows", [1, 7, 1531])
def test_backward_16bit_staged_rows(dtype, op, d, rows):
    xb, xw, dyb, dyw, gb, gw, bw = _inputs(rows, d, dtype, 817, "offset")
    m32, r32 = _stats(xw, gw, bw)
    capi.device_error(clear=True)
    out = _run(op, dtype, xb, dyb, gb, m32, r32)
    _check(op, dtype, xw, dyw, gw, bw, out, chain=max(4, -(-rows // 152)) + 16)
    assert capi.device_error() == 0


@pytest.mark.parametrize("op", [LN, RMS])
@pytest.mark.parametrize("d", [4096, 8192])
def test_backward_16bit_staged_one_cta_and_no_grads(op, d):
    rows = 613
    xb, xw, dyb, dyw, gb, gw, bw = _inputs(rows, d, "bf16", 819, "normal")
    m32, r32 = _stats(xw, gw, bw)
    width = 2 * d if op == LN else d
    out = _run(op, "bf16", xb, dyb, gb, m32, r32, ws_bytes=width * 4)   # one CTA
    _check(op, "bf16", xw, dyw, gw, bw, out, chain=rows + 16)
    out = _run(op, "bf16", xb, dyb, gb, m32, r32, grads=False)
    _check(op, "bf16", xw, dyw, gw, bw, out, chain=0)
    assert capi.device_error() == 0


# 16-bit rows of 64 or 128 threads run the staged backward when every CTA
# walks at least 8 rows (one CTA per row group there): calls large enough
# to take that path, LayerNorm and RMSNorm, both thread counts.
@pytest.mark.parametrize("dtype,op,d,rows", [("bf16", LN, 1536, 5000), ("bf16", LN, 1024, 10000),
                                             ("f16", RMS, 1536, 10000),
                                             ("bf16", RMS, 520, 20000)])
def test_backward_16bit_staged_narrow_rows(dtype, op, d, rows):
    xb, xw, dyb, dyw, gb, gw, bw = _inputs(rows, d, dtype, 821, "offset")
    m32, r32 = _stats(xw, gw, bw)
    capi.device_error(clear=True)
    out = _run(op, dtype, xb, dyb, gb, m32, r32)
    _check(op, dtype, xw, dyw, gw, bw, out, chain=max(4, -(-rows // 152)) + 16)
    assert capi.device_error() == 0


# 16-bit RMSNorm rows of 1024 threads (8193-16384 wide) run staged too, with
# the parameters in shared memory ahead of a 2-4 stage ring: several rows per
# CTA, and a one-CTA grid whose ring wraps once per row.
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("d", [12288, 16384])
def test_backward_16bit_staged_wide_rms(dtype, d):
    rows = 500
    xb, xw, dyb, dyw, gb, gw, bw = _inputs(rows, d, dtype, 823, "offset")
    m32, r32 = _stats(xw, gw, bw)
    capi.device_error(clear=True)
    out = _run(RMS, dtype, xb, dyb, gb, m32, r32)
    _check(RMS, dtype, xw, dyw, gw, bw, out, chain=max(4, -(-rows // 152)) + 16)
    out = _run(RMS, dtype, xb, dyb, gb, m32, r32, ws_bytes=d * 4)   # one CTA
    _check(RMS, dtype, xw, dyw, gw, bw, out, chain=rows + 16)
    assert capi.device_error() == 0
