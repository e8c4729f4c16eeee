"""Strided rows (ln_fwd_strided / rms_fwd_strided) against the oracle (GPU).

x lives in a wider matrix (row stride ldx >= d) whose gap elements hold NaN,
so that a kernel reading outside its rows poisons the statistics; y is written
into a matrix of row stride ldy whose gaps hold a sentinel, and every gap and
guard element must come back untouched. Each strided call runs through every
variant that accepts its phases (plus AUTO); values follow the forward
tolerances of tests/parity.py.
"""
import numpy as np
import pytest

import gpu_util as G
import parity
import workloads
from oracle import reference
from row_wise_normalization_gb300 import capi

pytestmark = pytest.mark.gpu

F32, BF16 = capi.RN_DTYPE_F32, capi.RN_DTYPE_BF16
NAN32 = np.uint32(0x7FC00000)
NAN16 = np.uint16(0x7FC0)


def _variants(dtype, op, d, ldx, ldy, x_off, y_off):
    es = 4 if dtype == F32 else 2
    xa, ya = (1 << 20) + es * x_off, (1 << 30) + es * y_off
    out = [capi.RN_VARIANT_AUTO]
    for v in range(1, capi.RN_VARIANT_COUNT):
        try:
            capi.plan_strided(dtype, op, v, d, xa, ldx, ya, ldy)
        except capi.RowNormError:
            continue
        out.append(v)
    return out


def _run(op, dtype, x, params, ldx, ldy, variant, x_off=0, y_off=0):
    """One strided call; returns (y rows as FP32 values or 16-bit patterns,
    mean, rstd) after checking gaps and guards."""
    torch = G.torch_cuda()
    rows, d = x.shape
    if dtype == F32:
        xs = np.full((rows, ldx), NAN32, np.uint32).view(np.float32)
        xs[:, :d] = x
        xflat, yfill, tdt = xs.reshape(-1).view(np.int32), parity.SENTINEL_BITS, torch.int32
        pvals = [np.ascontiguousarray(p, np.float32).view(np.int32) for p in params]
    else:
        xb, _ = workloads.to_storage(x, "bf16")
        xs = np.full((rows, ldx), NAN16, np.uint16)
        xs[:, :d] = xb
        xflat, yfill, tdt = xs.reshape(-1).view(np.int16), 0x7FC1, torch.int16
        pvals = [workloads.to_storage(p, "bf16")[0].view(np.int16) for p in params]
    xbuf = torch.zeros(xflat.size + x_off + 16, dtype=tdt, device="cuda")
    xbuf[x_off:x_off + xflat.size].copy_(torch.from_numpy(xflat.copy()))
    pbufs = [torch.from_numpy(p.copy()).to("cuda") for p in pvals]
    ny = (rows - 1) * ldy + d if rows else 0
    head = parity.GUARD + y_off
    fill = np.array([yfill], np.uint32 if dtype == F32 else np.uint16).view(
        np.int32 if dtype == F32 else np.int16)[0]
    ybuf = torch.full((head + ny + parity.GUARD,), int(fill), dtype=tdt, device="cuda")
    es = xbuf.element_size()
    xp, yp = xbuf.data_ptr() + es * x_off, ybuf.data_ptr() + es * head
    s = G.stream_handle()
    if op == capi.RN_OP_LN:
        m, r = G.Guarded(rows), G.Guarded(rows)
        st = capi.ln_fwd_strided(dtype, variant, xp, ldx, pbufs[0].data_ptr(), pbufs[1].data_ptr(),
                                 yp, ldy, m.ptr, r.ptr, rows, d, float(np.float32(1e-5)), s)
    else:
        m = r = None
        st = capi.rms_fwd_strided(dtype, variant, xp, ldx, pbufs[0].data_ptr(), yp, ldy, rows, d,
                                  float(np.float32(1e-5)), s)
    capi.check(st)
    torch.cuda.synchronize()
    yh = ybuf.cpu().numpy()
    untouched = np.ones(yh.size, bool)
    body = np.zeros(yh.size, bool)
    for i in range(rows):
        body[head + i * ldy: head + i * ldy + d] = True
    untouched &= ~body
    if not np.all(yh[untouched] == fill):
        bad = np.nonzero(untouched & (yh != fill))[0]
        raise parity.ParityError(f"{bad.size} elements outside the rows of y were written "
                                 f"(first at offset {bad[0] - head})")
    rows_out = np.stack([yh[head + i * ldy: head + i * ldy + d] for i in range(rows)])
    if dtype == F32:
        rows_out = rows_out.view(np.float32)
    else:
        rows_out = rows_out.view(np.uint16)
    return (rows_out, m.fetch("mean guard") if m else None, r.fetch("rstd guard") if r else None)


def _check(op, dtype, x, params, out):
    y, mean, rstd = out
    xw = x if dtype == F32 else workloads.to_storage(x, "bf16")[1]
    pw = params if dtype == F32 else [workloads.to_storage(p, "bf16")[1] for p in params]
    if op == capi.RN_OP_LN:
        yr, mr, sr = reference.layer_norm(xw, *pw)
        parity.check_mean(mean, mr, xw)
        parity.check_rstd(rstd, sr)
    else:
        yr, _ = reference.rms_norm(xw, *pw)
    if dtype == F32:
        parity.check_y(y, yr)
    else:
        parity.check_y_storage(y, yr, "bf16")


CASES = [  # d, ldx, ldy, x_off, y_off
    (1, 3, 1, 0, 0),
    (33, 40, 37, 1, 0),
    (768, 3 * 768, 768, 0, 0),        # a column block of a fused projection
    (768, 771, 775, 2, 2),            # strides agreeing modulo 4, unaligned rows
    (768, 770, 768, 0, 0),            # strides disagreeing modulo 4: scalar path
    (1000, 1024, 1000, 0, 0),
    (4096, 4100, 4096, 0, 0),
    (20000, 20004, 20008, 0, 0),      # staged / cluster / stream widths
    (40000, 40001, 40001, 3, 3),
]


@pytest.mark.parametrize("op", [capi.RN_OP_LN, capi.RN_OP_RMS])
@pytest.mark.parametrize("d,ldx,ldy,x_off,y_off", CASES)
def test_strided_f32_every_variant(op, d, ldx, ldy, x_off, y_off):
    rows = 37 if d > 8192 else 203
    wl = workloads.Workload("ln" if op == capi.RN_OP_LN else "rms", rows, d, seed=301,
                            x_dist="offset", x_std=2.0)
    x = wl.x()
    params = wl.params()
    for v in _variants(F32, op, d, ldx, ldy, x_off, y_off):
        _check(op, F32, x, params, _run(op, F32, x, params, ldx, ldy, v, x_off, y_off))


@pytest.mark.parametrize("op", [capi.RN_OP_LN, capi.RN_OP_RMS])
@pytest.mark.parametrize("d,ldx,ldy", [(768, 2304, 768), (1000, 1016, 1008), (1000, 1004, 1000),
                                       (4096, 4104, 4096), (40000, 40008, 40000)])
def test_strided_bf16(op, d, ldx, ldy):
    rows = 37 if d > 8192 else 203
    wl = workloads.Workload("ln" if op == capi.RN_OP_LN else "rms", rows, d, seed=303)
    x = wl.x()
    params = wl.params()
    for v in _variants(BF16, op, d, ldx, ldy, 0, 0):
        _check(op, BF16, x, params, _run(op, BF16, x, params, ldx, ldy, v))


def test_strided_views_through_the_torch_binding():
    torch = G.torch_cuda()
    import row_wise_normalization_gb300 as rn

    rows, d, heads = 300, 128, 6
    wl = workloads.Workload("ln", rows, heads * d, seed=305)
    big = torch.from_numpy(wl.x()).to("cuda")
    g, b = (torch.from_numpy(p[:d].copy()).to("cuda") for p in wl.params())
    out = torch.full_like(big, float("nan"))
    for h in range(heads):
        xv = big[:, h * d:(h + 1) * d]                 # row stride heads*d
        yv = out[:, h * d:(h + 1) * d]
        rn.ln_fwd(xv, g, b, y=yv)
        q = rn.rms_fwd(xv, g)                          # y allocated contiguous
        yr, _, _ = reference.layer_norm(xv.cpu().numpy(), g.cpu().numpy(), b.cpu().numpy())
        parity.check_y(yv.cpu().numpy(), yr, what=f"head {h}")
        qr, _ = reference.rms_norm(xv.cpu().numpy(), g.cpu().numpy())
        parity.check_y(q.cpu().numpy(), qr, what=f"rms head {h}")
    assert not torch.isnan(out).any()


def test_strided_views_of_pinned_host_matrices():
    """Column blocks of a wider matrix in pinned host memory, read and
    written in place by the kernel over the host link (the persistent grid
    host-resident rows get), each against the oracle; the gaps between the
    blocks' rows stay untouched."""
    torch = G.torch_cuda()
    import row_wise_normalization_gb300 as rn

    rows, d, heads = 4000, 256, 3
    wl = workloads.Workload("ln", rows, heads * d, seed=307, x_dist="offset", x_std=2.0)
    big = torch.from_numpy(wl.x()).pin_memory()
    g, b = (torch.from_numpy(p[:d].copy()).to("cuda") for p in wl.params())
    out = torch.full(big.shape, float("nan")).pin_memory()
    for h in (0, 2):
        xv = big[:, h * d:(h + 1) * d]                 # row stride heads*d
        yv = out[:, h * d:(h + 1) * d]
        rn.ln_fwd(xv, g, b, y=yv)
        torch.cuda.synchronize()
        yr, _, _ = reference.layer_norm(xv.numpy(), g.cpu().numpy(), b.cpu().numpy())
        parity.check_y(yv.numpy(), yr, what=f"host head {h}")
    assert torch.isnan(out[:, d:2 * d]).all(), "a gap column was written"
    assert not torch.isnan(out[:, :d]).any() and not torch.isnan(out[:, 2 * d:]).any()
