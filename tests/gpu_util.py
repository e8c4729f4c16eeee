"""Device-side helpers for the GPU parity tests: buffers at chosen 4-byte
phases, guarded outputs, and calls straight through the C ABI."""
from __future__ import annotations

import numpy as np

import parity
from row_wise_normalization_gb300 import capi


def torch_cuda():
    import torch

    if not torch.cuda.is_available():
        raise RuntimeError("a CUDA device is required for the gpu tests")
    return torch


def dev_copy(a, offset=0, pad=16):
    """Upload FP32 array ``a`` into a fresh allocation, ``offset`` floats in.

    Allocations are 256-byte aligned, so the data starts at 16-byte phase
    ``offset % 4``. Returns (buffer, device pointer of the data).
    """
    torch = torch_cuda()
    a = np.ascontiguousarray(a, np.float32).reshape(-1)
    buf = torch.empty(a.size + offset + pad, dtype=torch.float32, device="cuda")
    buf.fill_(0.0)
    if a.size:
        buf[offset:offset + a.size].copy_(torch.from_numpy(a))
    return buf, buf.data_ptr() + 4 * offset


class Guarded:
    """A device output of n floats framed by sentinel guards.

    The data starts ``parity.GUARD + offset`` floats into the allocation (16-
    byte phase ``offset % 4``); every element, the output region included,
    starts as the sentinel so that unwritten outputs fail the y check.
    """

    def __init__(self, n, offset=0):
        torch = torch_cuda()
        self.n = n
        self.head = parity.GUARD + offset
        host = parity.guarded(n, head=self.head)
        self.buf = torch.from_numpy(host.copy()).to("cuda")
        self.ptr = self.buf.data_ptr() + 4 * self.head

    def fetch(self, what):
        h = self.buf.cpu().numpy()
        parity.check_guards(h, self.n, what=what, head=self.head)
        return h[self.head:self.head + self.n]


def stream_handle():
    torch = torch_cuda()
    return torch.cuda.current_stream().cuda_stream


def run_ln(x, g, b, eps=1e-5, variant=capi.RN_VARIANT_AUTO, x_off=0, y_off=0, p_off=0,
           stats=True):
    """LayerNorm through ln_fwd_variant; returns (y, mean, rstd) as FP32 numpy
    (mean/rstd None when not requested) after checking every guard."""
    torch = torch_cuda()
    rows, d = x.shape
    xb, xp = dev_copy(x, x_off)
    gb, gp = dev_copy(g, p_off)
    bb, bp = dev_copy(b, p_off)
    y = Guarded(rows * d, y_off)
    m = Guarded(rows) if stats else None
    r = Guarded(rows) if stats else None
    st = capi.ln_fwd_variant(variant, xp, gp, bp, y.ptr, m.ptr if m else 0, r.ptr if r else 0,
                             rows, d, float(np.float32(eps)), stream_handle())
    capi.check(st)
    torch.cuda.synchronize()
    yo = y.fetch("y guard").reshape(rows, d)
    mo = m.fetch("mean guard") if m else None
    ro = r.fetch("rstd guard") if r else None
    return yo, mo, ro


def run_rms(x, w, eps=1e-5, variant=capi.RN_VARIANT_AUTO, x_off=0, y_off=0, p_off=0):
    torch = torch_cuda()
    rows, d = x.shape
    xb, xp = dev_copy(x, x_off)
    wb, wp = dev_copy(w, p_off)
    y = Guarded(rows * d, y_off)
    st = capi.rms_fwd_variant(variant, xp, wp, y.ptr, rows, d, float(np.float32(eps)),
                              stream_handle())
    capi.check(st)
    torch.cuda.synchronize()
    return y.fetch("y guard").reshape(rows, d)


def variants_for(op, d, x_off=0, y_off=0):
    """Every forced variant that accepts width d at these phases (plus AUTO)."""
    out = [capi.RN_VARIANT_AUTO]
    xa, ya = (1 << 20) + 4 * x_off, (1 << 30) + 4 * y_off
    for v in range(1, capi.RN_VARIANT_COUNT):
        try:
            capi.plan(op, v, d, xa, ya)
        except capi.RowNormError:
            continue
        out.append(v)
    return out


def run_residual(op, x, r, params, eps=1e-5, variant=capi.RN_VARIANT_AUTO, x_off=0, r_off=0,
                 y_off=0, h_off=0, p_off=0, want_h=True):
    """ln/rms_fwd_residual_variant through the C ABI; returns (h or None, y,
    mean, rstd) as FP32 numpy (mean/rstd None for RMSNorm), guards checked."""
    torch = torch_cuda()
    rows, d = x.shape
    xb, xp = dev_copy(x, x_off)
    rb, rp = dev_copy(r, r_off)
    pbs = [dev_copy(a, p_off) for a in params]
    y = Guarded(rows * d, y_off)
    h = Guarded(rows * d, h_off) if want_h else None
    if op == capi.RN_OP_LN:
        m, s = Guarded(rows), Guarded(rows)
        st = capi.ln_fwd_residual_variant(variant, xp, rp, pbs[0][1], pbs[1][1],
                                          h.ptr if h else 0, y.ptr, m.ptr, s.ptr, rows, d,
                                          float(np.float32(eps)), stream_handle())
    else:
        m = s = None
        st = capi.rms_fwd_residual_variant(variant, xp, rp, pbs[0][1], h.ptr if h else 0, y.ptr,
                                           rows, d, float(np.float32(eps)), stream_handle())
    capi.check(st)
    torch.cuda.synchronize()
    ho = h.fetch("h guard").reshape(rows, d) if h else None
    yo = y.fetch("y guard").reshape(rows, d)
    return (ho, yo, m.fetch("mean guard") if m else None, s.fetch("rstd guard") if s else None)


def residual_variants_for(op, d, x_off=0, y_off=0):
    """Every forced variant the residual entry points accept for width d."""
    out = [capi.RN_VARIANT_AUTO]
    xa, ya = (1 << 20) + 4 * x_off, (1 << 30) + 4 * y_off
    for v in range(1, capi.RN_VARIANT_COUNT):
        try:
            capi.plan_residual(op, v, d, xa, xa + (1 << 28), ya + (1 << 28), ya)
        except capi.RowNormError:
            continue
        out.append(v)
    return out


DTYPE_CODE = {"f32": capi.RN_DTYPE_F32, "bf16": capi.RN_DTYPE_BF16, "f16": capi.RN_DTYPE_F16}


def dev_copy16(bits, offset=0, pad=16):
    """Upload uint16 patterns, ``offset`` elements into a fresh allocation."""
    torch = torch_cuda()
    a = np.ascontiguousarray(bits, np.uint16).reshape(-1).view(np.int16)
    buf = torch.zeros(a.size + offset + pad, dtype=torch.int16, device="cuda")
    if a.size:
        buf[offset:offset + a.size].copy_(torch.from_numpy(a.copy()))
    return buf, buf.data_ptr() + 2 * offset


class Guarded16:
    """A device output of n 16-bit elements framed by sentinel guards."""

    def __init__(self, n, offset=0):
        torch = torch_cuda()
        self.n = n
        self.head = parity.GUARD + offset
        host = np.full(n + self.head + parity.GUARD, parity.SENTINEL16, np.uint16).view(np.int16)
        self.buf = torch.from_numpy(host).to("cuda")
        self.ptr = self.buf.data_ptr() + 2 * self.head

    def fetch(self, what):
        h = self.buf.cpu().numpy().view(np.uint16)
        if not (np.all(h[:self.head] == parity.SENTINEL16)
                and np.all(h[self.head + self.n:] == parity.SENTINEL16)):
            raise parity.ParityError(f"{what}: guard region overwritten")
        return h[self.head:self.head + self.n]


def run_typed(op, dtype, xbits, pbits, eps=1e-5, variant=capi.RN_VARIANT_AUTO, x_off=0, y_off=0,
              p_off=0, stats=True):
    """ln/rms_fwd_typed on 16-bit patterns; returns (y patterns, mean, rstd)."""
    torch = torch_cuda()
    rows, d = xbits.shape
    xb, xp = dev_copy16(xbits, x_off)
    pbs = [dev_copy16(p, p_off) for p in pbits]
    y = Guarded16(rows * d, y_off)
    code = DTYPE_CODE[dtype]
    if op == capi.RN_OP_LN:
        m = Guarded(rows) if stats else None
        r = Guarded(rows) if stats else None
        st = capi.ln_fwd_typed(code, variant, xp, pbs[0][1], pbs[1][1], y.ptr,
                               m.ptr if m else 0, r.ptr if r else 0, rows, d,
                               float(np.float32(eps)), stream_handle())
    else:
        m = r = None
        st = capi.rms_fwd_typed(code, variant, xp, pbs[0][1], y.ptr, rows, d,
                                float(np.float32(eps)), stream_handle())
    capi.check(st)
    torch.cuda.synchronize()
    return (y.fetch("y guard").reshape(rows, d), m.fetch("mean guard") if m else None,
            r.fetch("rstd guard") if r else None)


def typed_variants_for(dtype, op, d, x_off=0, y_off=0):
    out = [capi.RN_VARIANT_AUTO]
    es = 4 if dtype == "f32" else 2
    xa, ya = (1 << 20) + es * x_off, (1 << 30) + es * y_off
    for v in range(1, capi.RN_VARIANT_COUNT):
        try:
            capi.plan_typed(DTYPE_CODE[dtype], op, v, d, xa, ya)
        except capi.RowNormError:
            continue
        out.append(v)
    return out
