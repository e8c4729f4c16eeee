"""Seeded random configurations against the oracle (GPU).

The other parity tests walk chosen shapes; these draw the call itself: the
operation, the row count, the width (log-uniform from 1 to 70000, so every
kernel family and both sides of every dispatch boundary come up), the
16-byte phases of x, y and the parameters, the value distribution, the eps
and a forced variant among those that accept the call. The draws are fixed
by the case number, so a failure names a reproducible case. Sizes stay
small enough for the float64 oracle (at most ~2M elements per case). The
strided, batched and backward entry points are drawn the same way.
"""
import math

import numpy as np
import pytest

import gpu_util as G
import parity
import workloads
from oracle import reference
from row_wise_normalization_gb300 import capi

pytestmark = pytest.mark.gpu

LN, RMS = capi.RN_OP_LN, capi.RN_OP_RMS
DISTS = ("normal", "offset", "small", "zeros", "alternating")


def _draw(case):
    rng = np.random.default_rng([77, case])
    d = int(math.exp(rng.uniform(0.0, math.log(70000.0))))
    d = max(1, d)
    rows = int(rng.integers(1, max(2, min(700, 2_000_000 // d)) + 1))
    op = LN if rng.random() < 0.5 else RMS
    dist = DISTS[int(rng.integers(0, len(DISTS)))]
    x_off, y_off, p_off = (int(v) for v in rng.integers(0, 4, size=3))
    if rng.random() < 0.5:
        y_off = x_off          # half the cases keep x and y in one phase
    eps = float(np.float32(10.0 ** rng.uniform(-7, -2)))
    return rng, op, rows, d, dist, x_off, y_off, p_off, eps


@pytest.mark.parametrize("case", range(400))
def test_fuzz_forward(case):
    rng, op, rows, d, dist, x_off, y_off, p_off, eps = _draw(case)
    # spreads down to 0.05 on offset rows (|mean| up to 100): the output's
    # accuracy must not depend on |mean| / sigma
    x_std = float(math.exp(rng.uniform(math.log(0.05), math.log(3.0))))
    wl = workloads.Workload("ln" if op == LN else "rms", rows, d, seed=1000 + case,
                            x_dist=dist, x_std=x_std, eps=eps)
    x = wl.x()
    params = wl.params()
    variants = G.variants_for(op, d, x_off, y_off)
    v = variants[int(rng.integers(0, len(variants)))]
    if op == LN:
        y, m, r = G.run_ln(x, *params, eps=eps, variant=v, x_off=x_off, y_off=y_off, p_off=p_off)
        yr, mr, rr = reference.layer_norm(x, *params, eps)
        parity.check_y(y, yr, what=f"case {case} y")
        parity.check_mean(m, mr, x, what=f"case {case} mean")
        parity.check_rstd(r, rr, what=f"case {case} rstd")
    else:
        y = G.run_rms(x, *params, eps=eps, variant=v, x_off=x_off, y_off=y_off, p_off=p_off)
        yr, _ = reference.rms_norm(x, *params, eps)
        parity.check_y(y, yr, what=f"case {case} y")
    assert capi.device_error() == 0


@pytest.mark.parametrize("case", range(48))
def test_fuzz_residual(case):
    rng, op, rows, d, dist, x_off, y_off, p_off, eps = _draw(1000 + case)
    wl = workloads.Workload("ln" if op == LN else "rms", rows, d, seed=2000 + case,
                            x_dist=dist, x_std=_x_std(rng), eps=eps)
    x = wl.x()
    # a residual of random scale: h = x + res keeps x's offset and a spread
    # down to 0.05
    res = (workloads.Workload("ln", rows, d, seed=3000 + case).x()
           * np.float32(_x_std(rng))).astype(np.float32)
    params = wl.params()
    variants = G.residual_variants_for(op, d, x_off, y_off)
    v = variants[int(rng.integers(0, len(variants)))]
    h, y, m, r = G.run_residual(op, x, res, params, eps=eps, variant=v, x_off=x_off,
                                r_off=x_off, y_off=y_off, h_off=y_off, p_off=p_off)
    hr = reference.residual_sum(x, res)
    assert np.array_equal(h.view(np.uint32), hr.view(np.uint32)), f"case {case} h"
    if op == LN:
        _, yr, mr, rr = reference.layer_norm_residual(x, res, *params, eps)
        parity.check_mean(m, mr, hr, what=f"case {case} mean")
        parity.check_rstd(r, rr, what=f"case {case} rstd")
    else:
        _, yr, _ = reference.rms_norm_residual(x, res, *params, eps)
    parity.check_y(y, yr, what=f"case {case} y")


@pytest.mark.parametrize("case", range(48))
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_fuzz_16bit(case, dtype):
    rng, op, rows, d, dist, x_off, y_off, p_off, eps = _draw(2000 + case)
    if dist == "offset" and dtype == "f16":
        dist = "normal"            # FP16's range and step do not carry the +-100 offsets well
    wl = workloads.Workload("ln" if op == LN else "rms", rows, d, seed=4000 + case,
                            x_dist=dist, eps=eps)
    xb, xw = workloads.to_storage(wl.x(), dtype)
    pst = [workloads.to_storage(p_, dtype) for p_ in wl.params()]
    variants = G.typed_variants_for(dtype, op, d, x_off, y_off)
    v = variants[int(rng.integers(0, len(variants)))]
    y, m, r = G.run_typed(op, dtype, xb, [p_[0] for p_ in pst], eps=eps, variant=v, x_off=x_off,
                          y_off=y_off, p_off=p_off)
    pw = [p_[1] for p_ in pst]
    if op == LN:
        yr, mr, rr = reference.layer_norm(xw, *pw, eps)
        parity.check_mean(m, mr, xw, what=f"case {case} mean")
        parity.check_rstd(r, rr, what=f"case {case} rstd")
    else:
        yr, _ = reference.rms_norm(xw, *pw, eps)
    parity.check_y_storage(y, yr, dtype, what=f"case {case} y")


def _x_std(rng):
    return float(math.exp(rng.uniform(math.log(0.05), math.log(3.0))))


@pytest.mark.parametrize("case", range(64))
def test_fuzz_strided(case):
    """Random row strides (>= d) and phases through ln_fwd_strided /
    rms_fwd_strided, every accepted variant drawn; gaps must stay untouched."""
    import test_gpu_strided as S

    rng, op, rows, d, dist, x_off, y_off, p_off, eps = _draw(3000 + case)
    rows = min(rows, max(1, 400_000 // d))
    ldx = d + int(rng.integers(0, 9))
    ldy = d + int(rng.integers(0, 9))
    dtype = capi.RN_DTYPE_F32 if rng.random() < 0.75 else capi.RN_DTYPE_BF16
    wl = workloads.Workload("ln" if op == LN else "rms", rows, d, seed=5000 + case, x_dist=dist,
                            x_std=_x_std(rng))
    x = wl.x()
    params = wl.params()
    variants = S._variants(dtype, op, d, ldx, ldy, x_off, y_off)
    v = variants[int(rng.integers(0, len(variants)))]
    S._check(op, dtype, x, params, S._run(op, dtype, x, params, ldx, ldy, v, x_off, y_off))


@pytest.mark.parametrize("case", range(16))
def test_fuzz_batched(case):
    """A random table of problems (widths, rows, phases, empty ones) through
    ln_fwd_batched / rms_fwd_batched, each against the oracle and, bit for
    bit, against its single call."""
    import test_gpu_batched as B

    rng = np.random.default_rng([78, case])
    op = LN if rng.random() < 0.5 else RMS
    dtype = capi.RN_DTYPE_F32 if rng.random() < 0.75 else capi.RN_DTYPE_BF16
    n = int(rng.integers(1, 150))
    shapes = []
    for _ in range(n):
        d = int(math.exp(rng.uniform(0.0, math.log(1500.0))))
        rows = int(rng.integers(0, 40))
        xo = int(rng.integers(0, 4))
        yo = xo if rng.random() < 0.7 else int(rng.integers(0, 4))
        if dtype == capi.RN_DTYPE_BF16:
            xo, yo = 2 * xo, 2 * yo
        shapes.append((rows, max(1, d), xo, yo))
    B._run_batch(op, dtype, shapes, 7000 + 1000 * case)


@pytest.mark.parametrize("case", range(48))
def test_fuzz_backward(case):
    """Random LayerNorm / RMSNorm backward calls: widths up to 16384, offset
    rows with small spreads, aligned or not, and a random workspace size
    between one partial row and the full one."""
    import test_gpu_backward as W

    rng, op, rows, d, dist, x_off, y_off, p_off, eps = _draw(4000 + case)
    d = min(d, 16384)
    rows = max(1, min(rows, 600_000 // d))
    off = int(rng.integers(0, 4)) if d <= 8192 else 0
    wl = workloads.Workload("ln", rows, d, seed=9000 + case, x_dist=dist, x_std=_x_std(rng))
    x = wl.x()
    dy = workloads.Workload("ln", rows, d, seed=9500 + case).x()
    g, _ = wl.params()
    width = 2 * d if op == LN else d
    if d > 8192 and d % 4:
        # beyond the scalar layout's 8192 floats: a documented size error,
        # from the workspace query and from the call itself
        with pytest.raises(capi.RowNormError) as err:
            capi.bwd_workspace_size(op, rows, d)
        assert err.value.status == capi.RN_ERR_SIZE
        with pytest.raises(capi.RowNormError) as err:
            if op == LN:
                m32, r32 = W._stats(x, g)
                W._run_ln(x, dy, g, m32, r32, off=off, ws_bytes=4 * width * 4)
            else:
                W._run_rms(x, dy, g, off=off, ws_bytes=4 * width * 4)
        assert err.value.status == capi.RN_ERR_SIZE
        return
    full = capi.bwd_workspace_size(op, rows, d)
    ws = int(rng.integers(1, max(2, full // (4 * width)) + 1)) * 4 * width
    chain = max(4, -(-rows // 152)) + 16 if ws >= full else rows + 16
    if op == LN:
        m32, r32 = W._stats(x, g)
        W._check_ln(x, dy, g, W._run_ln(x, dy, g, m32, r32, off=off, ws_bytes=ws), chain=chain)
    else:
        dx, dw = W._run_rms(x, dy, g, off=off, ws_bytes=ws)
        dxr, dwr = reference.rms_norm_backward(dy, x, g)
        parity.check_y(dx, dxr, what=f"case {case} dx")
        _, r = reference.rms_norm(x, g)
        terms = np.abs(dy.astype(np.float64) * x * r[:, None]).sum(axis=0)
        parity.check_colsum(dw, dwr, terms, chain, f"case {case} dw")


@pytest.mark.parametrize("case", range(40))
def test_fuzz_backward_staged(case):
    """Random backward calls in the staged range (rows of 256 or 512
    threads on the vector layout: FP32 widths 3073-8192, 16-bit 2049-8192),
    any storage type, row counts from one row to several ring cycles per CTA,
    and a random workspace size (down to one partial row: one CTA whose ring
    wraps once per row)."""
    import test_gpu_backward as W
    import test_gpu_backward_16bit as H

    rng = np.random.default_rng([79, case])
    dtype = ("f32", "bf16", "f16")[int(rng.integers(0, 3))]
    vec = 4 if dtype == "f32" else 8
    lo = 3073 if dtype == "f32" else 2049
    d = int(rng.integers(lo // vec + 1, 8192 // vec + 1)) * vec
    rows = int(rng.integers(1, min(2500, 3_000_000 // d) + 1))
    op = LN if rng.random() < 0.5 else RMS
    dist = DISTS[int(rng.integers(0, len(DISTS)))]
    width = 2 * d if op == LN else d
    full = capi.bwd_workspace_size(op, rows, d)
    ws = int(rng.integers(1, max(2, full // (4 * width)) + 1)) * 4 * width
    chain = max(4, -(-rows // 152)) + 16 if ws >= full else rows + 16
    capi.device_error(clear=True)
    if dtype == "f32":
        wl = workloads.Workload("ln", rows, d, seed=9700 + case, x_dist=dist, x_std=_x_std(rng))
        x = wl.x()
        dy = workloads.Workload("ln", rows, d, seed=9800 + case).x()
        g, _ = wl.params()
        if op == LN:
            m32, r32 = W._stats(x, g)
            W._check_ln(x, dy, g, W._run_ln(x, dy, g, m32, r32, ws_bytes=ws), chain=chain)
        else:
            dx, dw = W._run_rms(x, dy, g, ws_bytes=ws)
            dxr, dwr = reference.rms_norm_backward(dy, x, g)
            parity.check_y(dx, dxr, what=f"case {case} dx")
            _, r = reference.rms_norm(x, g)
            terms = np.abs(dy.astype(np.float64) * x * r[:, None]).sum(axis=0)
            parity.check_colsum(dw, dwr, terms, chain, f"case {case} dw")
    else:
        xb, xw, dyb, dyw, gb, gw, bw = H._inputs(rows, d, dtype, 9900 + case,
                                                 "offset" if dist == "offset" else "normal")
        m32, r32 = H._stats(xw, gw, bw)
        out = H._run(op, dtype, xb, dyb, gb, m32, r32, ws_bytes=ws)
        H._check(op, dtype, xw, dyw, gw, bw, out, chain=chain)
    assert capi.device_error() == 0


def _pinned_at(torch, a, off, pad=16):
    """A pinned FP32 buffer holding ``a`` (flattened) ``off`` elements in,
    NaN everywhere else; returns (buffer, address of the first element)."""
    n = a.size
    buf = torch.full((n + off + pad,), float("nan")).pin_memory()
    if n:
        buf[off:off + n] = torch.from_numpy(np.ascontiguousarray(a, np.float32).reshape(-1))
    return buf, buf.data_ptr() + 4 * off


@pytest.mark.parametrize("case", range(96))
def test_fuzz_forward_host_resident(case):
    """x and y in pinned host memory (read and written over the host link,
    on the grid host-resident rows get), at random phases, with any variant
    that accepts the call except the staged one (which refuses host rows);
    the parameters and statistics in device memory. Every element of the
    host buffers outside y's rows must stay NaN."""
    torch = G.torch_cuda()
    rng, op, rows, d, dist, x_off, y_off, p_off, eps = _draw(5000 + case)
    rows = min(rows, max(1, 400_000 // d))     # pinned buffers of a few MB at most
    wl = workloads.Workload("ln" if op == LN else "rms", rows, d, seed=6000 + case,
                            x_dist=dist, x_std=_x_std(rng), eps=eps)
    x = wl.x()
    params = wl.params()
    variants = [v for v in G.variants_for(op, d, x_off, y_off) if v != capi.RN_VARIANT_STAGED]
    v = variants[int(rng.integers(0, len(variants)))]
    dev = torch.device("cuda", 0)
    xbuf, xp = _pinned_at(torch, x, x_off)
    ybuf, yp = _pinned_at(torch, np.full_like(x, np.nan), y_off)
    pts = [G.dev_copy(p, p_off) for p in params]
    m = torch.full((rows,), float("nan"), device=dev)
    r = torch.full((rows,), float("nan"), device=dev)
    s = torch.cuda.current_stream().cuda_stream
    if op == LN:
        st = capi.ln_fwd_variant(v, xp, pts[0][1], pts[1][1], yp, m.data_ptr(), r.data_ptr(),
                                 rows, d, eps, s)
    else:
        st = capi.rms_fwd_variant(v, xp, pts[0][1], yp, rows, d, eps, s)
    capi.check(st)
    torch.cuda.synchronize()
    yb = ybuf.numpy()
    y = yb[y_off:y_off + rows * d].reshape(rows, d)
    assert np.isnan(yb[:y_off]).all() and np.isnan(yb[y_off + rows * d:]).all(), \
        f"case {case}: a write outside y"
    if op == LN:
        yr, mr, rr = reference.layer_norm(x, *params, eps)
        parity.check_y(y, yr, what=f"case {case} y")
        parity.check_mean(m.cpu().numpy(), mr, x, what=f"case {case} mean")
        parity.check_rstd(r.cpu().numpy(), rr, what=f"case {case} rstd")
    else:
        yr, _ = reference.rms_norm(x, *params, eps)
        parity.check_y(y, yr, what=f"case {case} y")
    assert capi.device_error() == 0
