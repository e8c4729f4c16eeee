"""BF16 / FP16 storage with FP32 arithmetic against the float64 oracle (GPU).

The oracle normalises the exact values of the 16-bit inputs in float64; the
kernels widen to FP32, accumulate in FP32 and round y once to the storage
type, so y must be within one unit in the last place of the rounded
reference (tests/parity.py, check_y_storage) and mean / rstd within the FP32
tolerances.
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
DTYPES = ("bf16", "f16")


def _case(rows, d, seed, dtype, dist="offset", std=2.0):
    wl = workloads.Workload("ln", rows, d, seed=seed, x_dist=dist, x_std=std)
    xb, xw = workloads.to_storage(wl.x(), dtype)
    g, b = wl.params()
    gb, gw = workloads.to_storage(g, dtype)
    bb, bw = workloads.to_storage(b, dtype)
    return (xb, gb, bb), (xw, gw, bw)


def _check(op, dtype, wide, out):
    y, m, s = out
    xw, gw, bw = wide
    if op == LN:
        yr, mr, sr = reference.layer_norm(xw, gw, bw)
        if m is not None:
            parity.check_mean(m, mr, xw)
            parity.check_rstd(s, sr)
    else:
        yr, _ = reference.rms_norm(xw, gw)
    parity.check_y_storage(y, yr, dtype)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("d", [1, 7, 8, 9, 33, 128, 768, 1029, 3072, 4099, 8193, 20000,
                               40003])
def test_16bit_every_variant_and_phase(dtype, d):
    bits, wide = _case(23, d, seed=71, dtype=dtype)
    for x_off, y_off, p_off in ((0, 0, 0), (1, 1, 3), (5, 5, 1), (7, 7, 0), (0, 3, 0)):
        for op in (LN, RMS):
            pb = bits[1:] if op == LN else bits[1:2]
            for v in G.typed_variants_for(dtype, op, d, x_off, y_off):
                out = G.run_typed(op, dtype, bits[0], pb, variant=v, x_off=x_off, y_off=y_off,
                                  p_off=p_off)
                _check(op, dtype, wide, out)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("wl", [workloads.ln_4096x768(), workloads.Workload("ln", 4096, 3072, seed=74),
                                workloads.Workload("ln", 32768, 4096, seed=73)],
                         ids=lambda w: f"{w.rows}x{w.d}")
def test_16bit_larger_shapes(dtype, wl):
    xb, xw = workloads.to_storage(wl.x(), dtype)
    g, b = wl.params()
    gb, gw = workloads.to_storage(g, dtype)
    bb, bw = workloads.to_storage(b, dtype)
    for op in (LN, RMS):
        pb = (gb, bb) if op == LN else (gb,)
        _check(op, dtype, (xw, gw, bw), G.run_typed(op, dtype, xb, pb))


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("pattern", workloads.PATTERNS)
def test_16bit_rms_case_matrix_patterns(dtype, pattern):
    for d in workloads.RMS_WIDTHS:
        wl = workloads.Workload("rms", 512, d, seed=2, x_dist=pattern)
        xb, xw = workloads.to_storage(wl.x(), dtype)
        (w,) = wl.params()
        wb, ww = workloads.to_storage(w, dtype)
        _check(RMS, dtype, (xw, ww, None), G.run_typed(RMS, dtype, xb, (wb,)))


def test_16bit_refuses_residual_and_fp32_only_variants():
    bits, _ = _case(4, 40000, seed=75, dtype="bf16")
    for v in (capi.RN_VARIANT_STAGED, capi.RN_VARIANT_CLUSTER):
        with pytest.raises(capi.RowNormError):
            G.run_typed(LN, "bf16", bits[0], bits[1:], variant=v)


def test_16bit_torch_binding():
    torch = G.torch_cuda()
    import row_wise_normalization_gb300 as rn

    wl = workloads.Workload("ln", 333, 1000, seed=77)
    x = torch.from_numpy(wl.x()).cuda()
    g, b = (torch.from_numpy(a).cuda() for a in wl.params())
    for tdt, name in ((torch.bfloat16, "bf16"), (torch.float16, "f16")):
        xt, gt, bt = x.to(tdt), g.to(tdt), b.to(tdt)
        y, m, s = rn.ln_fwd(xt, gt, bt)
        yq = rn.rms_fwd(xt, gt)
        assert y.dtype == tdt and m.dtype == torch.float32
        xw, gw, bw = (t.float().cpu().numpy() for t in (xt, gt, bt))
        yr, mr, sr = reference.layer_norm(xw, gw, bw)
        parity.check_y_storage(y.view(torch.int16).cpu().numpy().view(np.uint16), yr, name)
        parity.check_mean(m.cpu().numpy(), mr, xw)
        parity.check_rstd(s.cpu().numpy(), sr)
        yqr, _ = reference.rms_norm(xw, gw)
        parity.check_y_storage(yq.view(torch.int16).cpu().numpy().view(np.uint16), yqr, name)


# host-resident x and y (pinned; the kernel reads and writes them over the
# host link on a persistent grid), parameters and statistics on the device
@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("rows,d", [(4096, 1024), (1000, 4096), (333, 1029)])
def test_16bit_host_resident(dtype, rows, d):
    torch = G.torch_cuda()
    bits, wide = _case(rows, d, seed=77, dtype=dtype)
    dev = torch.device("cuda", 0)
    xh = torch.from_numpy(bits[0].view(np.int16)).pin_memory()
    pd = [torch.from_numpy(p.view(np.int16)).to(dev) for p in bits[1:]]
    code = G.DTYPE_CODE[dtype]
    s = torch.cuda.current_stream().cuda_stream
    for op in (LN, RMS):
        y = torch.full((rows, d), -1, dtype=torch.int16).pin_memory()
        m = torch.full((rows,), float("nan"), device=dev)
        r = torch.full((rows,), float("nan"), device=dev)
        if op == LN:
            st = capi.ln_fwd_typed(code, capi.RN_VARIANT_AUTO, xh.data_ptr(), pd[0].data_ptr(),
                                   pd[1].data_ptr(), y.data_ptr(), m.data_ptr(), r.data_ptr(),
                                   rows, d, float(np.float32(1e-5)), s)
        else:
            st = capi.rms_fwd_typed(code, capi.RN_VARIANT_AUTO, xh.data_ptr(), pd[0].data_ptr(),
                                    y.data_ptr(), rows, d, float(np.float32(1e-5)), s)
        capi.check(st)
        torch.cuda.synchronize()
        yb = y.numpy().view(np.uint16)
        out = (yb, m.cpu().numpy(), r.cpu().numpy()) if op == LN else (yb, None, None)
        _check(op, dtype, wide, out)
