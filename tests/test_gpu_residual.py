"""Residual add fused with LayerNorm / RMSNorm against the oracle (GPU).

h = x + res must be bit-for-bit the FP32 sum (an FP32 add rounds the same
way everywhere); y, mean and rstd follow the tolerances of tests/parity.py.
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


def _inputs(rows, d, seed):
    wl = workloads.Workload("ln", rows, d, seed=seed, x_dist="offset", x_std=2.0)
    x = wl.x()
    r = workloads.Workload("ln", rows, d, seed=seed + 1000).x()
    g, b = wl.params()
    return x, r, g, b


def _check(op, x, r, g, b, out, want_h=True):
    h, y, m, s = out
    if op == LN:
        hr, yr, mr, sr = reference.layer_norm_residual(x, r, g, b)
        parity.check_mean(m, mr, hr)
        parity.check_rstd(s, sr)
    else:
        hr, yr, _ = reference.rms_norm_residual(x, r, g)
    parity.check_y(y, yr)
    if want_h:
        assert np.array_equal(h.view(np.uint32), hr.view(np.uint32)), "h is not the FP32 sum"


@pytest.mark.parametrize("d", [1, 3, 31, 128, 768, 1029, 4099, 8193, 20000, 40003])
def test_residual_every_variant_and_phase(d):
    rows = 29
    x, r, g, b = _inputs(rows, d, seed=51)
    for x_off, y_off in ((0, 0), (1, 1), (3, 3), (0, 2)):
        for op in (LN, RMS):
            params = (g, b) if op == LN else (g,)
            for v in G.residual_variants_for(op, d, x_off, y_off):
                out = G.run_residual(op, x, r, params, variant=v, x_off=x_off, r_off=x_off,
                                     y_off=y_off, h_off=y_off, p_off=1)
                _check(op, x, r, g, b, out)


@pytest.mark.parametrize("rows,d", [(4096, 768), (8192, 1024), (1000, 4096)])
def test_residual_without_h(rows, d):
    x, r, g, b = _inputs(rows, d, seed=53)
    for op in (LN, RMS):
        params = (g, b) if op == LN else (g,)
        out = G.run_residual(op, x, r, params, want_h=False)
        _check(op, x, r, g, b, out, want_h=False)


def test_residual_staged_and_cluster_refuse():
    x, r, g, b = _inputs(4, 40000, seed=55)
    for v in (capi.RN_VARIANT_STAGED, capi.RN_VARIANT_CLUSTER):
        with pytest.raises(capi.RowNormError):
            G.run_residual(LN, x, r, (g, b), variant=v)


def test_residual_cancels_to_beta():
    """x + (-x) = 0 exactly, so y = beta and rstd = eps^-1/2."""
    x, _, g, b = _inputs(64, 768, seed=57)
    h, y, m, s = G.run_residual(LN, x, -x, (g, b))
    assert not h.any()
    assert np.array_equal(y, np.broadcast_to(b, y.shape))
    np.testing.assert_allclose(s, np.float32(1e-5) ** -0.5, rtol=1e-6)


def test_residual_torch_binding():
    torch = G.torch_cuda()
    import row_wise_normalization_gb300 as rn

    x, r, g, b = _inputs(300, 1000, seed=59)
    dev = torch.device("cuda", 0)
    xt, rt, gt, bt = (torch.from_numpy(a).to(dev) for a in (x, r, g, b))
    h, y, m, s = rn.ln_fwd_residual(xt.view(3, 100, 1000), rt.view(3, 100, 1000), gt, bt)
    assert h.shape == (3, 100, 1000) and m.shape == (3, 100)
    _check(LN, x, r, g, b, (h.view(300, 1000).cpu().numpy(), y.view(300, 1000).cpu().numpy(),
                            m.view(300).cpu().numpy(), s.view(300).cpu().numpy()))
    h2, y2 = rn.rms_fwd_residual(xt, rt, gt, write_h=False)
    assert h2 is None
    _check(RMS, x, r, g, b, (None, y2.cpu().numpy(), None, None), want_h=False)


# x, res, h and y in pinned host memory: the kernel reads and writes them over
# the host link, on the persistent grid host-resident rows get
@pytest.mark.parametrize("rows,d", [(4096, 768), (1000, 4096), (333, 1029)])
def test_residual_host_resident(rows, d):
    torch = G.torch_cuda()
    import row_wise_normalization_gb300 as rn  # noqa: F401  (loads the library)

    x, r, g, b = _inputs(rows, d, seed=57)
    dev = torch.device("cuda", 0)
    xh = torch.from_numpy(x).pin_memory()
    rh = torch.from_numpy(r).pin_memory()
    gt, bt = torch.from_numpy(g).to(dev), torch.from_numpy(b).to(dev)
    s = torch.cuda.current_stream().cuda_stream
    for op in (LN, RMS):
        h = torch.full((rows, d), float("nan")).pin_memory()
        y = torch.full((rows, d), float("nan")).pin_memory()
        m = torch.full((rows,), float("nan"), device=dev)
        sd = torch.full((rows,), float("nan"), device=dev)
        if op == LN:
            st = capi.ln_fwd_residual(xh.data_ptr(), rh.data_ptr(), gt.data_ptr(), bt.data_ptr(),
                                      h.data_ptr(), y.data_ptr(), m.data_ptr(), sd.data_ptr(),
                                      rows, d, float(np.float32(1e-5)), s)
        else:
            st = capi.rms_fwd_residual(xh.data_ptr(), rh.data_ptr(), gt.data_ptr(), h.data_ptr(),
                                       y.data_ptr(), rows, d, float(np.float32(1e-5)), s)
        capi.check(st)
        torch.cuda.synchronize()
        _check(op, x, r, g, b, (h.numpy(), y.numpy(), m.cpu().numpy(), sd.cpu().numpy()))
