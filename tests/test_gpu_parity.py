"""CUDA path against the float64 oracle, element by element (GPU required).

Every call goes through the C ABI (ln_fwd_variant / rms_fwd_variant, AUTO and
each forced kernel variant that accepts the width). Outputs are framed by
sentinel guards that must survive, and the output region starts as
sentinels, so a dropped element fails. Tolerances are those of
``tests/parity.py``.
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


def _check_ln(x, g, b, out, eps=1e-5):
    y, mean, rstd = out
    yr, mr, rr = reference.layer_norm(x, g, b, eps)
    parity.check_y(y, yr)
    if mean is not None:
        parity.check_mean(mean, mr, x)
        parity.check_rstd(rstd, rr)


def _check_rms(x, w, y, eps=1e-5):
    yr, _ = reference.rms_norm(x, w, eps)
    parity.check_y(y, yr)


# ---------------------------------------------------------------------------
# the LayerNorm shapes: 512 x 128 (seed 0) and the harness shape 4096 x 768
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("wl", [workloads.ln_512x128(), workloads.ln_4096x768()],
                         ids=lambda w: w.tag)
def test_ln_configs_every_variant(wl):
    x = wl.x()
    g, b = wl.params()
    for v in G.variants_for(LN, wl.d):
        _check_ln(x, g, b, G.run_ln(x, g, b, wl.eps, variant=v))


# ---------------------------------------------------------------------------
# the RMSNorm case matrix: 512 rows x 7 widths x 4 patterns x every variant
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("wl", workloads.rms_512_matrix(), ids=lambda w: w.tag)
def test_rms_case_matrix(wl):
    x = wl.x()
    (w,) = wl.params()
    for v in G.variants_for(RMS, wl.d):
        _check_rms(x, w, G.run_rms(x, w, wl.eps, variant=v))


@pytest.mark.parametrize("d", workloads.RMS_WIDTHS)
@pytest.mark.parametrize("pattern", workloads.PATTERNS)
def test_ln_on_the_rms_case_matrix(d, pattern):
    """LayerNorm over the same widths and patterns (zeros give y = beta)."""
    wl = workloads.Workload("ln", 512, d, seed=2, x_dist=pattern)
    x = wl.x()
    g, b = wl.params()
    for v in G.variants_for(LN, d):
        _check_ln(x, g, b, G.run_ln(x, g, b, wl.eps, variant=v))


# ---------------------------------------------------------------------------
# the offset-row sweep (centred variance under a large per-row mean)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("wl", workloads.sweep_offset(), ids=lambda w: w.tag)
def test_sweep_offset_rows(wl):
    x = wl.x()
    if wl.op == "ln":
        g, b = wl.params()
        for v in G.variants_for(LN, wl.d):
            _check_ln(x, g, b, G.run_ln(x, g, b, wl.eps, variant=v))
    else:
        (w,) = wl.params()
        for v in G.variants_for(RMS, wl.d):
            _check_rms(x, w, G.run_rms(x, w, wl.eps, variant=v))


# ---------------------------------------------------------------------------
# ragged widths and every 16-byte phase of x, y and the parameters
# ---------------------------------------------------------------------------
PHASE_WIDTHS = [1, 2, 3, 5, 7, 31, 33, 127, 130, 769, 1027, 1029, 4099, 8193, 9000, 16387,
                20000, 20003, 24576, 24579, 32768, 32771, 33001]


@pytest.mark.parametrize("d", PHASE_WIDTHS)
def test_phases_and_ragged_widths(d):
    rows = 37
    wl = workloads.Workload("ln", rows, d, seed=17, x_dist="offset", x_std=2.0)
    x = wl.x()
    g, b = wl.params()
    for x_off, y_off, p_off in ((0, 0, 0), (1, 1, 0), (2, 2, 3), (3, 3, 1), (0, 1, 2), (3, 0, 0)):
        for v in G.variants_for(LN, d, x_off, y_off):
            _check_ln(x, g, b, G.run_ln(x, g, b, variant=v, x_off=x_off, y_off=y_off,
                                        p_off=p_off))
        for v in G.variants_for(RMS, d, x_off, y_off):
            _check_rms(x, g, G.run_rms(x, g, variant=v, x_off=x_off, y_off=y_off, p_off=p_off))


# ---------------------------------------------------------------------------
# rows too wide for registers: staged (bulk copy into shared memory) and
# streaming kernels, up to the largest row one CTA can stage
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("d", [24577, 40000, 57856, 57860, 100003])
def test_wide_rows(d):
    wl = workloads.Workload("ln", 67, d, seed=29, x_dist="offset", x_std=2.0)
    x = wl.x()
    g, b = wl.params()
    for x_off, y_off in ((0, 0), (3, 3), (1, 2)):
        for v in G.variants_for(LN, d, x_off, y_off):
            _check_ln(x, g, b, G.run_ln(x, g, b, variant=v, x_off=x_off, y_off=y_off, p_off=1))
        for v in G.variants_for(RMS, d, x_off, y_off):
            _check_rms(x, g, G.run_rms(x, g, variant=v, x_off=x_off, y_off=y_off))
    assert capi.device_error() == 0


@pytest.mark.parametrize("rows,d", [(9, 65539), (5, 131072), (3, 200003), (3, 524288),
                                    (7, 524291)])
def test_very_wide_rows(rows, d):
    """Rows split over 8-16 CTA clusters (and the streaming kernel beyond)."""
    wl = workloads.Workload("ln", rows, d, seed=37, x_dist="offset", x_std=2.0)
    x = wl.x()
    g, b = wl.params()
    for x_off, y_off in ((0, 0), (1, 1)):
        for v in G.variants_for(LN, d, x_off, y_off):
            _check_ln(x, g, b, G.run_ln(x, g, b, variant=v, x_off=x_off, y_off=y_off, p_off=2))
        for v in G.variants_for(RMS, d, x_off, y_off):
            _check_rms(x, g, G.run_rms(x, g, variant=v, x_off=x_off, y_off=y_off))


def _cluster_shapes():
    # every compiled cluster shape at the widest row it takes: 256-thread CTAs
    # of 4 (2 CTAs only), 6 or 8 quads a thread over 2-16 CTAs, then 16 CTAs
    # of 512 and 1024 threads
    out = [(2, 256, 4)] + [(c, 256, s) for c in (2, 4, 8, 16) for s in (6, 8)]
    return out + [(16, 512, 8), (16, 1024, 8)]


@pytest.mark.parametrize("cl,threads,slots", _cluster_shapes())
def test_every_cluster_shape(cl, threads, slots):
    """The cluster kernel at every compiled shape (parameters in shared
    memory on aligned 256-thread shapes, 16-96 KB of it), LayerNorm and
    RMSNorm, aligned and at another 16-byte phase, at the widest row of the
    shape, through the forced variant."""
    rows = 3
    d_al = 4 * cl * threads * slots                    # the widest aligned row
    for d, x_off, y_off in ((d_al, 0, 0), (d_al - 4 * (cl - 1) - 2, 1, 1)):
        wl = workloads.Workload("ln", rows, d, seed=43, x_dist="offset", x_std=2.0)
        x = wl.x()
        g, b = wl.params()
        pl = capi.plan(LN, capi.RN_VARIANT_CLUSTER, d, (1 << 20) + 4 * x_off,
                       (1 << 30) + 4 * y_off)
        assert (pl.cluster, pl.threads_per_cta, pl.slots) == (cl, threads, slots)
        assert pl.aligned == (1 if x_off == 0 else 0)
        _check_ln(x, g, b, G.run_ln(x, g, b, variant=capi.RN_VARIANT_CLUSTER, x_off=x_off,
                                    y_off=y_off, p_off=2 * x_off))
        _check_rms(x, g, G.run_rms(x, g, variant=capi.RN_VARIANT_CLUSTER, x_off=x_off,
                                   y_off=y_off, p_off=2 * x_off))


@pytest.mark.parametrize("rows,d", [(40000, 16384), (5000, 65536)])
def test_cluster_rows_beyond_resident_clusters(rows, d):
    """More rows than resident clusters: every cluster walks many rows."""
    wl = workloads.Workload("rms", rows, d, seed=41)
    x = wl.x()
    (w,) = wl.params()
    _check_rms(x, w, G.run_rms(x, w, variant=capi.RN_VARIANT_CLUSTER))


# ---------------------------------------------------------------------------
# rows far beyond the resident grid: every CTA walks many rows
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("rows,d", [(200003, 64), (60001, 200), (20011, 1500), (3001, 40000)])
def test_many_rows_per_cta(rows, d):
    wl = workloads.Workload("ln", rows, d, seed=23)
    x = wl.x()
    g, b = wl.params()
    _check_ln(x, g, b, G.run_ln(x, g, b))
    _check_rms(x, g, G.run_rms(x, g))


# ---------------------------------------------------------------------------
# optional statistics, empty input, eps = 0
# ---------------------------------------------------------------------------
def test_no_device_error_reported():
    """No staged kernel of the runs above hit its bounded wait."""
    assert capi.device_error() == 0


def test_statistics_optional():
    wl = workloads.Workload("ln", 300, 768, seed=5)
    x = wl.x()
    g, b = wl.params()
    for v in G.variants_for(LN, 768):
        _check_ln(x, g, b, G.run_ln(x, g, b, variant=v, stats=False))


def test_empty_rows_is_noop_on_device():
    torch = G.torch_cuda()
    y = G.Guarded(16)
    xb, xp = G.dev_copy(np.ones(16, np.float32))
    assert capi.ln_fwd(xp, xp, xp, y.ptr, 0, 0, 0, 16, 1e-5, G.stream_handle()) == capi.RN_OK
    assert capi.rms_fwd(xp, xp, y.ptr, 0, 16, 1e-5, G.stream_handle()) == capi.RN_OK
    torch.cuda.synchronize()
    out = y.fetch("guard")
    assert np.all(out.view(np.uint32) == parity.SENTINEL_BITS)


def test_eps_zero_matches_oracle_including_nan():
    """eps = 0 is accepted: zero rows then give NaN exactly where the oracle does."""
    x = np.zeros((4, 33), np.float32)
    x[1] = np.arange(33, dtype=np.float32) - 16
    g = np.ones(33, np.float32)
    b = np.zeros(33, np.float32)
    y, mean, rstd = G.run_ln(x, g, b, eps=0.0)
    with np.errstate(all="ignore"):
        yr, mr, rr = reference.layer_norm(x, g, b, 0.0)
    assert np.array_equal(np.isnan(y), np.isnan(yr))
    parity.check_y(y[1], yr[1])
    assert np.all(np.isinf(rstd[[0, 2, 3]]))
    yq = G.run_rms(x, g, eps=0.0)
    with np.errstate(all="ignore"):
        yqr, _ = reference.rms_norm(x, g, 0.0)
    assert np.array_equal(np.isnan(yq), np.isnan(yqr))


def test_torch_binding_and_side_stream():
    torch = G.torch_cuda()
    import row_wise_normalization_gb300 as rn

    wl = workloads.Workload("ln", 1000, 1000, seed=8)
    x = wl.x()
    g, b = wl.params()
    s = torch.cuda.Stream()
    xt = torch.from_numpy(x).cuda()
    gt = torch.from_numpy(g).cuda()
    bt = torch.from_numpy(b).cuda()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        y, mean, rstd = rn.ln_fwd(xt, gt, bt)
        yq = rn.rms_fwd(xt, gt)
    s.synchronize()
    _check_ln(x, g, b, (y.cpu().numpy(), mean.cpu().numpy(), rstd.cpu().numpy()))
    _check_rms(x, g, yq.cpu().numpy())
    # a 3-D input normalises its last dimension
    y3, m3, r3 = rn.ln_fwd(xt.view(10, 100, 1000), gt, bt)
    assert y3.shape == (10, 100, 1000) and m3.shape == (10, 100)
    torch.testing.assert_close(y3.view(1000, 1000), y, rtol=0, atol=0)


# ---------------------------------------------------------------------------
# host-resident buffers: pinned host memory read and written by the kernel
# over the host link (no staging copies)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("where", ["host_in", "host_out", "host_both"])
@pytest.mark.parametrize("rows,d", [(4096, 768), (333, 1029), (64, 40000), (2000, 4096),
                                    (1500, 8192), (20000, 256)])
def test_host_resident_buffers(where, rows, d):
    torch = G.torch_cuda()
    import row_wise_normalization_gb300 as rn

    wl = workloads.Workload("ln", rows, d, seed=31, x_dist="offset", x_std=2.0)
    x = wl.x()
    g, b = wl.params()
    dev = torch.device("cuda", 0)
    xin = torch.from_numpy(x).pin_memory() if where != "host_out" else torch.from_numpy(x).to(dev)
    gt, bt = torch.from_numpy(g).to(dev), torch.from_numpy(b).to(dev)

    def out(shape):
        if where == "host_in":
            return torch.full(shape, float("nan"), device=dev)
        return torch.full(shape, float("nan")).pin_memory()

    y, m, r = out((rows, d)), out((rows,)), out((rows,))
    rn.ln_fwd(xin, gt, bt, y=y, mean=m, rstd=r)
    yq = rn.rms_fwd(xin, gt, y=out((rows, d)))
    torch.cuda.synchronize()
    _check_ln(x, g, b, (y.cpu().numpy(), m.cpu().numpy(), r.cpu().numpy()))
    _check_rms(x, g, yq.cpu().numpy())
    if where == "host_both":
        # outputs allocated by the binding live where x lives
        y2, m2, _ = rn.ln_fwd(xin, gt, bt)
        torch.cuda.synchronize()
        assert not y2.is_cuda and y2.is_pinned() and m2.is_pinned()
        parity.check_y(y2.numpy(), reference.layer_norm(x, g, b)[0])


def _pageable_access_supported(torch):
    """cudaDevAttrPageableMemoryAccess (88) of device 0 through the CUDA
    runtime torch has loaded; None when that library cannot be reached."""
    import ctypes
    torch.cuda.init()
    for name in ("libcudart.so.13", "libcudart.so"):
        try:
            rt = ctypes.CDLL(name)
        except OSError:
            continue
        v = ctypes.c_int(0)
        if rt.cudaDeviceGetAttribute(ctypes.byref(v), 88, 0) != 0:
            return None
        return v.value == 1
    return None


@pytest.mark.parametrize("rows,d", [(4096, 768), (333, 1029), (1000, 4096)])
def test_pageable_host_buffers_through_the_c_entry_point(rows, d):
    """Ordinary (pageable, unregistered) host memory for x and y, on a GPU
    that reads host page tables (checked first: on any other GPU such an
    access is not allowed, and the test does not run it)."""
    torch = G.torch_cuda()
    import row_wise_normalization_gb300 as rn  # noqa: F401  (loads the library)

    ok = _pageable_access_supported(torch)
    if not ok:
        pytest.skip("the GPU does not read pageable host memory" if ok is False
                    else "CUDA runtime library not reachable through ctypes")
    wl = workloads.Workload("ln", rows, d, seed=37, x_dist="offset", x_std=2.0)
    x = np.ascontiguousarray(wl.x(), np.float32)
    g, b = wl.params()
    dev = torch.device("cuda", 0)
    gt, bt = torch.from_numpy(g).to(dev), torch.from_numpy(b).to(dev)
    y = np.full((rows, d), np.nan, np.float32)
    yq = np.full((rows, d), np.nan, np.float32)
    m = torch.full((rows,), float("nan"), device=dev)
    r = torch.full((rows,), float("nan"), device=dev)
    s = torch.cuda.current_stream().cuda_stream
    capi.check(capi.ln_fwd(x.ctypes.data, gt.data_ptr(), bt.data_ptr(), y.ctypes.data,
                           m.data_ptr(), r.data_ptr(), rows, d, 1e-5, s))
    capi.check(capi.rms_fwd(x.ctypes.data, gt.data_ptr(), yq.ctypes.data, rows, d, 1e-5, s))
    torch.cuda.synchronize()
    _check_ln(x, g, b, (y, m.cpu().numpy(), r.cpu().numpy()))
    _check_rms(x, g, yq)


def test_forward_parameters_in_host_memory_are_refused():
    """The forward kernels stage gamma/beta (w) in shared memory with the
    bulk-copy engine, which is given device memory only: host-resident
    parameters return RN_ERR_HOSTMEM before anything is launched."""
    torch = G.torch_cuda()
    import row_wise_normalization_gb300 as rn  # noqa: F401  (loads the library)

    rows, d = 64, 768
    dev = torch.device("cuda", 0)
    x = torch.ones(rows, d, device=dev)
    y = torch.empty_like(x)
    m = torch.empty(rows, device=dev)
    r = torch.empty(rows, device=dev)
    g_dev = torch.ones(d, device=dev)
    g_pin = torch.ones(d).pin_memory()
    s = torch.cuda.current_stream().cuda_stream
    assert capi.ln_fwd(x.data_ptr(), g_pin.data_ptr(), g_dev.data_ptr(), y.data_ptr(),
                       m.data_ptr(), r.data_ptr(), rows, d, 1e-5, s) == capi.RN_ERR_HOSTMEM
    assert capi.ln_fwd(x.data_ptr(), g_dev.data_ptr(), g_pin.data_ptr(), y.data_ptr(),
                       m.data_ptr(), r.data_ptr(), rows, d, 1e-5, s) == capi.RN_ERR_HOSTMEM
    assert capi.rms_fwd(x.data_ptr(), g_pin.data_ptr(), y.data_ptr(), rows, d, 1e-5,
                        s) == capi.RN_ERR_HOSTMEM
    g_np = np.ones(d, np.float32)                       # pageable
    assert capi.rms_fwd(x.data_ptr(), g_np.ctypes.data, y.data_ptr(), rows, d, 1e-5,
                        s) == capi.RN_ERR_HOSTMEM
    torch.cuda.synchronize()


def test_staged_kernel_refuses_rows_in_host_memory():
    """The staged kernel's ring is filled by bulk copies: a call forced onto
    it with x in host memory returns RN_ERR_VARIANT (AUTO never plans it for
    such rows)."""
    torch = G.torch_cuda()
    import row_wise_normalization_gb300 as rn  # noqa: F401

    rows, d = 16, 5000
    dev = torch.device("cuda", 0)
    xh = torch.ones(rows, d).pin_memory()
    y = torch.empty(rows, d, device=dev)
    g = torch.ones(d, device=dev)
    s = torch.cuda.current_stream().cuda_stream
    assert capi.rms_fwd_variant(capi.RN_VARIANT_STAGED, xh.data_ptr(), g.data_ptr(),
                                y.data_ptr(), rows, d, 1e-5, s) == capi.RN_ERR_VARIANT
    xd = xh.to(dev)                                     # the same call on device rows runs
    assert capi.rms_fwd_variant(capi.RN_VARIANT_STAGED, xd.data_ptr(), g.data_ptr(),
                                y.data_ptr(), rows, d, 1e-5, s) == capi.RN_OK
    torch.cuda.synchronize()
    parity.check_y(y.cpu().numpy(), reference.rms_norm(np.ones((rows, d), np.float32),
                                                       np.ones(d, np.float32))[0])


def test_pageable_cpu_tensors_through_the_torch_binding():
    """On a GPU that reads pageable host memory the binding takes ordinary
    CPU tensors for x (and allocates y, mean and rstd beside it); the
    parameters stay on the device."""
    torch = G.torch_cuda()
    import row_wise_normalization_gb300 as rn

    if not capi.pageable_host_access():
        pytest.skip("the GPU does not read pageable host memory")
    wl = workloads.Workload("ln", 2000, 768, seed=39, x_dist="offset", x_std=2.0)
    x = wl.x()
    g, b = wl.params()
    dev = torch.device("cuda", 0)
    gt, bt = torch.from_numpy(g).to(dev), torch.from_numpy(b).to(dev)
    xt = torch.from_numpy(x)
    y, m, r = rn.ln_fwd(xt, gt, bt)
    yq = rn.rms_fwd(xt, gt)
    torch.cuda.synchronize()
    assert not y.is_cuda and not y.is_pinned() and not m.is_cuda
    _check_ln(x, g, b, (y.numpy(), m.numpy(), r.numpy()))
    _check_rms(x, g, yq.numpy())
    with pytest.raises(capi.RowNormError):
        rn.ln_fwd(xt, torch.from_numpy(g), bt)          # parameters in host memory


# ---------------------------------------------------------------------------
# full size, in the launch configuration the benchmark times
# ---------------------------------------------------------------------------
@pytest.mark.slow
@pytest.mark.parametrize("op", ["ln", "rms"])
def test_full_size_32768x8192(op):
    torch = G.torch_cuda()
    import row_wise_normalization_gb300 as rn

    wl = workloads.large_32768x8192(op)
    x = wl.x()
    xt = torch.from_numpy(x).cuda()
    params = [torch.from_numpy(p).cuda() for p in wl.params()]
    if op == "ln":
        y, mean, rstd = rn.ln_fwd(xt, *params)
        mean, rstd = mean.cpu().numpy(), rstd.cpu().numpy()
    else:
        y = rn.rms_fwd(xt, *params)
    torch.cuda.synchronize()
    yh = y.cpu().numpy()
    del xt, y
    p = [t.cpu().numpy() for t in params]
    step = 2048
    for r0 in range(0, wl.rows, step):
        xs = x[r0:r0 + step]
        if op == "ln":
            yr, mr, rr = reference.layer_norm(xs, p[0], p[1], wl.eps)
            parity.check_y(yh[r0:r0 + step], yr, what=f"y rows {r0}+")
            parity.check_mean(mean[r0:r0 + step], mr, xs)
            parity.check_rstd(rstd[r0:r0 + step], rr)
        else:
            yr, _ = reference.rms_norm(xs, p[0], wl.eps)
            parity.check_y(yh[r0:r0 + step], yr, what=f"y rows {r0}+")


# ---------------------------------------------------------------------------
# rows far from zero with a tiny spread: |mean| / sigma = 1e6
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("d", [5, 127, 768, 4096, 20000, 70001])
def test_large_offset_tiny_spread_every_variant(d):
    """x = 1e4 + N(0, 0.01^2): an FP32 mean is only good to half an ulp of
    1e4 (5e-4, 5% of sigma), so deviations taken from the rounded mean would
    miss rstd by ~1e-3 and y by far more than the tolerance; the kernels take
    every deviation in the frame shifted by the row's first element."""
    rng = np.random.default_rng([97, d])
    rows = 24
    x = (1e4 + 0.01 * rng.standard_normal((rows, d))).astype(np.float32)
    g = (1.0 + 0.1 * rng.standard_normal(d)).astype(np.float32)
    b = (0.1 * rng.standard_normal(d)).astype(np.float32)
    for x_off, y_off in ((0, 0), (1, 1), (0, 2)):
        for v in G.variants_for(LN, d, x_off, y_off):
            _check_ln(x, g, b, G.run_ln(x, g, b, variant=v, x_off=x_off, y_off=y_off))
