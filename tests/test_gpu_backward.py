"""LayerNorm / RMSNorm backward against the float64 oracle (GPU).

dx follows the element rule of tests/parity.py; the parameter gradients are
sums over rows and follow the recursive-summation bound of check_colsum. The
longest chain of plain additions a column sum goes through is the rows one row
group takes (at most max(4, rows / 152) on a 152-SM GB300 with the full
workspace) plus the up to 8 groups of a CTA; the CTAs' partials are added with
compensation. CHAIN_PAD covers the last two parts.
"""
import numpy as np
import pytest

import gpu_util as G
import parity
import workloads
from oracle import reference
from row_wise_normalization_gb300 import capi

pytestmark = pytest.mark.gpu
CHAIN_PAD = 16


def _chain(rows):
    return max(4, -(-rows // 152)) + CHAIN_PAD


def _case(rows, d, seed, dist="offset"):
    wl = workloads.Workload("ln", rows, d, seed=seed, x_dist=dist, x_std=2.0)
    x = wl.x()
    dy = workloads.Workload("ln", rows, d, seed=seed + 500).x()
    g, b = wl.params()
    return x, dy, g, b


def _run_ln(x, dy, g, mean32, rstd32, off=0, ws_bytes=None, param_grads=True):
    torch = G.torch_cuda()
    rows, d = x.shape
    bufs = [G.dev_copy(a, off) for a in (dy, x, g, mean32, rstd32)]
    dx = G.Guarded(rows * d, off)
    dg, db = (G.Guarded(d), G.Guarded(d)) if param_grads else (None, None)
    need = capi.bwd_workspace_size(capi.RN_OP_LN, rows, d) if ws_bytes is None else ws_bytes
    ws = torch.empty(max(need // 4, 4), dtype=torch.float32, device="cuda")
    st = capi.ln_bwd(bufs[0][1], bufs[1][1], bufs[2][1], bufs[3][1], bufs[4][1], dx.ptr,
                     dg.ptr if dg else 0, db.ptr if db else 0, rows, d,
                     ws.data_ptr() if param_grads else 0, need if param_grads else 0,
                     G.stream_handle())
    capi.check(st)
    torch.cuda.synchronize()
    return (dx.fetch("dx guard").reshape(rows, d), dg.fetch("dgamma guard") if dg else None,
            db.fetch("dbeta guard") if db else None)


def _run_rms(x, dy, w, off=0, ws_bytes=None):
    torch = G.torch_cuda()
    rows, d = x.shape
    bufs = [G.dev_copy(a, off) for a in (dy, x, w)]
    dx = G.Guarded(rows * d, off)
    dw = G.Guarded(d)
    need = capi.bwd_workspace_size(capi.RN_OP_RMS, rows, d) if ws_bytes is None else ws_bytes
    ws = torch.empty(max(need // 4, 4), dtype=torch.float32, device="cuda")
    st = capi.rms_bwd(bufs[0][1], bufs[1][1], bufs[2][1], dx.ptr, dw.ptr, rows, d,
                      float(np.float32(1e-5)), ws.data_ptr(), need, G.stream_handle())
    capi.check(st)
    torch.cuda.synchronize()
    return dx.fetch("dx guard").reshape(rows, d), dw.fetch("dw guard")


def _check_ln(x, dy, g, out, chain):
    _, mean, rstd = reference.layer_norm(x, g, np.zeros_like(g))
    m32, r32 = mean.astype(np.float32), rstd.astype(np.float32)
    dxr, dgr, dbr = reference.layer_norm_backward(dy, x, g, m32, r32)
    dx, dg, db = out
    parity.check_y(dx, dxr, what="dx")
    if dg is not None:
        xhat = (x.astype(np.float64) - m32[:, None].astype(np.float64)) * r32[:, None]
        parity.check_colsum(dg, dgr, np.abs(dy * xhat).sum(axis=0), chain, "dgamma")
        parity.check_colsum(db, dbr, np.abs(dy.astype(np.float64)).sum(axis=0), chain, "dbeta")


def _stats(x, g):
    _, mean, rstd = reference.layer_norm(x, g, np.zeros_like(g))
    return mean.astype(np.float32), rstd.astype(np.float32)


@pytest.mark.parametrize("d", [1, 3, 31, 128, 768, 1029, 4096, 8192, 12288, 16384])
@pytest.mark.parametrize("off", [0, 1])
def test_ln_backward(d, off):
    rows = 300
    x, dy, g, _ = _case(rows, d, seed=81)
    if off and d > 8192:
        pytest.skip("the scalar layout holds rows of up to 8192 floats")
    m32, r32 = _stats(x, g)
    out = _run_ln(x, dy, g, m32, r32, off=off)
    _check_ln(x, dy, g, out, chain=_chain(rows))


@pytest.mark.parametrize("d", [1, 33, 768, 4096, 8192, 12288, 16384])
@pytest.mark.parametrize("off", [0, 3])
def test_rms_backward(d, off):
    rows = 257
    x, dy, w, _ = _case(rows, d, seed=83)
    if off and d > 8192:
        pytest.skip("the scalar layout holds rows of up to 8192 floats")
    dx, dw = _run_rms(x, dy, w, off=off)
    dxr, dwr = reference.rms_norm_backward(dy, x, w)
    parity.check_y(dx, dxr, what="dx")
    _, r = reference.rms_norm(x, w)
    terms = np.abs(dy.astype(np.float64) * x * r[:, None]).sum(axis=0)
    parity.check_colsum(dw, dwr, terms, _chain(rows), "dw")


@pytest.mark.parametrize("rows,d", [(4096, 768), (32768, 1024), (8192, 4096), (1000, 12288),
                                    (700, 16384)])
def test_backward_larger(rows, d):
    x, dy, g, _ = _case(rows, d, seed=85, dist="normal")
    m32, r32 = _stats(x, g)
    _check_ln(x, dy, g, _run_ln(x, dy, g, m32, r32), chain=_chain(rows))
    dx, dw = _run_rms(x, dy, g)
    dxr, dwr = reference.rms_norm_backward(dy, x, g)
    parity.check_y(dx, dxr, what="rms dx")


def test_backward_small_workspace_and_no_param_grads():
    rows, d = 1000, 512
    x, dy, g, _ = _case(rows, d, seed=87)
    m32, r32 = _stats(x, g)
    # one partial row only: a single CTA takes every row
    out = _run_ln(x, dy, g, m32, r32, ws_bytes=2 * d * 4)
    _check_ln(x, dy, g, out, chain=rows)
    with pytest.raises(capi.RowNormError):
        _run_ln(x, dy, g, m32, r32, ws_bytes=2 * d * 4 - 4)   # less than one partial row
    out = _run_ln(x, dy, g, m32, r32, param_grads=False)
    _check_ln(x, dy, g, out, chain=rows)


@pytest.mark.parametrize("d", [8196, 12288, 16384])
def test_wide_backward_without_param_grads(d):
    """1024-thread rows without parameter gradients: the parameters alone
    take the dynamic shared memory (exactly 48 KB at 12288 floats)."""
    rows = 64
    x, dy, g, _ = _case(rows, d, seed=89)
    m32, r32 = _stats(x, g)
    _check_ln(x, dy, g, _run_ln(x, dy, g, m32, r32, param_grads=False), chain=0)


def test_backward_torch_binding_and_autograd_match():
    torch = G.torch_cuda()
    import row_wise_normalization_gb300 as rn

    rows, d = 500, 1000
    x, dy, g, b = _case(rows, d, seed=89)
    dev = torch.device("cuda", 0)
    xt, dyt, gt, bt = (torch.from_numpy(a).to(dev) for a in (x, dy, g, b))
    _, mean, rstd = rn.ln_fwd(xt, gt, bt)
    dx, dg, db = rn.ln_bwd(dyt, xt, gt, mean, rstd)
    # torch autograd on the same FP32 inputs, in float64
    xr = xt.double().requires_grad_()
    gr = gt.double().requires_grad_()
    br = bt.double().requires_grad_()
    torch.nn.functional.layer_norm(xr, [d], gr, br, 1e-5).backward(dyt.double())
    parity.check_y(dx.cpu().numpy(), xr.grad.cpu().numpy(), what="dx vs autograd")
    np.testing.assert_allclose(dg.cpu().numpy(), gr.grad.cpu().numpy(), rtol=1e-4, atol=2e-4)
    np.testing.assert_allclose(db.cpu().numpy(), br.grad.cpu().numpy(), rtol=1e-4, atol=2e-4)
    dxq, dwq = rn.rms_bwd(dyt, xt, gt)
    xr = xt.double().requires_grad_()
    wr = gt.double().requires_grad_()
    torch.nn.functional.rms_norm(xr, [d], wr, 1e-5).backward(dyt.double())
    parity.check_y(dxq.cpu().numpy(), xr.grad.cpu().numpy(), what="rms dx vs autograd")
    np.testing.assert_allclose(dwq.cpu().numpy(), wr.grad.cpu().numpy(), rtol=1e-4, atol=2e-4)


def test_backward_empty_batch_zeroes_param_grads():
    torch = G.torch_cuda()
    g = torch.ones(64, device="cuda")
    dg = torch.full((64,), 7.0, device="cuda")
    db = torch.full((64,), 7.0, device="cuda")
    buf = torch.zeros(64, device="cuda")
    st = capi.ln_bwd(buf.data_ptr(), buf.data_ptr(), g.data_ptr(), buf.data_ptr(), buf.data_ptr(),
                     0, dg.data_ptr(), db.data_ptr(), 0, 64, 0, 0, G.stream_handle())
    capi.check(st)
    torch.cuda.synchronize()
    assert not dg.any() and not db.any()


def test_backward_repeatable():
    rows, d = 5000, 1024
    x, dy, g, _ = _case(rows, d, seed=91, dist="normal")
    m32, r32 = _stats(x, g)
    a = _run_ln(x, dy, g, m32, r32)
    b = _run_ln(x, dy, g, m32, r32)
    for u, v in zip(a, b):
        assert np.array_equal(u.view(np.uint32), v.view(np.uint32))


# FP32 rows of 256 or 512 threads (3 or 4 quads a thread) on the vector
# layout run the staged backward: single rows, ragged row counts, and a
# one-CTA grid (a workspace of one partial row) whose ring wraps many times.
@pytest.mark.parametrize("d", [3072, 4096, 6144, 8192])
@pytest.mark.parametrize("rows", [1, 9, 1207])
def test_backward_staged_fp32(d, rows):
    x, dy, g, _ = _case(rows, d, seed=93)
    m32, r32 = _stats(x, g)
    capi.device_error(clear=True)
    _check_ln(x, dy, g, _run_ln(x, dy, g, m32, r32), chain=_chain(rows))
    dx, dw = _run_rms(x, dy, g)
    dxr, dwr = reference.rms_norm_backward(dy, x, g)
    parity.check_y(dx, dxr, what="rms dx")
    _, r = reference.rms_norm(x, g)
    terms = np.abs(dy.astype(np.float64) * x * r[:, None]).sum(axis=0)
    parity.check_colsum(dw, dwr, terms, _chain(rows), "dw")
    assert capi.device_error() == 0


def test_backward_staged_fp32_one_cta():
    rows, d = 517, 4096
    x, dy, g, _ = _case(rows, d, seed=95)
    m32, r32 = _stats(x, g)
    _check_ln(x, dy, g, _run_ln(x, dy, g, m32, r32, ws_bytes=2 * d * 4), chain=rows + CHAIN_PAD)
    _check_ln(x, dy, g, _run_ln(x, dy, g, m32, r32, param_grads=False), chain=0)
    dx, dw = _run_rms(x, dy, g, ws_bytes=d * 4)
    dxr, dwr = reference.rms_norm_backward(dy, x, g)
    parity.check_y(dx, dxr, what="rms dx")
    _, r = reference.rms_norm(x, g)
    terms = np.abs(dy.astype(np.float64) * x * r[:, None]).sum(axis=0)
    parity.check_colsum(dw, dwr, terms, rows + CHAIN_PAD, "dw")
    assert capi.device_error() == 0


def test_backward_graph_capture_and_replay_with_new_inputs():
    """The backward launches only on the given stream (row kernel, then the
    column reduction as its programmatic dependent), takes its workspace from
    the caller and neither allocates nor synchronises, so calls can be
    captured into a CUDA graph once (after one ordinary call of each
    configuration) and replayed on new data; a replay gives bit for bit what
    a direct call on the same inputs gives. Register-held and staged rows,
    FP32 and BF16."""
    torch = G.torch_cuda()
    import row_wise_normalization_gb300 as rn

    cases = [(torch.float32, 512, 768), (torch.float32, 600, 4096), (torch.bfloat16, 600, 4096),
             (torch.bfloat16, 12000, 1024)]
    bufs = []
    for i, (dt, rows, d) in enumerate(cases):
        wl = workloads.Workload("ln", rows, d, seed=1100 + i)
        x = torch.from_numpy(wl.x()).to("cuda").to(dt)
        dy = torch.from_numpy(workloads.Workload("ln", rows, d, seed=1150 + i).x()).to("cuda").to(dt)
        g, b = (torch.from_numpy(p_).to("cuda").to(dt) for p_ in wl.params())
        _, m, s = rn.ln_fwd(x, g, b)
        ws = torch.empty(max(capi.bwd_workspace_size(capi.RN_OP_LN, rows, d),
                             capi.bwd_workspace_size(capi.RN_OP_RMS, rows, d)) // 4 + 4,
                         device="cuda")
        outs = (torch.empty_like(x), torch.empty_like(g), torch.empty_like(b),
                torch.empty_like(x), torch.empty_like(g))
        bufs.append((x, dy, g, b, m, s, ws, outs))

    def step():
        for x, dy, g, b, m, s, ws, (dx, dg, db, dxq, dw) in bufs:
            rn.ln_bwd(dy, x, g, m, s, dx=dx, dgamma=dg, dbeta=db, workspace=ws)
            rn.rms_bwd(dy, x, g, dx=dxq, dw=dw, workspace=ws)

    step()                      # one ordinary call of each configuration
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for k in range(2):          # new data in the same buffers, then replay
        for i, ((dt, rows, d), (x, dy, g, b, m, s, ws, outs)) in enumerate(zip(cases, bufs)):
            x.copy_(torch.from_numpy(workloads.Workload("ln", rows, d, seed=1200 + 10 * k + i).x()))
            dy.copy_(torch.from_numpy(workloads.Workload("ln", rows, d, seed=1250 + 10 * k + i).x()))
            rn.ln_fwd(x, g, b, mean=m, rstd=s)
        graph.replay()
        torch.cuda.synchronize()
        for x, dy, g, b, m, s, ws, outs in bufs:
            got = [t.clone() for t in outs]
            dx, dg, db = rn.ln_bwd(dy, x, g, m, s, workspace=ws)
            dxq, dw = rn.rms_bwd(dy, x, g, workspace=ws)
            torch.cuda.synchronize()
            for a, b_ in zip(got, (dx, dg, db, dxq, dw)):
                assert torch.equal(a, b_)
    assert capi.device_error() == 0


@pytest.mark.parametrize("rows,d", [(1024, 4096), (300, 8192), (4096, 768)])
def test_ln_backward_rows_in_pinned_host_memory(rows, d):
    """x, dy and dx in pinned host memory (read and written over the host
    link): the rows that would take the staged ring, which the bulk-copy
    engine fills from device memory only, run the register form instead."""
    torch = G.torch_cuda()
    x, dy, g, _ = _case(rows, d, seed=87)
    m32, r32 = _stats(x, g)
    dev = torch.device("cuda", 0)
    xh = torch.from_numpy(x).pin_memory()
    dyh = torch.from_numpy(dy).pin_memory()
    dxh = torch.full((rows, d), float("nan")).pin_memory()
    gt = torch.from_numpy(g).to(dev)
    mt, rt = torch.from_numpy(m32).to(dev), torch.from_numpy(r32).to(dev)
    dg = torch.full((d,), float("nan"), device=dev)
    db = torch.full((d,), float("nan"), device=dev)
    need = capi.bwd_workspace_size(capi.RN_OP_LN, rows, d)
    ws = torch.empty(max(need // 4, 4), dtype=torch.float32, device=dev)
    capi.check(capi.ln_bwd(dyh.data_ptr(), xh.data_ptr(), gt.data_ptr(), mt.data_ptr(),
                           rt.data_ptr(), dxh.data_ptr(), dg.data_ptr(), db.data_ptr(), rows, d,
                           ws.data_ptr(), need, G.stream_handle()))
    torch.cuda.synchronize()
    _check_ln(x, dy, g, (dxh.numpy(), dg.cpu().numpy(), db.cpu().numpy()), chain=_chain(rows))
