"""Batched small problems (ln_fwd_batched / rms_fwd_batched) and CUDA-graph
capture of the single-call entry points (GPU).

A batch mixes every kind of problem the call sorts: widths the batched
kernel takes (d <= 1024, x and y in one 16-byte phase, at any phase) and
ones that get launches of their own (wider rows, x and y in different
phases), empty problems, and more than one table's worth (128) of problems.
Every output is checked against the oracle and, bit for bit, against the
single call (ln_fwd_typed / rms_fwd_typed) on the same inputs.
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
F32, BF16 = capi.RN_DTYPE_F32, capi.RN_DTYPE_BF16

# rows, d, x_off, y_off (elements)
SHAPES = [(512, 128, 0, 0), (7, 1, 0, 0), (33, 3, 1, 1), (64, 31, 0, 2), (100, 33, 3, 3),
          (300, 768, 0, 0), (17, 1000, 2, 2), (9, 1024, 0, 0), (5, 1024, 1, 1), (0, 64, 0, 0),
          (11, 1025, 0, 0), (40, 4096, 0, 0), (13, 768, 1, 0), (3, 128, 2, 3)]


class _Problem:
    def __init__(self, op, dtype, rows, d, x_off, y_off, seed):
        torch = G.torch_cuda()
        self.rows, self.d = rows, d
        wl = workloads.Workload("ln" if op == LN else "rms", rows, d, seed=seed, x_dist="offset",
                                x_std=2.0)
        x = wl.x()
        params = wl.params()
        if dtype == F32:
            self.xw, self.pw = x, params
            self.xbuf, xp = G.dev_copy(x, x_off)
            self.pbufs = [G.dev_copy(p_) for p_ in params]
            self.es, fill, tdt = 4, parity.SENTINEL_BITS, torch.int32
        else:
            xb, self.xw = workloads.to_storage(x, "bf16")
            pb = [workloads.to_storage(p_, "bf16") for p_ in params]
            self.pw = [b[1] for b in pb]
            self.xbuf, xp = G.dev_copy16(xb, x_off)
            self.pbufs = [G.dev_copy16(b[0]) for b in pb]
            self.es, fill, tdt = 2, 0x7FC1, torch.int16
        self.fill = int(np.array([fill], np.uint32 if dtype == F32 else np.uint16).view(
            np.int32 if dtype == F32 else np.int16)[0])
        self.head = parity.GUARD + y_off
        n = rows * d
        self.ybuf = torch.full((self.head + n + parity.GUARD,), self.fill, dtype=tdt, device="cuda")
        self.m, self.s = G.Guarded(max(rows, 1)), G.Guarded(max(rows, 1))
        self.xp = xp
        self.yp = self.ybuf.data_ptr() + self.es * self.head
        self.item = (xp, self.pbufs[0][1], self.pbufs[1][1] if op == LN else 0, self.yp,
                     self.m.ptr if op == LN else 0, self.s.ptr if op == LN else 0, rows, d)

    def y(self):
        h = self.ybuf.cpu().numpy()
        n = self.rows * self.d
        if not (np.all(h[:self.head] == self.fill) and np.all(h[self.head + n:] == self.fill)):
            raise parity.ParityError("y guard overwritten")
        return h[self.head:self.head + n].reshape(self.rows, self.d)


def _single(op, dtype, pb):
    """The single call on the same inputs, its y at the same 16-byte phase as
    the batch's (the phase picks the kernel path)."""
    torch = G.torch_cuda()
    n = pb.rows * pb.d
    y = torch.empty(pb.head + n + 16, dtype=pb.ybuf.dtype, device="cuda")
    yp = y.data_ptr() + pb.es * pb.head
    m = torch.empty(max(pb.rows, 1), device="cuda")
    s = torch.empty(max(pb.rows, 1), device="cuda")
    if op == LN:
        st = capi.ln_fwd_typed(dtype, 0, pb.xp, pb.pbufs[0][1], pb.pbufs[1][1], yp,
                               m.data_ptr(), s.data_ptr(), pb.rows, pb.d, float(np.float32(1e-5)),
                               G.stream_handle())
    else:
        st = capi.rms_fwd_typed(dtype, 0, pb.xp, pb.pbufs[0][1], yp, pb.rows, pb.d,
                                float(np.float32(1e-5)), G.stream_handle())
    capi.check(st)
    torch.cuda.synchronize()
    return y.cpu().numpy()[pb.head:pb.head + n].reshape(pb.rows, pb.d), \
        m.cpu().numpy()[:pb.rows], s.cpu().numpy()[:pb.rows]


def _run_batch(op, dtype, shapes, seed0):
    torch = G.torch_cuda()
    probs = [_Problem(op, dtype, *sh, seed=seed0 + i) for i, sh in enumerate(shapes)]
    fn = capi.ln_fwd_batched if op == LN else capi.rms_fwd_batched
    capi.check(fn(dtype, capi.problems([p_.item for p_ in probs]), len(probs),
                  float(np.float32(1e-5)), G.stream_handle()))
    torch.cuda.synchronize()
    for i, pb in enumerate(probs):
        if pb.rows == 0:
            pb.y()
            continue
        y = pb.y()
        yv = y.view(np.float32) if dtype == F32 else y.view(np.uint16)
        if op == LN:
            yr, mr, sr = reference.layer_norm(pb.xw, *pb.pw)
            m, s = pb.m.fetch("mean guard")[:pb.rows], pb.s.fetch("rstd guard")[:pb.rows]
            parity.check_mean(m, mr, pb.xw, what=f"problem {i} mean")
            parity.check_rstd(s, sr, what=f"problem {i} rstd")
        else:
            yr, _ = reference.rms_norm(pb.xw, *pb.pw)
        if dtype == F32:
            parity.check_y(yv, yr, what=f"problem {i} y")
        else:
            parity.check_y_storage(yv, yr, "bf16", what=f"problem {i} y")
        ys, ms, ss = _single(op, dtype, pb)
        assert np.array_equal(y.reshape(-1).view(np.uint8),
                              np.ascontiguousarray(ys).reshape(-1).view(np.uint8)), \
            f"problem {i}: batched and single-call y differ"
        if op == LN:
            assert np.array_equal(m.view(np.uint32), ms.view(np.uint32)), f"problem {i} mean bits"
            assert np.array_equal(s.view(np.uint32), ss.view(np.uint32)), f"problem {i} rstd bits"


@pytest.mark.parametrize("op", [LN, RMS])
def test_batched_f32_mixed(op):
    _run_batch(op, F32, SHAPES, 401)


@pytest.mark.parametrize("op", [LN, RMS])
def test_batched_bf16_mixed(op):
    shapes = [(rows, d, 2 * xo, 2 * yo) for rows, d, xo, yo in SHAPES]
    _run_batch(op, BF16, shapes, 451)


def test_batched_more_than_one_table():
    # 300 problems: three tables, some rows empty, widths 1..1024
    rng = np.random.default_rng(7)
    shapes = [(int(rng.integers(0, 20)), int(rng.integers(1, 1025)), 0, 0) for _ in range(300)]
    _run_batch(LN, F32, shapes, 1000)


def test_batched_torch_binding():
    torch = G.torch_cuda()
    import row_wise_normalization_gb300 as rn

    probs, refs = [], []
    for i in range(64):
        wl = workloads.Workload("ln", 512, 128, seed=500 + i)
        x = torch.from_numpy(wl.x()).to("cuda")
        g, b = (torch.from_numpy(p_).to("cuda") for p_ in wl.params())
        probs.append((x, g, b))
    outs = rn.ln_fwd_batched(probs)
    for (x, g, b), (y, m, s) in zip(probs, outs):
        yr, mr, sr = reference.layer_norm(x.cpu().numpy(), g.cpu().numpy(), b.cpu().numpy())
        parity.check_y(y.cpu().numpy(), yr)
        parity.check_rstd(s.cpu().numpy(), sr)
    qs = rn.rms_fwd_batched([(x, g) for x, g, _ in probs])
    for (x, g, _), q in zip(probs, qs):
        parity.check_y(q.cpu().numpy(), reference.rms_norm(x.cpu().numpy(), g.cpu().numpy())[0])


def test_graph_capture_and_replay_with_new_inputs():
    """The forward entry points launch kernels only on the given stream and
    neither allocate nor synchronise, so a sequence of calls can be captured
    into a CUDA graph once (after one ordinary call of each configuration,
    which sets up the per-device launch tables) and replayed on new data."""
    torch = G.torch_cuda()
    import row_wise_normalization_gb300 as rn

    shapes = [(512, 128), (4096, 768), (64, 8193), (1024, 20000)]
    ins = []
    for i, (rows, d) in enumerate(shapes):
        wl = workloads.Workload("ln", rows, d, seed=600 + i)
        ins.append([torch.from_numpy(a).to("cuda") for a in (wl.x(),) + wl.params()])
    tiny = [(torch.from_numpy(workloads.Workload("ln", 256, 64, seed=650 + i).x()).to("cuda"),)
            for i in range(8)]
    wt = torch.ones(64, device="cuda")
    outs = [(torch.empty_like(x), torch.empty(x.shape[0], device="cuda"),
             torch.empty(x.shape[0], device="cuda"), torch.empty_like(x)) for x, g, b in ins]

    def step():
        for (x, g, b), (y, m, s, q) in zip(ins, outs):
            rn.ln_fwd(x, g, b, y=y, mean=m, rstd=s)
            rn.rms_fwd(x, g, y=q)
        return rn.rms_fwd_batched([(t[0], wt) for t in tiny])

    step()                      # one ordinary call of each configuration
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        batched_out = step()
    for k in range(2):          # new data in the same buffers, then replay
        for i, ((x, g, b), (rows, d)) in enumerate(zip(ins, shapes)):
            x.copy_(torch.from_numpy(workloads.Workload("ln", rows, d, seed=700 + 10 * k + i).x()))
        for i, t in enumerate(tiny):
            t[0].copy_(torch.from_numpy(workloads.Workload("ln", 256, 64, seed=800 + 10 * k + i).x()))
        graph.replay()
        torch.cuda.synchronize()
        for (x, g, b), (y, m, s, q) in zip(ins, outs):
            xh, gh, bh = x.cpu().numpy(), g.cpu().numpy(), b.cpu().numpy()
            yr, mr, sr = reference.layer_norm(xh, gh, bh)
            parity.check_y(y.cpu().numpy(), yr)
            parity.check_mean(m.cpu().numpy(), mr, xh)
            parity.check_rstd(s.cpu().numpy(), sr)
            parity.check_y(q.cpu().numpy(), reference.rms_norm(xh, gh)[0])
        for t, q in zip(tiny, batched_out):
            parity.check_y(q.cpu().numpy(), reference.rms_norm(t[0].cpu().numpy(),
                                                               wt.cpu().numpy())[0])


def test_batched_parameters_in_host_memory_are_refused_before_any_launch():
    """A table whose last problem has its gamma in pinned host memory
    returns RN_ERR_HOSTMEM, and the earlier problems' outputs stay
    untouched: the check runs before the first launch."""
    torch = G.torch_cuda()
    import row_wise_normalization_gb300 as rn  # noqa: F401  (loads the library)

    dev = torch.device("cuda", 0)
    items, ys = [], []
    for i, d in enumerate((128, 700, 5000)):
        x = torch.ones(16, d, device=dev)
        g = torch.ones(d, device=dev) if i < 2 else torch.ones(d).pin_memory()
        b = torch.zeros(d, device=dev)
        y = torch.full((16, d), float("nan"), device=dev)
        m = torch.full((16,), float("nan"), device=dev)
        r = torch.full((16,), float("nan"), device=dev)
        items.append((x, g, b, y, m, r))
        ys.append(y)
    table = capi.problems([(x.data_ptr(), g.data_ptr(), b.data_ptr(), y.data_ptr(),
                            m.data_ptr(), r.data_ptr(), 16, x.shape[1])
                           for x, g, b, y, m, r in items])
    st = capi.ln_fwd_batched(capi.RN_DTYPE_F32, table, len(items), 1e-5,
                             torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == capi.RN_ERR_HOSTMEM
    assert all(torch.isnan(y).all() for y in ys), "a problem was launched before the refusal"
