"""Calls that depend on one another, back to back on one stream (GPU).

The forward kernels are launched with programmatic stream serialization: a
kernel may be scheduled while the kernel ahead of it is still running, and
it waits (griddepcontrol.wait) for that kernel to complete before its first
global access. These tests give that wait something to protect:

* a chain in which every call reads the previous call's output (a
  read-after-write across launches), each step checked against the float64
  oracle applied to the previous step's result;
* a ping-pong chain in which every call also overwrites the buffer the call
  before it read (a write-after-read across launches), checked at the end
  against the oracle chain;
* both chains captured once into a CUDA graph and replayed on new inputs;
* ping-pong chains (FP32, 16-bit, with a residual, on pinned host buffers)
  run back to back hundreds of times, directly and from a CUDA graph, each
  result compared bit for bit
  with the same chain run with a device synchronisation after every call
  (the kernels are deterministic, so any difference is a read that the
  dependency wait did not order).

Every output buffer starts as sentinel values, so a call that read its input
before the previous call had written it would see sentinels, not data.
"""
import numpy as np
import pytest

import gpu_util as G
import parity
import workloads
from oracle import reference
from row_wise_normalization_gb300 import capi

pytestmark = pytest.mark.gpu

EPS = float(np.float32(1e-5))

# (variant, rows, d): every forward kernel family, each on a width it takes
CASES = [
    (capi.RN_VARIANT_WARP, 4096, 768),
    (capi.RN_VARIANT_WARP, 512, 128),
    (capi.RN_VARIANT_BLOCK, 1024, 4096),
    (capi.RN_VARIANT_BLOCK, 300, 771),
    (capi.RN_VARIANT_STAGED, 256, 5000),
    (capi.RN_VARIANT_STREAM, 256, 3001),
    (capi.RN_VARIANT_CLUSTER, 64, 65536),
    (capi.RN_VARIANT_AUTO, 16, 200000),
]
STEPS = 4   # alternating LayerNorm and RMSNorm


def _params(d, seed):
    wl = workloads.Workload("ln", 1, d, seed=seed)
    return wl.params()


def _step_call(k, variant, src, dst, params, rows, d, mean, rstd, stream):
    g, b = params
    if k % 2 == 0:
        return capi.ln_fwd_variant(variant, src, g, b, dst, mean, rstd, rows, d, EPS, stream)
    return capi.rms_fwd_variant(variant, src, g, dst, rows, d, EPS, stream)


def _oracle_step(k, x, gh, bh):
    if k % 2 == 0:
        return reference.layer_norm(x, gh, bh, EPS)
    y, _ = reference.rms_norm(x, gh, EPS)
    return y, None, None


def _check_step(k, x, gh, bh, y, mean, rstd):
    yr, mr, rr = _oracle_step(k, x, gh, bh)
    parity.check_y(y, yr, what=f"step {k} y")
    if mr is not None:
        parity.check_mean(mean, mr, x)
        parity.check_rstd(rstd, rr)


@pytest.mark.parametrize("variant,rows,d", CASES)
def test_each_call_reads_the_previous_output(variant, rows, d):
    torch = G.torch_cuda()
    x0 = workloads.Workload("ln", rows, d, seed=900 + d % 97, x_dist="offset", x_std=2.0).x()
    gh, bh = _params(d, seed=901)
    g = G.dev_copy(gh)
    b = G.dev_copy(bh)
    src = G.dev_copy(x0)
    ys = [G.Guarded(rows * d) for _ in range(STEPS)]
    means = [G.Guarded(rows) for _ in range(STEPS)]
    rstds = [G.Guarded(rows) for _ in range(STEPS)]
    s = G.stream_handle()
    prev = src[1]
    for k in range(STEPS):
        capi.check(_step_call(k, variant, prev, ys[k].ptr, (g[1], b[1]), rows, d,
                              means[k].ptr, rstds[k].ptr, s))
        prev = ys[k].ptr
    torch.cuda.synchronize()
    x = x0
    for k in range(STEPS):
        y = ys[k].fetch(f"step {k} guard").reshape(rows, d)
        m = means[k].fetch("mean guard") if k % 2 == 0 else None
        r = rstds[k].fetch("rstd guard") if k % 2 == 0 else None
        _check_step(k, x, gh, bh, y, m, r)
        x = y


def _oracle_chain(x, gh, bh, steps):
    for k in range(steps):
        y, _, _ = _oracle_step(k, x, gh, bh)
        x = y.astype(np.float32)   # each step stores FP32, the next reads it
    return x


@pytest.mark.parametrize("variant,rows,d", CASES[:7])
def test_ping_pong_chain_and_its_graph_replay(variant, rows, d):
    """A <- op(B) <- op(A) ...: every call overwrites the buffer that the
    call before it read. Run directly, then captured into a CUDA graph (after
    that ordinary run, which sets up the launch tables) and replayed twice on
    new inputs."""
    torch = G.torch_cuda()
    import row_wise_normalization_gb300 as rn  # noqa: F401  (loads the library)

    gh, bh = _params(d, seed=911)
    g = torch.from_numpy(gh).to("cuda")
    b = torch.from_numpy(bh).to("cuda")
    a_buf = torch.empty(rows * d, dtype=torch.float32, device="cuda")
    b_buf = torch.empty_like(a_buf)
    mean = torch.empty(rows, dtype=torch.float32, device="cuda")
    rstd = torch.empty_like(mean)

    def chain():
        s = torch.cuda.current_stream().cuda_stream
        bufs = (a_buf, b_buf)
        for k in range(STEPS):
            src, dst = bufs[k % 2], bufs[(k + 1) % 2]
            capi.check(_step_call(k, variant, src.data_ptr(), dst.data_ptr(),
                                  (g.data_ptr(), b.data_ptr()), rows, d, mean.data_ptr(),
                                  rstd.data_ptr(), s))

    def load(seed):
        x0 = workloads.Workload("ln", rows, d, seed=seed, x_dist="offset", x_std=2.0).x()
        a_buf.copy_(torch.from_numpy(x0.reshape(-1)))
        b_buf.fill_(float("nan"))
        return x0

    def check(x0):
        torch.cuda.synchronize()
        got = (a_buf if STEPS % 2 == 0 else b_buf).cpu().numpy().reshape(rows, d)
        parity.check_y(got, _oracle_chain(x0, gh, bh, STEPS), what="chain result")

    x0 = load(913)
    chain()
    check(x0)

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        chain()
    for seed in (915, 917):
        x0 = load(seed)
        graph.replay()
        check(x0)


def test_batched_calls_chained():
    """ln_fwd_batched then rms_fwd_batched on its outputs, then again."""
    torch = G.torch_cuda()
    shapes = [(512, 128), (100, 1000), (33, 96), (7, 1024)]
    xs, params = [], []
    for i, (rows, d) in enumerate(shapes):
        wl = workloads.Workload("ln", rows, d, seed=930 + i, x_dist="offset", x_std=2.0)
        xs.append(wl.x())
        params.append(wl.params())
    dev_x = [G.dev_copy(x) for x in xs]
    dev_p = [(G.dev_copy(g), G.dev_copy(b)) for g, b in params]
    outs = [[G.Guarded(r * d) for (r, d) in shapes] for _ in range(STEPS)]
    s = G.stream_handle()
    src = [p for _, p in dev_x]
    for k in range(STEPS):
        items = [(src[i], dev_p[i][0][1], dev_p[i][1][1], outs[k][i].ptr, 0, 0, r, d)
                 for i, (r, d) in enumerate(shapes)]
        table = capi.problems(items)
        fn = capi.ln_fwd_batched if k % 2 == 0 else capi.rms_fwd_batched
        capi.check(fn(capi.RN_DTYPE_F32, table, len(items), EPS, s))
        src = [o.ptr for o in outs[k]]
    torch.cuda.synchronize()
    for i, (rows, d) in enumerate(shapes):
        gh, bh = params[i]
        x = xs[i]
        for k in range(STEPS):
            y = outs[k][i].fetch(f"problem {i} step {k} guard").reshape(rows, d)
            yr, _, _ = _oracle_step(k, x, gh, bh)
            parity.check_y(y, yr, what=f"problem {i} step {k}")
            x = y


# ---------------------------------------------------------------------------
# back to back against synchronised, bit for bit
# ---------------------------------------------------------------------------
RACE_STEPS = 8
RACE_DIRECT = 200    # chains enqueued behind a device sleep, so they run back to back
RACE_GRAPH = 600     # replays of one captured chain


def _race(torch, reset, chain, outs, graph=True):
    """Runs reset + chain with a sync after every call (twice: the kernels
    must be deterministic), then back to back RACE_DIRECT times and (graph)
    from a CUDA graph RACE_GRAPH times; returns how many of those results
    differ from the synchronised one in any bit of any tensor of ``outs``."""
    capi.device_error(clear=True)
    reset()
    chain(True)
    ref = [o.clone() for o in outs]
    reset()
    chain(True)
    assert all(torch.equal(o, r) for o, r in zip(outs, ref)), \
        "the synchronised chain is not deterministic"
    bad = torch.zeros((), dtype=torch.int64, device="cuda")

    def count():
        diff = torch.zeros((), dtype=torch.bool, device="cuda")
        for o, r in zip(outs, ref):
            diff |= (o != r).any()
        bad.add_(diff.to(torch.int64))

    for _ in range(RACE_DIRECT):
        torch.cuda._sleep(2_000_000)   # the host enqueues the chain meanwhile
        reset()
        chain(False)
        count()
    if graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            reset()
            chain(False)
        for _ in range(RACE_GRAPH):
            g.replay()
            count()
    torch.cuda.synchronize()
    # no bounded wait (parameter copy, cluster exchange, staging ring) ran out
    assert capi.device_error() == 0
    return int(bad.item())


def _race_buffers(torch, rows, d, dtype, seed):
    x0 = workloads.Workload("ln", rows, d, seed=seed, x_dist="offset", x_std=2.0).x()
    gh, bh = _params(d, seed=seed + 1)
    t = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[dtype]
    x0 = torch.from_numpy(x0.reshape(-1)).to("cuda", t)
    g = torch.from_numpy(gh).to("cuda", t)
    b = torch.from_numpy(bh).to("cuda", t)
    mean = torch.empty(rows, dtype=torch.float32, device="cuda")
    rstd = torch.empty_like(mean)
    return x0, g, b, mean, rstd


@pytest.mark.parametrize("dtype,variant,rows,d", [
    ("f32", v, r, d) for (v, r, d) in CASES[:7]] + [
    ("f32", capi.RN_VARIANT_AUTO, 4096, 768),
    ("f32", capi.RN_VARIANT_AUTO, 8192, 768),
    ("f32", capi.RN_VARIANT_AUTO, 2048, 4096),
    ("f32", capi.RN_VARIANT_AUTO, 200, 8192),    # three 256-thread rows a CTA
    ("f32", capi.RN_VARIANT_AUTO, 700, 2001),    # unaligned rows, parameters by bulk copy
    ("bf16", capi.RN_VARIANT_AUTO, 4096, 768),
    ("bf16", capi.RN_VARIANT_AUTO, 1024, 4096),
    ("f16", capi.RN_VARIANT_AUTO, 2048, 2048),
    ("bf16", capi.RN_VARIANT_AUTO, 32, 40000),
])
def test_back_to_back_chains_match_synchronised_ones(dtype, variant, rows, d):
    """A <- op(B) <- op(A) ..., LayerNorm and RMSNorm alternating: every call
    reads what the call before it wrote and overwrites what it read."""
    torch = G.torch_cuda()
    import row_wise_normalization_gb300 as rn  # noqa: F401  (loads the library)

    code = {"f32": capi.RN_DTYPE_F32, "bf16": capi.RN_DTYPE_BF16, "f16": capi.RN_DTYPE_F16}[dtype]
    x0, g, b, mean, rstd = _race_buffers(torch, rows, d, dtype, seed=941)
    bufs = (torch.empty_like(x0), torch.empty_like(x0))

    def reset():
        bufs[0].copy_(x0)
        bufs[1].fill_(float("nan"))

    def chain(sync):
        s = torch.cuda.current_stream().cuda_stream
        for k in range(RACE_STEPS):
            src, dst = bufs[k % 2], bufs[(k + 1) % 2]
            if k % 2 == 0:
                st = capi.ln_fwd_typed(code, variant, src.data_ptr(), g.data_ptr(), b.data_ptr(),
                                       dst.data_ptr(), mean.data_ptr(), rstd.data_ptr(), rows, d,
                                       EPS, s)
            else:
                st = capi.rms_fwd_typed(code, variant, src.data_ptr(), g.data_ptr(),
                                        dst.data_ptr(), rows, d, EPS, s)
            capi.check(st)
            if sync:
                torch.cuda.synchronize()

    assert _race(torch, reset, chain, (bufs[RACE_STEPS % 2],)) == 0


@pytest.mark.parametrize("variant,rows,d", [
    (capi.RN_VARIANT_AUTO, 4096, 768),
    (capi.RN_VARIANT_BLOCK, 1024, 4096),
    (capi.RN_VARIANT_AUTO, 64, 20000),
])
def test_back_to_back_residual_chains_match_synchronised_ones(variant, rows, d):
    """Residual calls: each reads the previous call's y as x and its h as the
    residual, and writes h and y over the two buffers the previous call read."""
    torch = G.torch_cuda()
    import row_wise_normalization_gb300 as rn  # noqa: F401

    x0, g, b, mean, rstd = _race_buffers(torch, rows, d, "f32", seed=951)
    r0 = torch.flip(x0, (0,)).contiguous()
    pair = ((torch.empty_like(x0), torch.empty_like(x0)),
            (torch.empty_like(x0), torch.empty_like(x0)))   # (x or y, residual or h)

    def reset():
        pair[0][0].copy_(x0)
        pair[0][1].copy_(r0)
        pair[1][0].fill_(float("nan"))
        pair[1][1].fill_(float("nan"))

    def chain(sync):
        s = torch.cuda.current_stream().cuda_stream
        for k in range(RACE_STEPS):
            (xi, ri), (yo, ho) = pair[k % 2], pair[(k + 1) % 2]
            if k % 2 == 0:
                st = capi.ln_fwd_residual_variant(variant, xi.data_ptr(), ri.data_ptr(),
                                                  g.data_ptr(), b.data_ptr(), ho.data_ptr(),
                                                  yo.data_ptr(), mean.data_ptr(),
                                                  rstd.data_ptr(), rows, d, EPS, s)
            else:
                st = capi.rms_fwd_residual_variant(variant, xi.data_ptr(), ri.data_ptr(),
                                                   g.data_ptr(), ho.data_ptr(), yo.data_ptr(),
                                                   rows, d, EPS, s)
            capi.check(st)
            if sync:
                torch.cuda.synchronize()

    assert _race(torch, reset, chain, pair[RACE_STEPS % 2]) == 0


@pytest.mark.parametrize("dtype,rows,d", [
    ("f32", 4096, 768),    # warp rows
    ("f32", 2048, 4096),   # a CTA per row
    ("f32", 200, 8192),    # three 256-thread rows a CTA
    ("bf16", 1024, 4096),
    ("f32", 700, 2001),    # unaligned rows
])
def test_back_to_back_host_resident_chains_match_synchronised_ones(dtype, rows, d):
    """The ping-pong chain on pinned host buffers, which the kernels read and
    write over the host link on their persistent grid: every call reads
    what the call before it wrote to host memory. The buffers are reset and
    the result brought back by stream-ordered copies, so that the chain and
    its checks stay on the stream (not captured into a graph: the copies
    between pinned and device memory are torch's, outside the library)."""
    torch = G.torch_cuda()
    import row_wise_normalization_gb300 as rn  # noqa: F401

    code = {"f32": capi.RN_DTYPE_F32, "bf16": capi.RN_DTYPE_BF16}[dtype]
    x0, g, b, mean, rstd = _race_buffers(torch, rows, d, dtype, seed=961)
    nan = torch.full_like(x0, float("nan"))
    bufs = (torch.empty(x0.shape, dtype=x0.dtype).pin_memory(),
            torch.empty(x0.shape, dtype=x0.dtype).pin_memory())
    mirror = torch.empty_like(x0)

    def reset():
        bufs[0].copy_(x0, non_blocking=True)
        bufs[1].copy_(nan, non_blocking=True)

    def chain(sync):
        s = torch.cuda.current_stream().cuda_stream
        for k in range(RACE_STEPS):
            src, dst = bufs[k % 2], bufs[(k + 1) % 2]
            if k % 2 == 0:
                st = capi.ln_fwd_typed(code, capi.RN_VARIANT_AUTO, src.data_ptr(), g.data_ptr(),
                                       b.data_ptr(), dst.data_ptr(), mean.data_ptr(),
                                       rstd.data_ptr(), rows, d, EPS, s)
            else:
                st = capi.rms_fwd_typed(code, capi.RN_VARIANT_AUTO, src.data_ptr(), g.data_ptr(),
                                        dst.data_ptr(), rows, d, EPS, s)
            capi.check(st)
            if sync:
                torch.cuda.synchronize()
        mirror.copy_(bufs[RACE_STEPS % 2], non_blocking=True)
        if sync:
            torch.cuda.synchronize()

    assert _race(torch, reset, chain, (mirror,), graph=False) == 0
    # and the chain's result is the oracle chain's
    torch.cuda.synchronize()
    if dtype == "f32":
        got = mirror.cpu().numpy().reshape(rows, d)
        want = _oracle_chain(x0.cpu().numpy().reshape(rows, d), g.cpu().numpy(),
                             b.cpu().numpy(), RACE_STEPS)
        parity.check_y(got, want, what="host chain")
