#!/usr/bin/env python3
"""Benchmark of the row-wise normalization forward pass on GB300.

Headline workload: LayerNorm FP32 forward, rows = 4096, d = 768 (the pages'
harness shape), x ~ N(0,1), gamma ~ N(1,0.1), beta ~ N(0,0.1), seed 1,
eps = 1e-5. One step = one ln_fwd call (one kernel) over one batch of that
shape. The K timed steps run back to back over distinct copies of the batch
that together hold more than twice the L2, so that every step reads an x
that is not in L2 (inputs larger than L2, no flush inside the timed
region); one pair of CUDA events brackets all K steps, and `value` is the
whole job's throughput. Metric: algorithmic GB/s (4*rows*d read +
4*rows*d written + 8*d parameters + 8*rows statistics) per step time, and
its fraction of the measured HBM copy bandwidth.

Also reported in the same JSON line: the e2e number (the same K steps
through the C entry point with x read from, and the results written to,
pinned host memory), the oracle on the host cores (``cpu_baseline``), the
headline shape timed one launch at a time after an L2 flush (a 2x-L2 buffer
written before every launch, outside the events), with a clean L2, warm, as
a CUDA graph, the empty-kernel launch floor, a device copy of the same
bytes under the same protocols, the large / sweep shapes under three
protocols for both LayerNorm and RMSNorm, the small shapes against the
launch-latency floor, the fused residual add against add-then-normalise,
BF16/FP16 storage, the backward (dx plus parameter gradients), and 64 small
problems as single calls, a CUDA graph of them and one batched call. The
line ends with ``summary``: every fraction the targets are judged on, each
named with its protocol.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank normalises its own batches of the same
shape (rows are independent, so there is no collective on the data path);
the step time is the max over ranks and ``value`` counts the bytes of all
ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import glob
import json
import os
import platform
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads  # noqa: E402

METRIC = "LayerNorm/RMSNorm FP32 GB/s and % of HBM roofline (cold L2) at 1 GB300"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
PROFILES = os.path.join(ROOT, "profiles")


# ---------------------------------------------------------------------------
# bytes and peaks
# ---------------------------------------------------------------------------
def algorithmic_bytes(op: str, rows: int, d: int) -> int:
    """Bytes the operation must move at least once: x in, y out, the
    parameter vectors, and (LayerNorm) the per-row mean and rstd."""
    if op == "ln":
        return 8 * rows * d + 8 * d + 8 * rows
    return 8 * rows * d + 4 * d


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# Sources of the FP32 register-held forward kernels (the headline kernel's
# family): a change to any of them invalidates recorded ncu counters.
KERNEL_SOURCES = ("rn_reg.cuh", "rn_device.cuh", "rn_params.h", "reg_ln_v4.cu", "reg_ln_v4_al.cu",
                  "reg_ln_v4_pp.cu", "reg_ln_v1.cu", "reg_rms_v4.cu", "reg_rms_v4_al.cu",
                  "reg_rms_v4_pp.cu", "reg_rms_v1.cu", "reg_ps_f32.cu")


CLOCK_WINDOW_S = 0.3


def source_hash() -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        h.update(name.encode())
        h.update(open(os.path.join(ROOT, "row_wise_normalization_gb300", "csrc", name), "rb").read())
    return h.hexdigest()[:16]


def plan_key(pl: dict) -> str:
    return "{variant}/vec{vec}/slots{slots}/tpr{threads_per_row}/cta{threads_per_cta}".format(**pl)


def recorded_traffic(kernel_tag: str, current_hash: str, plan: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel sources and launch plan (else None)."""
    path = os.path.join(PROFILES, f"{kernel_tag}.traffic.txt")
    if not os.path.exists(path):
        return None
    kv = {}
    for line in open(path):
        if "=" in line and not line.lstrip().startswith("#"):
            k, v = line.split("=", 1)
            kv[k.strip()] = v.strip()
    if kv.get("source_hash") != current_hash or kv.get("plan") != plan:
        return None
    try:
        return int(kv["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, interval_ms: int = 20):
        self.gpu = gpu_index
        self.interval = interval_ms
        self.proc = None
        self.out = None
        self.windows = []

    def start(self):
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.interval)],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)

    def mark(self, name, t0, t1):
        self.windows.append((name, t0, t1))

    def stop(self):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.out.flush()

    def _samples(self):
        rows = []
        try:
            with open(self.out.name) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) < 10:
                        continue
                    try:
                        ts = time.mktime(time.strptime(parts[0].split(".")[0],
                                                       "%Y/%m/%d %H:%M:%S"))
                        frac = float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                        rows.append(dict(t=ts + frac, sm=float(parts[2]), smax=float(parts[3]),
                                         active=parts[5], hw=parts[6], hwt=parts[7],
                                         swt=parts[8], swp=parts[9]))
                    except (ValueError, IndexError):
                        continue
        finally:
            try:
                os.unlink(self.out.name)
            except OSError:
                pass
        return rows

    def summary(self, window: str):
        rows = self._samples()
        sel = []
        for name, t0, t1 in self.windows:
            if name == window:
                sel = [r for r in rows if t0 - 0.01 <= r["t"] <= t1 + 0.01]
        label = (f"{window} steps (continued untimed with the same step to "
                 f"{int(CLOCK_WINDOW_S * 1000)} ms when shorter)")
        if len(sel) < 3:
            # the timed region is shorter than a few sampling intervals: use
            # every sample taken while the benchmark kept the GPU busy
            sel = [r for r in rows
                   if any(t0 <= r["t"] <= t1 for _, t0, t1 in self.windows)]
            label = "all measured regions"
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "window": "none (nvidia-smi unavailable)"}
        reasons = set()
        for r in sel:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("swp", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in sel),
                "sm_max_mhz": max(r["smax"] for r in sel),
                "reasons": sorted(reasons), "samples": len(sel), "window": label}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
class Flusher:
    """Writes a buffer of twice the L2 size, leaving no input in L2.

    mode "write": L2 is left full of dirty lines of that buffer, which the
    timed kernel's own traffic must write back (the conservative cold case).
    mode "clean": a second buffer of twice the L2 size is then read, so the
    timed kernel starts with clean, unrelated lines in L2.
    """

    def __init__(self, torch, device, mode="write"):
        props = torch.cuda.get_device_properties(device)
        l2 = getattr(props, "L2_cache_size", 0) or (128 << 20)
        self.nbytes = 2 * l2
        self.mode = mode
        self.buf = torch.empty(self.nbytes // 4, dtype=torch.float32, device=device)
        self.rbuf = (torch.ones(self.nbytes // 4, dtype=torch.float32, device=device)
                     if mode == "clean" else None)
        self.sink = torch.empty(1, dtype=torch.float32, device=device)

    def __call__(self):
        self.buf.fill_(1.0)
        if self.rbuf is not None:
            self.sink.copy_(self.rbuf.amax().view(1))


HOST_LEAD_CYCLES_PER_STEP = 100_000  # ~50 us of SM clock per step


def time_launches(torch, launch, steps, flush=None):
    """Per-launch device time (ms) of `launch`, CUDA events on the current
    stream; `flush` (if any) runs before each launch, outside the events.

    Without a flush the GPU would finish each short launch before the host
    has enqueued the next event and launch (a call through Python costs
    several microseconds of host time), and the events would time the host.
    So a spin kernel that keeps the stream busy for about 50 us per step is
    enqueued first: the host runs ahead of the GPU and every event pair
    brackets GPU work only. With a flush, the flush itself keeps the GPU
    busy for longer than the host needs per step."""
    s = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    if flush is None:
        torch.cuda._sleep(HOST_LEAD_CYCLES_PER_STEP * steps)
    for a, b in ev:
        if flush is not None:
            flush()
        a.record(s)
        launch()
        b.record(s)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


class LnCase:
    """Device-resident inputs/outputs of one workload and its C-ABI launch."""

    def __init__(self, torch, wl, device):
        from row_wise_normalization_gb300 import capi

        self.capi = capi
        self.wl = wl
        self.torch = torch
        x = wl.x()
        self.x = torch.from_numpy(x).to(device)
        self.params = [torch.from_numpy(p).to(device) for p in wl.params()]
        self.y = torch.empty_like(self.x)
        self.mean = torch.empty(wl.rows, dtype=torch.float32, device=device)
        self.rstd = torch.empty(wl.rows, dtype=torch.float32, device=device)
        self.bytes = algorithmic_bytes(wl.op, wl.rows, wl.d)
        self.x_host = x

    def launch(self):
        s = self.torch.cuda.current_stream().cuda_stream
        c = self.capi
        if self.wl.op == "ln":
            st = c.ln_fwd(self.x.data_ptr(), self.params[0].data_ptr(), self.params[1].data_ptr(),
                          self.y.data_ptr(), self.mean.data_ptr(), self.rstd.data_ptr(),
                          self.wl.rows, self.wl.d, self.wl.eps, s)
        else:
            st = c.rms_fwd(self.x.data_ptr(), self.params[0].data_ptr(), self.y.data_ptr(),
                           self.wl.rows, self.wl.d, self.wl.eps, s)
        if st != c.RN_OK:
            c.check(st)

    def plan(self):
        c = self.capi
        op = c.RN_OP_LN if self.wl.op == "ln" else c.RN_OP_RMS
        p = c.plan(op, c.RN_VARIANT_AUTO, self.wl.d, self.x.data_ptr(), self.y.data_ptr())
        return {"variant": c.variant_name(p.variant), "vec": p.vec, "slots": p.slots,
                "threads_per_row": p.threads_per_row, "threads_per_cta": p.threads_per_cta}


NAMED = {
    "ln_512x128": workloads.ln_512x128,
    "ln_4096x768": workloads.ln_4096x768,
    "ln_32768x8192": lambda: workloads.large_32768x8192("ln"),
    "rms_32768x8192": lambda: workloads.large_32768x8192("rms"),
}


def latency_bound_check(torch, capi, wl, device, flush, peak, steps):
    """Is a small shape launch-latency-bound? Its cold time must be within
    the same-grid empty kernel's time plus its bytes at the measured HBM
    bandwidth plus 1 us, and its CUDA-graph-replayed time per launch within
    1.5x the empty kernel's replayed the same way. A device copy of the same
    bytes, timed both ways, is reported beside it: unlike the empty kernel
    it pays the DRAM round trip and the store drain a real kernel pays."""
    c = LnCase(torch, wl, device)
    pl = c.plan()
    rpc = max(1, pl["threads_per_cta"] // pl["threads_per_row"])
    grid = max(1, -(-wl.rows // rpc))

    def empty():
        capi.check(capi.launch_empty(grid, pl["threads_per_cta"],
                                     torch.cuda.current_stream().cuda_stream))

    def graph_per_launch(f):
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            f()
            torch.cuda.synchronize()
            with torch.cuda.graph(g, stream=s):
                for _ in range(64):
                    f()
        torch.cuda.current_stream().wait_stream(s)
        g.replay()
        torch.cuda.synchronize()
        return statistics.median(time_launches(torch, g.replay, 15)) / 64

    ycopy = torch.empty_like(c.x)

    def copy():
        ycopy.copy_(c.x)

    out = {}
    for name, f in (("kernel", c.launch), ("empty", empty), ("copy", copy)):
        for _ in range(3):
            flush()
            f()
        out[name] = statistics.median(time_launches(torch, f, steps, flush))
        out[name + "_graph"] = graph_per_launch(f)
    at_peak_ms = c.bytes / (peak * 1e9) * 1e3
    ok = (out["kernel"] <= out["empty"] + at_peak_ms + 1e-3 and
          out["kernel_graph"] <= 1.5 * out["empty_graph"])
    return {"workload": wl.tag or f"{wl.op}_{wl.rows}x{wl.d}", "plan": pl, "grid": grid,
            "kernel_cold_us": 1e3 * out["kernel"], "empty_cold_us": 1e3 * out["empty"],
            "bytes_at_measured_peak_us": 1e3 * at_peak_ms,
            "kernel_graph_us_per_launch": 1e3 * out["kernel_graph"],
            "empty_graph_us_per_launch": 1e3 * out["empty_graph"],
            "launch_latency_bound": ok,
            "same_size_copy_cold_us": 1e3 * out["copy"],
            "same_size_copy_graph_us_per_launch": 1e3 * out["copy_graph"],
            "kernel_over_copy_cold": out["kernel"] / out["copy"],
            "kernel_over_copy_graph": out["kernel_graph"] / out["copy_graph"]}


class BatchSets:
    """Distinct copies of one workload's batch (x, y, mean, rstd), enough of
    them that together they are larger than twice the L2, used round robin:
    a call on set i reads an x that later calls have pushed out of L2 (the
    dirty y lines of earlier calls are written back during later ones, as in
    a real pipeline). `host` keeps the sets in pinned host memory instead
    (the kernel then reads x and writes y over the host link)."""

    def __init__(self, torch, case, device, host=False):
        props = torch.cuda.get_device_properties(device)
        l2 = getattr(props, "L2_cache_size", 0) or (128 << 20)
        wl = case.wl
        self.torch, self.case, self.wl = torch, case, wl
        self.per_set = 2 * case.x.numel() * case.x.element_size() + 8 * wl.rows
        self.n = max(2, -(-2 * l2 // self.per_set) + 1)
        src = torch.from_numpy(case.x_host) if host else case.x
        self.sets = []
        for _ in range(self.n):
            if host:
                x = src.clone().pin_memory()
                y = torch.empty_like(x).pin_memory()
                m = torch.empty(wl.rows, dtype=torch.float32).pin_memory()
                r = torch.empty(wl.rows, dtype=torch.float32).pin_memory()
            else:
                x = src.clone()
                y = torch.empty_like(x)
                m = torch.empty(wl.rows, dtype=torch.float32, device=device)
                r = torch.empty(wl.rows, dtype=torch.float32, device=device)
            self.sets.append((x, y, m, r))

    def launch(self, i):
        """One call of the C entry point (ln_fwd / rms_fwd) on set i mod n."""
        x, y, m, r = self.sets[i % self.n]
        c = self.case.capi
        wl = self.wl
        s = self.torch.cuda.current_stream().cuda_stream
        p = self.case.params
        if wl.op == "ln":
            st = c.ln_fwd(x.data_ptr(), p[0].data_ptr(), p[1].data_ptr(), y.data_ptr(),
                          m.data_ptr(), r.data_ptr(), wl.rows, wl.d, wl.eps, s)
        else:
            st = c.rms_fwd(x.data_ptr(), p[0].data_ptr(), y.data_ptr(), wl.rows, wl.d, wl.eps, s)
        if st != c.RN_OK:
            c.check(st)

    def span(self, steps, first=0):
        """Device time (ms) of `steps` calls back to back (sets first, first +
        1, ...), one event pair around all of them; a GPU spin enqueued first
        lets the host enqueue every call before the GPU reaches them, so the
        events time GPU work only."""
        torch = self.torch
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(HOST_LEAD_CYCLES_PER_STEP * steps)
        a.record()
        for i in range(steps):
            self.launch(first + i)
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b)


def graph_span(torch, sets, steps, reps=5):
    """The same `steps` back-to-back calls captured once into a CUDA graph
    and replayed; median device time per call (ms) over `reps` replays."""
    g = torch.cuda.CUDAGraph()
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(st):
        sets.launch(0)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=st):
            for i in range(steps):
                sets.launch(i)
    torch.cuda.current_stream().wait_stream(st)
    g.replay()
    torch.cuda.synchronize()
    per = []
    for _ in range(reps):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        torch.cuda.synchronize()
        per.append(a.elapsed_time(b) / steps)
    del g
    return statistics.median(per)


def pick_workload(name: str) -> workloads.Workload:
    """A named workload, or op:rows:d (seed 1, x ~ N(0,1))."""
    if name in NAMED:
        return NAMED[name]()
    try:
        op, rows, d = name.split(":")
        assert op in ("ln", "rms")
        return workloads.Workload(op, int(rows), int(d), seed=1, tag=f"{op}_{rows}x{d}")
    except (ValueError, AssertionError):
        raise SystemExit(f"unknown workload {name!r}: one of {sorted(NAMED)} or op:rows:d")


def gbs(nbytes, ms):
    return nbytes / (ms * 1e-3) / 1e9


def parity_gate(case_wl, out, gpu_result):
    """The oracle's output for the batch against the GPU's: "pass" or the
    first failure."""
    import parity as P

    x = case_wl.x()
    try:
        P.check_y(gpu_result[0], out[0])
        if case_wl.op == "ln":
            P.check_mean(gpu_result[1], out[1], x)
            P.check_rstd(gpu_result[2], out[2])
        return "pass"
    except AssertionError as e:
        return f"FAIL: {e}"


def oracle_once(case_wl):
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from oracle import c_oracle

    fn = c_oracle.layer_norm if case_wl.op == "ln" else c_oracle.rms_norm
    return fn(case_wl.x(), *case_wl.params(), case_wl.eps)


def cpu_baseline_leg(case_wl, gpu_result=None, seconds=10.0):
    """Time the C oracle (as it stands) on the host: whole passes over the
    headline batch, once on one thread (about `seconds`) and once on every
    host core, the rows split into one block per core (about `seconds` / 2;
    the reported value). Also the parity gate: the oracle's output for that
    batch is compared with the GPU's."""
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from oracle import c_oracle

    x = case_wl.x()
    params = case_wl.params()
    fn = c_oracle.layer_norm if case_wl.op == "ln" else c_oracle.rms_norm
    out = fn(x, *params, case_wl.eps)
    t0 = time.perf_counter()
    n = 0
    while True:
        fn(x, *params, case_wl.eps)
        n += 1
        if time.perf_counter() - t0 >= seconds:
            break
    el = time.perf_counter() - t0
    nbytes = algorithmic_bytes(case_wl.op, case_wl.rows, case_wl.d)

    # the same oracle function on every host core at once: the rows split
    # into one contiguous block per thread (ctypes releases the GIL during
    # the call), whole passes for about half the single-thread time
    from concurrent.futures import ThreadPoolExecutor

    cores = len(os.sched_getaffinity(0))
    bounds = [(case_wl.rows * i // cores, case_wl.rows * (i + 1) // cores) for i in range(cores)]
    parts = [(np.ascontiguousarray(x[a:b]), a, b) for a, b in bounds if b > a]

    def one(part):
        fn(part[0], *params, case_wl.eps)

    with ThreadPoolExecutor(len(parts)) as ex:
        list(ex.map(one, parts))
        t1 = time.perf_counter()
        n_all = 0
        while True:
            list(ex.map(one, parts))
            n_all += 1
            if time.perf_counter() - t1 >= seconds / 2:
                break
        el_all = time.perf_counter() - t1
    all_cores = {"value": nbytes * n_all / el_all / 1e9, "unit": UNIT, "cores": len(parts),
                 "sample": f"{n_all} whole passes over {case_wl.rows}x{case_wl.d}, rows split "
                           f"over {len(parts)} threads, {el_all:.1f} s"}
    parity = parity_gate(case_wl, out, gpu_result) if gpu_result is not None else None
    single = {"value": nbytes * n / el / 1e9, "unit": UNIT, "cores": 1,
              "sample": f"{n} whole passes over {case_wl.rows}x{case_wl.d}, one thread, "
                        f"{el:.1f} s"}
    return {"value": all_cores["value"], "unit": UNIT, "cores": all_cores["cores"],
            "kind": "oracle",
            "sample": f"the C float64 oracle as it stands: {all_cores['sample']} "
                      f"({case_wl.op})",
            "cpu": platform.processor() or platform.machine(),
            "host_cores_available": cores, "single_thread": single}, parity


def environment(torch, device) -> dict:
    """What the numbers were measured on."""
    props = torch.cuda.get_device_properties(device)
    env = {"gpu": torch.cuda.get_device_name(device), "sms": props.multi_processor_count,
           "l2_bytes": getattr(props, "L2_cache_size", None),
           "compute_capability": f"{props.major}.{props.minor}",
           "torch": torch.__version__, "cuda_runtime": torch.version.cuda,
           "host": platform.machine(), "host_cores": len(os.sched_getaffinity(0))}
    try:
        out = subprocess.run(["nvidia-smi", "--query-gpu=driver_version,memory.total",
                              "--format=csv,noheader", f"--id={device.index or 0}"],
                             capture_output=True, text=True, timeout=20)
        drv, mem = [v.strip() for v in out.stdout.strip().split(",")[:2]]
        env.update({"driver": drv, "gpu_memory": mem})
    except (OSError, ValueError, subprocess.SubprocessError):
        pass
    return env


def rank_workload(base: workloads.Workload, rank: int) -> workloads.Workload:
    """Weak scaling: every rank normalises its own batch of the base shape;
    the rows are independent, so a rank's batch is just other seeded data
    (seed shifted by 1000 per rank) and no data crosses ranks."""
    return workloads.Workload(base.op, base.rows, base.d, base.seed + 1000 * rank, base.x_dist,
                              base.x_std, base.eps, tag=base.tag)


def max_over_ranks(value: float, dist, device) -> float:
    """The slowest rank's time (one all-reduce of a scalar; not on the data
    path). Without a process group, the value itself."""
    if dist is None:
        return value
    import torch

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


L2_PROTOCOL = ("inputs larger than L2: the K steps run back to back over distinct copies of "
               "the batch, more than twice the L2 in all, one event pair around them")


def headline_config(wl, world):
    """The `config` of the headline line (the same for both arms)."""
    return {"workload": f"{'layernorm' if wl.op == 'ln' else 'rmsnorm'}_fwd_fp32_"
                        f"{wl.rows}x{wl.d}", "rows": wl.rows, "d": wl.d,
            "eps": wl.eps, "seed": wl.seed, "op": f"{wl.op}_fwd", "l2": L2_PROTOCOL,
            "rows_per_rank": wl.rows, "parallelism": f"rows sharded, {world} rank(s)"}


def _r(v, n=3):
    return None if v is None else float(f"{v:.{n}g}")


def summary(line, peak):
    """A compact record of every fraction of the measured HBM peak the
    targets are judged on, each named with its protocol: "b2b" (calls back
    to back over distinct batches larger than twice the L2, one span: the
    headline protocol), "cold" (a 2x-L2 buffer written before each launch,
    the launch timed alone), "clean" (that buffer written, then another
    2x-L2 buffer read), and the kernel's time over a device copy of the same
    bytes timed the "cold" way. Rows of numbers follow the column names
    given beside them."""
    ex = line["extra"]
    cold = ex["headline_cold_per_launch"]
    out = {"peak_GBps": peak,
           "protocols": {"b2b": "back to back, distinct batches > 2x L2, one span",
                         "cold": "alone after a 2x-L2 write",
                         "clean": "alone after a 2x-L2 write and a 2x-L2 read"},
           "headline": {"workload": line["config"]["workload"],
                        "b2b_frac": _r(line["roofline"]["frac"]),
                        "b2b_us": _r(1e3 * line["ms_per_step"]),
                        "b2b_over_copy": _r(line["roofline"]["same_size_copy"]
                                            ["kernel_over_copy_time"]),
                        "graph_frac": _r(ex["headline_stream_graph"]["frac_of_measured_hbm"]),
                        "cold_frac": _r(cold["frac_of_measured_hbm"]),
                        "cold_us": _r(1e3 * cold["ms_mean"])}}
    shapes = {}
    for w in ex.get("sweep_cold_l2", []):
        shapes[f"{w['op']}_{w['rows']}x{w['d']}"] = [
            _r(w["back_to_back"]["frac_of_measured_hbm"]), _r(w["frac_of_measured_hbm"]),
            _r(w["clean_l2"]["frac_of_measured_hbm"]), _r(w["kernel_over_copy_time"])]
    if shapes:
        out["shape_cols"] = ["b2b", "cold", "clean", "cold_over_copy"]
        out["shapes"] = shapes
    small = {}
    for w in ex.get("small_shapes_latency_bound", []):
        small[w["workload"]] = [
            w["launch_latency_bound"], _r(w["kernel_cold_us"]),
            _r(w["empty_cold_us"] + w["bytes_at_measured_peak_us"] + 1.0),
            _r(w["kernel_graph_us_per_launch"]), _r(1.5 * w["empty_graph_us_per_launch"])]
    if small:
        out["small_cols"] = ["latency_bound", "cold_us", "cold_bound_us", "graph_us",
                             "graph_bound_us"]
        out["small"] = small
    return out


def run_ours(args, rank, world, local_rank):
    import torch

    from row_wise_normalization_gb300 import capi

    capi.load()
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    dist = None
    if world > 1:
        import torch.distributed as dist

        # the shape sweep and the other context numbers are one-GPU figures;
        # under several ranks they would hold every GPU while rank 0 alone
        # measures them
        args.no_sweep = True
    peak, peak_src = hbm_peak()

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    wl = rank_workload(pick_workload(args.workload), rank)
    case = LnCase(torch, wl, device)
    flush = Flusher(torch, device)
    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        sampler.start()

    # correctness gate before any timing: one call, checked against the
    # oracle on this rank's batch; a failing call is not timed
    case.launch()
    torch.cuda.synchronize()
    gate = parity_gate(wl, oracle_once(wl), (case.y.cpu().numpy(), case.mean.cpu().numpy(),
                                             case.rstd.cpu().numpy()))
    if gate != "pass":
        print(f"parity gate failed before timing (rank {rank}): {gate}", file=sys.stderr)
        if sampler:
            sampler.stop()
        raise SystemExit(3)

    # The timed steps run back to back over distinct copies of the batch,
    # more than twice the L2 in all (BatchSets): every step reads an x that
    # is not in L2, and the whole job's throughput is timed as one span.
    sets = BatchSets(torch, case, device)
    for i in range(args.warmup):
        sets.launch(i)
    barrier()

    # ---- timed region: exactly K steps, back to back ------------------------
    t0 = time.time()
    span_ms = sets.span(args.steps, first=args.warmup)
    barrier()
    t1 = time.time()
    if sampler:
        # nvidia-smi samples every few tens of ms: when the K steps end
        # sooner than CLOCK_WINDOW_S, keep running the same step (untimed)
        # until the window is that long, so that the clock record covers
        # this load and not idle time
        i = 0
        while time.time() - t0 < CLOCK_WINDOW_S:
            for _ in range(200):
                sets.launch(i)
                i += 1
            torch.cuda.synchronize()
        sampler.mark("timed", t0, time.time())
    step_ms = max_over_ranks(span_ms / args.steps, dist, device)
    value = gbs(case.bytes * world, step_ms)
    same_as_gate = bool(torch.equal(sets.sets[0][1], case.y))

    # ---- e2e through the C entry point on pinned host buffers ---------------
    # x lives in pinned host memory and y/mean/rstd are written to pinned host
    # memory: ln_fwd's kernel reads x from the host and writes the results
    # back over the host link (NVLink-C2C on GB300) every step, with no
    # staging copies -- on this machine that beats copy-in/kernel/copy-out.
    # The same protocol as the headline: K calls back to back over distinct
    # host copies of the batch.
    import row_wise_normalization_gb300 as rn

    hsets = BatchSets(torch, case, device, host=True)
    for i in range(3):
        hsets.launch(i)
    barrier()
    t2 = time.time()
    e2e_span = hsets.span(args.steps, first=3)
    barrier()
    if sampler:
        sampler.mark("e2e", t2, time.time())
    e2e_ms = max_over_ranks(e2e_span / args.steps, dist, device)
    # the host-resident result must equal the device-resident one (same x)
    e2e_match = bool(torch.equal(hsets.sets[0][1], case.y.cpu()))
    xh, yh, mh, rh = hsets.sets[0]

    # the same through explicit copies (context): pinned x -> device, kernel,
    # device results -> pinned host, serially on one stream
    xd = torch.empty_like(case.x)

    def copy_step():
        xd.copy_(xh, non_blocking=True)
        if wl.op == "ln":
            y, m, r = rn.ln_fwd(xd, case.params[0], case.params[1], wl.eps,
                                y=case.y, mean=case.mean, rstd=case.rstd)
            mh.copy_(m, non_blocking=True)
            rh.copy_(r, non_blocking=True)
        else:
            y = rn.rms_fwd(xd, case.params[0], wl.eps, y=case.y)
        yh.copy_(y, non_blocking=True)

    for _ in range(3):
        copy_step()
    copy_ms = statistics.fmean(time_launches(torch, copy_step, args.steps, flush))
    h2d = 4 * wl.rows * wl.d
    d2h = 4 * wl.rows * wl.d + (8 * wl.rows if wl.op == "ln" else 0)
    del hsets

    if rank != 0:
        return None

    # ---- context measurements (rank 0 only) ---------------------------------
    extra = {}
    # one launch at a time with the L2 flushed before each (a 2x-L2 buffer
    # written outside the events): the per-launch cold protocol, which pays
    # the whole launch latency, the first DRAM round trip and the write-back
    # of the flush's dirty lines in every launch
    for _ in range(3):
        flush()
        case.launch()
    times = time_launches(torch, case.launch, args.steps, flush)
    extra["headline_cold_per_launch"] = {
        "ms_mean": statistics.fmean(times), "ms_median": statistics.median(times),
        "GBps": gbs(case.bytes, statistics.fmean(times)),
        "frac_of_measured_hbm": gbs(case.bytes, statistics.fmean(times)) / peak,
        "samples_ms": [round(t_, 6) for t_ in times]}
    clean = Flusher(torch, device, "clean")
    ct = time_launches(torch, case.launch, args.steps, clean)
    extra["headline_cold_clean_l2"] = {"ms_median": statistics.median(ct),
                                       "GBps": gbs(case.bytes, statistics.median(ct))}
    del clean
    warm = time_launches(torch, case.launch, args.steps)
    extra["headline_warm_l2"] = {"ms_median": statistics.median(warm),
                                 "GBps": gbs(case.bytes, statistics.median(warm))}
    # the timed stream of calls replayed from one CUDA graph (launch cost
    # taken off the host and the GPU's front end)
    g_ms = graph_span(torch, sets, args.steps)
    extra["headline_stream_graph"] = {"ms_per_step": g_ms, "GBps": gbs(case.bytes, g_ms),
                                      "frac_of_measured_hbm": gbs(case.bytes, g_ms) / peak,
                                      "calls_per_graph": args.steps}
    # CUDA graph of 64 back-to-back launches (warm), per-launch average
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        case.launch()
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            for _ in range(64):
                case.launch()
    torch.cuda.current_stream().wait_stream(s)
    g.replay()
    torch.cuda.synchronize()
    gt = time_launches(torch, g.replay, 15)
    extra["headline_graph64_warm"] = {"us_per_launch_median": 1e3 * statistics.median(gt) / 64}
    del g
    pl = case.plan()
    n_sm = torch.cuda.get_device_properties(device).multi_processor_count
    empty = time_launches(torch, lambda: capi.check(capi.launch_empty(
        n_sm, pl["threads_per_cta"], torch.cuda.current_stream().cuda_stream)), args.steps)
    extra["empty_kernel_us_median"] = 1e3 * statistics.median(empty)
    extra["batch_sets"] = {"distinct_batches": sets.n, "resident_bytes": sets.n * sets.per_set,
                           "same_result_as_gate_call": same_as_gate}

    # the same bytes moved by a device-to-device copy of x, timed the same ways:
    # back to back over distinct copies (the headline protocol) and alone after
    # a flush -- the practical floor for a kernel that reads x and writes y
    ysets = [(x_, torch.empty_like(x_)) for x_, _, _, _ in sets.sets]

    def copy_i(i):
        x_, y_ = ysets[i % len(ysets)]
        y_.copy_(x_)

    for i in range(3):
        copy_i(i)
    torch.cuda.synchronize()
    torch.cuda._sleep(HOST_LEAD_CYCLES_PER_STEP * args.steps)
    ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ea.record()
    for i in range(args.steps):
        copy_i(i)
    eb.record()
    torch.cuda.synchronize()
    same_copy_stream_ms = ea.elapsed_time(eb) / args.steps
    for _ in range(3):
        flush()
        copy_i(0)
    same_copy_ms = statistics.median(time_launches(torch, lambda: copy_i(0), args.steps, flush))
    del ysets, sets

    sweep = []
    if not args.no_sweep:
        cases = [workloads.large_32768x8192("ln"), workloads.large_32768x8192("rms")]
        cases += [w for w in workloads.sweep_offset()]
        t3 = time.time()
        clean = Flusher(torch, device, mode="clean")
        for w in cases:
            c = LnCase(torch, w, device)
            for _ in range(3):
                flush()
                c.launch()
            ts = time_launches(torch, c.launch, args.sweep_steps, flush)
            med = statistics.median(ts)
            # the same with the L2 holding clean, unrelated lines (no
            # write-backs of the flush buffer during the kernel)
            tc = statistics.median(time_launches(torch, c.launch, args.sweep_steps, clean))
            # a device copy of x into a y-sized buffer, timed the same way
            yc = torch.empty_like(c.x)
            tcp = statistics.median(time_launches(torch, lambda: yc.copy_(c.x), args.sweep_steps,
                                                  flush))
            del yc
            # back to back over distinct copies of the batch (the headline
            # protocol): no flush, no input in L2, the whole span timed
            bs = BatchSets(torch, c, device)
            for i in range(2):
                bs.launch(i)
            ts_ = bs.span(args.sweep_steps, first=2) / args.sweep_steps
            del bs
            sweep.append({"workload": w.tag, "op": w.op, "rows": w.rows, "d": w.d,
                          "same_size_copy_ms_median": tcp, "kernel_over_copy_time": med / tcp,
                          "plan": c.plan(), "ms_median": med, "GBps": gbs(c.bytes, med),
                          "frac_of_measured_hbm": gbs(c.bytes, med) / peak,
                          "clean_l2": {"ms_median": tc, "GBps": gbs(c.bytes, tc),
                                       "frac_of_measured_hbm": gbs(c.bytes, tc) / peak},
                          "back_to_back": {"ms_per_call": ts_, "GBps": gbs(c.bytes, ts_),
                                           "frac_of_measured_hbm": gbs(c.bytes, ts_) / peak}})
            del c
        del clean
        # same-session roofline control: a device-to-device copy of 1 GiB
        src = torch.empty(1 << 28, dtype=torch.float32, device=device)
        dst = torch.empty_like(src)
        ts = time_launches(torch, lambda: dst.copy_(src), args.sweep_steps, flush)
        med = statistics.median(ts)
        extra["d2d_copy_1GiB"] = {"ms_median": med, "GBps": gbs(2 * src.numel() * 4, med)}
        del src, dst
        if sampler:
            sampler.mark("sweep", t3, time.time())
    extra["sweep_cold_l2"] = sweep

    # the small shapes against the launch-latency floor
    if not args.no_sweep:
        small = [workloads.ln_512x128()]
        small += [w for w in workloads.rms_512_matrix() if w.x_dist == "normal"]
        extra["small_shapes_latency_bound"] = [
            latency_bound_check(torch, capi, w, device, flush, peak, args.sweep_steps)
            for w in small]

    # residual add fused with the normalization, against the same work done
    # as a separate add followed by the normalization (cold L2)
    if not args.no_sweep:
        import row_wise_normalization_gb300 as rn

        fused = []
        for op, rows_, d_ in (("ln", 4096, 768), ("ln", 16384, 4096), ("rms", 16384, 4096)):
            xw = workloads.Workload(op, rows_, d_, seed=61)
            xt = torch.from_numpy(xw.x()).to(device)
            rt = torch.from_numpy(workloads.Workload(op, rows_, d_, seed=62).x()).to(device)
            pt = [torch.from_numpy(p_).to(device) for p_ in xw.params()]
            ht, yt = torch.empty_like(xt), torch.empty_like(xt)
            mt = torch.empty(rows_, device=device)
            st_ = torch.empty(rows_, device=device)
            if op == "ln":
                f_fused = lambda: rn.ln_fwd_residual(xt, rt, *pt, h=ht, y=yt, mean=mt, rstd=st_)
                f_split = lambda: (torch.add(xt, rt, out=ht),
                                   rn.ln_fwd(ht, *pt, y=yt, mean=mt, rstd=st_))
            else:
                f_fused = lambda: rn.rms_fwd_residual(xt, rt, *pt, h=ht, y=yt)
                f_split = lambda: (torch.add(xt, rt, out=ht), rn.rms_fwd(ht, *pt, y=yt))
            res_ = {}
            for name, f in (("fused", f_fused), ("add_then_norm", f_split)):
                for _ in range(3):
                    flush()
                    f()
                res_[name] = statistics.median(time_launches(torch, f, args.sweep_steps, flush))
            nb = 16 * rows_ * d_ + (8 if op == "ln" else 4) * d_ + (8 * rows_ if op == "ln" else 0)
            fused.append({"workload": f"{op}_residual_{rows_}x{d_}",
                          "fused_ms": res_["fused"], "add_then_norm_ms": res_["add_then_norm"],
                          "fused_GBps": gbs(nb, res_["fused"]),
                          "speedup": res_["add_then_norm"] / res_["fused"]})
            del xt, rt, ht, yt
        extra["residual_fused_cold_l2"] = fused

        # 16-bit storage (FP32 arithmetic): algorithmic bytes at 2 bytes per element
        typed = []
        for op, rows_, d_, dt in (("ln", 4096, 768, torch.bfloat16), ("ln", 32768, 8192, torch.bfloat16),
                                  ("rms", 32768, 8192, torch.bfloat16),
                                  ("ln", 32768, 8192, torch.float16)):
            xw = workloads.Workload(op, rows_, d_, seed=63)
            xt = torch.from_numpy(xw.x()).to(device).to(dt)
            pt = [torch.from_numpy(p_).to(device).to(dt) for p_ in xw.params()]
            yt = torch.empty_like(xt)
            if op == "ln":
                mt = torch.empty(rows_, device=device)
                st_ = torch.empty(rows_, device=device)
                f = lambda: rn.ln_fwd(xt, *pt, y=yt, mean=mt, rstd=st_)
            else:
                f = lambda: rn.rms_fwd(xt, *pt, y=yt)
            for _ in range(3):
                flush()
                f()
            ms_ = statistics.median(time_launches(torch, f, args.sweep_steps, flush))
            nb = 4 * rows_ * d_ + (4 if op == "ln" else 2) * d_ + (8 * rows_ if op == "ln" else 0)
            typed.append({"workload": f"{op}_{str(dt).split('.')[-1]}_{rows_}x{d_}",
                          "ms_median": ms_, "GBps": gbs(nb, ms_),
                          "frac_of_measured_hbm": gbs(nb, ms_) / peak})
            del xt, yt
        extra["storage_16bit_cold_l2"] = typed

        # backward (dx plus the parameter gradients through the workspace);
        # algorithmic bytes: read dy and x, write dx, read the parameters (and
        # LN's saved mean/rstd), write the parameter gradients
        bwd = []
        for op, rows_, d_, dt in (("ln", 4096, 768, torch.float32),
                                  ("ln", 32768, 1024, torch.float32),
                                  ("ln", 16384, 4096, torch.float32),
                                  ("rms", 16384, 4096, torch.float32),
                                  ("ln", 16384, 4096, torch.bfloat16),
                                  ("rms", 16384, 4096, torch.bfloat16)):
            xw = workloads.Workload(op, rows_, d_, seed=65)
            xt = torch.from_numpy(xw.x()).to(device).to(dt)
            dyt = torch.from_numpy(workloads.Workload(op, rows_, d_, seed=66).x()).to(device).to(dt)
            pt = [torch.from_numpy(p_).to(device).to(dt) for p_ in xw.params()]
            dxt = torch.empty_like(xt)
            g0 = torch.empty(d_, device=device, dtype=dt)
            g1 = torch.empty(d_, device=device, dtype=dt)
            wst = torch.empty(capi.bwd_workspace_size(capi.RN_OP_LN if op == "ln" else capi.RN_OP_RMS,
                                                      rows_, d_) // 4 + 4, device=device)
            es = xt.element_size()
            if op == "ln":
                _, mt, st_ = rn.ln_fwd(xt, *pt)
                f = lambda: rn.ln_bwd(dyt, xt, pt[0], mt, st_, dx=dxt, dgamma=g0, dbeta=g1,
                                      workspace=wst)
                nb = 3 * es * rows_ * d_ + 3 * es * d_ + 8 * rows_
            else:
                f = lambda: rn.rms_bwd(dyt, xt, pt[0], dx=dxt, dw=g0, workspace=wst)
                nb = 3 * es * rows_ * d_ + 2 * es * d_
            for _ in range(3):
                flush()
                f()
            ms_ = statistics.median(time_launches(torch, f, args.sweep_steps, flush))
            bwd.append({"workload": f"{op}_bwd_{str(dt).split('.')[-1]}_{rows_}x{d_}",
                        "ms_median": ms_,
                        "GBps": gbs(nb, ms_), "frac_of_measured_hbm": gbs(nb, ms_) / peak,
                        "launches_per_call": 2})
            del xt, dyt, dxt, wst
        extra["backward_cold_l2"] = bwd

        # 64 small problems (LayerNorm 512x128 each): 64 single calls, the
        # same 64 calls replayed from a CUDA graph, and one batched call
        nprob, rows_, d_ = 64, 512, 128
        probs = []
        for i in range(nprob):
            xw = workloads.Workload("ln", rows_, d_, seed=70 + i)
            xt = torch.from_numpy(xw.x()).to(device)
            gt, bt = (torch.from_numpy(p_).to(device) for p_ in xw.params())
            probs.append((xt, gt, bt, torch.empty_like(xt), torch.empty(rows_, device=device),
                          torch.empty(rows_, device=device)))
        table = capi.problems([(x_.data_ptr(), g_.data_ptr(), b_.data_ptr(), y_.data_ptr(),
                                m_.data_ptr(), s_.data_ptr(), rows_, d_)
                               for x_, g_, b_, y_, m_, s_ in probs])
        eps32 = float(np.float32(1e-5))

        def singles():
            s_ = torch.cuda.current_stream().cuda_stream
            for x_, g_, b_, y_, m_, r_ in probs:
                capi.ln_fwd(x_.data_ptr(), g_.data_ptr(), b_.data_ptr(), y_.data_ptr(),
                            m_.data_ptr(), r_.data_ptr(), rows_, d_, eps32, s_)

        def batched():
            capi.ln_fwd_batched(capi.RN_DTYPE_F32, table, nprob, eps32,
                                torch.cuda.current_stream().cuda_stream)

        singles()
        batched()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            singles()
        graph_b = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph_b):
            batched()
        tiny = {}
        for name, f in (("single_calls", singles), ("graph_of_single_calls", graph.replay),
                        ("batched_call", batched), ("batched_call_from_graph", graph_b.replay)):
            for _ in range(3):
                flush()
                f()
            tiny[name + "_us"] = 1e3 * statistics.median(time_launches(torch, f, args.sweep_steps,
                                                                        flush))
        nb = nprob * algorithmic_bytes("ln", rows_, d_)
        tiny.update({"workload": f"{nprob} x ln_{rows_}x{d_}", "cold_l2": True,
                     "batched_GBps": gbs(nb, tiny["batched_call_us"] / 1e3),
                     "launches": {"single_calls": nprob, "graph_of_single_calls": nprob,
                                  "batched_call": 1, "batched_call_from_graph": 1}})
        extra["many_small_problems"] = tiny
        del probs, graph, graph_b

    clocks = None
    if sampler:
        sampler.stop()
        clocks = sampler.summary("timed")

    # ---- CPU baseline + parity gate (oracle on the host cores) --------------
    gpu_out = (case.y.cpu().numpy(), case.mean.cpu().numpy(), case.rstd.cpu().numpy())
    if world == 1:
        cpu, parity = cpu_baseline_leg(wl, gpu_out, seconds=args.cpu_seconds)
    else:
        # the CPU baseline is a one-GPU figure; with several ranks rank 0
        # only checks its batch against the oracle (one pass)
        cpu, parity = None, parity_gate(wl, oracle_once(wl), gpu_out)
    if parity != "pass":
        print(f"parity gate failed: {parity}", file=sys.stderr)

    h = source_hash()
    traffic = recorded_traffic(wl.tag, h, plan_key(pl))
    achieved = gbs(case.bytes, span_ms / args.steps)   # this rank's launches
    line = {
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": step_ms,
        "rows_per_s": wl.rows * world / (step_ms * 1e-3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded NumPy: x ~ N(0,1), gamma ~ N(1,0.1), beta ~ N(0,0.1))",
        "config": headline_config(wl, world),
        "e2e": {"value": gbs(case.bytes * world, e2e_ms), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms,
                "path": f"the C entry point {wl.op}_fwd on pinned host buffers: its kernel "
                        "reads x from host memory and writes the outputs to host memory over "
                        "NVLink-C2C every step (host-resident rows walk a persistent grid "
                        "holding about 1.25 MB in flight); K steps back to back over "
                        "distinct host copies of the batch, one event pair",
                "same_result_as_device_path": e2e_match,
                "explicit_copies": {"value": gbs(case.bytes * world, copy_ms), "unit": UNIT,
                                    "ms_per_step": copy_ms,
                                    "path": "pinned x -> device copy, kernel, results -> "
                                            "pinned host copies, one stream, L2 flushed "
                                            "before each step"}},
        "gpu_launches": args.steps,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": UNIT,
                     "frac": achieved / peak, "traffic": traffic,
                     "frac_of_nominal_8000": achieved / 8000.0,
                     "same_size_copy": {"ms_per_step": same_copy_stream_ms,
                                        "kernel_over_copy_time": (span_ms / args.steps)
                                        / same_copy_stream_ms,
                                        "alone_after_flush_ms_median": same_copy_ms,
                                        "what": "device copy of x into a y-sized buffer, the "
                                                "same back-to-back protocol over the same "
                                                "distinct batches"},
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_src == "measured" else "fallback 6800 GB/s",
                     "kernel": f"reg_kernel ({pl['variant']} per row; at 4096 x 768 the "
                               "instance with gamma/beta staged in shared memory, every row "
                               "in flight in one wave), one launch per step",
                     "plan": pl},
        "cpu_baseline": cpu,
        "parity": parity,
        "clocks": clocks,
        "environment": environment(torch, device),
        "samples_ms": [round(span_ms, 6)],
        "samples_what": "one span: the K timed steps back to back",
        "extra": extra,
        "source_hash": h,
    }
    # last in the line (whose tail is what a log keeps): every fraction the
    # targets are judged on, each with its protocol
    line["summary"] = summary(line, peak)
    print(json.dumps(line), flush=True)
    return line


# ---------------------------------------------------------------------------
# reference arm: the oracle as it stands, on the host cores
# ---------------------------------------------------------------------------
def run_reference(args, rank, world):
    """The oracle as it stands, timed on the host's cores: each step is one
    whole pass over the workload, its rows split into one contiguous block
    per core (the unchanged C oracle called per block from a thread pool;
    ctypes releases the GIL during each call)."""
    if rank != 0:
        return None
    from concurrent.futures import ThreadPoolExecutor

    from oracle import c_oracle

    wl = pick_workload(args.workload)
    x = wl.x()
    params = wl.params()
    fn = c_oracle.layer_norm if wl.op == "ln" else c_oracle.rms_norm
    nbytes = algorithmic_bytes(wl.op, wl.rows, wl.d)
    cores = len(os.sched_getaffinity(0))
    blocks = [np.ascontiguousarray(x[wl.rows * i // cores: wl.rows * (i + 1) // cores])
              for i in range(cores)]
    blocks = [b_ for b_ in blocks if b_.shape[0] > 0]

    def one(block):
        fn(block, *params, wl.eps)

    with ThreadPoolExecutor(len(blocks)) as ex:
        for _ in range(args.warmup):
            list(ex.map(one, blocks))
        times = []
        for _ in range(args.steps):
            t0 = time.perf_counter()
            list(ex.map(one, blocks))
            times.append(time.perf_counter() - t0)
    ms = 1e3 * statistics.fmean(times)
    value = gbs(nbytes, ms)
    line = {
        "impl": "reference",
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded NumPy)",
        "config": headline_config(wl, world),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": len(blocks), "kind": "oracle",
                         "sample": f"each step one whole pass of the C float64 oracle over "
                                   f"{wl.rows}x{wl.d}, rows split over {len(blocks)} threads"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return line


VARIANTS = ("auto", "warp", "block", "staged", "stream", "cluster")


def run_case(args):
    """One forward call, variant forced: W warm-up launches, K launches each
    after the L2 flush (cold), K launches back to back on the same buffers
    behind a GPU spin (warm), then (forward calls) n launches over n
    distinct copies of x and y, more than twice the L2 in all, and K more
    back to back over them, one event pair around the K (back_to_back).
    Prints one JSON line. The launch order is fixed so that an ncu capture
    can select a cold launch (any launch under --cache-control all), a warm
    one (launch W + K + 2 under --cache-control none: a warm launch that
    follows another) or a back-to-back one (W + 2K + n + 2 and on, under
    --cache-control none)."""
    import torch

    import row_wise_normalization_gb300 as rn
    from row_wise_normalization_gb300 import capi

    capi.load()
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    peak, _ = hbm_peak()
    op, rows, d = args.case.split(":")
    rows, d = int(rows), int(d)
    if op not in ("ln", "rms"):
        raise SystemExit("--case takes ln:rows:d or rms:rows:d")
    dt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[args.dtype]
    esz = 4 if args.dtype == "f32" else 2
    wl = workloads.Workload(op, rows, d, seed=1)
    x = torch.from_numpy(wl.x()).to(device).to(dt)
    ps = [torch.from_numpy(p_).to(device).to(dt) for p_ in wl.params()]
    y = torch.empty_like(x)
    variant = VARIANTS.index(args.variant)
    if args.residual:
        r = torch.from_numpy(workloads.Workload(op, rows, d, seed=2).x()).to(device).to(dt)
        h = torch.empty_like(x)
    if op == "ln":
        mean = torch.empty(rows, device=device)
        rstd = torch.empty(rows, device=device)
        if args.residual:
            f = lambda: rn.ln_fwd_residual(x, r, ps[0], ps[1], wl.eps, h=h, y=y, mean=mean,
                                           rstd=rstd, variant=variant)
        else:
            f = lambda: rn.ln_fwd(x, ps[0], ps[1], wl.eps, y=y, mean=mean, rstd=rstd,
                                  variant=variant)
        nbytes = (2 * esz * rows * d + 2 * esz * d + 8 * rows)
    else:
        if args.residual:
            f = lambda: rn.rms_fwd_residual(x, r, ps[0], wl.eps, h=h, y=y, variant=variant)
        else:
            f = lambda: rn.rms_fwd(x, ps[0], wl.eps, y=y, variant=variant)
        nbytes = 2 * esz * rows * d + esz * d
    if args.residual:
        nbytes += 2 * esz * rows * d
    if args.backward:
        # the backward of the same call: dy, x (and the saved statistics) in,
        # dx and the parameter gradients out, through a caller workspace
        dy = torch.from_numpy(workloads.Workload(op, rows, d, seed=3).x()).to(device).to(dt)
        dx = torch.empty_like(x)
        g0 = torch.empty_like(ps[0])
        opc_ = capi.RN_OP_LN if op == "ln" else capi.RN_OP_RMS
        ws = torch.empty(capi.bwd_workspace_size(opc_, rows, d) // 4 + 4, device=device)
        if op == "ln":
            _, sm, sr = rn.ln_fwd(x, ps[0], ps[1], wl.eps)
            g1 = torch.empty_like(ps[1])
            f = lambda: rn.ln_bwd(dy, x, ps[0], sm, sr, dx=dx, dgamma=g0, dbeta=g1, workspace=ws)
            nbytes = 3 * esz * rows * d + 3 * esz * d + 8 * rows
        else:
            f = lambda: rn.rms_bwd(dy, x, ps[0], wl.eps, dx=dx, dw=g0, workspace=ws)
            nbytes = 3 * esz * rows * d + 2 * esz * d
    for _ in range(args.warmup):
        f()
    torch.cuda.synchronize()
    flush = Flusher(torch, device)
    cold = time_launches(torch, f, args.steps, flush)
    warm = time_launches(torch, f, args.steps)
    b2b = None
    if not (args.backward or args.residual):
        # back to back over distinct copies of x (and y), more than twice the
        # L2 in all, one event pair around K calls
        l2 = getattr(torch.cuda.get_device_properties(device), "L2_cache_size", 0) or (128 << 20)
        n = max(2, -(-2 * l2 // (2 * x.numel() * x.element_size())) + 1)
        xs = [(x.clone(), torch.empty_like(y)) for _ in range(n)]

        def fi(i):
            xi, yi = xs[i % n]
            if op == "ln":
                rn.ln_fwd(xi, ps[0], ps[1], wl.eps, y=yi, mean=mean, rstd=rstd, variant=variant)
            else:
                rn.rms_fwd(xi, ps[0], wl.eps, y=yi, variant=variant)

        for i in range(n):
            fi(i)
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(HOST_LEAD_CYCLES_PER_STEP * args.steps)
        a.record()
        for i in range(args.steps):
            fi(i)
        b.record()
        torch.cuda.synchronize()
        b2b = [a.elapsed_time(b) / args.steps]
        del xs
    opc = capi.RN_OP_LN if op == "ln" else capi.RN_OP_RMS
    if args.residual:
        pl = capi.plan_residual(opc, variant, d, x.data_ptr(), r.data_ptr(), h.data_ptr(),
                                y.data_ptr())
    else:
        pl = capi.plan_typed(("f32", "bf16", "f16").index(args.dtype), opc, variant, d,
                             x.data_ptr(), y.data_ptr())
    kind = "_backward" if args.backward else ("_residual" if args.residual else "")
    out = {"case": f"{op}{kind}_{args.dtype}_{rows}x{d}",
           "variant": args.variant,
           "planned": ("backward row kernel + column reduction" if args.backward
                       else capi.variant_name(pl.variant)),
           "bytes": nbytes}
    for name, ts in (("cold", cold), ("warm", warm), ("back_to_back", b2b)):
        if ts is None:
            continue
        med = statistics.median(ts)
        out[name] = {"ms_median": med, "GBps": gbs(nbytes, med),
                     "frac_of_measured_hbm": gbs(nbytes, med) / peak}
    print(json.dumps(out))


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--sweep-steps", type=int, default=20)
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--workload", default="ln_4096x768",
                    help="named workload or op:rows:d (default: the 4096x768 LayerNorm)")
    ap.add_argument("--case", default=None,
                    help="op:rows:d -- time one forward call alone, cold and warm (see run_case)")
    ap.add_argument("--variant", choices=VARIANTS, default="auto")
    ap.add_argument("--dtype", choices=("f32", "bf16", "f16"), default="f32")
    ap.add_argument("--residual", action="store_true")
    ap.add_argument("--backward", action="store_true",
                    help="with --case: time the backward (dx and parameter gradients)")
    args = ap.parse_args(argv)
    if args.case is not None:
        run_case(args)
        return 0
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return 0
    if world > 1:
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist

            dist.barrier()
            dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
