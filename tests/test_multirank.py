"""The multi-rank bench path on CPU: two gloo ranks (no GPU).

Rows are independent, so ranks shard by taking batches of their own
(different seeded data, the same shape: weak scaling) with no collective on
the data path; the only exchange is the max over ranks of the step time.
These tests run that host logic in two spawned processes over gloo.
"""
import multiprocessing as mp
import os
import socket
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, local_ms, out):
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        base = bench.pick_workload("ln_4096x768")
        wl = bench.rank_workload(base, rank)
        step_ms = bench.max_over_ranks(local_ms[rank], dist, torch.device("cpu"))
        value = bench.gbs(bench.algorithmic_bytes(wl.op, wl.rows, wl.d) * world, step_ms)
        first_row = wl.x_rows(0, 1)[0, :8].tolist()
        out.put((rank, wl.rows, wl.d, wl.seed, step_ms, value, first_row))
    finally:
        dist.destroy_process_group()


def _run(world, local_ms):
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, local_ms, out))
             for r in range(world)]
    for p in procs:
        p.start()
    res = [out.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return sorted(res)


def test_two_ranks_shard_rows_and_agree_on_the_slowest_time():
    res = _run(2, [0.011, 0.017])
    (r0, rows0, d0, seed0, ms0, v0, row0), (r1, rows1, d1, seed1, ms1, v1, row1) = res
    assert (r0, r1) == (0, 1)
    # weak scaling: same shape per rank, different data
    assert (rows0, d0) == (rows1, d1) == (4096, 768)
    assert seed0 != seed1 and row0 != row1
    # both ranks report the slowest rank's time, and the value counts all ranks' bytes
    assert ms0 == ms1 == pytest.approx(0.017)
    assert v0 == v1 == pytest.approx(2 * (8 * 4096 * 768 + 8 * 768 + 8 * 4096) / 0.017e-3 / 1e9)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(0.5, None, None) == 0.5
    base = bench.pick_workload("ln_4096x768")
    assert bench.rank_workload(base, 0).seed == base.seed


def test_reference_arm_runs_on_rank_zero_only(capsys):
    sys.path.insert(0, ROOT)
    import bench

    class Args:
        workload = "ln_512x128"
        warmup = 3
        steps = 1

    assert bench.run_reference(Args, 1, 2) is None
    assert capsys.readouterr().out == ""


def test_parity_gate_of_several_ranks():
    """With several ranks rank 0 checks its batch against one oracle pass
    instead of timing the oracle: the gate passes on the oracle's own output
    (rounded to FP32, as a GPU writes it) and names the first failure when
    one output is off by more than the tolerance."""
    sys.path.insert(0, ROOT)
    import bench

    wl = bench.pick_workload("ln_512x128")
    out = bench.oracle_once(wl)
    got = tuple(a.astype("float32") for a in out)
    assert bench.parity_gate(wl, out, got) == "pass"
    bad = got[0].copy()
    bad[7, 3] += 1e-2
    verdict = bench.parity_gate(wl, out, (bad, got[1], got[2]))
    assert verdict.startswith("FAIL")
