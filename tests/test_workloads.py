"""The seeded input generators (no GPU)."""
import numpy as np

import golden_cases
import parity
import workloads


def test_blocks_regenerate_identically():
    w = workloads.Workload("ln", 700, 33, seed=9, x_dist="offset", x_std=2.0)
    full = w.x()
    assert full.dtype == np.float32 and full.shape == (700, 33)
    np.testing.assert_array_equal(w.x_rows(250, 530), full[250:530])
    idx = [699, 0, 256, 255, 511, 3]
    np.testing.assert_array_equal(w.x_take(idx), full[idx])
    np.testing.assert_array_equal(w.x(threads=8), full)


def test_patterns():
    d = 33
    z = workloads.Workload("rms", 10, d, seed=2, x_dist="zeros").x()
    assert not z.any()
    a = workloads.Workload("rms", 10, d, seed=2, x_dist="alternating").x()
    assert np.all(a[:, 0::2] == 1) and np.all(a[:, 1::2] == -1)
    s = workloads.Workload("rms", 300, d, seed=2, x_dist="small").x()
    assert np.abs(s).max() <= 1e-3 and np.abs(s).max() > 5e-4
    o = workloads.Workload("ln", 512, 256, seed=3, x_dist="offset", x_std=2.0).x()
    m = o.mean(axis=1)
    assert np.abs(m).max() < 101 and np.abs(m).max() > 50
    assert 1.7 < o.std(axis=1).mean() < 2.3


def test_params_distributions():
    g, b = workloads.Workload("ln", 1, 20000, seed=1).params()
    assert abs(g.mean() - 1) < 0.01 and abs(g.std() - 0.1) < 0.01
    assert abs(b.mean()) < 0.01 and abs(b.std() - 0.1) < 0.01
    (w,) = workloads.Workload("rms", 1, 20000, seed=2).params()
    assert abs(w.mean() - 1) < 0.01


def test_case_matrix_covers_the_pages():
    kv = golden_cases.read_kv("rms_case_matrix.txt")
    widths = {int(v) for v in kv["widths"] + kv["extra_widths"]}
    mat = workloads.rms_512_matrix()
    assert {w.d for w in mat} == widths
    assert {w.x_dist for w in mat} == set(kv["patterns"])
    assert all(w.rows == 512 for w in mat)
    assert float(kv["atol"][0]) == parity.Y_ATOL and float(kv["rtol"][0]) == parity.Y_RTOL
    assert float(kv["eps"][0]) == workloads.EPS
    sweep = set(golden_cases.shapes("ln_shapes.txt", "sweep"))
    assert sweep - {(4096, 768)} <= set(workloads.SWEEP_SHAPES)
