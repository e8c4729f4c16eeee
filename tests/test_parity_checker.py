"""The parity checker must fail on the pages' two negative controls (no GPU).

"RMSNorm on an RTX 5070 ..." (section "Correctness before timing") removes
epsilon, which gives NaN on zero rows, and drops the final column, which
leaves a sentinel in the output; both must stop the run. Here the mistakes
are planted in oracle output on the CPU and fed to the same checker the GPU
tests use.
"""
import numpy as np
import pytest

import parity
import workloads
from oracle import reference


def _rms_case(d, pattern):
    w = workloads.Workload("rms", 64, d, seed=2, x_dist=pattern)
    return w.x(), w.params()[0]


def test_correct_fp32_output_passes():
    x, w = _rms_case(127, "normal")
    y, _ = reference.rms_norm(x, w)
    parity.check_y(y.astype(np.float32), y)
    wl = workloads.Workload("ln", 64, 129, seed=3, x_dist="offset", x_std=2.0)
    x = wl.x()
    g, b = wl.params()
    y, m, r = reference.layer_norm(x, g, b)
    parity.check_y(y.astype(np.float32), y)
    parity.check_mean(m.astype(np.float32), m, x)
    parity.check_rstd(r.astype(np.float32), r)


def test_negative_control_eps_removed():
    x, w = _rms_case(33, "zeros")
    y_ref, _ = reference.rms_norm(x, w, 1e-5)
    with np.errstate(all="ignore"):
        x64 = x.astype(np.float64)
        ms = (x64 * x64).mean(axis=1)
        y_bad = (x64 * w * (1.0 / np.sqrt(ms))[:, None]).astype(np.float32)
    assert np.isnan(y_bad).all()
    with pytest.raises(parity.ParityError):
        parity.check_y(y_bad, y_ref)


def test_negative_control_tail_dropped():
    x, w = _rms_case(8193, "normal")
    y_ref, _ = reference.rms_norm(x, w)
    n = y_ref.size
    buf = parity.guarded(n)
    out = buf[parity.GUARD:parity.GUARD + n].reshape(y_ref.shape)
    out[:, :-1] = y_ref[:, :-1]          # every column but the last written
    parity.check_guards(buf, n)          # guards intact ...
    with pytest.raises(parity.ParityError):
        parity.check_y(out, y_ref)       # ... but the sentinel remains in y


def test_guard_overwrite_detected():
    buf = parity.guarded(100)
    buf[parity.GUARD + 100] = 0.0        # one element past the end
    with pytest.raises(parity.ParityError):
        parity.check_guards(buf, 100)
    buf = parity.guarded(100)
    buf[parity.GUARD - 1] = 1.0          # one element before the start
    with pytest.raises(parity.ParityError):
        parity.check_guards(buf, 100)


def test_stat_tolerances_reject_slips():
    wl = workloads.Workload("ln", 32, 768, seed=1)
    x = wl.x()
    g, b = wl.params()
    _, m, r = reference.layer_norm(x, g, b)
    with pytest.raises(parity.ParityError):
        parity.check_rstd(r * (1 + 3e-6), r)
    with pytest.raises(parity.ParityError):
        parity.check_mean(m + 1e-3, m, x)
    # a biased-vs-unbiased slip in rstd is far outside the bound
    with pytest.raises(parity.ParityError):
        parity.check_rstd(r * np.sqrt(767 / 768), r)
