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


def test_storage_rounding_matches_torch():
    """The input generator's BF16/FP16 rounding is torch's (round to nearest even)."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(5)
    a = (rng.standard_normal(100000) * 10.0 ** rng.integers(-6, 6, 100000)).astype(np.float32)
    bits, wide = workloads.to_storage(a, "bf16")
    t = torch.from_numpy(a).to(torch.bfloat16)
    assert np.array_equal(bits.view(np.int16), t.view(torch.int16).numpy())
    assert np.array_equal(wide, t.float().numpy())
    bits, wide = workloads.to_storage(a[np.abs(a) < 6e4], "f16")
    t = torch.from_numpy(a[np.abs(a) < 6e4]).to(torch.float16)
    assert np.array_equal(bits.view(np.int16), t.view(torch.int16).numpy())


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_storage_checker(dtype):
    rng = np.random.default_rng(6)
    ref = rng.standard_normal(5000) * 3
    bits, _ = workloads.to_storage(ref.astype(np.float32), dtype)
    parity.check_y_storage(bits, ref, dtype)               # the rounded reference passes
    off1 = bits.copy()
    off1[::7] += 1                                           # 1 ulp away: still accepted
    parity.check_y_storage(off1, ref, dtype)
    off2 = bits.copy()
    off2[3] += 2                                             # 2 ulp away: rejected
    with pytest.raises(parity.ParityError):
        parity.check_y_storage(off2, ref, dtype)
    sent = bits.copy()
    sent[10] = parity.SENTINEL16                             # an unwritten element: rejected
    with pytest.raises(parity.ParityError):
        parity.check_y_storage(sent, ref, dtype)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_storage_checker_near_zero_uses_fp32_rule(dtype):
    """Tiny outputs: an absolute error inside the FP32 rule passes even when it is
    many 16-bit ulps; a large one does not."""
    ref = np.array([4.6e-6, -3.0e-5, 1e-3])
    bits, _ = workloads.to_storage(np.array([2.3e-6, -2.8e-5, 1e-3], np.float32), dtype)
    parity.check_y_storage(bits, ref, dtype)
    bits, _ = workloads.to_storage(np.array([4.6e-6, -3.0e-5, 1.2e-3], np.float32), dtype)
    with pytest.raises(parity.ParityError):
        parity.check_y_storage(bits, ref, dtype)
