"""The CPU oracle against what the pages and the mathematics fix (no GPU)."""
import numpy as np
import pytest

import oracle_pins as P
from oracle import c_oracle, reference

IMPLS = {
    "numpy": (reference.layer_norm, reference.rms_norm),
    "c": (c_oracle.layer_norm, c_oracle.rms_norm),
}


@pytest.mark.parametrize("impl", sorted(IMPLS))
@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin, impl):
    ln, rms = IMPLS[impl]
    pin(ln, rms)


@pytest.mark.parametrize("rows,d", [(1, 1), (37, 31), (64, 768), (9, 8193)])
def test_numpy_and_c_oracles_agree(rows, d):
    """Two independent restatements of the definitions agree to float64 rounding."""
    rng = np.random.default_rng(rows * 100003 + d)
    x = (rng.standard_normal((rows, d)) * 2 + rng.uniform(-100, 100, (rows, 1))).astype(np.float32)
    g = (1 + 0.1 * rng.standard_normal(d)).astype(np.float32)
    b = (0.1 * rng.standard_normal(d)).astype(np.float32)
    a = reference.layer_norm(x, g, b, 1e-5)
    c = c_oracle.layer_norm(x, g, b, 1e-5)
    for u, v in zip(a, c):
        np.testing.assert_allclose(u, v, rtol=1e-11, atol=1e-11)
    a = reference.rms_norm(x, g, 1e-5)
    c = c_oracle.rms_norm(x, g, 1e-5)
    for u, v in zip(a, c):
        np.testing.assert_allclose(u, v, rtol=1e-11, atol=1e-11)


def test_zero_width_rejected():
    for f in (reference.layer_norm, c_oracle.layer_norm):
        with pytest.raises(ValueError):
            f(np.zeros((2, 0), np.float32), np.zeros(0, np.float32), np.zeros(0, np.float32))
    for f in (reference.rms_norm, c_oracle.rms_norm):
        with pytest.raises(ValueError):
            f(np.zeros((2, 0), np.float32), np.zeros(0, np.float32))


def test_empty_rows():
    y, m, r = reference.layer_norm(np.zeros((0, 5), np.float32), np.ones(5, np.float32),
                                   np.zeros(5, np.float32))
    assert y.shape == (0, 5) and m.shape == (0,) and r.shape == (0,)
    y, m, r = c_oracle.layer_norm(np.zeros((0, 5), np.float32), np.ones(5, np.float32),
                                  np.zeros(5, np.float32))
    assert y.shape == (0, 5) and m.shape == (0,) and r.shape == (0,)
