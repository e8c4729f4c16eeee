"""Pins for the residual-add oracle (no GPU).

The residual form is the plain composition h = x + res (rounded to FP32, the
stored residual stream), then the normalization of h; the pins check the
composition against independent routes to the same numbers.
"""
import numpy as np
import pytest

import oracle_pins as P
from oracle import reference


def _inputs(rows=7, d=33, seed=0):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((rows, d)) * 3 + rng.uniform(-50, 50, (rows, 1))).astype(np.float32)
    r = (rng.standard_normal((rows, d)) * 0.5).astype(np.float32)
    g = (1 + 0.1 * rng.standard_normal(d)).astype(np.float32)
    b = (0.1 * rng.standard_normal(d)).astype(np.float32)
    return x, r, g, b


def test_residual_sum_is_the_fp32_add():
    """float64 sum rounded once == IEEE FP32 add (numpy float32 arithmetic)."""
    rng = np.random.default_rng(1)
    x = (rng.standard_normal(100000) * 10.0 ** rng.integers(-8, 8, 100000)).astype(np.float32)
    r = (rng.standard_normal(100000) * 10.0 ** rng.integers(-8, 8, 100000)).astype(np.float32)
    h = reference.residual_sum(x, r)
    assert h.dtype == np.float32
    assert np.array_equal(h.view(np.uint32), (x + r).view(np.uint32))


def test_zero_residual_is_plain_norm():
    x, r, g, b = _inputs()
    z = np.zeros_like(r)
    h, y, m, s = reference.layer_norm_residual(x, z, g, b)
    assert np.array_equal(h, x)
    y2, m2, s2 = reference.layer_norm(x, g, b)
    assert np.array_equal(y, y2) and np.array_equal(m, m2) and np.array_equal(s, s2)
    h, y, rr = reference.rms_norm_residual(z, x, g)
    y2, rr2 = reference.rms_norm(x, g)
    assert np.array_equal(y, y2) and np.array_equal(rr, rr2)


def test_residual_operands_commute():
    x, r, g, b = _inputs(seed=2)
    a = reference.layer_norm_residual(x, r, g, b)
    c = reference.layer_norm_residual(r, x, g, b)
    for u, v in zip(a, c):
        assert np.array_equal(u, v)


def test_residual_brute_force():
    """Exact rationals on dyadic inputs whose FP32 sum is exact."""
    rng = np.random.default_rng(3)
    x = (rng.integers(-40, 40, (3, 5)) / 8).astype(np.float32)
    r = (rng.integers(-40, 40, (3, 5)) / 8).astype(np.float32)
    g = (rng.integers(-16, 16, 5) / 4).astype(np.float32)
    b = (rng.integers(-16, 16, 5) / 4).astype(np.float32)
    h, y, m, s = reference.layer_norm_residual(x, r, g, b, P.EPS32)
    for i in range(3):
        hs = [float(x[i, j]) + float(r[i, j]) for j in range(5)]     # exact in float64
        assert list(h[i].astype(np.float64)) == hs
        ye, me, re = P.exact_ln_row(np.array(hs), g, b, P.EPS)
        np.testing.assert_allclose(y[i], ye, rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(s[i], re, rtol=1e-14)
    h, y, rr = reference.rms_norm_residual(x, r, g, P.EPS32)
    for i in range(3):
        ye, re = P.exact_rms_row(h[i], g, P.EPS)
        np.testing.assert_allclose(y[i], ye, rtol=1e-13, atol=1e-13)


def test_residual_cancellation_is_exact():
    """x + (-x) = 0 exactly: the normalized output is beta (LN) or 0 (RMS)."""
    x, _, g, b = _inputs(seed=4)
    h, y, m, s = reference.layer_norm_residual(x, -x, g, b)
    assert not h.any()
    assert np.array_equal(y, np.broadcast_to(b.astype(np.float64), y.shape))
    h, y, _ = reference.rms_norm_residual(x, -x, g)
    assert not y.any()


@pytest.mark.parametrize("mutant", ["drop_residual", "subtract", "norm_before_add"])
def test_residual_mutants_are_caught(mutant):
    """Planted mistakes in a copy of the residual composition fail the pins."""
    x, r, g, b = _inputs(seed=5)
    ref = reference.layer_norm_residual(x, r, g, b)
    if mutant == "drop_residual":
        bad = reference.layer_norm(x, g, b)[0]
    elif mutant == "subtract":
        bad = reference.layer_norm((x - r).astype(np.float32), g, b)[0]
    else:
        bad = reference.layer_norm(x, g, b)[0] + r
    assert not np.allclose(bad, ref[1], rtol=1e-4, atol=1e-5)
