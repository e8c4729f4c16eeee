"""Pins for the CPU oracle: checks that do not trust the oracle itself.

Every pin takes the two oracle entry points as callables,
``ln(x, gamma, beta, eps) -> (y, mean, rstd)`` and
``rms(x, w, eps) -> (y, r)``, and raises ``AssertionError`` on a mismatch.
The same pins run against the NumPy oracle, the C oracle and, in
``test_oracle_mutants.py``, against copies of the oracle with a planted
mistake, each of which must fail at least one pin.

What pins what:

* exact brute force on tiny rows (``fractions`` + 50-digit ``decimal``,
  element by element in Python loops, rows != d so a transposed operand
  shows) -- the LayerNorm statistics equation of "Rewriting the layer norm
  and matmul kernels" (section "A reduction has to meet somewhere") and the
  RMSNorm equation of "RMSNorm on an RTX 5070 ..." (section "The operator and
  the change");
* closed forms: zero rows, width 1, alternating +/-1 rows, constant rows;
* invariants: normalised moments with gamma = 1 and beta = 0, row and column
  permutation equivariance, shift invariance, scale invariance with
  eps -> eps * a^2;
* a float64 library special case: ``torch.ops.aten.native_layer_norm`` and
  ``torch.nn.functional.rms_norm`` on CPU float64 tensors.
"""
from __future__ import annotations

from decimal import Decimal, localcontext
from fractions import Fraction

import numpy as np

EPS32 = np.float32(1e-5)
EPS = float(EPS32)


def _close(a, b, rtol, atol=0.0, what=""):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} != {b.shape}"
    ok = np.abs(a - b) <= atol + rtol * np.abs(b)
    assert np.all(ok), f"{what}: max |diff| {np.max(np.abs(a - b)):.3e}"


# ---------------------------------------------------------------------------
# exact arithmetic helpers (independent of NumPy reductions)
# ---------------------------------------------------------------------------

def _dec(fr: Fraction) -> Decimal:
    return Decimal(fr.numerator) / Decimal(fr.denominator)


def exact_ln_row(xr, g, b, eps):
    """One LayerNorm row in exact rationals, rstd and y to 50 digits."""
    xs = [Fraction(float(v)) for v in xr]
    d = len(xs)
    mu = sum(xs, Fraction(0)) / d
    var = sum(((v - mu) ** 2 for v in xs), Fraction(0)) / d
    with localcontext() as ctx:
        ctx.prec = 50
        rstd = Decimal(1) / (_dec(var) + _dec(Fraction(float(eps)))).sqrt()
        y = [float(_dec(v - mu) * rstd * _dec(Fraction(float(g[j])))
                   + _dec(Fraction(float(b[j])))) for j, v in enumerate(xs)]
        return y, float(_dec(mu)), float(rstd)


def exact_rms_row(xr, w, eps):
    """One RMSNorm row in exact rationals, scale and y to 50 digits."""
    xs = [Fraction(float(v)) for v in xr]
    d = len(xs)
    ms = sum((v * v for v in xs), Fraction(0)) / d
    with localcontext() as ctx:
        ctx.prec = 50
        r = Decimal(1) / (_dec(ms) + _dec(Fraction(float(eps)))).sqrt()
        y = [float(_dec(v) * _dec(Fraction(float(w[j]))) * r) for j, v in enumerate(xs)]
        return y, float(r)


def _dyadic(rng, shape, lo=-40, hi=40, den=8):
    return (rng.integers(lo, hi, size=shape) / den).astype(np.float32)


# ---------------------------------------------------------------------------
# pins
# ---------------------------------------------------------------------------

def pin_ln_hand_row(ln, rms):
    """Row [1,2,3,4]: mu = 2.5 and sigma^2 = 1.25 by hand."""
    x = np.array([[1, 2, 3, 4]], np.float32)
    y, mean, rstd = ln(x, np.ones(4, np.float32), np.zeros(4, np.float32), EPS32)
    assert mean[0] == 2.5, mean
    _close(rstd, [1.0 / np.sqrt(1.25 + EPS)], 1e-15, what="rstd")
    _close(y[0], np.array([-1.5, -0.5, 0.5, 1.5]) / np.sqrt(1.25 + EPS), 1e-15, what="y")
    # non-trivial affine: gamma and beta per column
    g = np.array([2.0, 0.5, 1.0, -1.0], np.float32)
    b = np.array([0.25, 0.0, -1.0, 3.0], np.float32)
    y, _, _ = ln(x, g, b, EPS32)
    s = 1.0 / np.sqrt(1.25 + EPS)
    _close(y[0], [-3.0 * s + 0.25, -0.25 * s, 0.5 * s - 1.0, -1.5 * s + 3.0], 1e-15,
           what="y affine")


def pin_ln_bruteforce(ln, rms):
    """Exact rational LayerNorm on tiny non-square inputs."""
    rng = np.random.default_rng(1234)
    for rows, d in ((1, 1), (3, 2), (2, 3), (4, 5), (3, 8), (5, 7)):
        x = _dyadic(rng, (rows, d))
        g = _dyadic(rng, d, -16, 16, 4)
        b = _dyadic(rng, d, -16, 16, 4)
        y, mean, rstd = ln(x, g, b, EPS32)
        for i in range(rows):
            ye, me, re = exact_ln_row(x[i], g, b, EPS)
            _close(y[i], ye, 1e-13, 1e-13, what=f"y[{i}] ({rows}x{d})")
            _close(mean[i], me, 1e-14, 1e-15, what=f"mean[{i}]")
            _close(rstd[i], re, 1e-14, what=f"rstd[{i}]")


def pin_rms_bruteforce(ln, rms):
    """Exact rational RMSNorm on tiny non-square inputs."""
    rng = np.random.default_rng(4321)
    for rows, d in ((1, 1), (3, 2), (2, 3), (4, 5), (3, 8), (5, 7)):
        x = _dyadic(rng, (rows, d))
        w = _dyadic(rng, d, -16, 16, 4)
        y, r = rms(x, w, EPS32)
        for i in range(rows):
            ye, re = exact_rms_row(x[i], w, EPS)
            _close(y[i], ye, 1e-13, 1e-13, what=f"y[{i}] ({rows}x{d})")
            _close(r[i], re, 1e-14, what=f"r[{i}]")


def pin_zero_rows(ln, rms):
    """Zero rows: LayerNorm gives beta, mean 0, rstd eps^-1/2; RMSNorm gives 0."""
    rng = np.random.default_rng(7)
    d = 9
    x = np.zeros((3, d), np.float32)
    g = (1 + 0.1 * rng.standard_normal(d)).astype(np.float32)
    b = (0.1 * rng.standard_normal(d)).astype(np.float32)
    y, mean, rstd = ln(x, g, b, EPS32)
    assert np.all(np.isfinite(y)), "non-finite output on zero rows"
    assert np.array_equal(y, np.broadcast_to(b.astype(np.float64), y.shape)), "y != beta"
    assert np.all(mean == 0.0)
    _close(rstd, np.full(3, EPS ** -0.5), 1e-15, what="rstd")
    y, r = rms(x, g, EPS32)
    assert np.all(np.isfinite(y)) and np.all(y == 0.0), "RMS of zero rows != 0"
    _close(r, np.full(3, EPS ** -0.5), 1e-15, what="r")


def pin_width_one(ln, rms):
    """d = 1: LayerNorm y = beta, mean = x; RMSNorm y = x w / sqrt(x^2 + eps)."""
    x = np.array([[3.5], [-2.0], [0.0], [1e-3]], np.float32)
    g = np.array([1.5], np.float32)
    b = np.array([0.25], np.float32)
    y, mean, rstd = ln(x, g, b, EPS32)
    assert np.all(y == 0.25), y
    assert np.array_equal(mean, x[:, 0].astype(np.float64))
    _close(rstd, np.full(4, EPS ** -0.5), 1e-15, what="rstd")
    y, r = rms(x, g, EPS32)
    xv = x[:, 0].astype(np.float64)
    _close(y[:, 0], xv * 1.5 / np.sqrt(xv * xv + EPS), 1e-15, 1e-300, what="rms y")


def pin_alternating(ln, rms):
    """Rows +1,-1,+1,...: RMS mean square is exactly 1; LN (even d) mu 0, sigma^2 1."""
    rng = np.random.default_rng(11)
    for d in (1, 2, 7, 128, 1001):
        x = np.broadcast_to(np.where(np.arange(d) % 2 == 0, 1.0, -1.0),
                            (3, d)).astype(np.float32)
        w = (1 + 0.1 * rng.standard_normal(d)).astype(np.float32)
        y, r = rms(x, w, EPS32)
        s = 1.0 / np.sqrt(1.0 + EPS)
        _close(r, np.full(3, s), 1e-15, what=f"rms r d={d}")
        _close(y, x * w.astype(np.float64) * s, 1e-15, what=f"rms y d={d}")
        if d % 2 == 0:
            b = (0.1 * rng.standard_normal(d)).astype(np.float32)
            y, mean, rstd = ln(x, w, b, EPS32)
            assert np.all(mean == 0.0)
            _close(rstd, np.full(3, s), 1e-15, what=f"ln rstd d={d}")
            _close(y, x * s * w.astype(np.float64) + b, 1e-14, 1e-15, what=f"ln y d={d}")


def pin_constant_rows(ln, rms):
    """Constant rows c (short mantissas): LN y = beta, mean c; RMS scale 1/sqrt(c^2+eps)."""
    rng = np.random.default_rng(5)
    d = 33
    cs = np.array([1.0, -3.5, 0.25, 1024.0], np.float32)
    x = np.repeat(cs[:, None], d, axis=1)
    g = (1 + 0.1 * rng.standard_normal(d)).astype(np.float32)
    b = (0.1 * rng.standard_normal(d)).astype(np.float32)
    y, mean, rstd = ln(x, g, b, EPS32)
    assert np.array_equal(mean, cs.astype(np.float64))
    assert np.array_equal(y, np.broadcast_to(b.astype(np.float64), y.shape))
    _close(rstd, np.full(4, EPS ** -0.5), 1e-15, what="rstd")
    y, r = rms(x, g, EPS32)
    c = cs.astype(np.float64)
    _close(r, 1.0 / np.sqrt(c * c + EPS), 1e-15, what="rms r")
    _close(y, np.sign(c)[:, None] * g * (np.abs(c) / np.sqrt(c * c + EPS))[:, None],
           1e-14, what="rms y")


def pin_ln_normalised_moments(ln, rms):
    """gamma=1, beta=0: each y row has mean 0 and variance sigma^2/(sigma^2+eps) = 1 - eps rstd^2.

    The mean output is also checked against the textbook mean of the row.
    """
    rng = np.random.default_rng(21)
    for rows, d in ((6, 2), (5, 3), (4, 17), (3, 256)):
        x = (rng.standard_normal((rows, d)) * rng.uniform(1e-3, 10.0, (rows, 1))
             + rng.uniform(-5, 5, (rows, 1))).astype(np.float32)
        y, mean, rstd = ln(x, np.ones(d, np.float32), np.zeros(d, np.float32), EPS32)
        x64 = x.astype(np.float64)
        _close(mean, x64.mean(axis=1), 1e-13, 1e-13, what="mean vs textbook mean")
        ym = y.mean(axis=1)
        assert np.all(np.abs(ym) <= 1e-12), f"row means {ym}"
        yv = ((y - ym[:, None]) ** 2).mean(axis=1)
        _close(yv, 1.0 - EPS * rstd ** 2, 1e-11, 1e-13, what=f"var(y) d={d}")


def pin_rms_normalised_moments(ln, rms):
    """Each RMS row has mean((y/w)^2) = ms/(ms+eps) = 1 - eps r^2."""
    rng = np.random.default_rng(22)
    for rows, d in ((5, 1), (4, 3), (3, 64)):
        x = (rng.standard_normal((rows, d)) * rng.uniform(1e-3, 10.0, (rows, 1))).astype(np.float32)
        w = (1 + 0.1 * rng.standard_normal(d)).astype(np.float32)
        y, r = rms(x, w, EPS32)
        q = ((y / w.astype(np.float64)) ** 2).mean(axis=1)
        _close(q, 1.0 - EPS * r ** 2, 1e-12, 1e-14, what=f"mean (y/w)^2 d={d}")


def pin_permutations(ln, rms):
    """Row permutations commute with the op; column permutations with gamma/beta/w permuted too."""
    rng = np.random.default_rng(31)
    rows, d = 6, 10
    x = rng.standard_normal((rows, d)).astype(np.float32)
    g = (1 + 0.1 * rng.standard_normal(d)).astype(np.float32)
    b = (0.1 * rng.standard_normal(d)).astype(np.float32)
    pr = rng.permutation(rows)
    pc = rng.permutation(d)
    y, mean, rstd = ln(x, g, b, EPS32)
    y2, m2, r2 = ln(x[pr], g, b, EPS32)
    _close(y2, y[pr], 1e-14, 1e-15, what="ln row perm")
    _close(m2, mean[pr], 1e-14, 1e-15, what="ln row perm mean")
    y3, m3, r3 = ln(x[:, pc], g[pc], b[pc], EPS32)
    _close(y3, y[:, pc], 1e-13, 1e-14, what="ln col perm")
    _close(r3, rstd, 1e-13, what="ln col perm rstd")
    yr, rr = rms(x, g, EPS32)
    yr2, _ = rms(x[pr], g, EPS32)
    _close(yr2, yr[pr], 1e-14, 1e-15, what="rms row perm")
    yr3, rr3 = rms(x[:, pc], g[pc], EPS32)
    _close(yr3, yr[:, pc], 1e-13, 1e-14, what="rms col perm")


def pin_shift(ln, rms):
    """LN(x + c) = LN(x), with the mean shifted by c (x and c integers, so x + c is exact)."""
    rng = np.random.default_rng(41)
    rows, d = 4, 12
    x = rng.integers(-50, 50, (rows, d)).astype(np.float32)
    g = (1 + 0.1 * rng.standard_normal(d)).astype(np.float32)
    b = (0.1 * rng.standard_normal(d)).astype(np.float32)
    c = np.float32(64.0)
    y, mean, rstd = ln(x, g, b, EPS32)
    y2, m2, r2 = ln(x + c, g, b, EPS32)
    _close(y2, y, 1e-12, 1e-13, what="shift y")
    _close(m2, mean + 64.0, 1e-14, what="shift mean")
    _close(r2, rstd, 1e-12, what="shift rstd")


def pin_scale(ln, rms):
    """op_{eps a^2}(a x) = op_eps(x) for a > 0 (a = 4, exact in FP32)."""
    rng = np.random.default_rng(51)
    rows, d = 5, 9
    x = rng.standard_normal((rows, d)).astype(np.float32)
    g = (1 + 0.1 * rng.standard_normal(d)).astype(np.float32)
    b = (0.1 * rng.standard_normal(d)).astype(np.float32)
    a = np.float32(4.0)
    e2 = np.float32(EPS32 * a * a)
    y, mean, rstd = ln(x, g, b, EPS32)
    y2, m2, r2 = ln(a * x, g, b, e2)
    _close(y2, y, 1e-12, 1e-13, what="scale ln y")
    _close(m2, 4.0 * mean, 1e-14, 1e-15, what="scale ln mean")
    _close(r2, rstd / 4.0, 1e-13, what="scale ln rstd")
    yr, rr = rms(x, g, EPS32)
    yr2, rr2 = rms(a * x, g, e2)
    _close(yr2, yr, 1e-12, 1e-13, what="scale rms y")
    _close(rr2, rr / 4.0, 1e-13, what="scale rms r")


def pin_torch_float64(ln, rms):
    """Special case that reduces to a library routine: torch CPU float64."""
    import torch

    rng = np.random.default_rng(61)
    for rows, d in ((7, 1), (5, 33), (3, 300)):
        x = (rng.standard_normal((rows, d)) * 3 + rng.uniform(-10, 10, (rows, 1))).astype(np.float32)
        g = (1 + 0.1 * rng.standard_normal(d)).astype(np.float32)
        b = (0.1 * rng.standard_normal(d)).astype(np.float32)
        y, mean, rstd = ln(x, g, b, EPS32)
        xt = torch.from_numpy(x.astype(np.float64))
        yt, mt, rt = torch.ops.aten.native_layer_norm(
            xt, [d], torch.from_numpy(g.astype(np.float64)),
            torch.from_numpy(b.astype(np.float64)), EPS)
        _close(y, yt.numpy(), 1e-12, 1e-12, what="torch ln y")
        _close(mean, mt.numpy().reshape(-1), 1e-12, 1e-12, what="torch ln mean")
        _close(rstd, rt.numpy().reshape(-1), 1e-12, what="torch ln rstd")
        if hasattr(torch.nn.functional, "rms_norm"):
            yr, _ = rms(x, g, EPS32)
            ytr = torch.nn.functional.rms_norm(xt, [d], torch.from_numpy(g.astype(np.float64)), EPS)
            _close(yr, ytr.numpy(), 1e-12, 1e-12, what="torch rms y")


ALL_PINS = [
    pin_ln_hand_row,
    pin_ln_bruteforce,
    pin_rms_bruteforce,
    pin_zero_rows,
    pin_width_one,
    pin_alternating,
    pin_constant_rows,
    pin_ln_normalised_moments,
    pin_rms_normalised_moments,
    pin_permutations,
    pin_shift,
    pin_scale,
    pin_torch_float64,
]
