"""Planted mistakes in a copy of the oracle must each fail at least one pin.

Each mutant below is the NumPy oracle with one plausible slip (a dropped
term, a wrong sign, a wrong divisor, a swapped or mis-indexed operand). If a
mutant passed every pin, the pins would not be able to tell that slip from
the definition. The mistakes live only in these test-local copies, on the
CPU.
"""
import numpy as np
import pytest

import oracle_pins as P
from oracle import reference


def _w(a):
    return np.asarray(a, np.float32).astype(np.float64)


def _ln(x, g, b, eps, *, var_div=0, eps_mode="inside", sign=-1, centred=True,
        beta=True, swap=False, rev_gamma=False, rstd_pow=0.5, mean_div=0, apply_rstd=True):
    x64, g64, b64 = _w(x), _w(g), _w(b)
    if swap:
        g64, b64 = b64, g64
    if rev_gamma:
        g64 = g64[::-1]
    rows, d = x64.shape
    mu = x64.sum(axis=1) / (d + mean_div)
    dev = x64 + sign * mu[:, None]
    if centred:
        var = (dev * dev).sum(axis=1) / (d + var_div)
    else:
        var = (x64 * x64).sum(axis=1) / (d + var_div)
    e = float(np.float32(eps))
    if eps_mode == "inside":
        rstd = 1.0 / (var + e) ** rstd_pow
    elif eps_mode == "outside":
        rstd = 1.0 / (np.sqrt(var) + e)
    else:
        with np.errstate(divide="ignore", invalid="ignore"):
            rstd = 1.0 / np.sqrt(var)
    with np.errstate(invalid="ignore"):
        y = dev * (rstd[:, None] if apply_rstd else 1.0) * g64[None, :]
    if beta:
        y = y + b64[None, :]
    return y, mu, rstd


def _rms(x, w, eps, *, square=True, mean=True, use_w=True, eps_mode="inside", centred=False):
    x64, w64 = _w(x), _w(w)
    rows, d = x64.shape
    v = x64 - x64.mean(axis=1, keepdims=True) if centred else x64
    q = (v * v) if square else np.abs(v)
    ms = q.sum(axis=1) / (d if mean else 1)
    e = float(np.float32(eps))
    if eps_mode == "inside":
        r = 1.0 / np.sqrt(ms + e)
    else:
        r = 1.0 / (np.sqrt(ms) + e)
    y = x64 * (w64[None, :] if use_w else 1.0) * r[:, None]
    return y, r


LN_MUTANTS = {
    "unbiased_variance": dict(var_div=-1),
    "eps_outside_root": dict(eps_mode="outside"),
    "eps_dropped": dict(eps_mode="none"),
    "beta_dropped": dict(beta=False),
    "gamma_beta_swapped": dict(swap=True),
    "gamma_reversed_index": dict(rev_gamma=True),
    "plus_mean": dict(sign=+1),
    "uncentred_variance": dict(centred=False),
    "mean_over_d_plus_1": dict(mean_div=1),
    "rstd_not_rooted": dict(rstd_pow=1.0),
    "rstd_not_applied": dict(apply_rstd=False),
}

RMS_MUTANTS = {
    "mean_abs_not_square": dict(square=False),
    "sum_not_mean": dict(mean=False),
    "weight_dropped": dict(use_w=False),
    "eps_outside_root": dict(eps_mode="outside"),
    "centred": dict(centred=True),
}


def _fails_some_pin(ln, rms):
    failed = []
    for pin in P.ALL_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(ln, rms)
        except (AssertionError, FloatingPointError, ValueError):
            failed.append(pin.__name__)
    return failed


@pytest.mark.parametrize("name", sorted(LN_MUTANTS))
def test_ln_mutant_is_caught(name):
    kw = LN_MUTANTS[name]
    failed = _fails_some_pin(lambda x, g, b, e: _ln(x, g, b, e, **kw), reference.rms_norm)
    assert failed, f"LayerNorm mutant {name!r} passed every pin"


@pytest.mark.parametrize("name", sorted(RMS_MUTANTS))
def test_rms_mutant_is_caught(name):
    kw = RMS_MUTANTS[name]
    failed = _fails_some_pin(reference.layer_norm, lambda x, w, e: _rms(x, w, e, **kw))
    assert failed, f"RMSNorm mutant {name!r} passed every pin"


def test_unmutated_copies_pass():
    """The mutation harness itself: with no mistake planted, every pin passes."""
    assert not _fails_some_pin(lambda x, g, b, e: _ln(x, g, b, e),
                               lambda x, w, e: _rms(x, w, e))
