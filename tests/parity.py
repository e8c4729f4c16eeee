"""Element-by-element comparison of a device result with the float64 oracle.

Tolerances:

* y: ``|y - y_ref| <= 1e-5 + 1e-4 * |y_ref|`` for every element, the rule of
  "RMSNorm on an RTX 5070 ..." (section "Correctness before timing"); a NaN
  or Inf where the reference is finite fails.
* mean: ``|mean - mu_ref| <= 1e-6 * max(|mu_ref|, mean_j |x_ij|)``. A bare
  1e-6 relative bound is ill-posed for rows whose mean is near zero (an
  N(0,1) row of width 768 has |mu| ~ 1e-5 while FP32 summation error is
  ~1e-9 absolute), so the bound is taken relative to the row's magnitude.
* rstd: ``|rstd - rstd_ref| <= 1e-6 * rstd_ref``.

Guard regions (the same page) are stretches of sentinel values before and
after each output; they must be bit-for-bit unchanged after the call, and a
sentinel left inside the output region fails the y check.
"""
from __future__ import annotations

import numpy as np

Y_ATOL = 1e-5
Y_RTOL = 1e-4
STAT_RTOL = 1e-6
GUARD = 1024                     # elements of guard before and after an output
SENTINEL_BITS = 0x7FC0DEAD       # a quiet NaN with a payload


def sentinel_f32():
    return np.array([SENTINEL_BITS], np.uint32).view(np.float32)[0]


class ParityError(AssertionError):
    pass


def _first_bad(bad):
    idx = np.argwhere(bad)
    return tuple(int(i) for i in idx[0]) if len(idx) else None


def check_y(y, y_ref, what="y"):
    y = np.asarray(y, np.float64)
    y_ref = np.asarray(y_ref, np.float64)
    if y.shape != y_ref.shape:
        raise ParityError(f"{what}: shape {y.shape} != {y_ref.shape}")
    err = np.abs(y - y_ref)
    lim = Y_ATOL + Y_RTOL * np.abs(y_ref)
    bad = ~(err <= lim)           # NaN in y fails
    if bad.any():
        i = _first_bad(bad)
        raise ParityError(f"{what}: {int(bad.sum())} elements out of tolerance; first at {i}: "
                          f"got {y[i]!r}, want {y_ref[i]!r}")
    return float(err.max()) if err.size else 0.0


def check_mean(mean, mu_ref, x, what="mean"):
    mean = np.asarray(mean, np.float64)
    mu_ref = np.asarray(mu_ref, np.float64)
    scale = np.maximum(np.abs(mu_ref), np.abs(np.asarray(x, np.float64)).mean(axis=1))
    err = np.abs(mean - mu_ref)
    bad = ~(err <= STAT_RTOL * scale)
    if bad.any():
        i = _first_bad(bad)
        raise ParityError(f"{what}: {int(bad.sum())} rows out of tolerance; first row {i}: "
                          f"got {mean[i]!r}, want {mu_ref[i]!r}")
    with np.errstate(invalid="ignore", divide="ignore"):
        rel = np.where(scale > 0, err / scale, err)
    return float(rel.max()) if rel.size else 0.0


def check_rstd(rstd, rstd_ref, what="rstd"):
    rstd = np.asarray(rstd, np.float64)
    rstd_ref = np.asarray(rstd_ref, np.float64)
    err = np.abs(rstd - rstd_ref)
    bad = ~(err <= STAT_RTOL * np.abs(rstd_ref))
    if bad.any():
        i = _first_bad(bad)
        raise ParityError(f"{what}: {int(bad.sum())} rows out of tolerance; first row {i}: "
                          f"got {rstd[i]!r}, want {rstd_ref[i]!r}")
    rel = err / np.abs(rstd_ref)
    return float(rel.max()) if rel.size else 0.0


def check_guards(buf, n, what="guard", head=GUARD):
    """``buf`` holds ``head`` sentinels, n outputs, GUARD sentinels (as FP32)."""
    bits = np.asarray(buf, np.float32).view(np.uint32)
    if bits.shape[0] != n + head + GUARD:
        raise ParityError(f"{what}: buffer length {bits.shape[0]} != {n + head + GUARD}")
    head, tail = bits[:head], bits[head + n:]
    if not (np.all(head == SENTINEL_BITS) and np.all(tail == SENTINEL_BITS)):
        raise ParityError(f"{what}: guard region overwritten")


def guarded(n, head=GUARD):
    """A host buffer of n outputs framed by guards, every element a sentinel."""
    return np.full(n + head + GUARD, SENTINEL_BITS, np.uint32).view(np.float32)


# --------------------------------------------------------------------------
# 16-bit storage: y is computed in FP32 and rounded once to the storage type.
# An element passes if it is within one unit in the last place of the float64
# reference rounded to that type (the FP32 value can sit on the other side of
# a rounding boundary, never further), or within the FP32 rule plus one unit
# in the last place: near-zero outputs of LayerNorm (beta cancelling the
# normalised term) carry the FP32 computation's absolute error, ~u_32 |mu|
# rstd, which exceeds one 16-bit ulp there and is what the FP32 rule's
# absolute term already allows.
# --------------------------------------------------------------------------
SENTINEL16 = 0x7FC1   # a NaN in both BF16 and FP16


def _round_storage(ref64, dtype):
    import workloads

    bits, _ = workloads.to_storage(np.asarray(ref64, np.float64).astype(np.float32), dtype)
    return bits


def check_y_storage(bits, y_ref, dtype, what="y"):
    bits = np.asarray(bits, np.uint16)
    y_ref = np.asarray(y_ref, np.float64)
    want = _round_storage(y_ref, dtype)
    if bits.shape != want.shape:
        raise ParityError(f"{what}: shape {bits.shape} != {want.shape}")
    # ordered integer keys: ULP distance of same-type values
    def key(b):
        b = b.astype(np.int32)
        return np.where(b & 0x8000, 0x8000 - b, b)
    dist = np.abs(key(bits) - key(want))
    nan = np.isnan(y_ref)
    import workloads

    got = workloads.from_storage(bits, dtype).astype(np.float64)
    ulp = np.abs(workloads.from_storage(want ^ np.uint16(0), dtype).astype(np.float64)
                 - workloads.from_storage((want + np.uint16(1)) & np.uint16(0x7FFF) |
                                          (want & np.uint16(0x8000)), dtype).astype(np.float64))
    with np.errstate(invalid="ignore"):
        loose = np.abs(got - y_ref) <= Y_ATOL + Y_RTOL * np.abs(y_ref) + ulp
    bad = ((dist > 1) & ~loose & ~nan) | (np.isnan(got) & ~nan)
    if bad.any():
        i = _first_bad(bad)
        raise ParityError(f"{what}: {int(bad.sum())} elements more than 1 ulp off; first at {i}: "
                          f"got {got[i]!r}, want {y_ref[i]!r}")
    return int(dist.max()) if dist.size else 0


# --------------------------------------------------------------------------
# Sums over rows (parameter gradients). FP32 recursive summation of n terms
# errs by at most about n u |terms|_1 (Higham, "Accuracy and Stability of
# Numerical Algorithms", recursive summation bound); the kernels sum at most
# `chain` rows in sequence per partial and add the partials with Kahan
# compensation, so |err_j| <= (chain + 4) u sum_i |term_ij| + 1e-4 |ref_j|.
# --------------------------------------------------------------------------
U32 = 2.0 ** -24


def check_colsum(got, ref, abs_terms, chain, what="colsum"):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    lim = (chain + 4) * U32 * np.asarray(abs_terms, np.float64) + 1e-4 * np.abs(ref) + 1e-7
    err = np.abs(got - ref)
    bad = ~(err <= lim)
    if bad.any():
        i = _first_bad(bad)
        raise ParityError(f"{what}: {int(bad.sum())} columns out of tolerance; first {i}: "
                          f"got {got[i]!r}, want {ref[i]!r} (limit {lim[i]:.3e})")
    return float((err / np.maximum(lim, 1e-300)).max()) if err.size else 0.0
