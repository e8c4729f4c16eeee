"""NumPy float64 oracle for row-wise normalization (test infrastructure only).

Each function restates one definition in the order the pages give it; no
blocking, fusion or reordering is added beyond what NumPy does inside a
single ``sum``.
"""
from __future__ import annotations

import numpy as np


def _eps64(eps) -> float:
    # The GPU receives eps as an FP32 value; the oracle widens that exact value.
    return float(np.float32(eps))


def layer_norm(x, gamma, beta, eps=1e-5):
    """LayerNorm forward of every row of ``x`` in float64.

    Statistics, from "Rewriting the layer norm and matmul kernels", section
    "A reduction has to meet somewhere" (the displayed equation)::

        mu_i      = (1/d) * sum_j x_ij
        sigma_i^2 = (1/d) * sum_j (x_ij - mu_i)^2        (biased, centred)

    The pages print only these two statistics. The output step is the
    standard layer-normalization affine map, with eps inside the root as in
    the RMSNorm equation of "RMSNorm on an RTX 5070 ..." (section "The
    operator and the change")::

        rstd_i = (sigma_i^2 + eps)^(-1/2)
        y_ij   = (x_ij - mu_i) * rstd_i * gamma_j + beta_j

    Returns float64 (y [rows, d], mean [rows], rstd [rows]).
    """
    x64 = np.asarray(x, dtype=np.float32).astype(np.float64)
    g64 = np.asarray(gamma, dtype=np.float32).astype(np.float64)
    b64 = np.asarray(beta, dtype=np.float32).astype(np.float64)
    rows, d = x64.shape
    if d == 0:
        raise ValueError("d must be positive")
    mu = x64.sum(axis=1) / d
    dev = x64 - mu[:, None]
    var = (dev * dev).sum(axis=1) / d
    rstd = 1.0 / np.sqrt(var + _eps64(eps))
    y = dev * rstd[:, None] * g64[None, :] + b64[None, :]
    return y, mu, rstd


def rms_norm(x, w, eps=1e-5):
    """RMSNorm forward of every row of ``x`` in float64.

    From "RMSNorm on an RTX 5070 ...", section "The operator and the change"
    (the displayed equation)::

        y_rc = x_rc * w_c * ( (1/D) * sum_j x_rj^2 + eps )^(-1/2)

    Returns float64 (y [rows, d], r [rows]) where r is the per-row scale
    ``(mean(x^2) + eps)^(-1/2)``.
    """
    x64 = np.asarray(x, dtype=np.float32).astype(np.float64)
    w64 = np.asarray(w, dtype=np.float32).astype(np.float64)
    rows, d = x64.shape
    if d == 0:
        raise ValueError("d must be positive")
    ms = (x64 * x64).sum(axis=1) / d
    r = 1.0 / np.sqrt(ms + _eps64(eps))
    y = x64 * w64[None, :] * r[:, None]
    return y, r


def residual_sum(x, res):
    """h = x + res, rounded to FP32 (the stored residual stream).

    The sum of two FP32 values rounded to nearest FP32 is what an FP32 add
    produces; computing it in float64 first and rounding once gives the same
    bits (the exact sum of two FP32 values fits in float64).
    """
    x64 = np.asarray(x, dtype=np.float32).astype(np.float64)
    r64 = np.asarray(res, dtype=np.float32).astype(np.float64)
    return (x64 + r64).astype(np.float32)


def layer_norm_residual(x, res, gamma, beta, eps=1e-5):
    """Residual add followed by LayerNorm: h = x + res (FP32), then
    ``layer_norm(h)``. Returns (h FP32, y, mean, rstd) with y/mean/rstd in
    float64."""
    h = residual_sum(x, res)
    y, mean, rstd = layer_norm(h, gamma, beta, eps)
    return h, y, mean, rstd


def rms_norm_residual(x, res, w, eps=1e-5):
    """Residual add followed by RMSNorm: h = x + res (FP32), then
    ``rms_norm(h)``. Returns (h FP32, y, r)."""
    h = residual_sum(x, res)
    y, r = rms_norm(h, w, eps)
    return h, y, r


def layer_norm_backward(dy, x, gamma, mean, rstd):
    """Gradients of LayerNorm for upstream gradient ``dy``, from the saved
    per-row mean and rstd (float64 of the given values).

    With xhat = (x - mean) * rstd and g = dy * gamma (the derivative of the
    output definition above, written out):

        dbeta_j  = sum_i dy_ij
        dgamma_j = sum_i dy_ij * xhat_ij
        dx_ij    = rstd_i * (g_ij - (1/d) sum_k g_ik - xhat_ij (1/d) sum_k g_ik xhat_ik)

    Returns float64 (dx [rows, d], dgamma [d], dbeta [d]).
    """
    dy64 = np.asarray(dy, dtype=np.float32).astype(np.float64)
    x64 = np.asarray(x, dtype=np.float32).astype(np.float64)
    g64 = np.asarray(gamma, dtype=np.float32).astype(np.float64)
    mu = np.asarray(mean, dtype=np.float64).reshape(-1, 1)
    rs = np.asarray(rstd, dtype=np.float64).reshape(-1, 1)
    xhat = (x64 - mu) * rs
    g = dy64 * g64[None, :]
    dx = rs * (g - g.mean(axis=1, keepdims=True) - xhat * (g * xhat).mean(axis=1, keepdims=True))
    return dx, (dy64 * xhat).sum(axis=0), dy64.sum(axis=0)


def rms_norm_backward(dy, x, w, eps=1e-5):
    """Gradients of RMSNorm for upstream gradient ``dy`` (the per-row scale r
    recomputed from x as in the forward definition).

    With r = (mean_j x^2 + eps)^(-1/2) and g = dy * w:

        dw_j  = sum_i dy_ij * x_ij * r_i
        dx_ij = r_i * g_ij - x_ij * r_i^3 * (1/d) sum_k g_ik x_ik

    Returns float64 (dx [rows, d], dw [d]).
    """
    dy64 = np.asarray(dy, dtype=np.float32).astype(np.float64)
    x64 = np.asarray(x, dtype=np.float32).astype(np.float64)
    w64 = np.asarray(w, dtype=np.float32).astype(np.float64)
    _, r = rms_norm(x, w, eps)
    r = r.reshape(-1, 1)
    g = dy64 * w64[None, :]
    dx = r * g - x64 * r ** 3 * (g * x64).mean(axis=1, keepdims=True)
    return dx, (dy64 * x64 * r).sum(axis=0)
