"""Pins for the backward oracle (no GPU).

The backward is the derivative of the forward definitions; it is pinned to
things that do not share its algebra: central finite differences of the
forward oracle on small float64 problems, torch's CPU float64 autograd of
its own layer_norm / rms_norm, and identities of the gradient.
"""
import numpy as np
import pytest

from oracle import reference

EPS = float(np.float32(1e-5))


def _case(rows, d, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((rows, d)) * scale + rng.uniform(-3, 3, (rows, 1))).astype(np.float32)
    dy = rng.standard_normal((rows, d)).astype(np.float32)
    g = (1 + 0.3 * rng.standard_normal(d)).astype(np.float32)
    b = (0.3 * rng.standard_normal(d)).astype(np.float32)
    return x, dy, g, b


def _ln_loss(x, g, b, dy):
    # forward in float64 on float64 inputs (no FP32 rounding of perturbed values)
    mu = x.mean(axis=1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=1, keepdims=True)
    y = (x - mu) / np.sqrt(var + EPS) * g + b
    return (y * dy).sum()


def _rms_loss(x, w, dy):
    r = 1.0 / np.sqrt((x * x).mean(axis=1, keepdims=True) + EPS)
    return (x * w * r * dy).sum()


def _fd(f, a, h=1e-6):
    g = np.zeros_like(a)
    it = np.nditer(a, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        ap, am = a.copy(), a.copy()
        ap[i] += h
        am[i] -= h
        g[i] = (f(ap) - f(am)) / (2 * h)
    return g


@pytest.mark.parametrize("rows,d", [(1, 1), (2, 3), (3, 5), (4, 8)])
def test_ln_backward_matches_finite_differences(rows, d):
    x, dy, g, b = _case(rows, d, seed=rows * 10 + d)
    x64, dy64, g64, b64 = (a.astype(np.float64) for a in (x, dy, g, b))
    _, mean, rstd = reference.layer_norm(x, g, b)
    dx, dg, db = reference.layer_norm_backward(dy, x, g, mean, rstd)
    np.testing.assert_allclose(dx, _fd(lambda a: _ln_loss(a, g64, b64, dy64), x64), rtol=1e-6,
                               atol=1e-6)
    np.testing.assert_allclose(dg, _fd(lambda a: _ln_loss(x64, a, b64, dy64), g64), rtol=1e-6,
                               atol=1e-6)
    np.testing.assert_allclose(db, _fd(lambda a: _ln_loss(x64, g64, a, dy64), b64), rtol=1e-6,
                               atol=1e-6)


@pytest.mark.parametrize("rows,d", [(1, 1), (2, 3), (3, 5), (4, 8)])
def test_rms_backward_matches_finite_differences(rows, d):
    x, dy, w, _ = _case(rows, d, seed=rows * 7 + d)
    x64, dy64, w64 = (a.astype(np.float64) for a in (x, dy, w))
    dx, dw = reference.rms_norm_backward(dy, x, w)
    np.testing.assert_allclose(dx, _fd(lambda a: _rms_loss(a, w64, dy64), x64), rtol=1e-6,
                               atol=1e-6)
    np.testing.assert_allclose(dw, _fd(lambda a: _rms_loss(x64, a, dy64), w64), rtol=1e-6,
                               atol=1e-6)


def test_backward_against_torch_autograd_float64():
    torch = pytest.importorskip("torch")
    x, dy, g, b = _case(6, 37, seed=3, scale=2.0)
    _, mean, rstd = reference.layer_norm(x, g, b)
    dx, dg, db = reference.layer_norm_backward(dy, x, g, mean, rstd)
    xt = torch.from_numpy(x.astype(np.float64)).requires_grad_()
    gt = torch.from_numpy(g.astype(np.float64)).requires_grad_()
    bt = torch.from_numpy(b.astype(np.float64)).requires_grad_()
    torch.nn.functional.layer_norm(xt, [37], gt, bt, EPS).backward(torch.from_numpy(
        dy.astype(np.float64)))
    np.testing.assert_allclose(dx, xt.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dg, gt.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(db, bt.grad.numpy(), rtol=1e-11, atol=1e-12)
    if hasattr(torch.nn.functional, "rms_norm"):
        dx, dw = reference.rms_norm_backward(dy, x, g)
        xt = torch.from_numpy(x.astype(np.float64)).requires_grad_()
        wt = torch.from_numpy(g.astype(np.float64)).requires_grad_()
        torch.nn.functional.rms_norm(xt, [37], wt, EPS).backward(torch.from_numpy(
            dy.astype(np.float64)))
        np.testing.assert_allclose(dx, xt.grad.numpy(), rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(dw, wt.grad.numpy(), rtol=1e-11, atol=1e-12)


def test_backward_identities():
    """LN's dx rows sum to zero and are orthogonal to xhat (the output is
    shift- and scale-invariant in x); RMS's dx is orthogonal to x when dy is
    proportional to the output (a pure scale of x leaves the direction fixed)."""
    x, dy, g, b = _case(5, 64, seed=4)
    _, mean, rstd = reference.layer_norm(x, g, b)
    dx, _, _ = reference.layer_norm_backward(dy, x, g, mean, rstd)
    xhat = (x.astype(np.float64) - mean[:, None]) * rstd[:, None]
    assert np.all(np.abs(dx.sum(axis=1)) < 1e-10)
    # orthogonality to xhat holds up to the eps term: var/(var+eps) close to 1
    np.testing.assert_allclose((dx * xhat).sum(axis=1), 0.0, atol=1e-3)
    y, _ = reference.rms_norm(x, g)
    dxr, _ = reference.rms_norm_backward(y.astype(np.float32) / np.float32(1.0), x, g)
    np.testing.assert_allclose((dxr * x.astype(np.float64)).sum(axis=1), 0.0, atol=1e-2)


@pytest.mark.parametrize("mutant", ["no_centering", "missing_xhat_term", "dgamma_without_xhat",
                                    "rms_missing_cube"])
def test_backward_mutants_are_caught(mutant):
    """Planted mistakes in copies of the backward fail the finite-difference pin."""
    x, dy, g, b = _case(3, 6, seed=5)
    x64, dy64, g64, b64 = (a.astype(np.float64) for a in (x, dy, g, b))
    _, mean, rstd = reference.layer_norm(x, g, b)
    mu, rs = mean[:, None], rstd[:, None]
    xhat = (x64 - mu) * rs
    gg = dy64 * g64
    if mutant == "no_centering":
        bad = rs * (gg - xhat * (gg * xhat).mean(axis=1, keepdims=True))
        ref = _fd(lambda a: _ln_loss(a, g64, b64, dy64), x64)
    elif mutant == "missing_xhat_term":
        bad = rs * (gg - gg.mean(axis=1, keepdims=True))
        ref = _fd(lambda a: _ln_loss(a, g64, b64, dy64), x64)
    elif mutant == "dgamma_without_xhat":
        bad = (dy64 * x64).sum(axis=0)
        ref = _fd(lambda a: _ln_loss(x64, a, b64, dy64), g64)
    else:
        r = 1.0 / np.sqrt((x64 * x64).mean(axis=1, keepdims=True) + EPS)
        gw = dy64 * g64
        bad = r * gw - x64 * r * (gw * x64).mean(axis=1, keepdims=True)
        ref = _fd(lambda a: _rms_loss(a, g64, dy64), x64)
    assert not np.allclose(bad, ref, rtol=1e-4, atol=1e-4)
