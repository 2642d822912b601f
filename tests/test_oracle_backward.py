"""Pins of the oracle's backward passes (the gradients of softmax, cross-entropy,
RMSNorm and LayerNorm; the pages define the forward operators only).

* central differences of the pinned FP64 forward definitions: inputs and steps
  on a dyadic grid, so x +- h is exact in binary32 and the forward stays FP64;
* invariants of the gradients (softmax and LayerNorm gradients sum to zero,
  LayerNorm's is orthogonal to xh, RMSNorm's to x when eps = 0, cross-entropy
  rows sum to 0 or to dloss);
* the OT-1024 emulations on inputs where every binary32 step is exact, so they
  must equal the FP64 definitions bit for bit, and within a rounding bound on
  random inputs.
"""
import numpy as np
import pytest

import oracle

H = 2.0 ** -8


def grid(rng, shape, lo=-2.0, hi=2.0):
    """Values on a 2^-12 grid (exact in binary32 after adding +-2^-8)."""
    return (np.round(rng.uniform(lo, hi, shape) * 4096) / 4096).astype(np.float32)


def numgrad(f, x):
    g = np.zeros(x.shape, np.float64)
    for idx in np.ndindex(*x.shape):
        xp, xm = x.copy(), x.copy()
        xp[idx] += np.float32(H)
        xm[idx] -= np.float32(H)
        g[idx] = (f(xp) - f(xm)) / (2 * H)
    return g


def close(a, b, rel=2e-4):
    scale = max(np.abs(b).max(), 1e-30)
    assert np.abs(a - b).max() <= rel * scale, (np.abs(a - b).max(), scale)


def test_softmax_backward_is_the_derivative():
    rng = np.random.default_rng(1)
    x, dy = grid(rng, (3, 7)), grid(rng, (3, 7))
    y = oracle.softmax(x).astype(np.float32)
    dx = oracle.softmax_backward(y, dy)
    # y is rounded to binary32, so compare with the derivative through that y
    close(dx, numgrad(lambda v: float((oracle.softmax(v) * dy).sum()), x), rel=1e-3)


def test_cross_entropy_backward_is_the_derivative():
    rng = np.random.default_rng(2)
    x = grid(rng, (4, 9))
    labels = np.array([0, 8, 3, 20])                 # the last is outside [0, 9)
    dl = grid(rng, (4,), 0.5, 1.5)
    dx = oracle.cross_entropy_backward(x, labels, dl)
    close(dx, numgrad(lambda v: float((oracle.cross_entropy(v, labels) * dl).sum()), x))
    s = dx.sum(axis=1)
    assert np.allclose(s[:3], 0, atol=1e-12) and np.isclose(s[3], dl[3])
    assert np.allclose(oracle.cross_entropy_backward(x, labels), dx / dl[:, None])


@pytest.mark.parametrize("affine", [True, False])
def test_rmsnorm_backward_is_the_derivative(affine):
    rng = np.random.default_rng(3)
    x, dy = grid(rng, (3, 8)), grid(rng, (3, 8))
    w = grid(rng, (8,), 0.5, 1.5) if affine else None
    eps = 1e-3
    dx, dw = oracle.rmsnorm_backward(x, w, dy, eps)
    close(dx, numgrad(lambda v: float((oracle.rmsnorm(v, w, eps) * dy).sum()), x))
    if affine:
        close(dw, numgrad(lambda v: float((oracle.rmsnorm(x, v, eps) * dy).sum()), w))
    dx0, _ = oracle.rmsnorm_backward(x, w, dy, 0.0)
    assert np.allclose((dx0 * x).sum(axis=1), 0, atol=1e-12)       # scale invariance


@pytest.mark.parametrize("affine", [True, False])
def test_layernorm_backward_is_the_derivative(affine):
    rng = np.random.default_rng(4)
    x, dy = grid(rng, (3, 8)), grid(rng, (3, 8))
    g = grid(rng, (8,), 0.5, 1.5) if affine else None
    b = grid(rng, (8,), -0.5, 0.5) if affine else None
    eps = 1e-3
    dx, dg, db = oracle.layernorm_backward(x, g, dy, eps)
    close(dx, numgrad(lambda v: float((oracle.layernorm(v, g, b, eps) * dy).sum()), x))
    if affine:
        close(dg, numgrad(lambda v: float((oracle.layernorm(x, v, b, eps) * dy).sum()), g))
        close(db, numgrad(lambda v: float((oracle.layernorm(x, g, v, eps) * dy).sum()), b))
    assert np.allclose(dx.sum(axis=1), 0, atol=1e-12)               # shift invariance
    xh = (x - x.astype(np.float64).mean(1, keepdims=True))
    dx0, _, _ = oracle.layernorm_backward(x, g, dy, 0.0)
    assert np.allclose((dx0 * xh).sum(axis=1), 0, atol=1e-10)       # scale invariance


def bits(a):
    return np.asarray(a, np.float32).view(np.uint32)


def test_ordered_backward_exact_cases():
    # every binary32 step exact: the emulations must equal the FP64 definitions
    rng = np.random.default_rng(5)
    dy = rng.integers(-4, 5, (6, 8)).astype(np.float32)
    # RMSNorm: x = +-1, eps = 0 -> rms = 1; N = 8 keeps the means dyadic
    x = np.where(rng.integers(0, 2, (6, 8)) == 1, 1.0, -1.0).astype(np.float32)
    dx, dw = oracle.ot_rmsnorm_backward(x, None, dy, 0.0)
    ex, ew = oracle.rmsnorm_backward(x, None, dy, 0.0)
    assert np.array_equal(dx, ex.astype(np.float32)) and np.array_equal(dw, ew.astype(np.float32))
    # LayerNorm: rows a + (+-1) with as many + as -, so mean = a, var = 1
    a = rng.integers(-3, 4, (6, 1)).astype(np.float32)
    s = np.tile(np.array([1, -1, -1, 1, 1, -1, 1, -1], np.float32), (6, 1))
    x = a + s
    dx, dg, db = oracle.ot_layernorm_backward(x, None, dy, 0.0)
    ex, eg, eb = oracle.layernorm_backward(x, None, dy, 0.0)
    for got, want in ((dx, ex), (dg, eg), (db, eb)):
        assert np.array_equal(got, want.astype(np.float32))
    # softmax: dyadic y
    y = np.tile(np.array([0.5, 0.25, 0.125, 0.125], np.float32), (3, 1))
    d = rng.integers(-4, 5, (3, 4)).astype(np.float32)
    assert np.array_equal(oracle.ot_softmax_backward(y, d), oracle.softmax_backward(y, d).astype(np.float32))


def test_ordered_backward_within_rounding_bounds():
    rng = np.random.default_rng(6)
    x = rng.standard_normal((5, 3000)).astype(np.float32)
    dy = rng.standard_normal((5, 3000)).astype(np.float32)
    w = rng.uniform(0.5, 1.5, 3000).astype(np.float32)
    u = 2.0 ** -24
    dx, dw = oracle.ot_rmsnorm_backward(x, w, dy)
    ex, ew = oracle.rmsnorm_backward(x, w, dy)
    assert np.abs(dx - ex).max() <= 64 * u * np.abs(ex).max()
    assert np.all(np.abs(dw - ew) <= 32 * u * np.abs(dy * x).sum(0) * 2)
    dx, dg, db = oracle.ot_layernorm_backward(x, w, dy)
    ex, eg, eb = oracle.layernorm_backward(x, w, dy)
    assert np.abs(dx - ex).max() <= 64 * u * np.abs(ex).max()
    assert np.all(np.abs(db - eb) <= 32 * u * np.abs(dy).sum(0))
    y = oracle.softmax(x).astype(np.float32)
    assert np.abs(oracle.ot_softmax_backward(y, dy) - oracle.softmax_backward(y, dy)).max() <= 64 * u * 1e-2
    labels = rng.integers(0, 3000, 5)
    got = oracle.ot_cross_entropy_backward(x, labels)
    want = oracle.cross_entropy_backward(x, labels)
    assert np.abs(got - want).max() <= 1e-6
