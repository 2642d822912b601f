"""Pins of the oracle's fold policies ("TIRx Metal reduction lowering" §1,
ReductionPolicy fold_left / fold_right): hand-derived binary32 cases that only
the intended fold order produces, exact sums, direction symmetry, and every
operator under both folds within the rounding bound of its FP64 definition."""
import numpy as np
import pytest

import oracle

U = 2.0 ** -24


def test_the_three_orders_differ_as_derived():
    # [1, u, u, u], u = 2^-24:
    #   fold_left  ((1 + u) + u) + u: each add rounds back to 1           -> 1
    #   fold_right 1 + (u + (u + u)) = 1 + 3u = 1 + 1.5 ulp, a tie to even -> 1 + 2^-22
    #   OT-1024    (1 + u) + (u + u) = 1 + 2u = 1 + 2^-23
    v = np.array([1.0, U, U, U], np.float32)
    assert oracle.fold_sum(v, "left") == np.float32(1.0)
    assert oracle.fold_sum(v, "right") == np.float32(1.0 + 2.0 ** -22)
    assert oracle.ot_sum(v) == np.float32(1.0 + 2.0 ** -23)


def test_right_fold_is_the_left_fold_of_the_reversed_row():
    rng = np.random.default_rng(31)
    for n in (1, 2, 7, 1000, 4099):
        v = rng.standard_normal(n).astype(np.float32)
        assert oracle.fold_sum(v, "right") == oracle.fold_sum(v[::-1].copy(), "left")


def test_exact_cases():
    v = np.arange(-300, 301, dtype=np.float32)
    assert oracle.fold_sum(v, "left") == 0.0 and oracle.fold_sum(v, "right") == 0.0
    rng = np.random.default_rng(32)
    x = rng.standard_normal((5, 1537)).astype(np.float32)
    for d in ("left", "right"):
        assert np.array_equal(oracle.fold_row_max(x, d), x.max(1))
        assert np.array_equal(oracle.fold_row_min(x, d), x.min(1))
    z = np.array([[-0.0, 0.0, -1.0]], np.float32)
    assert not np.signbit(oracle.fold_row_max(z, "left")[0]) and not np.signbit(oracle.fold_row_max(z, "right")[0])
    assert oracle.fold_sum(np.array([-0.0], np.float32)) == 0.0               # the fold starts from +0
    assert not np.signbit(oracle.fold_sum(np.array([-0.0], np.float32)))


@pytest.mark.parametrize("direction", ["left", "right"])
def test_operators_within_the_fold_bound(direction):
    rng = np.random.default_rng(33)
    n = 3000
    x = (rng.standard_normal((4, n)) + rng.uniform(-3, 3, (4, 1))).astype(np.float32)
    w = rng.uniform(0.5, 1.5, n).astype(np.float32)
    b = (0.3 * rng.standard_normal(n)).astype(np.float32)
    # a fold of n terms: relative error of the sum at most (n + 4) u of sum|terms|
    tol = (n + 16) * U
    y = oracle.fold_softmax(x, direction)
    want = oracle.softmax(x)
    assert np.all(np.abs(y - want) <= tol * want + 1e-12)
    y = oracle.fold_rmsnorm(x, w, 1e-5, direction)
    want = oracle.rmsnorm(x, w, 1e-5)
    assert np.all(np.abs(y - want) <= tol * np.abs(want) + 1e-6)
    y = oracle.fold_layernorm(x, w, b, 1e-5, direction)
    want = oracle.layernorm(x, w, b, 1e-5)
    assert np.all(np.abs(y - want) <= 4 * tol * (np.abs(want) + 1.0))
    labels = rng.integers(0, n, 4)
    got = oracle.fold_cross_entropy(3 * x, labels, direction)
    want = oracle.cross_entropy(3 * x, labels)
    assert np.all(np.abs(got - want) <= tol * np.abs(want) + 1e-5)
    s = oracle.fold_softmax(x, direction).astype(np.float64).sum(1)
    assert np.all(np.abs(s - 1.0) <= tol + n * U)
