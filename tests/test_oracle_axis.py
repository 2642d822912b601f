"""Pins of the oracle's reductions over a non-last axis ("TIRx Metal reduction
lowering", Reductions inside composed groups: the reduced axis need not be the
last memory dimension; tests exercise both axis positions and extent one).

The oracle applies the row definitions to the vectors along the reduced axis;
these pins check that it picks the right vectors (brute force over every
output), and that the ordered tree is the one the tree's definition fixes for
short vectors: with at most four elements only quad 0 holds data, so OT-1024
gives (l0 + l1) + (l2 + l3) with l_k = 0 + v_k, and every other node adds +0."""
import itertools

import numpy as np
import pytest

import oracle


def ot_short(v):
    """OT-1024 of a vector of at most 4 floats, written out from the tree's definition."""
    z = np.float32(0.0)
    l = [np.float32(z + np.float32(v[k])) if k < len(v) else z for k in range(4)]
    return np.float32(np.float32(l[0] + l[1]) + np.float32(l[2] + l[3]))


def brute(x, dim, f):
    """f applied to every vector along `dim`, by explicit index loops."""
    shape = x.shape[:dim] + x.shape[dim + 1:]
    out = np.empty(shape, np.float64)
    for idx in itertools.product(*[range(n) for n in shape]):
        sl = list(idx)
        sl.insert(dim, slice(None))
        out[idx] = f(x[tuple(sl)])
    return out


@pytest.mark.parametrize("dim", [0, 1, 2, 3])
def test_axis_results_take_the_vectors_along_dim(dim):
    rng = np.random.default_rng(21 + dim)
    x = rng.standard_normal((2, 3, 4, 5)).astype(np.float32)
    assert np.allclose(oracle.axis_sum(x, dim), brute(x, dim, lambda v: sum(float(t) for t in v)), rtol=1e-13, atol=0)
    assert np.array_equal(oracle.axis_max(x, dim), brute(x, dim, lambda v: max(float(t) for t in v)))
    assert np.array_equal(oracle.axis_min(x, dim), brute(x, dim, lambda v: min(float(t) for t in v)))
    assert np.array_equal(oracle.ot_axis_max(x, dim), oracle.axis_max(x, dim))
    assert np.array_equal(oracle.ot_axis_min(x, dim), oracle.axis_min(x, dim))
    if x.shape[dim] <= 4:
        want = brute(x, dim, ot_short).astype(np.float32)
        assert np.array_equal(oracle.ot_axis_sum(x, dim).view(np.uint32), want.view(np.uint32))


def test_short_ordered_sum_is_the_pairwise_tree():
    # sequential: ((1 + u) + u) + u = 1 (each add of u = 2^-24 to 1 rounds back
    # to 1); the tree (1 + u) + (u + u) = 1 + 2^-23
    u = np.float32(2.0 ** -24)
    x = np.array([[[1.0]], [[u]], [[u]], [[u]]], np.float32)   # [extent 4, 1, 1] reduced over dim 0
    got = oracle.ot_axis_sum(x.reshape(4, 1), 0)[0]
    assert got == np.float32(1.0 + 2.0 ** -23)
    assert got == ot_short(x.ravel())


def test_closed_form_sums():
    # x[o, r, i] = r + 1: every vector sums to R (R + 1) / 2, exact in FP32 below 2^24
    for R in (1, 3, 257, 1025, 3000):
        x = np.broadcast_to(np.arange(1, R + 1, dtype=np.float32)[None, :, None], (2, R, 3)).copy()
        want = R * (R + 1) / 2
        assert np.all(oracle.axis_sum(x, 1) == want)
        assert np.all(oracle.ot_axis_sum(x, 1) == np.float32(want))


def test_extent_one_and_signed_zeros():
    x = np.array([[3.5, -0.0, -2.0]], np.float32)            # extent 1 along dim 0
    assert np.array_equal(oracle.ot_axis_max(x, 0), x[0])
    # the tree's leaves start at +0, so an ordered sum is never -0
    s = oracle.ot_axis_sum(x, 0)
    assert s[1] == 0 and not np.signbit(s[1]) and s[0] == 3.5 and s[2] == -2.0
    z = np.array([[-0.0], [0.0], [-0.0]], np.float32)
    assert not np.signbit(oracle.ot_axis_max(z, 0)[0]) and np.signbit(oracle.ot_axis_min(z, 0)[0])
