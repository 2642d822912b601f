"""Pins for the FP64 oracle: closed forms, invariants and brute force.

Each test checks the oracle against something other than itself, chosen so
that a plausible slip (a dropped term, a wrong sign, index or divisor, a
transposed operand) fails at least one of them.  Passages: "TIRx Metal
reduction lowering" §1 (softmax and cross-entropy programs), §5.1 (LayerNorm
mean/variance), §5.2 (guarded label gather), §8 (FP64 reference checks).
"""
import math

import numpy as np
import pytest

import oracle

RNG = np.random.default_rng(1234)


def rows_f32(r, c, scale=1.0, rng=RNG):
    return (rng.standard_normal((r, c)) * scale).astype(np.float32)


# --------------------------------------------------------------------- softmax

@pytest.mark.parametrize("n", [1, 2, 7, 257, 1537])
def test_softmax_constant_row_is_uniform(n):
    x = np.full((3, n), 0.7, np.float32)
    y = oracle.softmax(x)
    assert np.all(y == 1.0 / n)


def test_softmax_rows_sum_to_one_and_are_positive():
    y = oracle.softmax(rows_f32(5, 1537, 2.0))
    assert np.all(y > 0)
    assert np.allclose(y.sum(axis=1), 1.0, rtol=0, atol=1e-13)


def test_softmax_shift_invariance():
    # x on a 2^-10 grid in [-2, 2] so that x + 1 is exact in float32
    x = (RNG.integers(-2048, 2049, size=(4, 300)) / 1024.0).astype(np.float32)
    y0 = oracle.softmax(x)
    y1 = oracle.softmax(x + np.float32(1.0))
    assert np.allclose(y0, y1, rtol=1e-14, atol=0)


def test_softmax_two_element_is_logistic():
    x = rows_f32(50, 2, 3.0)
    y = oracle.softmax(x)
    d = x[:, 1].astype(np.float64) - x[:, 0].astype(np.float64)
    expect0 = 1.0 / (1.0 + np.exp(d))
    assert np.allclose(y[:, 0], expect0, rtol=1e-14, atol=0)
    assert np.allclose(y[:, 1], 1.0 / (1.0 + np.exp(-d)), rtol=1e-14, atol=0)


def test_softmax_ratio_and_order():
    x = rows_f32(2, 64)
    y = oracle.softmax(x)
    xd = x.astype(np.float64)
    ratio = y[:, :, None] / y[:, None, :]
    assert np.allclose(ratio, np.exp(xd[:, :, None] - xd[:, None, :]), rtol=1e-13)
    # order preserved: larger logit, larger probability
    o = np.argsort(x, axis=1)
    assert np.all(np.diff(np.take_along_axis(y, o, axis=1), axis=1) >= 0)


def test_softmax_dominant_element_is_one_hot():
    x = np.zeros((1, 10), np.float32)
    x[0, 3] = 200.0
    y = oracle.softmax(x)
    assert y[0, 3] == 1.0 and np.all(y[0, np.arange(10) != 3] < 1e-80)


def test_softmax_brute_force_mpmath():
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 40
    for n in range(1, 9):
        x = rows_f32(3, n, 2.0)
        y = oracle.softmax(x)
        for r in range(3):
            ex = [mp.e ** mp.mpf(float(v)) for v in x[r]]
            tot = mp.fsum(ex)
            for c in range(n):
                assert abs(float(ex[c] / tot) - y[r, c]) <= 4e-16 * abs(y[r, c])


# --------------------------------------------------------------------- RMSNorm

def test_rmsnorm_constant_row_closed_form():
    for c in (0.0, 0.25, -3.0, 1e-3):
        w = (RNG.random(33) + 0.5).astype(np.float32)
        x = np.full((1, 33), c, np.float32)
        y = oracle.rmsnorm(x, w, eps=1e-5)
        cd = float(np.float32(c))
        expect = cd / math.sqrt(cd * cd + float(np.float32(1e-5))) * w.astype(np.float64)
        assert np.allclose(y[0], expect, rtol=1e-15, atol=0)


def test_rmsnorm_single_column():
    x = rows_f32(20, 1, 5.0)
    w = np.array([1.5], np.float32)
    y = oracle.rmsnorm(x, w, eps=1e-5)
    xd = x[:, 0].astype(np.float64)
    expect = xd / np.sqrt(xd * xd + float(np.float32(1e-5))) * 1.5
    assert np.allclose(y[:, 0], expect, rtol=1e-15, atol=0)


def test_rmsnorm_unit_mean_square_without_eps():
    x = rows_f32(4, 999, 3.0)
    y = oracle.rmsnorm(x, None, eps=0.0)
    assert np.allclose((y * y).mean(axis=1), 1.0, rtol=0, atol=1e-13)


def test_rmsnorm_scale_invariance_and_weight():
    x = rows_f32(3, 100)
    w = (RNG.random(100) + 0.5).astype(np.float32)
    y1 = oracle.rmsnorm(x, w, eps=0.0)
    y8 = oracle.rmsnorm(x * np.float32(8.0), w, eps=0.0)  # exact scaling
    assert np.allclose(y1, y8, rtol=1e-14, atol=0)
    y_nw = oracle.rmsnorm(x, None, eps=0.0)
    assert np.allclose(y1, y_nw * w.astype(np.float64), rtol=1e-15, atol=0)


def test_rmsnorm_brute_force_mpmath():
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 40
    eps = np.float32(1e-5)
    for n in range(1, 9):
        x = rows_f32(2, n)
        w = (RNG.random(n) + 0.5).astype(np.float32)
        y = oracle.rmsnorm(x, w, eps=float(eps))
        for r in range(2):
            ms = mp.fsum(mp.mpf(float(v)) ** 2 for v in x[r]) / n
            rms = mp.sqrt(ms + mp.mpf(float(eps)))
            for c in range(n):
                ref = float(mp.mpf(float(x[r, c])) / rms * mp.mpf(float(w[c])))
                assert abs(ref - y[r, c]) <= 1e-15 * abs(ref) + 1e-300


# ------------------------------------------------------------------- LayerNorm

def test_layernorm_standardises_without_affine():
    x = (rows_f32(6, 3072) + RNG.uniform(-3, 3, (6, 1))).astype(np.float32)
    y = oracle.layernorm(x, None, None, eps=1e-5)
    assert np.all(np.abs(y.mean(axis=1)) < 1e-12)
    v = x.astype(np.float64).var(axis=1)  # population variance (numpy ddof=0)
    e = float(np.float32(1e-5))
    assert np.allclose(y.var(axis=1), v / (v + e), rtol=1e-12, atol=0)


def test_layernorm_population_variance_exact_without_eps():
    x = rows_f32(3, 17)
    y = oracle.layernorm(x, None, None, eps=0.0)
    # divisor is the width (population), so the output variance is exactly 1
    assert np.allclose((y * y).mean(axis=1), 1.0, rtol=0, atol=1e-14)


def test_layernorm_constant_row_gives_beta():
    g = (RNG.random(40) + 0.5).astype(np.float32)
    b = RNG.standard_normal(40).astype(np.float32)
    x = np.full((2, 40), -1.75, np.float32)
    y = oracle.layernorm(x, g, b, eps=1e-5)
    assert np.all(y == b.astype(np.float64))


def test_layernorm_two_columns_closed_form():
    x = rows_f32(30, 2, 2.0)
    y = oracle.layernorm(x, None, None, eps=1e-5)
    d = (x[:, 0].astype(np.float64) - x[:, 1].astype(np.float64)) / 2.0
    e = float(np.float32(1e-5))
    expect0 = d / np.sqrt(d * d + e)
    assert np.allclose(y[:, 0], expect0, rtol=1e-14, atol=1e-300)
    assert np.allclose(y[:, 1], -expect0, rtol=1e-14, atol=1e-300)


def test_layernorm_affine_and_shift_scale_invariance():
    x = rows_f32(3, 64)
    g = (RNG.random(64) + 0.5).astype(np.float32)
    b = RNG.standard_normal(64).astype(np.float32)
    plain = oracle.layernorm(x, None, None, eps=0.0)
    aff = oracle.layernorm(x, g, b, eps=0.0)
    assert np.allclose(aff, plain * g + b.astype(np.float64), rtol=1e-14, atol=1e-14)
    moved = oracle.layernorm(x * np.float32(4.0) + np.float32(0.5), None, None, eps=0.0)
    assert np.allclose(moved, plain, rtol=1e-6, atol=1e-6)  # x*4+0.5 rounds in float32


def test_layernorm_brute_force_mpmath():
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 40
    eps = np.float32(1e-5)
    for n in range(1, 9):
        x = rows_f32(2, n)
        g = (RNG.random(n) + 0.5).astype(np.float32)
        b = RNG.standard_normal(n).astype(np.float32)
        y = oracle.layernorm(x, g, b, eps=float(eps))
        for r in range(2):
            xs = [mp.mpf(float(v)) for v in x[r]]
            mu = mp.fsum(xs) / n
            var = mp.fsum((v - mu) ** 2 for v in xs) / n
            sd = mp.sqrt(var + mp.mpf(float(eps)))
            for c in range(n):
                ref = float((xs[c] - mu) / sd * mp.mpf(float(g[c])) + mp.mpf(float(b[c])))
                assert abs(ref - y[r, c]) <= 1e-14 * abs(ref) + 1e-15


# --------------------------------------------------------------- cross-entropy

@pytest.mark.parametrize("c", [1, 2, 10, 50257])
def test_cross_entropy_uniform_row_is_log_c(c):
    x = np.full((2, c), 1.25, np.float32)
    lab = np.array([0, c - 1], np.int64)
    loss = oracle.cross_entropy(x, lab)
    assert np.allclose(loss, math.log(c), rtol=1e-13, atol=1e-13)


def test_cross_entropy_confident_correct_is_near_zero():
    x = np.zeros((1, 100), np.float32)
    x[0, 42] = 30.0
    loss = oracle.cross_entropy(x, np.array([42], np.int64))
    # log(total) + peak - selected: 30 - 30 cancels, leaving ~1 ulp of 30
    assert abs(loss[0] - math.log1p(99 * math.exp(-30.0))) < 1e-13


def test_cross_entropy_two_classes_softplus():
    x = rows_f32(40, 2, 3.0)
    lab = RNG.integers(0, 2, 40)
    loss = oracle.cross_entropy(x, lab)
    xd = x.astype(np.float64)
    other = xd[np.arange(40), 1 - lab] - xd[np.arange(40), lab]
    assert np.allclose(loss, np.log1p(np.exp(other)), rtol=1e-13, atol=1e-15)


def test_cross_entropy_out_of_range_label_selects_zero():
    x = rows_f32(4, 37, 3.0)
    j = np.array([5, 0, 36, 11], np.int64)
    inside = oracle.cross_entropy(x, j)
    lse = inside + x[np.arange(4), j].astype(np.float64)  # logsumexp of each row
    for bad in (-1, 37, np.iinfo(np.int64).min, np.iinfo(np.int64).max):
        out = oracle.cross_entropy(x, np.full(4, bad, np.int64))
        assert np.allclose(out, lse, rtol=1e-14, atol=1e-14)


def test_cross_entropy_matches_negative_log_softmax():
    x = rows_f32(6, 300, 3.0)
    lab = RNG.integers(0, 300, 6)
    loss = oracle.cross_entropy(x, lab)
    p = oracle.softmax(x)[np.arange(6), lab]
    assert np.allclose(loss, -np.log(p), rtol=1e-12, atol=1e-13)
    assert np.all(loss >= 0)


def test_cross_entropy_brute_force_mpmath():
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 40
    for n in range(1, 9):
        x = rows_f32(3, n, 3.0)
        lab = RNG.integers(-1, n + 1, 3)
        loss = oracle.cross_entropy(x, lab)
        for r in range(3):
            lse = mp.log(mp.fsum(mp.e ** mp.mpf(float(v)) for v in x[r]))
            sel = mp.mpf(float(x[r, lab[r]])) if 0 <= lab[r] < n else mp.mpf(0)
            ref = float(lse - sel)
            assert abs(ref - loss[r]) <= 2e-15 * max(1.0, abs(ref))
