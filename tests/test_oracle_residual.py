"""Pins of the oracle's fused residual norms ("TIRx Metal reduction lowering"
§5.1: LayerNorm over combined = X + residual). The fused op is the base norm
applied to the FP32 sum h = x + r, so the pins check that sum and that the
composition passes h through unchanged."""
import numpy as np

import oracle


def test_residual_sum_is_one_rounded_float32_add():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((5, 37)).astype(np.float32)
    r = rng.standard_normal((5, 37)).astype(np.float32)
    h = oracle.residual_sum(x, r)
    assert h.dtype == np.float32
    exact = x.astype(np.float64) + r.astype(np.float64)
    # one rounding: |h - exact| <= half an ulp of h
    ulp = np.spacing(np.abs(h))
    assert np.all(np.abs(h.astype(np.float64) - exact) <= 0.5 * ulp)
    assert np.array_equal(oracle.residual_sum(r, x).view(np.uint32), h.view(np.uint32))   # commutative


def test_zero_residual_is_the_plain_norm():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((4, 100)).astype(np.float32)
    w = rng.uniform(0.5, 1.5, 100).astype(np.float32)
    b = rng.standard_normal(100).astype(np.float32)
    z = np.zeros_like(x)
    y, h = oracle.add_layernorm(x, z, w, b, 1e-5)
    assert np.array_equal(h, x) and np.array_equal(y, oracle.layernorm(x, w, b, 1e-5))
    y, h = oracle.add_rmsnorm(x, z, w, 1e-5)
    assert np.array_equal(y, oracle.rmsnorm(x, w, 1e-5))
    yo, _ = oracle.ot_add_layernorm(x, z, w, b, 1e-5)
    assert np.array_equal(yo.view(np.uint32), oracle.ot_layernorm(x, w, b, 1e-5).view(np.uint32))


def test_integer_rows_sum_exactly():
    # small integers: h is exact, so the fused op equals the norm of the exact sum
    rng = np.random.default_rng(3)
    x = rng.integers(-50, 51, (3, 257)).astype(np.float32)
    r = rng.integers(-50, 51, (3, 257)).astype(np.float32)
    exact = (x.astype(np.int64) + r.astype(np.int64)).astype(np.float32)
    y, h = oracle.add_rmsnorm(x, r, None, 0.0)
    assert np.array_equal(h, exact)
    ref = exact.astype(np.float64)
    want = ref / np.sqrt((ref * ref).mean(axis=1, keepdims=True))
    assert np.allclose(y, want, rtol=1e-12, atol=0)


def test_constant_sum_gives_beta():
    # x + r constant per row: centred values are 0, so LayerNorm returns beta exactly
    x = np.full((2, 64), 1.25, np.float32)
    r = np.full((2, 64), -0.5, np.float32)
    b = np.linspace(-1, 1, 64).astype(np.float32)
    y, h = oracle.add_layernorm(x, r, None, b, 1e-5)
    assert np.all(h == np.float32(0.75))
    assert np.array_equal(y, np.broadcast_to(b.astype(np.float64), y.shape))
