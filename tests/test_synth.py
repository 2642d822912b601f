"""The seeded input generator: SplitMix64 values, shapes and distributions."""
import math

import numpy as np
import torch

import synth


def test_splitmix64_published_first_outputs():
    # SplitMix64 seeded with 0: state advances by GOLDEN before each output
    got = [synth.mix64_int(i * synth.GOLDEN) for i in (1, 2, 3)]
    assert got == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_tensor_mixer_matches_integer_reference():
    seed, tag = 7, synth.TAG_X
    base = synth.stream_base(seed, tag)
    t = synth.raw_u64(seed, tag, 0, 1000)
    ref = [synth.mix64_int(base + (i + 1) * synth.GOLDEN) for i in range(1000)]
    assert [v & ((1 << 64) - 1) for v in t.tolist()] == ref
    # slices of a stream are the stream
    assert torch.equal(synth.raw_u64(seed, tag, 400, 100), t[400:500])


def test_workload_shapes_and_moments():
    x = synth.workload_inputs("softmax_37x1537")["x"]
    assert x.shape == (37, 1537) and x.dtype == torch.float32
    assert abs(x.double().std().item() - 2.0) < 0.05      # N(0, 2^2): sigma 2
    n = synth.norm_inputs(256, 3072, 1, row_offset=True)
    assert n["w"].min() >= 0.5 and n["w"].max() < 1.5
    assert abs(n["b"].double().var().item() - 0.1) < 0.02  # N(0, 0.1): variance 0.1
    row_means = n["x"].double().mean(dim=1)
    assert row_means.min() > -3.2 and row_means.max() < 3.2 and row_means.std() > 1.0
    ce = synth.xent_inputs(64, 50257, 3)
    assert ce["labels"].dtype == torch.int64
    assert int(ce["labels"].min()) >= 0 and int(ce["labels"].max()) < 50257
    assert abs(ce["x"].double().std().item() - 3.0) < 0.02


def test_generation_is_deterministic():
    a = synth.softmax_inputs(3, 100, 5)["x"]
    b = synth.softmax_inputs(3, 100, 5)["x"]
    c = synth.softmax_inputs(3, 100, 6)["x"]
    assert torch.equal(a, b) and not torch.equal(a, c)
    assert np.isfinite(a.numpy()).all() and math.isfinite(float(a.abs().max()))
