"""GPU parity of the wave plans (TR_PLAN_WAVE) against the CPU oracle.

A wave CTA serves 1 or 2 aligned rows with 256 threads; thread t caches the
16-byte slots t + 256 j of each row, which is the OT-1024 leaf layout
("TIRx Metal reduction lowering" §4.4 ownership with V = 4), so the same kernel
gives the ordered tree's bits. Unordered: |gpu - oracle| <= 1e-6 + 2e-6 |oracle|
against the FP64 oracle. Ordered: bit-identical to the OT-1024 emulation.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import fp32_row_reduction_gb300 as tr

pytestmark = pytest.mark.gpu

RTOL, ATOL = 2e-6, 1e-6
DEV = "cuda:0"
OPS = ["softmax", "rmsnorm", "layernorm"]
# aligned rows of 1024 .. 8192 columns, odd row counts (a half-empty last CTA when R = 2)
SHAPES = [(3, 1024), (5, 1028), (40, 2048), (21, 5000), (9, 6144), (11, 8192), (1, 4100)]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tr.load()
    yield
    tr.tr_plan_override(None)


def wave_plan(op, order, cols, rows_per_cta):
    k = min(k for k in (2, 4, 6, 8) if 1024 * k >= cols)
    return tr.tr_plan(op=tr.OPS[op], order=1 if order == "ordered" else 0, kind=tr.TR_PLAN_WAVE, lanes_per_row=32,
                      warps_per_row=8, rows_per_cta=rows_per_cta, cluster_ctas=1, vec_slots=k, block_threads=256)


def make(op, rows, cols, seed):
    if op == "softmax":
        return synth.make_inputs(op, rows, cols, seed, var=4.0, device=DEV)
    return synth.make_inputs(op, rows, cols, seed, row_offset=True, device=DEV)


def host(d):
    return {k: v.cpu().numpy() for k, v in d.items()}


def reference(op, h, eps=1e-5):
    if op == "softmax":
        return oracle.softmax(h["x"])
    if op == "rmsnorm":
        return oracle.rmsnorm(h["x"], h.get("w"), eps)
    return oracle.layernorm(h["x"], h.get("w"), h.get("b"), eps)


def emulated(op, h, eps=1e-5):
    if op == "softmax":
        return oracle.ot_softmax(h["x"])
    if op == "rmsnorm":
        return oracle.ot_rmsnorm(h["x"], h.get("w"), eps)
    return oracle.ot_layernorm(h["x"], h.get("w"), h.get("b"), eps)


def assert_close(got, ref, what):
    got = np.asarray(got, np.float64)
    err = np.abs(got - ref)
    bad = ~(err <= ATOL + RTOL * np.abs(ref))
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} outside tolerance"


def assert_bits(got, emu, what):
    g, e = np.asarray(got, np.float32), np.asarray(emu, np.float32)
    assert np.array_equal(np.isnan(g), np.isnan(e)), what
    ok = ~np.isnan(e)
    diff = int(np.sum(g[ok].view(np.uint32) != e[ok].view(np.uint32)))
    assert diff == 0, f"{what}: {diff} differing words"


def run_with(plan, op, d, order, out=None):
    assert tr.tr_plan_override(plan) == tr.TR_OK
    try:
        y = tr.run_op(op, d, out=out, order=order)
        torch.cuda.synchronize()
        # the override really selected the wave kernel
        assert tr.tr_plan_describe(tr.OPS[op], d["x"].shape[0], d["x"].shape[1], 1 if order == "ordered" else 0).kind \
            == tr.TR_PLAN_WAVE
    finally:
        tr.tr_plan_override(None)
    return y


@pytest.mark.parametrize("rows_per_cta", [1, 2])
@pytest.mark.parametrize("rows,cols", SHAPES)
@pytest.mark.parametrize("op", OPS)
def test_wave_unordered_matches_oracle(op, rows, cols, rows_per_cta):
    d = make(op, rows, cols, seed=rows * 31 + cols)
    y = run_with(wave_plan(op, "unordered", cols, rows_per_cta), op, d, "unordered")
    assert_close(y.cpu().numpy(), reference(op, host(d)), f"{op} {rows}x{cols} R={rows_per_cta}")


@pytest.mark.parametrize("rows_per_cta", [1, 2])
@pytest.mark.parametrize("rows,cols", SHAPES)
@pytest.mark.parametrize("op", OPS)
def test_wave_ordered_bit_exact(op, rows, cols, rows_per_cta):
    d = make(op, rows, cols, seed=rows * 977 + cols)
    h = host(d)
    y = run_with(wave_plan(op, "ordered", cols, rows_per_cta), op, d, "ordered").cpu().numpy()
    assert_bits(y, emulated(op, h), f"{op} {rows}x{cols} R={rows_per_cta}")
    assert_close(y, reference(op, h), f"ordered {op} {rows}x{cols}")


@pytest.mark.parametrize("order", ["unordered", "ordered"])
@pytest.mark.parametrize("op", OPS)
def test_wave_is_the_default_at_768x6144(op, order):
    p = tr.tr_plan_describe(tr.OPS[op], 768, 6144, 1 if order == "ordered" else 0)
    assert p.kind == tr.TR_PLAN_WAVE and p.vec_slots == 6


@pytest.mark.parametrize("rows_per_cta", [1, 2])
def test_wave_ordered_softmax_outside_the_fast_exp_range(rows_per_cta):
    # differences below -86 (and -inf, NaN, +inf) take the exp's general form for
    # the whole thread; every other thread keeps the branch-free form
    g = torch.Generator().manual_seed(5)
    x = torch.randn(7, 4096, generator=g) * 2.0
    x[0, 100] = 200.0                     # every other difference < -86
    x[1, ::5] = -1e30
    x[2] = -87.0 - torch.rand(4096, generator=g) * 30.0
    x[2, 0] = 0.0                         # subnormal and zero exponentials
    x[3, 17] = float("inf")
    x[4, 4095] = float("nan")
    x[5] = float("-inf")
    x[5, 1] = 0.0
    x[6, 2048] = -0.0
    d = {"x": x.to(DEV)}
    y = run_with(wave_plan("softmax", "ordered", 4096, rows_per_cta), "softmax", d, "ordered").cpu().numpy()
    assert_bits(y, oracle.ot_softmax(x.numpy()), "extreme rows")


@pytest.mark.parametrize("order", ["unordered", "ordered"])
@pytest.mark.parametrize("op", ["rmsnorm", "layernorm"])
def test_wave_norms_without_affine_and_partial_affine(op, order):
    d = make(op, 13, 3000, seed=8)
    variants = [dict(w=None, b=None), dict(b=None)]
    if op == "layernorm":
        variants.append(dict(w=None))
    for v in variants:
        dd = dict(d)
        for k, val in v.items():
            dd.pop(k, None)
        h = host(dd)
        y = run_with(wave_plan(op, order, 3000, 1), op, dd, order).cpu().numpy()
        if order == "ordered":
            assert_bits(y, emulated(op, h), f"{op} {sorted(v)}")
        else:
            assert_close(y, reference(op, h), f"{op} {sorted(v)}")


@pytest.mark.parametrize("order", ["unordered", "ordered"])
@pytest.mark.parametrize("yoff", [1, 2, 3])
def test_wave_output_at_another_phase_and_guard_bands(order, yoff):
    # y rows at another 16-byte phase than x take scalar stores; nothing outside y is written
    rows, cols = 9, 2052
    d = make("layernorm", rows, cols, seed=40 + yoff)
    guard = 64
    big = torch.full((guard + rows * cols + guard + 4,), 7.25, device=DEV)
    y = big[guard + yoff:guard + yoff + rows * cols].view(rows, cols)
    run_with(wave_plan("layernorm", order, cols, 2), "layernorm", d, order, out=y)
    h = host(d)
    got = y.cpu().numpy()
    if order == "ordered":
        assert_bits(got, emulated("layernorm", h), "phase-shifted y")
    else:
        assert_close(got, reference("layernorm", h), "phase-shifted y")
    b = big.cpu().numpy()
    assert np.all(b[:guard + yoff] == 7.25) and np.all(b[guard + yoff + rows * cols:] == 7.25)


def test_wave_refuses_what_it_cannot_serve():
    # unaligned weights, rows under 1024 columns, a vec_slots that is not the
    # smallest cover, the fused residual and cross-entropy operators
    d = make("rmsnorm", 4, 2048, seed=1)
    wbig = torch.empty(2049, device=DEV)
    w = wbig[1:]
    w.copy_(d["w"])
    assert tr.tr_plan_override(wave_plan("rmsnorm", "unordered", 2048, 1)) == tr.TR_OK
    try:
        with pytest.raises(tr.TrError) as e:
            tr.rmsnorm(d["x"], w)
        assert e.value.status == tr.TR_ERR_UNSUPPORTED
        with pytest.raises(tr.TrError):
            tr.rmsnorm(d["x"][:, :1000].contiguous(), d["w"][:1000].contiguous())
    finally:
        tr.tr_plan_override(None)
    p = wave_plan("softmax", "unordered", 2048, 1)
    p.vec_slots = 4
    assert tr.tr_plan_override(p) == tr.TR_OK
    try:
        with pytest.raises(tr.TrError):
            tr.softmax(make("softmax", 4, 2048, seed=2)["x"])
    finally:
        tr.tr_plan_override(None)
    for op in ("cross_entropy",):
        q = tr.tr_plan(op=tr.OPS[op], order=0, kind=tr.TR_PLAN_WAVE, lanes_per_row=32, warps_per_row=8,
                       rows_per_cta=1, cluster_ctas=1, vec_slots=2, block_threads=256)
        assert tr.tr_plan_override(q) == tr.TR_OK
        try:
            with pytest.raises(tr.TrError):
                tr.tr_plan_describe(tr.OPS[op], 4, 2048, 0)
        finally:
            tr.tr_plan_override(None)


@pytest.mark.parametrize("order", ["unordered", "ordered"])
@pytest.mark.parametrize("op", OPS)
def test_wave_full_size_768x6144(op, order):
    d = synth.workload_inputs(f"{op}_768x6144", device=DEV)
    h = host(d)
    y = tr.run_op(op, d, order=order)
    torch.cuda.synchronize()
    got = y.cpu().numpy()
    if order == "ordered":
        assert_bits(got, emulated(op, h), f"{op} 768x6144")
    else:
        assert_close(got, reference(op, h), f"{op} 768x6144")


@pytest.mark.parametrize("rows_per_cta", [1, 2])
def test_wave_ordered_softmax_dense_exp_range(rows_per_cta):
    # every difference x - max in (-86, 0], dense, plus a band where x / ln2 lies
    # within a few ulps of a half-integer (the rounding that picks the exp's k):
    # the packed exp must give the emulation's bits for all of them
    rng = np.random.default_rng(99 + rows_per_cta)
    rows, cols = 2048, 4096
    x = -(rng.random((rows, cols)) * 85.99).astype(np.float32)
    half = (rng.integers(-124, 0, size=(rows // 2, cols)) + 0.5) / np.log2(np.e)
    band = half.astype(np.float32).view(np.int32) + rng.integers(-3, 4, size=half.shape).astype(np.int32)
    x[: rows // 2] = np.maximum(band.view(np.float32), np.float32(-85.99))
    x[:, 0] = 0.0                                   # the row maximum, so x - max = x
    d = {"x": torch.from_numpy(x).to(DEV)}
    y = run_with(wave_plan("softmax", "ordered", cols, rows_per_cta), "softmax", d, "ordered").cpu().numpy()
    assert_bits(y, oracle.ot_softmax(x), "dense exp range")


@pytest.mark.parametrize("order", ["unordered", "ordered"])
@pytest.mark.parametrize("op", OPS)
def test_wave_two_rows_balanced_over_every_resident_cta(op, order):
    # rows between the resident CTAs (res) and twice as many: the grid is every
    # resident CTA, rows - res of them with two rows and the rest with one
    cols = 6000
    p = wave_plan(op, order, cols, 2)
    for extra in (1, 77, 1 << 20):
        assert tr.tr_plan_override(p) == tr.TR_OK
        try:
            res = tr.tr_plan_describe(tr.OPS[op], 10, cols, 1 if order == "ordered" else 0).resident_ctas
        finally:
            tr.tr_plan_override(None)
        rows = min(2 * res - 1, res + extra)
        d = make(op, rows, cols, seed=rows)
        y = run_with(p, op, d, order).cpu().numpy()
        assert tr.tr_plan_override(p) == tr.TR_OK
        try:
            assert tr.tr_plan_describe(tr.OPS[op], rows, cols, 1 if order == "ordered" else 0).grid_ctas == res
        finally:
            tr.tr_plan_override(None)
        h = host(d)
        if order == "ordered":
            assert_bits(y, emulated(op, h), f"{op} {rows}x{cols} balanced")
        else:
            assert_close(y, reference(op, h), f"{op} {rows}x{cols} balanced")

