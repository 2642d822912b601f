"""GPU parity of the segments plan (TR_PLAN_SEGMENTS) against the CPU oracle.
The selector picks it for the norms' long rows and for softmax's few long
rows; these tests force it with the plan override wherever it is legal.

Few long rows: every co-resident CTA (one per SM) owns one column segment of
every row and keeps its columns' weight and bias in registers for all rows;
the rows' partial statistics meet once in the stream's workspace ("TIRx Metal
reduction lowering" §4.2, the combine of cooperating workers one level above a
CTA). Unordered policy: |gpu - oracle| <= 1e-6 + 2e-6 |oracle| element by
element. Covered: rows with cached and streamed segments, 1 and 32 rows,
ragged segment boundaries, outputs at another 16-byte phase, guard bands,
repeated launches on one workspace (the arrival word is reset by the last CTA),
the give-up path of its wait for the other CTAs, and the refusals.
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


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tr.load()
    yield
    tr.tr_plan_override(None)
    tr.tr_debug_force_wait_timeout(0)


def sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def seg_plan(op, rows, cols):
    sq = -(-(cols // 4) // sms())
    k = -(-sq // 1024)
    return tr.tr_plan(op=tr.OPS[op], order=0, kind=tr.TR_PLAN_SEGMENTS, lanes_per_row=32, warps_per_row=32,
                      rows_per_cta=rows, cluster_ctas=1, vec_slots=k, block_threads=1024)


def make(op, rows, cols, seed):
    if op == "softmax":
        return synth.make_inputs(op, rows, cols, seed, var=4.0, device=DEV)
    return synth.make_inputs(op, rows, cols, seed, row_offset=True, device=DEV)


def reference(op, d, eps=1e-5):
    h = {k: v.cpu().numpy() for k, v in d.items()}
    if op == "softmax":
        return oracle.softmax(h["x"])
    if op == "rmsnorm":
        return oracle.rmsnorm(h["x"], h.get("w"), eps)
    return oracle.layernorm(h["x"], h.get("w"), h.get("b"), eps)


def assert_close(got, ref, what):
    got = np.asarray(got, np.float64)
    bad = ~(np.abs(got - ref) <= ATOL + RTOL * np.abs(ref))
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} outside tolerance"


def run_with(plan, op, d, out=None):
    assert tr.tr_plan_override(plan) == tr.TR_OK
    try:
        y = tr.run_op(op, d, out=out)
        torch.cuda.synchronize()
        r, c = d["x"].shape
        assert tr.tr_plan_describe(tr.OPS[op], r, c, 0).kind == tr.TR_PLAN_SEGMENTS
    finally:
        tr.tr_plan_override(None)
    assert tr.tr_last_device_error() == tr.TR_OK
    return y


# rows x cols: all rows cached, part cached, 1 row, 26 rows (26 x 152 partials fill
# most of the workspace), a segment count that does not divide the quads, the
# longest row one launch covers with 2 slots
SHAPES = [(4, 400000), (16, 400000), (16, 1048576), (1, 400000), (26, 320000), (7, 400004), (3, 1245184)]


@pytest.mark.parametrize("rows,cols", SHAPES)
@pytest.mark.parametrize("op", OPS)
def test_segments_match_oracle(op, rows, cols):
    d = make(op, rows, cols, seed=rows * 13 + cols % 1000)
    y = run_with(seg_plan(op, rows, cols), op, d)
    assert_close(y.cpu().numpy(), reference(op, d), f"{op} {rows}x{cols}")


@pytest.mark.parametrize("op", OPS)
def test_segments_selection_and_default_path(op):
    # the norms' 16 x 1048576 and every op's two rows of 1048576 run it unforced;
    # softmax's 16 rows keep the split plan (measured faster there)
    norm = op != "softmax"
    assert (tr.tr_plan_describe(tr.OPS[op], 16, 1048576, 0).kind == tr.TR_PLAN_SEGMENTS) == norm
    assert tr.tr_plan_describe(tr.OPS[op], 2, 1048576, 0).kind == tr.TR_PLAN_SEGMENTS
    assert any(c.kind == tr.TR_PLAN_SEGMENTS for c in tr.plan_candidates(tr.OPS[op], 2, 1048576, 0, 1))
    d = make(op, 2, 1048576, seed=31)
    y = tr.run_op(op, d)
    torch.cuda.synchronize()
    assert tr.tr_last_device_error() == tr.TR_OK
    assert_close(y.cpu().numpy(), reference(op, d), f"{op} 2x1048576 unforced")


@pytest.mark.parametrize("yoff", [1, 3])
def test_segments_output_at_another_phase_and_guard_bands(yoff):
    rows, cols = 5, 400000
    d = make("layernorm", rows, cols, seed=yoff)
    guard = 4096
    big = torch.full((guard + rows * cols + guard + 4,), 7.25, device=DEV)
    y = big[guard + yoff:guard + yoff + rows * cols].view(rows, cols)
    run_with(seg_plan("layernorm", rows, cols), "layernorm", d, out=y)
    assert_close(y.cpu().numpy(), reference("layernorm", d), "phase-shifted y")
    b = big.cpu().numpy()
    assert np.all(b[:guard + yoff] == 7.25) and np.all(b[guard + yoff + rows * cols:] == 7.25)


def test_segments_repeated_launches_and_norms_without_affine():
    rows, cols = 9, 400000
    d = make("rmsnorm", rows, cols, seed=4)
    first = run_with(seg_plan("rmsnorm", rows, cols), "rmsnorm", d).clone()
    for _ in range(3):
        again = run_with(seg_plan("rmsnorm", rows, cols), "rmsnorm", d)
        assert torch.equal(first.view(torch.int32), again.view(torch.int32))
    for op, drop in (("rmsnorm", ("w",)), ("layernorm", ("w", "b")), ("layernorm", ("b",))):
        dd = make(op, rows, cols, seed=5)
        for k in drop:
            dd.pop(k)
        y = run_with(seg_plan(op, rows, cols), op, dd)
        assert_close(y.cpu().numpy(), reference(op, dd), f"{op} without {drop}")


def test_segments_plan_has_no_copy_wait():
    # its segments stream through registers: the copy give-up mode changes nothing
    rows, cols = 16, 400000
    d = make("layernorm", rows, cols, seed=21)
    assert tr.tr_debug_force_wait_timeout(2) == tr.TR_OK
    try:
        y = run_with(seg_plan("layernorm", rows, cols), "layernorm", d)
    finally:
        tr.tr_debug_force_wait_timeout(0)
    assert_close(y.cpu().numpy(), reference("layernorm", d), "copy give-up mode")


@pytest.mark.parametrize("mode", [4, 6])
def test_segments_give_up_and_recover(mode):
    # a wait that gives up: the timeout is reported, no output is written, and
    # the next launch on the same workspace matches the oracle (nothing reset)
    rows, cols = 16, 400000
    d = make("softmax", rows, cols, seed=mode)
    ref = reference("softmax", d)
    y = torch.full_like(d["x"], 7.25)
    assert tr.tr_plan_override(seg_plan("softmax", rows, cols)) == tr.TR_OK
    try:
        tr.run_op("softmax", d)               # the stream's workspace exists before the forced launch
        torch.cuda.synchronize()
        assert tr.tr_debug_force_wait_timeout(mode) == tr.TR_OK
        tr.run_op("softmax", d, out=y)
        tr.run_op("softmax", d, out=y)
        assert tr.tr_debug_force_wait_timeout(0) == tr.TR_OK
        z = tr.run_op("softmax", d)
        torch.cuda.synchronize()
    finally:
        tr.tr_debug_force_wait_timeout(0)
        tr.tr_plan_override(None)
    assert bool((y == 7.25).all())
    assert_close(z.cpu().numpy(), ref, "after giving up")
    assert tr.tr_last_device_error() == tr.TR_ERR_DEVICE_TIMEOUT
    assert tr.tr_last_device_error() == tr.TR_OK


def test_segments_refusals():
    rows, cols = 4, 400000
    d = make("rmsnorm", rows, cols, seed=1)
    assert tr.tr_plan_override(seg_plan("rmsnorm", rows, cols)) == tr.TR_OK
    try:
        wbig = torch.empty(cols + 1, device=DEV)
        w = wbig[1:]
        w.copy_(d["w"])
        with pytest.raises(tr.TrError) as e:             # unaligned weights
            tr.rmsnorm(d["x"], w)
        assert e.value.status == tr.TR_ERR_UNSUPPORTED
        with pytest.raises(tr.TrError):                  # rows_per_cta must equal the rows
            tr.rmsnorm(d["x"][:3].contiguous(), d["w"])
        with pytest.raises(tr.TrError):                  # the ordered policy is not served
            tr.rmsnorm(d["x"], d["w"], order="ordered")
    finally:
        tr.tr_plan_override(None)
    p = seg_plan("softmax", 40, cols)
    assert tr.tr_plan_override(p) == tr.TR_OK
    try:
        with pytest.raises(tr.TrError):                  # more than 32 rows
            tr.tr_plan_describe(0, 40, cols, 0)
    finally:
        tr.tr_plan_override(None)
