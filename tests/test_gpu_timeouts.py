"""The give-up paths of the bounded device-side waits, run without a fault or hang.

"TIRx Metal reduction lowering" §1: failures are explicit errors, never a
fallback. Every device wait of the library has a time limit; when it passes,
the kernel records TR_ERR_DEVICE_TIMEOUT in the device error word and leaves
without trapping. The testing hook tr_debug_force_wait_timeout(mode) makes
the real waits give up at their first check (mode 2: waits for bulk copies;
mode 4: the split plan's wait for the other CTAs of a row), so these tests
check, for the split plan on its per-stream workspace, for the
no-allocation entry point on its static scratch, and for the staged rings:
  - the launch reports TR_ERR_DEVICE_TIMEOUT and the context stays usable;
  - a split row whose wait gave up skips its epilogue in every CTA (its
    outputs keep their previous contents);
  - the next launches on the same stream, workspace and scratch are correct
    against the oracle with nothing reset on the host in between.
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
SENTINEL = 7.25


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tr.load()
    yield
    tr.tr_debug_force_wait_timeout(0)
    tr.tr_plan_override(None)


@pytest.fixture(autouse=True)
def _reset():
    assert tr.tr_last_device_error() == tr.TR_OK
    yield
    tr.tr_debug_force_wait_timeout(0)
    tr.tr_plan_override(None)
    tr.tr_last_device_error()


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


def split_plan(op, C, T, K):
    return tr.tr_plan(op=tr.OPS[op], order=0, kind=tr.TR_PLAN_SPLIT, lanes_per_row=32, warps_per_row=T // 32,
                      rows_per_cta=1, cluster_ctas=C, vec_slots=K, block_threads=T)


@pytest.mark.parametrize("mode", [4, 6])
@pytest.mark.parametrize("op,C,K", [("softmax", 4, 4), ("layernorm", 3, 0), ("rmsnorm", 8, 2)])
def test_split_plan_gives_up_and_recovers(op, C, K, mode):
    rows, cols = 6, 20002
    d = make(op, rows, cols, seed=C * 10 + K + mode)
    ref = reference(op, d)
    s = torch.cuda.Stream()
    assert tr.tr_plan_override(split_plan(op, C, 256, K)) == tr.TR_OK
    with torch.cuda.stream(s):
        warm = tr.run_op(op, d)             # the stream's workspace exists before the forced launches
        s.synchronize()
        assert_close(warm.cpu().numpy(), ref, "before")
        y = torch.full_like(d["x"], SENTINEL)
        assert tr.tr_debug_force_wait_timeout(mode) == tr.TR_OK
        for _ in range(3):                  # counters must not drift over repeated give-ups
            tr.run_op(op, d, out=y)
        assert tr.tr_debug_force_wait_timeout(0) == tr.TR_OK
        z = tr.run_op(op, d)                # same stream, same workspace, no host-side reset
        s.synchronize()
    assert bool((y == SENTINEL).all()), "a row whose wait gave up wrote outputs"
    assert_close(z.cpu().numpy(), ref, f"{op} after giving up (mode {mode})")
    assert tr.tr_last_device_error() == tr.TR_ERR_DEVICE_TIMEOUT
    assert tr.tr_last_device_error() == tr.TR_OK
    with torch.cuda.stream(s):
        z2 = tr.run_op(op, d)
        s.synchronize()
    assert tr.tr_last_device_error() == tr.TR_OK
    assert torch.equal(z.view(torch.int32), z2.view(torch.int32))


@pytest.mark.parametrize("op", ["softmax", "rmsnorm", "layernorm"])
def test_split_plan_has_no_copy_wait(op):
    # mode 2 expires bulk-copy waits; the split plan streams its segments
    # through registers, so it runs normally under it
    rows, cols = 6, 20002
    d = make(op, rows, cols, seed=21)
    assert tr.tr_plan_override(split_plan(op, 4, 256, 4)) == tr.TR_OK
    try:
        tr.run_op(op, d)
        torch.cuda.synchronize()
        assert tr.tr_debug_force_wait_timeout(2) == tr.TR_OK
        y = tr.run_op(op, d)
        torch.cuda.synchronize()
    finally:
        tr.tr_debug_force_wait_timeout(0)
        tr.tr_plan_override(None)
    assert_close(y.cpu().numpy(), reference(op, d), f"{op} under mode 2")
    assert tr.tr_last_device_error() == tr.TR_OK


@pytest.mark.parametrize("mode", [4, 6])
@pytest.mark.parametrize("op", ["softmax", "rmsnorm", "layernorm"])
def test_no_alloc_entry_point_gives_up_and_recovers(op, mode):
    rows, cols = 16, 65536
    d = make(op, rows, cols, seed=3 + mode)
    ref = reference(op, d)
    w = d.get("w") if op != "softmax" else None
    b = d.get("b") if op == "layernorm" else None
    y = torch.full_like(d["x"], SENTINEL)
    z = torch.empty_like(d["x"])
    assert tr.tr_debug_force_wait_timeout(mode) == tr.TR_OK
    tr.split_rows_noalloc(op, d["x"], y, weight=w, bias=b)
    tr.split_rows_noalloc(op, d["x"], y, weight=w, bias=b)
    assert tr.tr_debug_force_wait_timeout(0) == tr.TR_OK
    tr.split_rows_noalloc(op, d["x"], z, weight=w, bias=b)   # the scratch is not reset in between
    torch.cuda.synchronize()
    assert bool((y == SENTINEL).all()), "a row whose wait gave up wrote outputs"
    assert_close(z.cpu().numpy(), ref, f"no-alloc {op} after giving up")
    assert tr.tr_last_device_error() == tr.TR_ERR_DEVICE_TIMEOUT
    assert tr.tr_last_device_error() == tr.TR_OK


@pytest.mark.parametrize("ordered", [False, True])
def test_staged_ring_gives_up_and_recovers(ordered):
    op = "layernorm"
    rows, cols = 40, 3000
    d = make(op, rows, cols, seed=21)
    kind = tr.TR_PLAN_ORDERED_STAGED if ordered else tr.TR_PLAN_STAGED
    p = tr.tr_plan(op=tr.OPS[op], order=1 if ordered else 0, kind=kind, lanes_per_row=32, warps_per_row=8,
                   rows_per_cta=3, cluster_ctas=1, vec_slots=4, block_threads=256)
    order = "ordered" if ordered else "unordered"
    assert tr.tr_plan_override(p) == tr.TR_OK
    assert tr.tr_debug_force_wait_timeout(2) == tr.TR_OK
    tr.run_op(op, d, order=order)           # outputs of the rows that gave up are undefined
    assert tr.tr_debug_force_wait_timeout(0) == tr.TR_OK
    z = tr.run_op(op, d, order=order)
    torch.cuda.synchronize()
    assert tr.tr_last_device_error() == tr.TR_ERR_DEVICE_TIMEOUT
    h = {k: v.cpu().numpy() for k, v in d.items()}
    if ordered:
        want = oracle.ot_layernorm(h["x"], h["w"], h["b"], 1e-5)
        assert np.array_equal(z.cpu().numpy().view(np.uint32), want.view(np.uint32))
    else:
        assert_close(z.cpu().numpy(), reference(op, d), "staged after giving up")


def test_hook_rejects_unknown_modes():
    assert tr.tr_debug_force_wait_timeout(8) == tr.TR_ERR_INVALID_ARG
    assert tr.tr_debug_force_wait_timeout(-1) == tr.TR_ERR_INVALID_ARG
    assert tr.tr_debug_force_wait_timeout(7) == tr.TR_OK
    assert tr.tr_debug_force_wait_timeout(0) == tr.TR_OK
