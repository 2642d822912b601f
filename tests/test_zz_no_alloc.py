"""The no-allocation entry point (tr_split_rows_noalloc_f32) against the CPU oracle.

Some callers cannot allocate device memory when they call: code that runs
inside a pre-sized arena in which every byte is accounted for, or a
latency-critical loop in which cudaMalloc (which may synchronise the device and
can fail under memory pressure) is not allowed. This entry point runs the
split-row plan over a fixed scratch array compiled into the library instead of
a workspace allocated on first use. Two calls in a row must each match the
FP64 oracle within the unordered tolerance (|gpu - oracle| <= 1e-6 + 2e-6
|oracle|) and give identical bits. Oversize inputs are refused before any
launch. The file is named to be collected last, and it holds no state that
depends on the tests before it.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import fp32_row_reduction_gb300 as tr

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
RTOL, ATOL = 2e-6, 1e-6


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tr.load()
    tr.tr_plan_override(None)
    tr.tr_debug_force_wait_timeout(0)


def reference(op, d, eps=1e-5):
    h = {k: v.cpu().numpy() for k, v in d.items()}
    if op == "softmax":
        return oracle.softmax(h["x"])
    if op == "rmsnorm":
        return oracle.rmsnorm(h["x"], h.get("w"), eps)
    return oracle.layernorm(h["x"], h.get("w"), h.get("b"), eps)


def assert_close(got, ref, what):
    got = got.cpu().numpy().astype(np.float64)
    err = np.abs(got - ref)
    bad = ~(err <= ATOL + RTOL * np.abs(ref))
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} elements outside tolerance"


CASES = [("softmax", 16, 65536), ("rmsnorm", 16, 262144), ("layernorm", 16, 65536), ("softmax", 3, 70001),
         ("layernorm", 5, 100003), ("rmsnorm", 1, 1), ("softmax", 150, 4096)]


@pytest.mark.parametrize("op,rows,cols", CASES)
def test_two_calls_match_the_oracle(op, rows, cols):
    d = synth.make_inputs(op, rows, cols, 41 + rows, var=4.0 if op == "softmax" else 1.0, device=DEV)
    ref = reference(op, d)
    a = torch.empty_like(d["x"])
    b = torch.empty_like(d["x"])
    w = d.get("w") if op != "softmax" else None
    bias = d.get("b") if op == "layernorm" else None
    tr.split_rows_noalloc(op, d["x"], a, weight=w, bias=bias)
    tr.split_rows_noalloc(op, d["x"], b, weight=w, bias=bias)
    torch.cuda.synchronize()
    assert tr.tr_last_device_error() == tr.TR_OK
    assert_close(a, ref, f"{op} {rows}x{cols}: first call")
    assert_close(b, ref, f"{op} {rows}x{cols}: second call")
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_matches_the_oracle_on_a_ragged_unaligned_row():
    rows, cols = 2, 40003
    d = synth.make_inputs("layernorm", rows, cols, 7, device=DEV)
    xbig = torch.empty(rows * cols + 4, device=DEV)
    x = xbig[1:1 + rows * cols].view(rows, cols)
    x.copy_(d["x"])
    y = torch.empty(rows, cols, device=DEV)
    tr.split_rows_noalloc("layernorm", x, y, weight=d["w"], bias=d["b"])
    torch.cuda.synchronize()
    ref = oracle.layernorm(d["x"].cpu().numpy(), d["w"].cpu().numpy(), d["b"].cpu().numpy(), 1e-5)
    got = y.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - ref) <= 1e-6 + 2e-6 * np.abs(ref))


def test_oversize_inputs_are_refused_without_a_launch():
    x = torch.zeros(300, 64, device=DEV)
    y = torch.full_like(x, 7.0)
    with pytest.raises(tr.TrError) as e:
        tr.split_rows_noalloc("softmax", x, y)
    assert e.value.status == tr.TR_ERR_UNSUPPORTED and "256 rows" in str(e.value)
    x = torch.zeros(200, 64, device=DEV)
    y = torch.full_like(x, 7.0)
    with pytest.raises(tr.TrError) as e:
        tr.split_rows_noalloc("rmsnorm", x, y)
    assert e.value.status == tr.TR_ERR_UNSUPPORTED and "co-resident" in str(e.value)
    torch.cuda.synchronize()
    assert float(y.min()) == 7.0 and float(y.max()) == 7.0   # nothing was written


def test_bad_arguments_are_refused():
    x = torch.zeros(4, 64, device=DEV)
    y = torch.empty_like(x)
    w = torch.ones(64, device=DEV)
    st = tr.tr_split_rows_noalloc_f32(0, x.data_ptr(), w.data_ptr(), None, y.data_ptr(), 4, 64, 0.0,
                                      torch.cuda.current_stream().cuda_stream)
    assert st == tr.TR_ERR_INVALID_ARG                         # softmax takes no weight
    st = tr.tr_split_rows_noalloc_f32(3, x.data_ptr(), None, None, y.data_ptr(), 4, 64, 0.0,
                                      torch.cuda.current_stream().cuda_stream)
    assert st == tr.TR_ERR_INVALID_ARG                         # cross-entropy is not offered
    st = tr.tr_split_rows_noalloc_f32(1, x.data_ptr(), None, None, x.data_ptr(), 4, 64, 1e-5,
                                      torch.cuda.current_stream().cuda_stream)
    assert st == tr.TR_ERR_INVALID_ARG                         # in place
