"""The C-ABI library without a GPU: it loads, exports every declared symbol,
and rejects bad arguments on the host before touching CUDA."""
import ctypes
import os
import re

import pytest

import fp32_row_reduction_gb300 as trlib
from fp32_row_reduction_gb300 import build as trbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tr.h")


@pytest.fixture(scope="module")
def lib():
    trbuild.build()
    return trlib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tr_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_four_operators():
    names = declared_functions()
    for n in ("tr_softmax_f32", "tr_rmsnorm_f32", "tr_layernorm_f32", "tr_cross_entropy_f32"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in trlib.SIGNATURES, f"binding lacks {name}"


def test_status_strings(lib):
    assert trlib.tr_status_string(0) == "TR_OK"
    assert trlib.tr_status_string(1) == "TR_ERR_INVALID_ARG"
    assert trlib.tr_status_string(4) == "TR_ERR_DEVICE_TIMEOUT"
    assert lib.tr_version() >= 100


def test_plan_struct_layout_matches_header():
    # int32 x 10, int64, double, int32 x 2, int64 -> 72 bytes with natural alignment
    assert ctypes.sizeof(trlib.tr_plan) == 72
    assert ctypes.sizeof(trlib.tr_device_desc) == 40


FAKE = 1 << 20  # host-side fake "device" addresses: validation runs before any CUDA call


@pytest.mark.parametrize("args,why", [
    ((FAKE, FAKE + 4096, 1, 1, 7, None), "bad order"),
    ((FAKE, FAKE + 4096, -1, 8, 0, None), "rows < 0"),
    ((FAKE, FAKE + 4096, 4, 0, 0, None), "cols < 1"),
    ((FAKE, FAKE + 4096, 4, 1 << 31, 0, None), "cols >= 2^31"),
    ((None, FAKE, 4, 8, 0, None), "null x"),
    ((FAKE, None, 4, 8, 0, None), "null y"),
    ((FAKE + 2, FAKE + 4096, 4, 8, 0, None), "x not 4-byte aligned"),
    ((FAKE, FAKE + 64, 4, 8, 0, None), "x and y overlap"),
    ((FAKE, FAKE, 4, 8, 0, None), "in place"),
])
def test_softmax_rejects(lib, args, why):
    assert trlib.tr_softmax_f32(*args) == trlib.TR_ERR_INVALID_ARG, why
    assert trlib.tr_last_error_message() != ""


def test_zero_rows_is_a_no_op(lib):
    assert trlib.tr_softmax_f32(None, None, 0, 5, 0, None) == trlib.TR_OK
    assert trlib.tr_cross_entropy_f32(None, None, None, 0, 5, 0, None) == trlib.TR_OK


@pytest.mark.parametrize("eps", [-1e-5, float("nan"), float("inf")])
def test_norms_reject_bad_eps(lib, eps):
    assert trlib.tr_rmsnorm_f32(FAKE, None, FAKE + 4096, 2, 8, eps, 0, None) == trlib.TR_ERR_INVALID_ARG
    assert trlib.tr_layernorm_f32(FAKE, None, None, FAKE + 4096, 2, 8, eps, 0, None) == trlib.TR_ERR_INVALID_ARG


def test_norm_output_must_not_alias_parameters(lib):
    # y overlaps w / beta
    assert trlib.tr_rmsnorm_f32(FAKE, FAKE + 4096, FAKE + 4096, 2, 8, 1e-5, 0, None) == trlib.TR_ERR_INVALID_ARG
    assert trlib.tr_layernorm_f32(FAKE, None, FAKE + 4100, FAKE + 4096, 2, 8, 1e-5, 0, None) \
        == trlib.TR_ERR_INVALID_ARG


def test_cross_entropy_rejects(lib):
    f = trlib.tr_cross_entropy_f32
    assert f(FAKE, None, FAKE + 8192, 4, 8, 0, None) == trlib.TR_ERR_INVALID_ARG       # null labels
    assert f(FAKE, FAKE + 8196, FAKE + 16384, 4, 8, 0, None) == trlib.TR_ERR_INVALID_ARG  # labels misaligned
    assert f(FAKE, FAKE + 8192, FAKE + 8, 4, 8, 0, None) == trlib.TR_ERR_INVALID_ARG   # losses inside logits
    assert f(FAKE, FAKE + 8192, FAKE + 8200, 4, 8, 0, None) == trlib.TR_ERR_INVALID_ARG  # losses inside labels


def test_calls_without_a_gpu_fail_loudly(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    # valid arguments: the library reaches CUDA and reports the missing device
    assert trlib.tr_softmax_f32(FAKE, FAKE + 4096, 4, 8, 0, None) == trlib.TR_ERR_CUDA


def test_override_rejects_malformed(lib):
    p = trlib.tr_plan(op=10)   # one past the last operator
    assert trlib.tr_plan_override(p) == trlib.TR_ERR_INVALID_ARG
    p = trlib.tr_plan(op=0, kind=17)
    assert trlib.tr_plan_override(p) == trlib.TR_ERR_INVALID_ARG
    assert trlib.tr_plan_override(None) == trlib.TR_OK


def test_noalloc_entry_rejects_bad_arguments_on_the_host(lib):
    f = trlib.tr_split_rows_noalloc_f32
    assert f(0, None, None, None, None, 0, 10, 0.0, None) == trlib.TR_OK          # empty: nothing to do
    assert f(3, None, None, None, None, 4, 10, 0.0, None) == trlib.TR_ERR_INVALID_ARG  # no cross-entropy
    assert f(0, 0x1000, 0x2000, None, 0x100000, 4, 10, 0.0, None) == trlib.TR_ERR_INVALID_ARG  # softmax + w
    assert f(1, 0x1000, None, None, 0x100000, 4, 10, float("nan"), None) == trlib.TR_ERR_INVALID_ARG
    assert f(2, 0x1000, None, None, 0x1010, 4, 10, 1e-5, None) == trlib.TR_ERR_INVALID_ARG  # y overlaps x
    assert f(2, 0x1002, None, None, 0x100000, 4, 10, 1e-5, None) == trlib.TR_ERR_INVALID_ARG  # misaligned
    # more rows than the fixed scratch holds: refused before any CUDA call
    assert f(0, 0x1000, None, None, 0x10000000, 257, 10, 0.0, None) == trlib.TR_ERR_UNSUPPORTED
    assert "256 rows" in lib.tr_last_error_message().decode()


def test_next_row_entry_points_validate_on_the_host(lib):
    L = trlib.load()
    E, U = trlib.TR_ERR_INVALID_ARG, trlib.TR_ERR_UNSUPPORTED
    # backward passes: null outputs, aliasing, bad order, fold orders refused
    assert L.tr_softmax_backward_f32(FAKE, FAKE + 4096, None, 2, 8, 0, None) == E
    assert L.tr_softmax_backward_f32(FAKE, FAKE + 4096, FAKE, 2, 8, 0, None) == E          # dx aliases y
    assert L.tr_softmax_backward_f32(FAKE, FAKE + 4096, FAKE + 8192, 2, 8, 9, None) == E
    assert L.tr_softmax_backward_f32(FAKE, FAKE + 4096, FAKE + 8192, 2, 8, 2, None) == U    # fold_left
    assert L.tr_cross_entropy_backward_f32(FAKE, None, None, FAKE + 8192, 2, 8, 0, None) == E
    assert L.tr_rmsnorm_backward_f32(FAKE, None, FAKE + 4096, FAKE + 8192, None, 2, 8, -1.0, 0, None, 0, None) == E
    assert L.tr_layernorm_backward_f32(FAKE, None, FAKE + 4096, FAKE + 8192, None, None, 2, 8, 1e-5, 3, None, 0,
                                       None) == U
    n = ctypes.c_size_t(0)
    assert L.tr_norm_backward_workspace_bytes(10, 100, ctypes.byref(n)) == trlib.TR_OK and n.value == 80
    # axis reductions: sizes, aliasing, fold orders refused
    assert L.tr_axis_sum_f32(FAKE, FAKE + 4096, 2, 0, 4, 0, None) == E
    assert L.tr_axis_sum_f32(FAKE, FAKE, 2, 3, 4, 0, None) == E
    assert L.tr_axis_max_f32(FAKE, FAKE + 4096, 2, 3, 4, 3, None) == U
    assert L.tr_axis_minmax_f32(FAKE, FAKE + 4096, None, 2, 3, 4, 0, None) == E
    # row reductions and the fused norms under bad arguments
    assert L.tr_row_minmax_f32(FAKE, FAKE + 4096, None, 2, 8, 0, None) == E
    assert L.tr_row_sum_f32(FAKE, FAKE + 4096, 2, 8, 4, None) == E
    assert L.tr_add_rmsnorm_f32(FAKE, None, None, FAKE + 4096, None, 2, 8, 1e-5, 0, None) == E


def test_axis_launch_shape_on_the_host(lib):
    sp, tl = trlib.axis_launch_shape("sum", 1, 768, 6144, 152)
    assert tl == 48 and 1 <= sp <= 32 and sp & (sp - 1) == 0
    sp, tl = trlib.axis_launch_shape("sum", 1, 768, 6144, 152, "ordered")
    assert tl == 192 and sp in (1, 2, 4, 8)
    sp, tl = trlib.axis_launch_shape("sum", 1, 20000, 7, 152)
    assert tl == 1 and sp == 32


def test_empty_inputs_are_a_no_op_on_every_entry_point(lib):
    L = trlib.load()
    ok = trlib.TR_OK
    ws = ctypes.c_size_t(0)
    assert L.tr_softmax_backward_f32(FAKE, FAKE + 4096, FAKE + 8192, 0, 8, 0, None) == ok
    assert L.tr_cross_entropy_backward_f32(FAKE, FAKE + 4096, None, FAKE + 8192, 0, 8, 1, None) == ok
    assert L.tr_rmsnorm_backward_f32(FAKE, None, FAKE + 4096, FAKE + 8192, FAKE + 12288, 0, 8, 1e-5, 0, None, 0,
                                     None) == ok
    assert L.tr_layernorm_backward_f32(FAKE, None, FAKE + 4096, FAKE + 8192, None, None, 0, 8, 1e-5, 1, None, 0,
                                       None) == ok
    assert L.tr_norm_backward_workspace_bytes(0, 8, ctypes.byref(ws)) == ok and ws.value == 0
    assert L.tr_axis_sum_f32(FAKE, FAKE + 4096, 0, 5, 3, 1, None) == ok
    for order in (0, 1, 2, 3):
        assert L.tr_row_sum_f32(FAKE, FAKE + 4096, 0, 8, order, None) == ok
        assert L.tr_softmax_f32(FAKE, FAKE + 4096, 0, 8, order, None) == ok


BIG = 1 << 24  # the first width the operators refuse: (float)cols must be exact


@pytest.mark.parametrize("call,name", [
    (lambda: trlib.tr_softmax_f32(FAKE, FAKE + 4 * BIG + 64, 1, BIG, 0, None), "softmax"),
    (lambda: trlib.tr_rmsnorm_f32(FAKE, None, FAKE + 4 * BIG + 64, 1, BIG, 1e-5, 0, None), "rmsnorm"),
    (lambda: trlib.tr_layernorm_f32(FAKE, None, None, FAKE + 4 * BIG + 64, 1, BIG, 1e-5, 1, None), "layernorm"),
    (lambda: trlib.tr_cross_entropy_f32(FAKE, FAKE + 4 * BIG + 64, FAKE + 4 * BIG + 256, 1, BIG, 0, None),
     "cross-entropy"),
    (lambda: trlib.tr_add_rmsnorm_f32(FAKE, FAKE + 4 * BIG + 64, None, FAKE + 8 * BIG + 128, None, 1, BIG,
                                      1e-5, 0, None), "fused residual RMSNorm"),
    (lambda: trlib.tr_split_rows_noalloc_f32(0, FAKE, None, None, FAKE + 4 * BIG + 64, 1, BIG, 0.0, None),
     "no-allocation entry point"),
])
def test_operators_refuse_cols_of_2_to_the_24(lib, call, name):
    # the operators take 1 <= cols < 2^24 (validation runs before any CUDA call)
    assert call() == trlib.TR_ERR_INVALID_ARG, name
    assert "2^24" in trlib.tr_last_error_message(), name


def test_debug_hook_takes_a_mask_of_known_modes(lib):
    # the hook only sets host state: no GPU is needed to check its arguments
    assert trlib.tr_debug_force_wait_timeout(8) == trlib.TR_ERR_INVALID_ARG
    assert trlib.tr_debug_force_wait_timeout(6) == trlib.TR_OK
    assert trlib.tr_debug_force_wait_timeout(0) == trlib.TR_OK
