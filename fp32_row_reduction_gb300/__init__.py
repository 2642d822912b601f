"""GB300-native FP32 row reductions: Python binding of libtr (ctypes).

The binding only marshals arguments: every operator runs in libtr's CUDA
kernels on the GPU. There is no CPU or PyTorch fallback: if libtr.so is
missing, importing the library functions raises, and on a machine without a
GPU the calls return TR_ERR_CUDA.

Two layers:

* the C-ABI, same names and arguments as ``include/tr.h``
  (``tr_softmax_f32(x_ptr, y_ptr, rows, cols, order, stream)`` ...), taking
  integer device pointers and returning a ``tr_status`` int;
* tensor helpers (``softmax``, ``rmsnorm``, ``layernorm``, ``cross_entropy``)
  that take CUDA float32 tensors, allocate the output with PyTorch (PyTorch is
  used for device memory and streams only) and raise ``TrError`` on failure.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libtr.so")

TR_OK = 0
TR_ERR_INVALID_ARG = 1
TR_ERR_UNSUPPORTED = 2
TR_ERR_CUDA = 3
TR_ERR_DEVICE_TIMEOUT = 4

TR_ORDER_UNORDERED_TREE = 0
TR_ORDER_ORDERED_TREE = 1
TR_ORDER_FOLD_LEFT = 2
TR_ORDER_FOLD_RIGHT = 3

TR_OP_SOFTMAX = 0
TR_OP_RMSNORM = 1
TR_OP_LAYERNORM = 2
TR_OP_CROSS_ENTROPY = 3

TR_PLAN_ROWS = 0
TR_PLAN_CLUSTER = 1
TR_PLAN_STREAM = 2
TR_PLAN_XENT = 3
TR_PLAN_ORDERED = 4
TR_PLAN_STAGED = 5
TR_PLAN_ORDERED_STAGED = 6
TR_PLAN_SPLIT = 7
TR_PLAN_FOLD = 8
COST_CONSTANTS = 16  # TR_COST_CONSTANTS
TR_PLAN_WAVE = 9
TR_PLAN_SEGMENTS = 10
TR_OP_ADD_RMSNORM = 4
TR_OP_ADD_LAYERNORM = 5
TR_OP_ROW_SUM = 6
TR_OP_ROW_MAX = 7
TR_OP_ROW_MIN = 8
TR_OP_ROW_MINMAX = 9
TR_PLAN_FLAG_PARAMS_IN_REGISTERS = 1
TR_PLAN_FLAG_PARAMS_IN_SHARED = 2
TR_PLAN_FLAG_TWO_ROWS = 4

OPS = {"softmax": TR_OP_SOFTMAX, "rmsnorm": TR_OP_RMSNORM, "layernorm": TR_OP_LAYERNORM,
       "cross_entropy": TR_OP_CROSS_ENTROPY, "add_rmsnorm": TR_OP_ADD_RMSNORM, "add_layernorm": TR_OP_ADD_LAYERNORM,
       "row_sum": TR_OP_ROW_SUM, "row_max": TR_OP_ROW_MAX, "row_min": TR_OP_ROW_MIN, "row_minmax": TR_OP_ROW_MINMAX}
REDUCE_OPS = ("row_sum", "row_max", "row_min", "row_minmax")
# reductions over axis 0 of a 2-D tensor (one value per column)
AXIS_OPS = ("axis_sum", "axis_max", "axis_min", "axis_minmax")
ORDERS = {"unordered": TR_ORDER_UNORDERED_TREE, "ordered": TR_ORDER_ORDERED_TREE,
          "fold_left": TR_ORDER_FOLD_LEFT, "fold_right": TR_ORDER_FOLD_RIGHT}


class tr_plan(ctypes.Structure):
    _fields_ = [
        ("op", ctypes.c_int32), ("order", ctypes.c_int32), ("kind", ctypes.c_int32),
        ("lanes_per_row", ctypes.c_int32), ("warps_per_row", ctypes.c_int32),
        ("rows_per_cta", ctypes.c_int32), ("cluster_ctas", ctypes.c_int32),
        ("vec_slots", ctypes.c_int32), ("block_threads", ctypes.c_int32),
        ("ctas_per_sm", ctypes.c_int32), ("grid_ctas", ctypes.c_int64), ("est_us", ctypes.c_double),
        ("candidates", ctypes.c_int32), ("flags", ctypes.c_int32), ("resident_ctas", ctypes.c_int64),
    ]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


class tr_device_desc(ctypes.Structure):
    _fields_ = [
        ("sm_count", ctypes.c_int32), ("max_threads_per_sm", ctypes.c_int32),
        ("max_ctas_per_sm", ctypes.c_int32), ("regs_per_sm", ctypes.c_int32),
        ("smem_per_sm", ctypes.c_int32), ("max_cluster_ctas", ctypes.c_int32),
        ("l2_bytes", ctypes.c_int64), ("hbm_gbs", ctypes.c_double),
    ]


def gb300_device_desc() -> tr_device_desc:
    """The GB300 as the plan selector models it (152 SMs, 2048 threads, 64K registers)."""
    return tr_device_desc(sm_count=152, max_threads_per_sm=2048, max_ctas_per_sm=32,
                          regs_per_sm=65536, smem_per_sm=233472, max_cluster_ctas=16,
                          l2_bytes=126 << 20, hbm_gbs=7000.0)


# The exported C-ABI and its argument types.
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32
_F = ctypes.c_float
SIGNATURES = {
    "tr_softmax_f32": ([_P, _P, _I64, _I64, _I32, _P], _I32),
    "tr_rmsnorm_f32": ([_P, _P, _P, _I64, _I64, _F, _I32, _P], _I32),
    "tr_layernorm_f32": ([_P, _P, _P, _P, _I64, _I64, _F, _I32, _P], _I32),
    "tr_cross_entropy_f32": ([_P, _P, _P, _I64, _I64, _I32, _P], _I32),
    "tr_add_rmsnorm_f32": ([_P, _P, _P, _P, _P, _I64, _I64, _F, _I32, _P], _I32),
    "tr_row_sum_f32": ([_P, _P, _I64, _I64, _I32, _P], _I32),
    "tr_row_max_f32": ([_P, _P, _I64, _I64, _I32, _P], _I32),
    "tr_row_min_f32": ([_P, _P, _I64, _I64, _I32, _P], _I32),
    "tr_row_minmax_f32": ([_P, _P, _P, _I64, _I64, _I32, _P], _I32),
    "tr_axis_sum_f32": ([_P, _P, _I64, _I64, _I64, _I32, _P], _I32),
    "tr_axis_max_f32": ([_P, _P, _I64, _I64, _I64, _I32, _P], _I32),
    "tr_axis_min_f32": ([_P, _P, _I64, _I64, _I64, _I32, _P], _I32),
    "tr_axis_minmax_f32": ([_P, _P, _P, _I64, _I64, _I64, _I32, _P], _I32),
    "tr_axis_launch_shape": ([_I32, _I32, _I32, _I64, _I64, _I64, ctypes.POINTER(_I32), ctypes.POINTER(_I64)],
                             _I32),
    "tr_softmax_backward_f32": ([_P, _P, _P, _I64, _I64, _I32, _P], _I32),
    "tr_cross_entropy_backward_f32": ([_P, _P, _P, _P, _I64, _I64, _I32, _P], _I32),
    "tr_rmsnorm_backward_f32": ([_P, _P, _P, _P, _P, _I64, _I64, _F, _I32, _P, ctypes.c_size_t, _P], _I32),
    "tr_layernorm_backward_f32": ([_P, _P, _P, _P, _P, _P, _I64, _I64, _F, _I32, _P, ctypes.c_size_t, _P], _I32),
    "tr_norm_backward_workspace_bytes": ([_I64, _I64, ctypes.POINTER(ctypes.c_size_t)], _I32),
    "tr_add_layernorm_f32": ([_P, _P, _P, _P, _P, _P, _I64, _I64, _F, _I32, _P], _I32),
    "tr_plan_describe": ([_I32, _I64, _I64, _I32, ctypes.POINTER(tr_plan)], _I32),
    "tr_plan_select_for": ([ctypes.POINTER(tr_device_desc), _I32, _I64, _I64, _I32, _I32,
                            ctypes.POINTER(tr_plan)], _I32),
    "tr_split_rows_noalloc_f32": ([_I32, _P, _P, _P, _P, _I64, _I64, ctypes.c_float, _P], _I32),
    "tr_plan_cost_constants": ([ctypes.POINTER(ctypes.c_double), _I32], _I32),
    "tr_plan_estimate_with": ([ctypes.POINTER(tr_device_desc), ctypes.POINTER(tr_plan), _I64, _I64, _I32,
                               ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double)], _I32),
    "tr_plan_candidates": ([_I32, _I64, _I64, _I32, _I32, ctypes.POINTER(tr_plan), _I32,
                            ctypes.POINTER(_I32)], _I32),
    "tr_plan_check_for": ([ctypes.POINTER(tr_device_desc), ctypes.POINTER(tr_plan), _I64, _I64, _I32], _I32),
    "tr_plan_override": ([ctypes.POINTER(tr_plan)], _I32),
    "tr_last_device_error": ([], _I32),
    "tr_debug_force_wait_timeout": ([_I32], _I32),
    "tr_status_string": ([_I32], ctypes.c_char_p),
    "tr_last_error_message": ([], ctypes.c_char_p),
    "tr_version": ([], _I32),
}

_lib = None


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libtr.so (built by ``fp32_row_reduction_gb300.build``). Raises if missing."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(
            f"libtr.so not found at {p}: build it with `python -m fp32_row_reduction_gb300.build` "
            "(there is no fallback implementation)")
    lib = ctypes.CDLL(p)
    for name, (args, res) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    if path is None:
        _lib = lib
    return lib


class TrError(RuntimeError):
    def __init__(self, status: int, where: str):
        lib = load()
        msg = lib.tr_last_error_message().decode()
        super().__init__(f"{where}: {lib.tr_status_string(status).decode()} ({msg})")
        self.status = status


def _check(status: int, where: str):
    if status != TR_OK:
        raise TrError(status, where)


# --------------------------------------------------------------------- C-ABI

def tr_softmax_f32(x, y, rows, cols, order, stream):
    return load().tr_softmax_f32(x, y, rows, cols, order, stream)


def tr_split_rows_noalloc_f32(op, x, w, b, y, rows, cols, eps, stream):
    return load().tr_split_rows_noalloc_f32(op, x, w, b, y, rows, cols, eps, stream)


def split_rows_noalloc(op, x, out, weight=None, bias=None, eps=1e-5, stream=None):
    """The no-allocation entry point on CUDA float32 tensors. ``out`` is
    required: this wrapper creates no tensor, and the library allocates no
    device memory."""
    code = OPS[op] if isinstance(op, str) else int(op)
    _check_matrix(x, "x")
    _check_matrix(out, "out")
    r, c = x.shape
    wp = _check_vector(weight, "weight", c)
    bp = _check_vector(bias, "bias", c)
    _check(tr_split_rows_noalloc_f32(code, x.data_ptr(), wp, bp, out.data_ptr(), r, c, eps, _stream_handle(stream)),
           "split_rows_noalloc")
    return out


def tr_rmsnorm_f32(x, w, y, rows, cols, eps, order, stream):
    return load().tr_rmsnorm_f32(x, w, y, rows, cols, eps, order, stream)


def tr_layernorm_f32(x, gamma, beta, y, rows, cols, eps, order, stream):
    return load().tr_layernorm_f32(x, gamma, beta, y, rows, cols, eps, order, stream)


def tr_cross_entropy_f32(logits, labels, losses, rows, cols, order, stream):
    return load().tr_cross_entropy_f32(logits, labels, losses, rows, cols, order, stream)


def tr_plan_describe(op, rows, cols, order) -> tr_plan:
    out = tr_plan()
    _check(load().tr_plan_describe(op, rows, cols, order, ctypes.byref(out)), "tr_plan_describe")
    return out


def tr_plan_select_for(dev: tr_device_desc, op, rows, cols, order, align16=1) -> tr_plan:
    out = tr_plan()
    _check(load().tr_plan_select_for(ctypes.byref(dev), op, rows, cols, order, align16, ctypes.byref(out)),
           "tr_plan_select_for")
    return out


def check_plan_for(dev: tr_device_desc, plan: tr_plan, rows, cols, align16=1):
    """Host-only legality check: (status, reason). Fills the plan's grid and estimate when legal."""
    lib = load()
    st = lib.tr_plan_check_for(ctypes.byref(dev), ctypes.byref(plan), rows, cols, align16)
    return st, ("" if st == TR_OK else lib.tr_last_error_message().decode())


def cost_constants():
    """The library's cost-model constants (TR_COST_CONSTANTS doubles)."""
    out = (ctypes.c_double * COST_CONSTANTS)()
    _check(load().tr_plan_cost_constants(out, COST_CONSTANTS), "tr_plan_cost_constants")
    return list(out)


def estimate_with(dev: tr_device_desc, plan: tr_plan, rows, cols, align16=1, constants=None) -> float:
    """The model's estimate (us) for a plan with grid_ctas/ctas_per_sm filled, under given constants."""
    c = None if constants is None else (ctypes.c_double * COST_CONSTANTS)(*constants)
    out = ctypes.c_double()
    _check(load().tr_plan_estimate_with(ctypes.byref(dev), ctypes.byref(plan), rows, cols, align16, c,
                                        ctypes.byref(out)), "tr_plan_estimate_with")
    return out.value


def plan_candidates(op, rows, cols, order=0, align16=1):
    """Every legal candidate plan on the current device, with estimates."""
    lib = load()
    n = ctypes.c_int32()
    _check(lib.tr_plan_candidates(op, rows, cols, order, align16, None, 0, ctypes.byref(n)), "tr_plan_candidates")
    buf = (tr_plan * max(1, n.value))()
    _check(lib.tr_plan_candidates(op, rows, cols, order, align16, buf, n.value, ctypes.byref(n)), "tr_plan_candidates")
    return list(buf[:n.value])


def tr_plan_override(plan: tr_plan | None) -> int:
    return load().tr_plan_override(None if plan is None else ctypes.byref(plan))


def tr_last_device_error() -> int:
    return load().tr_last_device_error()


def tr_debug_force_wait_timeout(mode) -> int:
    """Testing hook (tr.h): True / 1 adds a wait nothing completes; 2 expires the
    bulk-copy waits; 4 expires the split plan's waits for peer CTAs; 0 / False off."""
    return load().tr_debug_force_wait_timeout(int(mode))


def tr_status_string(status: int) -> str:
    return load().tr_status_string(status).decode()


def tr_last_error_message() -> str:
    return load().tr_last_error_message().decode()


# ------------------------------------------------------------ tensor helpers

def _stream_handle(stream=None):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _check_matrix(t, name):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.float32:
        raise TypeError(f"{name} must be a CUDA float32 tensor")
    if t.dim() != 2 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous 2-D (rows x cols) tensor")


def _check_vector(t, name, cols):
    import torch
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.float32:
        raise TypeError(f"{name} must be a CUDA float32 tensor")
    if t.numel() != cols or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous vector of {cols} floats")
    return t.data_ptr()


def _order(order):
    return ORDERS[order] if isinstance(order, str) else int(order)


def softmax(x, out=None, order="unordered", stream=None):
    """Row softmax of a CUDA float32 (rows, cols) tensor."""
    import torch
    _check_matrix(x, "x")
    y = torch.empty_like(x) if out is None else out
    _check_matrix(y, "out")
    r, c = x.shape
    _check(tr_softmax_f32(x.data_ptr(), y.data_ptr(), r, c, _order(order), _stream_handle(stream)), "softmax")
    return y


def rmsnorm(x, weight=None, eps=1e-5, out=None, order="unordered", stream=None):
    import torch
    _check_matrix(x, "x")
    r, c = x.shape
    wp = _check_vector(weight, "weight", c)
    y = torch.empty_like(x) if out is None else out
    _check_matrix(y, "out")
    _check(tr_rmsnorm_f32(x.data_ptr(), wp, y.data_ptr(), r, c, eps, _order(order), _stream_handle(stream)),
           "rmsnorm")
    return y


def layernorm(x, weight=None, bias=None, eps=1e-5, out=None, order="unordered", stream=None):
    import torch
    _check_matrix(x, "x")
    r, c = x.shape
    wp = _check_vector(weight, "weight", c)
    bp = _check_vector(bias, "bias", c)
    y = torch.empty_like(x) if out is None else out
    _check_matrix(y, "out")
    _check(tr_layernorm_f32(x.data_ptr(), wp, bp, y.data_ptr(), r, c, eps, _order(order),
                            _stream_handle(stream)), "layernorm")
    return y


def tr_add_rmsnorm_f32(x, r, w, y, h, rows, cols, eps, order, stream):
    return load().tr_add_rmsnorm_f32(x, r, w, y, h, rows, cols, eps, order, stream)


def tr_add_layernorm_f32(x, r, gamma, beta, y, h, rows, cols, eps, order, stream):
    return load().tr_add_layernorm_f32(x, r, gamma, beta, y, h, rows, cols, eps, order, stream)


def add_rmsnorm(x, residual, weight=None, eps=1e-5, out=None, h_out=None, order="unordered", stream=None):
    """y = RMSNorm(x + residual); h_out (optional) receives x + residual."""
    import torch
    _check_matrix(x, "x")
    _check_matrix(residual, "residual")
    r, c = x.shape
    wp = _check_vector(weight, "weight", c)
    y = torch.empty_like(x) if out is None else out
    _check_matrix(y, "out")
    hp = None
    if h_out is not None:
        _check_matrix(h_out, "h_out")
        hp = h_out.data_ptr()
    _check(tr_add_rmsnorm_f32(x.data_ptr(), residual.data_ptr(), wp, y.data_ptr(), hp, r, c, eps, _order(order),
                              _stream_handle(stream)), "add_rmsnorm")
    return y


def add_layernorm(x, residual, weight=None, bias=None, eps=1e-5, out=None, h_out=None, order="unordered",
                  stream=None):
    """y = LayerNorm(x + residual); h_out (optional) receives x + residual."""
    import torch
    _check_matrix(x, "x")
    _check_matrix(residual, "residual")
    r, c = x.shape
    wp = _check_vector(weight, "weight", c)
    bp = _check_vector(bias, "bias", c)
    y = torch.empty_like(x) if out is None else out
    _check_matrix(y, "out")
    hp = None
    if h_out is not None:
        _check_matrix(h_out, "h_out")
        hp = h_out.data_ptr()
    _check(tr_add_layernorm_f32(x.data_ptr(), residual.data_ptr(), wp, bp, y.data_ptr(), hp, r, c, eps,
                                _order(order), _stream_handle(stream)), "add_layernorm")
    return y


def row_reduce(x, op="row_sum", out=None, out2=None, order="unordered", stream=None):
    """Per-row sum, max or min of a CUDA float32 (rows, cols) tensor; op
    "row_minmax" writes the minima to ``out`` and the maxima to ``out2`` and
    returns both."""
    import torch
    _check_matrix(x, "x")
    r, c = x.shape
    y = torch.empty(r, device=x.device, dtype=torch.float32) if out is None else out
    lib = load()
    if op == "row_minmax":
        y2 = torch.empty(r, device=x.device, dtype=torch.float32) if out2 is None else out2
        _check(lib.tr_row_minmax_f32(x.data_ptr(), y.data_ptr(), y2.data_ptr(), r, c, _order(order),
                                     _stream_handle(stream)), "row_minmax")
        return y, y2
    fn = {"row_sum": lib.tr_row_sum_f32, "row_max": lib.tr_row_max_f32, "row_min": lib.tr_row_min_f32}[op]
    _check(fn(x.data_ptr(), y.data_ptr(), r, c, _order(order), _stream_handle(stream)), op)
    return y


def axis_launch_shape(op, outer, extent, inner, sm_count=152, order="unordered"):
    """(splits, tiles) of an axis reduction of an aligned x on a device with `sm_count` SMs (host only)."""
    sp, tl = ctypes.c_int32(0), ctypes.c_int64(0)
    code = OPS["row_" + op] if isinstance(op, str) else op
    _check(load().tr_axis_launch_shape(sm_count, code, _order(order), outer, extent, inner, ctypes.byref(sp),
                                       ctypes.byref(tl)), "axis_launch_shape")
    return sp.value, tl.value


def axis_reduce(x, dim=0, op="sum", out=None, out2=None, order="unordered", stream=None):
    """Sum, max, min, or min and max together, of a contiguous CUDA float32
    tensor over dimension `dim` (any position). The result has x's shape
    without `dim`; "minmax" returns (minima, maxima)."""
    import torch
    if not isinstance(x, torch.Tensor) or x.dtype != torch.float32 or not x.is_cuda or not x.is_contiguous():
        raise TypeError("x must be a contiguous CUDA float32 tensor")
    if x.dim() < 1:
        raise ValueError("x needs at least one dimension")
    d = dim % x.dim()
    shape = list(x.shape)
    outer = 1
    for n in shape[:d]:
        outer *= n
    inner = 1
    for n in shape[d + 1:]:
        inner *= n
    extent = shape[d]
    rshape = shape[:d] + shape[d + 1:]
    y = torch.empty(rshape, device=x.device, dtype=torch.float32) if out is None else out
    lib = load()
    if op == "minmax":
        y2 = torch.empty(rshape, device=x.device, dtype=torch.float32) if out2 is None else out2
        _check(lib.tr_axis_minmax_f32(x.data_ptr(), y.data_ptr(), y2.data_ptr(), outer, extent, inner,
                                      _order(order), _stream_handle(stream)), "axis_minmax")
        return y, y2
    fn = {"sum": lib.tr_axis_sum_f32, "max": lib.tr_axis_max_f32, "min": lib.tr_axis_min_f32}[op]
    _check(fn(x.data_ptr(), y.data_ptr(), outer, extent, inner, _order(order), _stream_handle(stream)),
           "axis_" + op)
    return y


# ------------------------------------------------------------ backward passes

def norm_backward_workspace_bytes(rows, cols):
    n = ctypes.c_size_t(0)
    _check(load().tr_norm_backward_workspace_bytes(rows, cols, ctypes.byref(n)), "norm_backward_workspace_bytes")
    return n.value


def softmax_backward(y, dy, out=None, order="unordered", stream=None):
    """dx = y * (dy - sum(dy * y)) per row, from the forward output y."""
    import torch
    _check_matrix(y, "y")
    _check_matrix(dy, "dy")
    r, c = y.shape
    dx = torch.empty_like(y) if out is None else out
    _check(load().tr_softmax_backward_f32(y.data_ptr(), dy.data_ptr(), dx.data_ptr(), r, c, _order(order),
                                          _stream_handle(stream)), "softmax_backward")
    return dx


def cross_entropy_backward(logits, labels, dloss=None, out=None, order="unordered", stream=None):
    """dlogits = dloss * (softmax(logits) - onehot(labels)); dloss None means 1."""
    import torch
    _check_matrix(logits, "logits")
    r, c = logits.shape
    dx = torch.empty_like(logits) if out is None else out
    _check(load().tr_cross_entropy_backward_f32(logits.data_ptr(), labels.data_ptr(),
                                                None if dloss is None else dloss.data_ptr(), dx.data_ptr(), r, c,
                                                _order(order), _stream_handle(stream)), "cross_entropy_backward")
    return dx


def _workspace(x, rows, cols, want):
    import torch
    if not want:
        return None, 0
    n = norm_backward_workspace_bytes(rows, cols)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=x.device), n


def rmsnorm_backward(x, w, dy, eps=1e-5, order="unordered", want_dw=True, dx=None, dw=None, workspace=None,
                     stream=None):
    """(dx, dw) of RMSNorm; dw is None when not wanted."""
    import torch
    _check_matrix(x, "x")
    _check_matrix(dy, "dy")
    r, c = x.shape
    dx = torch.empty_like(x) if dx is None else dx
    want = want_dw or dw is not None
    dw = (torch.empty(c, device=x.device, dtype=torch.float32) if dw is None else dw) if want else None
    ws, n = (workspace, workspace.numel()) if workspace is not None else _workspace(x, r, c, want)
    _check(load().tr_rmsnorm_backward_f32(x.data_ptr(), None if w is None else w.data_ptr(), dy.data_ptr(),
                                          dx.data_ptr(), None if dw is None else dw.data_ptr(), r, c, eps,
                                          _order(order), None if ws is None else ws.data_ptr(), n,
                                          _stream_handle(stream)), "rmsnorm_backward")
    return dx, dw


def layernorm_backward(x, gamma, dy, eps=1e-5, order="unordered", want_params=True, dx=None, dgamma=None,
                       dbeta=None, workspace=None, stream=None):
    """(dx, dgamma, dbeta) of LayerNorm; the parameter gradients are None when not wanted."""
    import torch
    _check_matrix(x, "x")
    _check_matrix(dy, "dy")
    r, c = x.shape
    dx = torch.empty_like(x) if dx is None else dx
    if want_params:
        dgamma = torch.empty(c, device=x.device, dtype=torch.float32) if dgamma is None else dgamma
        dbeta = torch.empty(c, device=x.device, dtype=torch.float32) if dbeta is None else dbeta
    want = dgamma is not None or dbeta is not None
    ws, n = (workspace, workspace.numel()) if workspace is not None else _workspace(x, r, c, want)
    _check(load().tr_layernorm_backward_f32(x.data_ptr(), None if gamma is None else gamma.data_ptr(),
                                            dy.data_ptr(), dx.data_ptr(),
                                            None if dgamma is None else dgamma.data_ptr(),
                                            None if dbeta is None else dbeta.data_ptr(), r, c, eps, _order(order),
                                            None if ws is None else ws.data_ptr(), n, _stream_handle(stream)),
           "layernorm_backward")
    return dx, dgamma, dbeta


def cross_entropy(logits, labels, out=None, order="unordered", stream=None):
    """Per-row loss log(sum exp(x)) - x[label] (label outside [0, cols) selects 0)."""
    import torch
    _check_matrix(logits, "logits")
    r, c = logits.shape
    if labels.dtype != torch.int64 or not labels.is_cuda or labels.numel() != r or not labels.is_contiguous():
        raise TypeError("labels must be a contiguous CUDA int64 tensor with one entry per row")
    loss = torch.empty(r, dtype=torch.float32, device=logits.device) if out is None else out
    _check(tr_cross_entropy_f32(logits.data_ptr(), labels.data_ptr(), loss.data_ptr(), r, c, _order(order),
                                _stream_handle(stream)), "cross_entropy")
    return loss


def plan_for(op, rows, cols, order="unordered") -> dict:
    """The plan the library would use on the current device, as a dict."""
    return tr_plan_describe(OPS[op] if isinstance(op, str) else op, rows, cols, _order(order)).as_dict()


def run_op(op, inputs, out=None, order="unordered", eps=1e-5, stream=None, h_out=None):
    """Dispatch one operator on a dict of inputs (keys as produced by ``synth``)."""
    if op == "softmax":
        return softmax(inputs["x"], out=out, order=order, stream=stream)
    if op == "rmsnorm":
        return rmsnorm(inputs["x"], inputs.get("w"), eps, out=out, order=order, stream=stream)
    if op == "layernorm":
        return layernorm(inputs["x"], inputs.get("w"), inputs.get("b"), eps, out=out, order=order, stream=stream)
    if op in REDUCE_OPS:
        return row_reduce(inputs["x"], op, out=out, out2=h_out, order=order, stream=stream)
    if op in AXIS_OPS:
        return axis_reduce(inputs["x"], 0, op[len("axis_"):], out=out, out2=h_out, order=order, stream=stream)
    if op == "add_rmsnorm":
        return add_rmsnorm(inputs["x"], inputs["r"], inputs.get("w"), eps, out=out, h_out=h_out, order=order,
                           stream=stream)
    if op == "add_layernorm":
        return add_layernorm(inputs["x"], inputs["r"], inputs.get("w"), inputs.get("b"), eps, out=out, h_out=h_out,
                             order=order, stream=stream)
    if op == "cross_entropy":
        return cross_entropy(inputs["x"], inputs["labels"], out=out, order=order, stream=stream)
    raise ValueError(f"unknown op {op!r}")
