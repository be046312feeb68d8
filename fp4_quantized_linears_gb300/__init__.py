"""Python binding of libfp4lin, the format-aware FP4 linear-layer boundary.

Argument marshalling only: every call goes through the C ABI declared in
``include/fp4lin.h`` and every step of the path runs in the library's CUDA
kernels.  PyTorch supplies device memory (``torch.Tensor.data_ptr()``) and the
current CUDA stream.  If the library cannot be loaded, every call raises: there
is no fallback path.

Functions keep the C names (``fp4_quantize``, ``fp4_linear_fprop`` ...).
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass
from typing import Optional

import torch

from ._build import LIB, build as _build_lib

# ---------------------------------------------------------------- constants --
FP4_OK = 0
FP4_ERR_INVALID_ARG = 1
FP4_ERR_UNSUPPORTED_SHAPE = 2
FP4_ERR_ROUTE_MISMATCH = 3
FP4_ERR_WORKSPACE = 4
FP4_ERR_CUDA = 5
FP4_ERR_TIMEOUT = 6
FP4_ERR_NONFINITE = 7

FP4_ROUTE_MXFP4 = 0
FP4_ROUTE_NVFP4_GLOBAL = 1
FP4_ROUTE_NVFP4_LOCAL = 2

FP4_VIEW_ROW = 1
FP4_VIEW_COL = 2

FP4_FLAG_WEIGHT_2D = 1
FP4_FLAG_SR_ROW = 2
FP4_FLAG_HADAMARD_COL = 4

FP4_OUT_F32 = 0
FP4_OUT_BF16 = 1

ROUTES = {"mx": FP4_ROUTE_MXFP4, "nv_global": FP4_ROUTE_NVFP4_GLOBAL, "nv_local": FP4_ROUTE_NVFP4_LOCAL}


class Fp4Error(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} (status {code})")


class fp4_tensor(ctypes.Structure):
    _fields_ = [
        ("codes", ctypes.c_void_p),
        ("scales", ctypes.c_void_p),
        ("outer", ctypes.c_void_p),
        ("rows", ctypes.c_int64),
        ("cols", ctypes.c_int64),
        ("route", ctypes.c_int32),
        ("outer_count", ctypes.c_int32),
    ]


_lib = None
_lock = threading.Lock()


def load(build_if_missing: bool = True):
    """Load libfp4lin.so (compiling it first if needed).  Raises if unavailable."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if build_if_missing:
            _build_lib()
        if not os.path.exists(LIB):
            raise RuntimeError(f"libfp4lin.so not found at {LIB}; run __graft_entry__.build()")
        L = ctypes.CDLL(LIB)
        _declare(L)
        _lib = L
        return L


def _declare(L):
    c_i64, c_u64, c_sz = ctypes.c_int64, ctypes.c_uint64, ctypes.c_size_t
    vp = ctypes.c_void_p
    tp = ctypes.POINTER(fp4_tensor)
    sig = {
        "fp4_version": (ctypes.c_int, []),
        "fp4_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "fp4_tensor_bytes": (ctypes.c_int, [ctypes.c_int, c_i64, c_i64, ctypes.c_uint, ctypes.POINTER(c_sz),
                                            ctypes.POINTER(c_sz), ctypes.POINTER(ctypes.c_int32)]),
        "fp4_quantize_workspace_bytes": (ctypes.c_int, [ctypes.c_int, c_i64, c_i64, ctypes.c_uint, ctypes.c_uint,
                                                        ctypes.POINTER(c_sz)]),
        "fp4_quantize": (ctypes.c_int, [vp, c_i64, c_i64, c_i64, ctypes.c_int, ctypes.c_uint, ctypes.c_uint, c_u64,
                                        c_u64, ctypes.POINTER(ctypes.c_int8), tp, tp, vp, c_sz, vp]),
        "fp4_linear_fprop": (ctypes.c_int, [tp, tp, vp, ctypes.c_int, ctypes.c_float, vp]),
        "fp4_linear_dgrad": (ctypes.c_int, [tp, tp, vp, ctypes.c_int, ctypes.c_float, vp]),
        "fp4_linear_wgrad": (ctypes.c_int, [tp, tp, vp, ctypes.c_float, vp]),
        "fp4_status": (ctypes.c_int, [vp, ctypes.POINTER(ctypes.c_int)]),
        "fp4_status_reset": (ctypes.c_int, [vp]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args


def status_string(code: int) -> str:
    try:
        return load(False).fp4_status_string(code).decode()
    except Exception:
        return f"status {code}"


def _check(code: int, where: str):
    if code != FP4_OK:
        raise Fp4Error(code, where)


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _route(route) -> int:
    return ROUTES[route] if isinstance(route, str) else int(route)


# ------------------------------------------------------------ quantized view --
@dataclass
class QView:
    """One quantized view: caller-side owner of the device buffers."""
    codes: torch.Tensor          # uint8 [rows, cols // 2]
    scales: torch.Tensor         # uint8 [rows * cols // bs] (atom layout)
    outer: Optional[torch.Tensor]  # float32 [outer_count] (NVFP4) or None
    route: int
    rows: int
    cols: int
    outer_count: int

    def struct(self) -> fp4_tensor:
        return fp4_tensor(self.codes.data_ptr(), self.scales.data_ptr(),
                          self.outer.data_ptr() if self.outer is not None else None,
                          self.rows, self.cols, self.route, self.outer_count)


def fp4_tensor_bytes(route, rows: int, cols: int, flags: int = 0):
    cb, sb, oc = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_int32()
    _check(load().fp4_tensor_bytes(_route(route), rows, cols, flags, ctypes.byref(cb), ctypes.byref(sb),
                                   ctypes.byref(oc)), "fp4_tensor_bytes")
    return cb.value, sb.value, oc.value


def alloc_view(route, rows: int, cols: int, flags: int = 0, device="cuda") -> QView:
    """Allocate (with torch) the buffers of a view with `rows` stored rows."""
    r = _route(route)
    cb, sb, oc = fp4_tensor_bytes(r, rows, cols, flags)
    codes = torch.empty((rows, cols // 2), dtype=torch.uint8, device=device)
    scales = torch.empty(sb, dtype=torch.uint8, device=device)
    outer = torch.empty(max(oc, 1), dtype=torch.float32, device=device) if r != FP4_ROUTE_MXFP4 else None
    return QView(codes, scales, outer, r, rows, cols, oc)


def fp4_quantize_workspace_bytes(route, rows: int, cols: int, views: int = 3, flags: int = 0) -> int:
    n = ctypes.c_size_t()
    _check(load().fp4_quantize_workspace_bytes(_route(route), rows, cols, views, flags, ctypes.byref(n)),
           "fp4_quantize_workspace_bytes")
    return n.value


def fp4_quantize(x: torch.Tensor, route, views: int = FP4_VIEW_ROW | FP4_VIEW_COL, flags: int = 0,
                 sr_seed: int = 0, sr_offset: int = 0, hadamard_signs=None, row_out: QView | None = None,
                 col_out: QView | None = None, workspace: torch.Tensor | None = None, stream=None):
    """Quantize a bf16 CUDA tensor [rows, cols] into the requested views.

    Returns (row_view or None, col_view or None)."""
    L = load()
    r = _route(route)
    if x.dtype != torch.bfloat16 or x.dim() != 2 or not x.is_cuda:
        raise ValueError("x must be a 2D bfloat16 CUDA tensor")
    if x.stride(1) != 1:
        raise ValueError("x must have unit stride along columns")
    R, C = x.shape
    if views & FP4_VIEW_ROW and row_out is None:
        row_out = alloc_view(r, R, C, flags, x.device)
    if views & FP4_VIEW_COL and col_out is None:
        col_out = alloc_view(r, C, R, flags, x.device)
    need = fp4_quantize_workspace_bytes(r, R, C, views, flags)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    signs = None
    if hadamard_signs is not None:
        arr = (ctypes.c_int8 * 16)(*[int(s) for s in hadamard_signs])
        signs = ctypes.cast(arr, ctypes.POINTER(ctypes.c_int8))
    rs = row_out.struct() if row_out is not None else None
    cs = col_out.struct() if col_out is not None else None
    code = L.fp4_quantize(ctypes.c_void_p(x.data_ptr()), R, C, x.stride(0), r, views, flags, sr_seed, sr_offset,
                          signs, ctypes.byref(rs) if rs else None, ctypes.byref(cs) if cs else None,
                          ctypes.c_void_p(workspace.data_ptr()) if workspace is not None else None,
                          workspace.numel() if workspace is not None else 0, _stream(stream))
    _check(code, "fp4_quantize")
    if rs:
        row_out.rows, row_out.cols, row_out.route, row_out.outer_count = rs.rows, rs.cols, rs.route, rs.outer_count
    if cs:
        col_out.rows, col_out.cols, col_out.route, col_out.outer_count = cs.rows, cs.cols, cs.route, cs.outer_count
    return row_out, col_out


def _out(a: QView, b: QView, out, out_dtype, device):
    if out is None:
        dt = torch.float32 if out_dtype == FP4_OUT_F32 else torch.bfloat16
        out = torch.empty((a.rows, b.rows), dtype=dt, device=device)
    return out


def fp4_linear_fprop(x_row: QView, w_row: QView, y: torch.Tensor | None = None, out_dtype: int = FP4_OUT_F32,
                     beta: float = 0.0, stream=None) -> torch.Tensor:
    y = _out(x_row, w_row, y, out_dtype, x_row.codes.device)
    a, b = x_row.struct(), w_row.struct()
    _check(load().fp4_linear_fprop(ctypes.byref(a), ctypes.byref(b), ctypes.c_void_p(y.data_ptr()), out_dtype,
                                   beta, _stream(stream)), "fp4_linear_fprop")
    return y


def fp4_linear_dgrad(dy_row: QView, w_col: QView, dx: torch.Tensor | None = None, out_dtype: int = FP4_OUT_F32,
                     beta: float = 0.0, stream=None) -> torch.Tensor:
    dx = _out(dy_row, w_col, dx, out_dtype, dy_row.codes.device)
    a, b = dy_row.struct(), w_col.struct()
    _check(load().fp4_linear_dgrad(ctypes.byref(a), ctypes.byref(b), ctypes.c_void_p(dx.data_ptr()), out_dtype,
                                   beta, _stream(stream)), "fp4_linear_dgrad")
    return dx


def fp4_linear_wgrad(dy_col: QView, x_col: QView, dw: torch.Tensor | None = None, beta: float = 0.0,
                     stream=None) -> torch.Tensor:
    dw = _out(dy_col, x_col, dw, FP4_OUT_F32, dy_col.codes.device)
    a, b = dy_col.struct(), x_col.struct()
    _check(load().fp4_linear_wgrad(ctypes.byref(a), ctypes.byref(b), ctypes.c_void_p(dw.data_ptr()), beta,
                                   _stream(stream)), "fp4_linear_wgrad")
    return dw


def fp4_status(stream=None) -> int:
    c = ctypes.c_int()
    _check(load().fp4_status(_stream(stream), ctypes.byref(c)), "fp4_status")
    return c.value


def fp4_status_reset(stream=None):
    _check(load().fp4_status_reset(_stream(stream)), "fp4_status_reset")


def fp4_version() -> int:
    return load().fp4_version()
