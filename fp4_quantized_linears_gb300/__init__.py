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
FP4_FLAG_HADAMARD16_COL = 8

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
        "fp4_quantize_hybrid": (ctypes.c_int, [vp, c_i64, c_i64, c_i64, ctypes.c_int, ctypes.c_int, ctypes.c_uint,
                                               ctypes.c_uint, c_u64, c_u64, ctypes.POINTER(ctypes.c_int8), tp, tp, vp,
                                               c_sz, vp]),
        "fp4_quantize_hybrid_workspace_bytes": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, c_i64, c_i64,
                                                               ctypes.c_uint, ctypes.c_uint, ctypes.POINTER(c_sz)]),
        "fp4_linear_fprop": (ctypes.c_int, [tp, tp, vp, ctypes.c_int, ctypes.c_float, vp]),
        "fp4_linear_dgrad": (ctypes.c_int, [tp, tp, vp, ctypes.c_int, ctypes.c_float, vp]),
        "fp4_linear_wgrad": (ctypes.c_int, [tp, tp, vp, ctypes.c_float, vp]),
        "fp4_linear_dgrad_rmsnorm": (ctypes.c_int, [tp, tp, vp, vp, vp, vp, vp, vp]),
        "fp4_residual_rmsnorm_fwd": (ctypes.c_int, [ctypes.c_int, ctypes.c_uint, vp, vp, vp, c_i64, c_i64, c_i64,
                                                    ctypes.c_float, vp, vp, tp, tp, vp, vp, c_sz, vp]),
        "fp4_residual_rmsnorm_bwd": (ctypes.c_int, [ctypes.c_int, ctypes.c_uint, ctypes.c_int, vp, vp, vp, vp, vp,
                                                    c_i64, c_i64, c_u64, c_u64, vp, tp, tp, vp, c_sz, vp]),
        "fp4_residual_rmsnorm_bwd_parts": (ctypes.c_int, [ctypes.c_int, ctypes.c_uint, ctypes.c_int, vp, vp, vp, vp,
                                                          vp, vp, c_i64, c_i64, c_u64, c_u64, vp, tp, tp, vp, c_sz,
                                                          vp]),
        "fp4_rmsnorm_bwd_workspace_bytes": (ctypes.c_int, [ctypes.c_int, c_i64, c_i64, ctypes.POINTER(c_sz)]),
        "fp4_swiglu_fwd": (ctypes.c_int, [tp, tp, c_i64, vp, vp, tp, tp, vp, vp, c_sz, vp]),
        "fp4_swiglu_bwd": (ctypes.c_int, [tp, tp, c_i64, vp, vp, c_u64, c_u64, tp, tp, vp, vp, vp, c_sz, vp]),
        "fp4_swiglu_workspace_bytes": (ctypes.c_int, [ctypes.c_int, c_i64, c_i64, ctypes.c_int, ctypes.c_int,
                                                      ctypes.POINTER(c_sz)]),
        "fp4_qkv_rope_fwd": (ctypes.c_int, [tp, tp, vp, vp, c_i64, ctypes.c_int, ctypes.c_int, vp, vp, vp, vp]),
        "fp4_qkv_rope_bwd": (ctypes.c_int, [ctypes.c_int, ctypes.c_uint, ctypes.c_int, vp, vp, vp, vp, vp, c_i64, c_i64,
                                            ctypes.c_int, ctypes.c_int, c_u64, c_u64, vp, tp, tp, vp, c_sz, vp]),
        "fp4_status": (ctypes.c_int, [vp, ctypes.POINTER(ctypes.c_int)]),
        "fp4_status_reset": (ctypes.c_int, [vp]),
        "fp4_set_wait_limit": (ctypes.c_int, [c_u64]),
        "fp4_test_skip_accumulator_release": (ctypes.c_int, [ctypes.c_int]),
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
    return _quantize(x, route, route, False, views, flags, sr_seed, sr_offset, hadamard_signs, row_out, col_out,
                     workspace, stream)


def fp4_quantize_hybrid(x: torch.Tensor, row_route, col_route, views: int = FP4_VIEW_ROW | FP4_VIEW_COL,
                        flags: int = 0, sr_seed: int = 0, sr_offset: int = 0, hadamard_signs=None,
                        row_out: QView | None = None, col_out: QView | None = None,
                        workspace: torch.Tensor | None = None, stream=None):
    """The operand-wise hybrid producer: the row view under row_route and the
    column view under col_route from one read of x.  Returns (row_view, col_view)."""
    return _quantize(x, row_route, col_route, True, views, flags, sr_seed, sr_offset, hadamard_signs, row_out,
                     col_out, workspace, stream)


def fp4_quantize_hybrid_workspace_bytes(row_route, col_route, rows: int, cols: int, views: int = 3,
                                        flags: int = 0) -> int:
    n = ctypes.c_size_t()
    _check(load().fp4_quantize_hybrid_workspace_bytes(_route(row_route), _route(col_route), rows, cols, views, flags,
                                                      ctypes.byref(n)), "fp4_quantize_hybrid_workspace_bytes")
    return n.value


def _quantize(x, row_route, col_route, hybrid, views, flags, sr_seed, sr_offset, hadamard_signs, row_out, col_out,
              workspace, stream):
    L = load()
    rr, cr = _route(row_route), _route(col_route)
    if x.dtype != torch.bfloat16 or x.dim() != 2 or not x.is_cuda:
        raise ValueError("x must be a 2D bfloat16 CUDA tensor")
    if x.stride(1) != 1:
        raise ValueError("x must have unit stride along columns")
    R, C = x.shape
    if views & FP4_VIEW_ROW and row_out is None:
        row_out = alloc_view(rr, R, C, flags, x.device)
    if views & FP4_VIEW_COL and col_out is None:
        col_out = alloc_view(cr, C, R, flags, x.device)
    need = fp4_quantize_hybrid_workspace_bytes(rr, cr, R, C, views, flags)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    signs = None
    if hadamard_signs is not None:
        arr = (ctypes.c_int8 * 16)(*[int(s) for s in hadamard_signs])
        signs = ctypes.cast(arr, ctypes.POINTER(ctypes.c_int8))
    rs = row_out.struct() if row_out is not None else None
    cs = col_out.struct() if col_out is not None else None
    ws_ptr = ctypes.c_void_p(workspace.data_ptr()) if workspace is not None else None
    ws_n = workspace.numel() if workspace is not None else 0
    args = (signs, ctypes.byref(rs) if rs else None, ctypes.byref(cs) if cs else None, ws_ptr, ws_n, _stream(stream))
    if hybrid:
        code = L.fp4_quantize_hybrid(ctypes.c_void_p(x.data_ptr()), R, C, x.stride(0), rr, cr, views, flags, sr_seed,
                                     sr_offset, *args)
    else:
        code = L.fp4_quantize(ctypes.c_void_p(x.data_ptr()), R, C, x.stride(0), rr, views, flags, sr_seed, sr_offset,
                              *args)
    _check(code, "fp4_quantize_hybrid" if hybrid else "fp4_quantize")
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


def fp4_linear_dgrad_rmsnorm(dy_row: QView, w_col: QView, r_prime: torch.Tensor, rstd: torch.Tensor,
                             g: torch.Tensor, dx: torch.Tensor | None = None, part: torch.Tensor | None = None,
                             stream=None):
    """dx = dY . W (bf16) and the adjacent RMSNorm backward's row terms
    part [rows][cols / 64] (binary32).  Returns (dx, part)."""
    dx = _out(dy_row, w_col, dx, FP4_OUT_BF16, dy_row.codes.device)
    if part is None:
        part = torch.empty((dy_row.rows, w_col.rows // 64), dtype=torch.float32, device=dy_row.codes.device)
    a, b = dy_row.struct(), w_col.struct()
    _check(load().fp4_linear_dgrad_rmsnorm(ctypes.byref(a), ctypes.byref(b), _ptr(dx), _ptr(r_prime), _ptr(rstd),
                                           _ptr(g), _ptr(part), _stream(stream)), "fp4_linear_dgrad_rmsnorm")
    return dx, part


def fp4_linear_wgrad(dy_col: QView, x_col: QView, dw: torch.Tensor | None = None, beta: float = 0.0,
                     stream=None) -> torch.Tensor:
    dw = _out(dy_col, x_col, dw, FP4_OUT_F32, dy_col.codes.device)
    a, b = dy_col.struct(), x_col.struct()
    _check(load().fp4_linear_wgrad(ctypes.byref(a), ctypes.byref(b), ctypes.c_void_p(dw.data_ptr()), beta,
                                   _stream(stream)), "fp4_linear_wgrad")
    return dw


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _views(route, R, C, views, flags, device, row_out, col_out):
    if views & FP4_VIEW_ROW and row_out is None:
        row_out = alloc_view(route, R, C, flags, device)
    if views & FP4_VIEW_COL and col_out is None:
        col_out = alloc_view(route, C, R, flags, device)
    return row_out, col_out


def _sync_fields(v, st):
    if st is not None:
        v.rows, v.cols, v.route, v.outer_count = st.rows, st.cols, st.route, st.outer_count


def fp4_residual_rmsnorm_fwd(r: torch.Tensor, b: torch.Tensor | None, g: torch.Tensor, route, views: int = 3,
                             eps: float = 1e-5, r_out=None, rstd=None, y_row=None, y_col=None, y_tap=None,
                             workspace=None, stream=None):
    """r' = bf16(r + b), rstd, and the FP4 views of y = bf16(r' * rstd * g).

    Returns (r_out, rstd, y_row, y_col)."""
    rt = _route(route)
    R, C = r.shape
    dev = r.device
    r_out = torch.empty((R, C), dtype=torch.bfloat16, device=dev) if r_out is None else r_out
    rstd = torch.empty(R, dtype=torch.float32, device=dev) if rstd is None else rstd
    y_row, y_col = _views(rt, R, C, views, 0, dev, y_row, y_col)
    need = fp4_quantize_workspace_bytes(rt, R, C, views, 0)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    rs = y_row.struct() if y_row is not None else None
    cs = y_col.struct() if y_col is not None else None
    _check(load().fp4_residual_rmsnorm_fwd(rt, views, _ptr(r), _ptr(b), _ptr(g), R, C, r.stride(0), eps, _ptr(r_out),
                                           _ptr(rstd), ctypes.byref(rs) if rs else None,
                                           ctypes.byref(cs) if cs else None, _ptr(y_tap), _ptr(workspace),
                                           workspace.numel() if workspace is not None else 0, _stream(stream)),
           "fp4_residual_rmsnorm_fwd")
    _sync_fields(y_row, rs)
    _sync_fields(y_col, cs)
    return r_out, rstd, y_row, y_col


def fp4_rmsnorm_bwd_workspace_bytes(route, rows: int, cols: int) -> int:
    n = ctypes.c_size_t()
    _check(load().fp4_rmsnorm_bwd_workspace_bytes(_route(route), rows, cols, ctypes.byref(n)),
           "fp4_rmsnorm_bwd_workspace_bytes")
    return n.value


def fp4_residual_rmsnorm_bwd(dy: torch.Tensor, r_prime: torch.Tensor, rstd: torch.Tensor, g: torch.Tensor,
                             dres: torch.Tensor | None, route, views: int = 3, sr: bool = True, sr_seed: int = 0,
                             sr_offset: int = 0, dr=None, dr_row=None, dr_col=None, workspace=None, stream=None):
    """dr = bf16(RMSNorm backward(dy) + dres) and its FP4 views (row view SR).

    Returns (dr, dr_row, dr_col)."""
    rt = _route(route)
    R, C = dy.shape
    dev = dy.device
    dr = torch.empty((R, C), dtype=torch.bfloat16, device=dev) if dr is None else dr
    flags = FP4_FLAG_SR_ROW if sr else 0
    dr_row, dr_col = _views(rt, R, C, views, flags, dev, dr_row, dr_col)
    if workspace is None:
        workspace = torch.empty(fp4_rmsnorm_bwd_workspace_bytes(rt, R, C), dtype=torch.uint8, device=dev)
    rs = dr_row.struct() if dr_row is not None else None
    cs = dr_col.struct() if dr_col is not None else None
    _check(load().fp4_residual_rmsnorm_bwd(rt, views, int(sr), _ptr(dy), _ptr(r_prime), _ptr(rstd), _ptr(g),
                                           _ptr(dres), R, C, sr_seed, sr_offset, _ptr(dr),
                                           ctypes.byref(rs) if rs else None, ctypes.byref(cs) if cs else None,
                                           _ptr(workspace), workspace.numel(), _stream(stream)),
           "fp4_residual_rmsnorm_bwd")
    _sync_fields(dr_row, rs)
    _sync_fields(dr_col, cs)
    return dr, dr_row, dr_col


def fp4_residual_rmsnorm_bwd_parts(dy: torch.Tensor, part: torch.Tensor, r_prime: torch.Tensor, rstd: torch.Tensor,
                                   g: torch.Tensor, dres: torch.Tensor | None, route, views: int = 3, sr: bool = True,
                                   sr_seed: int = 0, sr_offset: int = 0, dr=None, dr_row=None, dr_col=None,
                                   workspace=None, stream=None):
    """fp4_residual_rmsnorm_bwd with the row means from the row terms `part`
    that fp4_linear_dgrad_rmsnorm wrote for this dy.  Returns (dr, dr_row, dr_col)."""
    rt = _route(route)
    R, C = dy.shape
    dev = dy.device
    dr = torch.empty((R, C), dtype=torch.bfloat16, device=dev) if dr is None else dr
    flags = FP4_FLAG_SR_ROW if sr else 0
    dr_row, dr_col = _views(rt, R, C, views, flags, dev, dr_row, dr_col)
    if workspace is None:
        workspace = torch.empty(fp4_rmsnorm_bwd_workspace_bytes(rt, R, C), dtype=torch.uint8, device=dev)
    rs = dr_row.struct() if dr_row is not None else None
    cs = dr_col.struct() if dr_col is not None else None
    _check(load().fp4_residual_rmsnorm_bwd_parts(rt, views, int(sr), _ptr(dy), _ptr(part), _ptr(r_prime),
                                                 _ptr(rstd), _ptr(g), _ptr(dres), R, C, sr_seed, sr_offset, _ptr(dr),
                                                 ctypes.byref(rs) if rs else None, ctypes.byref(cs) if cs else None,
                                                 _ptr(workspace), workspace.numel(), _stream(stream)),
           "fp4_residual_rmsnorm_bwd_parts")
    _sync_fields(dr_row, rs)
    _sync_fields(dr_col, cs)
    return dr, dr_row, dr_col


def fp4_swiglu_workspace_bytes(route, T: int, f: int, backward: bool = False, with_tap: bool = False) -> int:
    n = ctypes.c_size_t()
    _check(load().fp4_swiglu_workspace_bytes(_route(route), T, f, 1 if backward else 0, 1 if with_tap else 0,
                                             ctypes.byref(n)), "fp4_swiglu_workspace_bytes")
    return n.value


def _ws_args(workspace):
    if workspace is None:
        return None, 0
    return ctypes.c_void_p(workspace.data_ptr()), workspace.numel() * workspace.element_size()


def fp4_swiglu_fwd(x_row: QView, w13_row: QView, f: int, a1=None, a3=None, h_row=None, h_col=None, h_tap=None,
                   quantize: bool = True, workspace=None, stream=None):
    """Fused W1/W3 contraction + SiLU gate.  Returns (a1, a3, h_row, h_col).

    With quantize (the default) the FP4 views of h are emitted for every
    route (NVFP4 through one bf16 copy of h; a workspace is allocated here
    when none is given); with quantize=False only h_tap is written."""
    T = x_row.rows
    dev = x_row.codes.device
    a1 = torch.empty((T, f), dtype=torch.bfloat16, device=dev) if a1 is None else a1
    a3 = torch.empty((T, f), dtype=torch.bfloat16, device=dev) if a3 is None else a3
    route = x_row.route
    if quantize:
        h_row = alloc_view(route, T, f, 0, dev) if h_row is None else h_row
        h_col = alloc_view(route, f, T, 0, dev) if h_col is None else h_col
        need = fp4_swiglu_workspace_bytes(route, T, f, False, h_tap is not None)
        if need and workspace is None:
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    else:
        h_row = h_col = None
    a, b = x_row.struct(), w13_row.struct()
    rs = h_row.struct() if h_row is not None else None
    cs = h_col.struct() if h_col is not None else None
    _check(load().fp4_swiglu_fwd(ctypes.byref(a), ctypes.byref(b), f, _ptr(a1), _ptr(a3),
                                 ctypes.byref(rs) if rs else None, ctypes.byref(cs) if cs else None, _ptr(h_tap),
                                 *_ws_args(workspace), _stream(stream)), "fp4_swiglu_fwd")
    if rs:
        _sync_fields(h_row, rs)
        _sync_fields(h_col, cs)
    return a1, a3, h_row, h_col


def fp4_swiglu_bwd(dy2_row: QView, w2_col: QView, f: int, a1: torch.Tensor, a3: torch.Tensor, sr_seed: int = 0,
                   sr_offset: int = 0, da13_row=None, da13_col=None, dh_tap=None, da13_tap=None,
                   quantize: bool = True, workspace=None, stream=None):
    """Fused W2 Dgrad + SiLU derivative.  Returns (da13_row, da13_col)."""
    T = dy2_row.rows
    dev = dy2_row.codes.device
    route = dy2_row.route
    if quantize:
        da13_row = alloc_view(route, T, 2 * f, FP4_FLAG_SR_ROW, dev) if da13_row is None else da13_row
        da13_col = alloc_view(route, 2 * f, T, 0, dev) if da13_col is None else da13_col
        need = fp4_swiglu_workspace_bytes(route, T, f, True, da13_tap is not None)
        if need and workspace is None:
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    else:
        da13_row = da13_col = None
    a, b = dy2_row.struct(), w2_col.struct()
    rs = da13_row.struct() if da13_row is not None else None
    cs = da13_col.struct() if da13_col is not None else None
    _check(load().fp4_swiglu_bwd(ctypes.byref(a), ctypes.byref(b), f, _ptr(a1), _ptr(a3), sr_seed, sr_offset,
                                 ctypes.byref(rs) if rs else None, ctypes.byref(cs) if cs else None, _ptr(dh_tap),
                                 _ptr(da13_tap), *_ws_args(workspace), _stream(stream)), "fp4_swiglu_bwd")
    if rs:
        _sync_fields(da13_row, rs)
        _sync_fields(da13_col, cs)
    return da13_row, da13_col


def fp4_qkv_rope_fwd(x_row: QView, wqkv_row: QView, rope_cos: torch.Tensor, rope_sin: torch.Tensor, seq_len: int,
                     heads_q: int, heads_kv: int, q=None, k=None, v=None, stream=None):
    """QKV projection with RoPE into head-major bf16 q [hq][T][128], k, v
    [hkv][T][128] (rope_cos / rope_sin: float32 CUDA [seq_len][64]).
    Returns (q, k, v)."""
    T = x_row.rows
    dev = x_row.codes.device
    q = torch.empty((heads_q, T, 128), dtype=torch.bfloat16, device=dev) if q is None else q
    k = torch.empty((heads_kv, T, 128), dtype=torch.bfloat16, device=dev) if k is None else k
    v = torch.empty((heads_kv, T, 128), dtype=torch.bfloat16, device=dev) if v is None else v
    a, b = x_row.struct(), wqkv_row.struct()
    _check(load().fp4_qkv_rope_fwd(ctypes.byref(a), ctypes.byref(b), _ptr(rope_cos), _ptr(rope_sin), seq_len, heads_q,
                                   heads_kv, _ptr(q), _ptr(k), _ptr(v), _stream(stream)), "fp4_qkv_rope_fwd")
    return q, k, v


def fp4_qkv_rope_bwd(dq: torch.Tensor, dk: torch.Tensor, dv: torch.Tensor, rope_cos: torch.Tensor,
                     rope_sin: torch.Tensor, seq_len: int, route, views: int = 3, sr: bool = True, sr_seed: int = 0,
                     sr_offset: int = 0, dqkv_tap=None, dqkv_row=None, dqkv_col=None, workspace=None, stream=None):
    """Head-major gradients of the turned Q, K and of V -> the QKV-layout
    gradient (dQ, dK turned back) quantized into its views.  Returns (row, col)."""
    rt = _route(route)
    heads_q, T, _ = dq.shape
    heads_kv = dk.shape[0]
    C = (heads_q + 2 * heads_kv) * 128
    dev = dq.device
    flags = FP4_FLAG_SR_ROW if sr else 0
    dqkv_row, dqkv_col = _views(rt, T, C, views, flags, dev, dqkv_row, dqkv_col)
    need = fp4_quantize_workspace_bytes(rt, T, C, views, 0)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    rs = dqkv_row.struct() if dqkv_row is not None else None
    cs = dqkv_col.struct() if dqkv_col is not None else None
    _check(load().fp4_qkv_rope_bwd(rt, views, 1 if sr else 0, _ptr(dq), _ptr(dk), _ptr(dv), _ptr(rope_cos),
                                   _ptr(rope_sin), T, seq_len, heads_q, heads_kv, sr_seed, sr_offset, _ptr(dqkv_tap),
                                   ctypes.byref(rs) if rs else None, ctypes.byref(cs) if cs else None,
                                   _ptr(workspace), workspace.numel() if workspace is not None else 0,
                                   _stream(stream)), "fp4_qkv_rope_bwd")
    _sync_fields(dqkv_row, rs)
    _sync_fields(dqkv_col, cs)
    return dqkv_row, dqkv_col


def fp4_status(stream=None) -> int:
    c = ctypes.c_int()
    _check(load().fp4_status(_stream(stream), ctypes.byref(c)), "fp4_status")
    return c.value


def fp4_status_reset(stream=None):
    _check(load().fp4_status_reset(_stream(stream)), "fp4_status_reset")


def fp4_set_wait_limit(cycles: int = 0):
    """Bound (SM clock cycles) of the GEMM kernels' barrier waits for the
    launches that follow; 0 restores the default."""
    _check(load().fp4_set_wait_limit(int(cycles)), "fp4_set_wait_limit")


def fp4_test_skip_accumulator_release(enable: bool):
    """Test hook: the following GEMM launches skip their first accumulator
    release, so a bounded wait runs out and reports FP4_ERR_TIMEOUT."""
    _check(load().fp4_test_skip_accumulator_release(1 if enable else 0), "fp4_test_skip_accumulator_release")


def fp4_version() -> int:
    return load().fp4_version()
