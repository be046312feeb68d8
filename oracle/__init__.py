"""CPU oracle of the format-aware FP4 linear boundary.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
CPU-baseline leg are the only callers.  The product library never imports
this package, and this package never imports the product library.

The arithmetic lives in ``fp4_oracle.c`` (plain scalar C, compiled with
``-ffp-contract=off``); this module compiles it on first use and composes its
primitives per route, following "Format-Aware Fusion for Fast FP4
Pretraining":

* Sec. 2.2 (Eq. 1)     E2M1 values, rounding and saturation
* Sec. 2.2.1           MXFP4 upward E8M0 scales, adaptive 2D32 weight rule
* Sec. 2.2.2 (Eq. 3)   global NVFP4 and CTA-local NVFP4 outer factors
* Sec. 2.3 (Eqs. 4-6)  row-facing / column-facing views of each operand
* Sec. 2.4 (Eqs. 7-8)  2D16 / 2D32 weight encodings shared by both views
* Sec. 2.5 (Eqs. 9-10) row-only SR and the paired fixed-sign H32
* Sec. 3.2             SwiGLU and residual-RMSNorm producers

Views are returned in their *stored* orientation: the row view of an R x C
tensor has R stored rows of C values; the column view has C stored rows of
R values (the transpose), so every operand is K-major for its contraction.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp4_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

ROUTES = ("mx", "nv_global", "nv_local")
STRIP = 128  # CTA-local strip height (rows of the stored view)


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C11, no FMA contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = ctypes.CDLL(build())
            _declare(_lib)
    return _lib


_u8p = ctypes.POINTER(ctypes.c_uint8)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_u32p = ctypes.POINTER(ctypes.c_uint32)
_i8p = ctypes.POINTER(ctypes.c_int8)
_i64p = ctypes.POINTER(ctypes.c_int64)
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)
_i64 = ctypes.c_int64
_u64 = ctypes.c_uint64


def _declare(L):
    sig = {
        "orc_bf16_round": (ctypes.c_uint16, [ctypes.c_double]),
        "orc_bf16_value": (ctypes.c_double, [ctypes.c_uint16]),
        "orc_e2m1_value": (ctypes.c_double, [ctypes.c_uint8]),
        "orc_e2m1_rn": (ctypes.c_uint8, [ctypes.c_double]),
        "orc_e2m1_sr": (ctypes.c_uint8, [ctypes.c_double, ctypes.c_uint32]),
        "orc_e8m0_exponent_up": (ctypes.c_int, [ctypes.c_double]),
        "orc_mx_weight_tile_exponent": (ctypes.c_int, [ctypes.c_double]),
        "orc_e4m3_value": (ctypes.c_double, [ctypes.c_uint8]),
        "orc_e4m3_rn_satfinite": (ctypes.c_uint8, [ctypes.c_double]),
        "orc_nv_senc": (ctypes.c_float, [ctypes.c_float]),
        "orc_nv_block_scale": (ctypes.c_uint8, [ctypes.c_float, ctypes.c_float, _f32p]),
        "orc_philox4x32_10": (None, [_u32p, _u32p, _u32p]),
        "orc_sr_uniform16": (ctypes.c_uint32, [_u64, _u64, _u64]),
        "orc_inv_sqrt32_f32": (ctypes.c_float, []),
        "orc_hadamard32_f32": (None, [_f32p, _i8p]),
        "orc_hadamard32_rows": (None, [_f32p, _i64, _i64, _i8p]),
        "orc_hadamard16_f32": (None, [_f32p, _i8p]),
        "orc_rope_tables": (None, [_i64, ctypes.c_int, ctypes.c_double, _f32p, _f32p]),
        "orc_qkv_rope_fwd": (None, [_u16p, _i64, _i64, ctypes.c_int, ctypes.c_int, ctypes.c_int, _f32p, _f32p,
                                    _u16p, _u16p, _u16p]),
        "orc_qkv_rope_bwd": (None, [_u16p, _u16p, _u16p, _i64, _i64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                    _f32p, _f32p, _u16p]),
        "orc_hadamard16_rows": (None, [_f32p, _i64, _i64, _i8p]),
        "orc_sylvester_h32": (None, [_i8p]),
        "orc_mx_quantize_rows": (None, [_f32p, _i64, _i64, ctypes.c_int, _u64, _u64, _u64, _i64, _u8p, _u8p]),
        "orc_mx_quantize_weight2d": (None, [_f32p, _i64, _i64, _u8p, _u8p]),
        "orc_nv_quantize_rows": (None, [_f32p, _i64, _i64, _f32p, ctypes.c_int, _u64, _u64, _u64, _i64, _u8p,
                                         _u8p]),
        "orc_nv_quantize_weight2d": (None, [_f32p, _i64, _i64, ctypes.c_float, _u8p, _u8p]),
        "orc_amax_f32": (ctypes.c_float, [_f32p, _i64]),
        "orc_bf16_to_f32": (None, [_u16p, _i64, _f32p]),
        "orc_dequantize": (None, [_u8p, _u8p, ctypes.c_int, _i64, _i64, _f32p, _f64p]),
        "orc_gemm_nt": (None, [_f64p, _f64p, _i64, _i64, _i64, _f64p]),
        "orc_gemm_sampled": (None, [_u8p, _u8p, _f32p, _u8p, _u8p, _f32p, ctypes.c_int, _i64,
                                    _i64p, _i64p, _i64, _f64p, _f64p]),
        "orc_swiglu_h": (None, [_u16p, _u16p, _i64, _u16p]),
        "orc_swiglu_bwd": (None, [_u16p, _u16p, _u16p, _i64, _u16p, _u16p]),
        "orc_residual_rmsnorm": (None, [_u16p, _u16p, _u16p, _i64, _i64, ctypes.c_double, ctypes.c_int,
                                        _f32p, _u16p, _f32p, _u16p]),
        "orc_rmsnorm_bwd": (None, [_u16p, _u16p, _f32p, _u16p, _u16p, _i64, _i64, _u16p]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args


def _p(a: np.ndarray, t):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(t)


def _opt(a, t):
    return None if a is None else _p(a, t)


# ---------------------------------------------------------------------------
# scalar helpers (used by the pins)
# ---------------------------------------------------------------------------

def e2m1_value(code: int) -> float:
    return lib().orc_e2m1_value(code)


def e2m1_rn(v: float) -> int:
    return lib().orc_e2m1_rn(v)


def e2m1_sr(v: float, u16: int) -> int:
    return lib().orc_e2m1_sr(v, u16)


def e8m0_exponent_up(amax: float) -> int:
    return lib().orc_e8m0_exponent_up(amax)


def mx_weight_tile_exponent(amax: float) -> int:
    return lib().orc_mx_weight_tile_exponent(amax)


def e4m3_value(code: int) -> float:
    return lib().orc_e4m3_value(code)


def e4m3_rn_satfinite(s: float) -> int:
    return lib().orc_e4m3_rn_satfinite(s)


def nv_senc(amax: float) -> float:
    return lib().orc_nv_senc(amax)


def nv_block_scale(block_amax: float, senc: float):
    m = ctypes.c_float(0.0)
    d = lib().orc_nv_block_scale(block_amax, senc, ctypes.byref(m))
    return d, m.value


def philox4x32_10(ctr, key):
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, np.uint32)
    lib().orc_philox4x32_10(_p(c, _u32p), _p(k, _u32p), _p(out, _u32p))
    return out


def sr_uniform16(seed: int, offset: int, index: int) -> int:
    return lib().orc_sr_uniform16(seed, offset, index)


def inv_sqrt32_f32() -> float:
    return lib().orc_inv_sqrt32_f32()


def hadamard32_f32(v, signs) -> np.ndarray:
    y = np.ascontiguousarray(v, dtype=np.float32).copy()
    s = np.ascontiguousarray(signs, dtype=np.int8)
    lib().orc_hadamard32_f32(_p(y, _f32p), _p(s, _i8p))
    return y


def hadamard16_f32(v, signs) -> np.ndarray:
    """Fixed-sign H16 of 16 binary32 values (signs of +-1; all +1 is plain H16)."""
    y = np.ascontiguousarray(v, dtype=np.float32).copy()
    s = np.ascontiguousarray(signs, dtype=np.int8)
    assert y.shape == (16,) and s.shape == (16,)
    lib().orc_hadamard16_f32(_p(y, _f32p), _p(s, _i8p))
    return y


def sylvester_h32() -> np.ndarray:
    h = np.zeros((32, 32), np.int8)
    lib().orc_sylvester_h32(_p(h, _i8p))
    return h


def bf16_round(v: float) -> int:
    return lib().orc_bf16_round(v)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(b.shape, np.float32)
    lib().orc_bf16_to_f32(_p(b, _u16p), b.size, _p(out, _f32p))
    return out


def amax_f32(x: np.ndarray) -> float:
    x = np.ascontiguousarray(x, dtype=np.float32)
    return lib().orc_amax_f32(_p(x, _f32p), x.size)


# ---------------------------------------------------------------------------
# tensor quantizers
# ---------------------------------------------------------------------------

def _mx_rows(xf: np.ndarray, sr: bool, seed: int, offset: int, index0: int = 0, ld: int | None = None):
    R, C = xf.shape
    codes = np.empty((R, C), np.uint8)
    scales = np.empty((R, C // 32), np.uint8)
    lib().orc_mx_quantize_rows(_p(xf, _f32p), R, C, int(sr), seed, offset, index0, C if ld is None else ld,
                               _p(codes, _u8p), _p(scales, _u8p))
    return codes, scales


def _nv_rows(xf: np.ndarray, senc_row: np.ndarray, sr: bool, seed: int, offset: int, index0: int = 0,
             ld: int | None = None):
    R, C = xf.shape
    codes = np.empty((R, C), np.uint8)
    scales = np.empty((R, C // 16), np.uint8)
    s = np.ascontiguousarray(senc_row, dtype=np.float32)
    lib().orc_nv_quantize_rows(_p(xf, _f32p), R, C, _p(s, _f32p), int(sr), seed, offset, index0,
                               C if ld is None else ld, _p(codes, _u8p), _p(scales, _u8p))
    return codes, scales


def _strip_senc(xf: np.ndarray) -> np.ndarray:
    """CTA-local outer factors: one S_enc per 128-row strip of the stored view,
    taken over the strip's full width (the whole K reduction)."""
    R = xf.shape[0]
    out = np.empty(R, np.float32)
    for s in range(0, R, STRIP):
        a = amax_f32(np.ascontiguousarray(xf[s:s + STRIP]))
        out[s:s + STRIP] = nv_senc(a)
    return out


def _sr_index(origin, cols, C):
    ld = C if cols is None else int(cols)
    return int(origin[0]) * ld + int(origin[1]), ld


def quantize(x_bits: np.ndarray, route: str, view: str, *, sr: bool = False, seed: int = 0,
             offset: int = 0, hadamard: bool = False, signs=None, weight2d: bool = False,
             hadamard16: bool = False,
             sr_origin: tuple[int, int] = (0, 0), sr_cols: int | None = None) -> dict:
    """Quantize a bf16 tensor (uint16 bits, R x C) into one view.

    route    'mx' | 'nv_global' | 'nv_local'
    view     'row' (scale blocks along C) | 'col' (blocks along R, stored transposed)
    sr       stochastic rounding; only allowed on the row view (Sec. 2.5)
    hadamard fixed-sign H32 before quantization; only on the MX column view
    hadamard16
             fixed-sign H16 (all signs +1: plain H16) on each aligned 16-value
             block of the column view before quantization, any route; an
             NVFP4 outer factor is then the transformed tensor's
    weight2d 2D32 (MX) or 2D16 (NV) shared weight encoding (Sec. 2.4)
    sr_origin, sr_cols
             when x is a block of a larger tensor: the (row, column) of its
             first element there and the larger tensor's row length, so that
             stochastic rounding draws the counters of the whole tensor's
             logical indices (defaults: x is the whole tensor)

    Returns dict(codes=uint8[rows, cols] 4-bit codes of the stored view,
                 scales=uint8[rows, cols // bs], senc=float32[rows] or None,
                 fmt=0 (MX) / 1 (NV), bs=block size).
    """
    assert route in ROUTES and view in ("row", "col")
    if sr and view != "row":
        raise ValueError("SR applies to the row-facing view only")
    if hadamard16 and (view != "col" or hadamard or weight2d):
        raise ValueError("H16 applies to a column-facing activation or gradient view only")
    if hadamard and (view != "col" or route != "mx"):
        raise ValueError("H32 applies to the MX column-facing view only")
    xf = bf16_to_f32(np.ascontiguousarray(x_bits))
    R, C = xf.shape
    if weight2d:
        if route == "mx":
            codes = np.empty((R, C), np.uint8)
            tiles = np.empty((R // 32, C // 32), np.uint8)
            lib().orc_mx_quantize_weight2d(_p(xf, _f32p), R, C, _p(codes, _u8p), _p(tiles, _u8p))
            bs, senc_all = 32, None
        else:
            senc = nv_senc(amax_f32(xf))
            codes = np.empty((R, C), np.uint8)
            tiles = np.empty((R // 16, C // 16), np.uint8)
            lib().orc_nv_quantize_weight2d(_p(xf, _f32p), R, C, senc, _p(codes, _u8p), _p(tiles, _u8p))
            bs, senc_all = 16, senc
        if view == "row":
            c = codes
            sc = np.repeat(tiles, bs, axis=0)
        else:
            c = np.ascontiguousarray(codes.T)
            sc = np.repeat(np.ascontiguousarray(tiles.T), bs, axis=0)
        senc_row = None if senc_all is None else np.full(c.shape[0], senc_all, np.float32)
        return dict(codes=np.ascontiguousarray(c), scales=np.ascontiguousarray(sc), senc=senc_row,
                    fmt=0 if route == "mx" else 1, bs=bs)

    v = xf if view == "row" else np.ascontiguousarray(xf.T)
    if hadamard:
        s = np.ascontiguousarray(signs, dtype=np.int8)
        assert s.shape == (16,)
        v = v.copy()
        lib().orc_hadamard32_rows(_p(v, _f32p), v.shape[0], v.shape[1], _p(s, _i8p))
    if hadamard16:
        s = np.ascontiguousarray(signs, dtype=np.int8)
        assert s.shape == (16,)
        v = v.copy()
        lib().orc_hadamard16_rows(_p(v, _f32p), v.shape[0], v.shape[1], _p(s, _i8p))
    if route == "mx":
        codes, scales = _mx_rows(v, sr, seed, offset, *_sr_index(sr_origin, sr_cols, C))
        return dict(codes=codes, scales=scales, senc=None, fmt=0, bs=32)
    if route == "nv_global":
        senc_row = np.full(v.shape[0], nv_senc(amax_f32(np.ascontiguousarray(v))), np.float32)
    else:
        senc_row = _strip_senc(v)
    codes, scales = _nv_rows(v, senc_row, sr, seed, offset, *_sr_index(sr_origin, sr_cols, C))
    return dict(codes=codes, scales=scales, senc=senc_row, fmt=1, bs=16)


def dequantize(q: dict) -> np.ndarray:
    codes, scales = q["codes"], q["scales"]
    R, C = codes.shape
    out = np.empty((R, C), np.float64)
    lib().orc_dequantize(_p(codes, _u8p), _p(scales, _u8p), q["fmt"], R, C, _opt(q["senc"], _f32p),
                         _p(out, _f64p))
    return out


def gemm(a: dict, b: dict) -> np.ndarray:
    """C[m, n] = sum_k A_hat[m, k] B_hat[n, k] in binary64 (Eqs. 4-6)."""
    A = dequantize(a)
    B = dequantize(b)
    M, K = A.shape
    N = B.shape[0]
    assert B.shape[1] == K
    C = np.empty((M, N), np.float64)
    lib().orc_gemm_nt(_p(A, _f64p), _p(B, _f64p), M, N, K, _p(C, _f64p))
    return C


def gemm_sampled(a: dict, b: dict, ms, ns):
    """Selected entries of the contraction and their sums of |products|."""
    assert a["fmt"] == b["fmt"]
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    K = a["codes"].shape[1]
    assert b["codes"].shape[1] == K
    out = np.empty(ms.size, np.float64)
    absout = np.empty(ms.size, np.float64)
    lib().orc_gemm_sampled(_p(a["codes"], _u8p), _p(a["scales"], _u8p), _opt(a["senc"], _f32p),
                           _p(b["codes"], _u8p), _p(b["scales"], _u8p), _opt(b["senc"], _f32p),
                           a["fmt"], K, _p(ms, _i64p), _p(ns, _i64p), ms.size, _p(out, _f64p),
                           _p(absout, _f64p))
    return out, absout


def gemm_abs(a: dict, b: dict) -> np.ndarray:
    """sum_k |A_hat[m, k] B_hat[n, k]| for every entry (the per-element error scale)."""
    A = np.abs(dequantize(a))
    B = np.abs(dequantize(b))
    M, K = A.shape
    N = B.shape[0]
    C = np.empty((M, N), np.float64)
    lib().orc_gemm_nt(_p(A, _f64p), _p(B, _f64p), M, N, K, _p(C, _f64p))
    return C


# ---------------------------------------------------------------------------
# fused-producer model arithmetic (Sec. 3.2)
# ---------------------------------------------------------------------------

def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round binary64 values to bf16 bits (nearest even), elementwise."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    f = np.vectorize(lambda v: lib().orc_bf16_round(float(v)), otypes=[np.uint16])
    return f(x) if x.size else np.zeros(x.shape, np.uint16)


def swiglu_h(a1: np.ndarray, a3: np.ndarray) -> np.ndarray:
    a1 = np.ascontiguousarray(a1, np.uint16)
    a3 = np.ascontiguousarray(a3, np.uint16)
    h = np.empty(a1.shape, np.uint16)
    lib().orc_swiglu_h(_p(a1, _u16p), _p(a3, _u16p), a1.size, _p(h, _u16p))
    return h


def swiglu_bwd(dh: np.ndarray, a1: np.ndarray, a3: np.ndarray):
    dh = np.ascontiguousarray(dh, np.uint16)
    a1 = np.ascontiguousarray(a1, np.uint16)
    a3 = np.ascontiguousarray(a3, np.uint16)
    da1 = np.empty(a1.shape, np.uint16)
    da3 = np.empty(a1.shape, np.uint16)
    lib().orc_swiglu_bwd(_p(dh, _u16p), _p(a1, _u16p), _p(a3, _u16p), a1.size, _p(da1, _u16p), _p(da3, _u16p))
    return da1, da3


def residual_rmsnorm(r, b, g, eps: float = 1e-5, rstd_in=None):
    """r' = bf16(r + b), rstd (binary32), y = bf16(r' * rstd * g) (Sec. 3.2)."""
    r = np.ascontiguousarray(r, np.uint16)
    b = np.ascontiguousarray(b, np.uint16)
    g = np.ascontiguousarray(g, np.uint16)
    R, C = r.shape
    r_out = np.empty((R, C), np.uint16)
    y = np.empty((R, C), np.uint16)
    rstd = np.empty(R, np.float32)
    ri = None if rstd_in is None else np.ascontiguousarray(rstd_in, np.float32)
    lib().orc_residual_rmsnorm(_p(r, _u16p), _p(b, _u16p), _p(g, _u16p), R, C, eps, int(ri is not None),
                               _opt(ri, _f32p), _p(r_out, _u16p), _p(rstd, _f32p), _p(y, _u16p))
    return r_out, rstd, y


def rmsnorm_bwd(dy, rp, rstd, g, dres):
    dy = np.ascontiguousarray(dy, np.uint16)
    rp = np.ascontiguousarray(rp, np.uint16)
    rstd = np.ascontiguousarray(rstd, np.float32)
    g = np.ascontiguousarray(g, np.uint16)
    dres = np.ascontiguousarray(dres, np.uint16)
    R, C = rp.shape
    dr = np.empty((R, C), np.uint16)
    lib().orc_rmsnorm_bwd(_p(dy, _u16p), _p(rp, _u16p), _p(rstd, _f32p), _p(g, _u16p), _p(dres, _u16p), R, C,
                          _p(dr, _u16p))
    return dr


# ---------------------------------------------------------------------------
# QKV producer with RoPE (Sec. 3.2)
# ---------------------------------------------------------------------------

ROPE_THETA = 500000.0  # Llama-3's base (the pages name RoPE but not its constants)


def rope_tables(S: int, D: int = 128, theta: float = ROPE_THETA):
    """cos, sin of p * theta^(-2i/D), binary64 rounded to binary32, [S][D/2] each."""
    c = np.empty((S, D // 2), np.float32)
    s_ = np.empty((S, D // 2), np.float32)
    lib().orc_rope_tables(S, D, theta, _p(c, _f32p), _p(s_, _f32p))
    return c, s_


def qkv_rope_fwd(qkv: np.ndarray, S: int, hq: int, hkv: int, cos_t, sin_t, D: int = 128):
    """qkv [T][(hq + 2 hkv) D] bf16 bits -> head-major q [hq][T][D], k, v
    [hkv][T][D]: Q and K turned by RoPE (rotate-half pairs, binary32 then
    bf16), V copied."""
    qkv = np.ascontiguousarray(qkv, dtype=np.uint16)
    T = qkv.shape[0]
    assert qkv.shape[1] == (hq + 2 * hkv) * D
    q = np.empty((hq, T, D), np.uint16)
    k = np.empty((hkv, T, D), np.uint16)
    v = np.empty((hkv, T, D), np.uint16)
    c, s_ = (np.ascontiguousarray(x, dtype=np.float32) for x in (cos_t, sin_t))
    lib().orc_qkv_rope_fwd(_p(qkv, _u16p), T, S, hq, hkv, D, _p(c, _f32p), _p(s_, _f32p), _p(q, _u16p), _p(k, _u16p),
                           _p(v, _u16p))
    return q, k, v


def qkv_rope_bwd(dq: np.ndarray, dk: np.ndarray, dv: np.ndarray, S: int, cos_t, sin_t, D: int = 128):
    """Head-major gradients of the turned Q, K and of V -> dqkv [T][(hq + 2 hkv) D]
    (the transposed rotation on dQ, dK; dV copied)."""
    dq, dk, dv = (np.ascontiguousarray(x, dtype=np.uint16) for x in (dq, dk, dv))
    hq, T, _ = dq.shape
    hkv = dk.shape[0]
    out = np.empty((T, (hq + 2 * hkv) * D), np.uint16)
    c, s_ = (np.ascontiguousarray(x, dtype=np.float32) for x in (cos_t, sin_t))
    lib().orc_qkv_rope_bwd(_p(dq, _u16p), _p(dk, _u16p), _p(dv, _u16p), T, S, hq, hkv, D, _p(c, _f32p),
                           _p(s_, _f32p), _p(out, _u16p))
    return out
