"""The C-ABI library builds, loads without a GPU, exports every function that
include/*.h declares, and rejects bad arguments on the host with the
documented status codes (no compute call is made)."""
import ctypes
import glob
import os
import re

import pytest

import fp4_quantized_linears_gb300 as F

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(fp4_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("fp4_quantize", "fp4_linear_fprop", "fp4_linear_dgrad", "fp4_linear_wgrad", "fp4_status"):
        assert n in names


def test_library_exports_every_declared_symbol():
    L = F.load()
    missing = [n for n in declared_functions() if not hasattr(L, n)]
    assert not missing, missing
    assert L.fp4_version() == 110


def test_tensor_bytes():
    assert F.fp4_tensor_bytes("mx", 256, 512) == (256 * 256, 256 * 16, 0)
    assert F.fp4_tensor_bytes("nv_global", 256, 512) == (256 * 256, 256 * 32, 1)
    assert F.fp4_tensor_bytes("nv_local", 256, 512) == (256 * 256, 256 * 32, 2)
    assert F.fp4_tensor_bytes("nv_local", 256, 512, F.FP4_FLAG_WEIGHT_2D)[2] == 1
    assert F.fp4_quantize_workspace_bytes("mx", 256, 512) == 0
    assert F.fp4_quantize_workspace_bytes("nv_local", 256, 512) == (1 + 2 + 4) * 4
    with pytest.raises(F.Fp4Error) as e:
        F.fp4_tensor_bytes("mx", 100, 512)
    assert e.value.code == F.FP4_ERR_UNSUPPORTED_SHAPE


def _t(rows=128, cols=128, route=0, oc=0):
    return F.fp4_tensor(16, 16, 16 if route else None, rows, cols, route, oc)


def test_host_validation_codes():
    L = F.load()
    q = L.fp4_quantize
    t = _t()
    sig = lambda *a: q(*a)
    # bad route / views / flags
    assert q(ctypes.c_void_p(16), 128, 128, 128, 9, 3, 0, 0, 0, None, ctypes.byref(t), ctypes.byref(t), None, 0, None) == F.FP4_ERR_INVALID_ARG
    assert q(ctypes.c_void_p(16), 128, 128, 128, 0, 0, 0, 0, 0, None, ctypes.byref(t), ctypes.byref(t), None, 0, None) == F.FP4_ERR_INVALID_ARG
    # shape rules
    assert q(ctypes.c_void_p(16), 100, 128, 128, 0, 3, 0, 0, 0, None, ctypes.byref(t), ctypes.byref(t), None, 0, None) == F.FP4_ERR_UNSUPPORTED_SHAPE
    # SR together with a 2D weight encoding; H32 on NVFP4
    assert q(ctypes.c_void_p(16), 128, 128, 128, 0, 3, 3, 0, 0, None, ctypes.byref(t), ctypes.byref(t), None, 0, None) == F.FP4_ERR_ROUTE_MISMATCH
    assert q(ctypes.c_void_p(16), 128, 128, 128, 1, 3, 4, 0, 0, None, ctypes.byref(t), ctypes.byref(t), None, 0, None) == F.FP4_ERR_ROUTE_MISMATCH
    # H32 without signs, and with a sign that is not +-1
    assert q(ctypes.c_void_p(16), 128, 128, 128, 0, 3, 4, 0, 0, None, ctypes.byref(t), ctypes.byref(t), None, 0, None) == F.FP4_ERR_INVALID_ARG
    bad = (ctypes.c_int8 * 16)(*([1] * 15 + [2]))
    assert q(ctypes.c_void_p(16), 128, 128, 128, 0, 3, 4, 0, 0, ctypes.cast(bad, ctypes.POINTER(ctypes.c_int8)), ctypes.byref(t), ctypes.byref(t), None, 0, None) == F.FP4_ERR_INVALID_ARG
    # NVFP4 without workspace
    tn = _t(route=1, oc=1)
    assert q(ctypes.c_void_p(16), 128, 128, 128, 1, 3, 0, 0, 0, None, ctypes.byref(tn), ctypes.byref(tn), None, 0, None) == F.FP4_ERR_WORKSPACE
    # misaligned input / leading dimension
    assert q(ctypes.c_void_p(18), 128, 128, 128, 0, 3, 0, 0, 0, None, ctypes.byref(t), ctypes.byref(t), None, 0, None) == F.FP4_ERR_INVALID_ARG
    assert q(ctypes.c_void_p(16), 128, 128, 132, 0, 3, 0, 0, 0, None, ctypes.byref(t), ctypes.byref(t), None, 0, None) == F.FP4_ERR_INVALID_ARG
    # empty tensors are a no-op
    assert q(ctypes.c_void_p(16), 0, 128, 128, 0, 3, 0, 0, 0, None, ctypes.byref(t), ctypes.byref(t), None, 0, None) == F.FP4_OK


def test_gemm_validation_codes():
    L = F.load()
    a, b = _t(128, 256), _t(256, 256)
    c = ctypes.c_void_p(16)
    assert L.fp4_linear_fprop(ctypes.byref(a), ctypes.byref(b), c, 7, 0.0, None) == F.FP4_ERR_INVALID_ARG
    bn = _t(256, 256, route=1, oc=1)
    assert L.fp4_linear_fprop(ctypes.byref(a), ctypes.byref(bn), c, 0, 0.0, None) == F.FP4_ERR_ROUTE_MISMATCH
    b2 = _t(256, 512)
    assert L.fp4_linear_fprop(ctypes.byref(a), ctypes.byref(b2), c, 0, 0.0, None) == F.FP4_ERR_UNSUPPORTED_SHAPE
    a3, b3 = _t(128, 128), _t(256, 128)  # K = 128 is below the 256-value K step
    assert L.fp4_linear_fprop(ctypes.byref(a3), ctypes.byref(b3), c, 0, 0.0, None) == F.FP4_ERR_UNSUPPORTED_SHAPE
    assert L.fp4_linear_fprop(None, ctypes.byref(b), c, 0, 0.0, None) == F.FP4_ERR_INVALID_ARG


def test_status_strings():
    assert F.status_string(0) == "ok"
    assert F.status_string(F.FP4_ERR_TIMEOUT) == "device wait timed out"


def test_dgrad_rmsnorm_validation_codes():
    """The Dgrad that emits RMSNorm row terms and the RMSNorm backward that
    consumes them reject missing or misaligned pointers and mismatched
    routes on the host."""
    L = F.load()
    dy, w = _t(128, 256), _t(256, 256)
    c, ok16, f4 = ctypes.c_void_p(16), ctypes.c_void_p(32), ctypes.c_void_p(64)
    d = L.fp4_linear_dgrad_rmsnorm
    assert d(ctypes.byref(dy), ctypes.byref(w), c, None, f4, ok16, f4, None) == F.FP4_ERR_INVALID_ARG   # no r'
    assert d(ctypes.byref(dy), ctypes.byref(w), c, ok16, None, ok16, f4, None) == F.FP4_ERR_INVALID_ARG  # no rstd
    assert d(ctypes.byref(dy), ctypes.byref(w), c, ok16, f4, None, f4, None) == F.FP4_ERR_INVALID_ARG    # no g
    assert d(ctypes.byref(dy), ctypes.byref(w), c, ok16, f4, ok16, None, None) == F.FP4_ERR_INVALID_ARG  # no terms
    assert d(ctypes.byref(dy), ctypes.byref(w), c, ctypes.c_void_p(18), f4, ok16, f4, None) == F.FP4_ERR_INVALID_ARG
    assert d(ctypes.byref(dy), ctypes.byref(w), c, ok16, f4, ctypes.c_void_p(40), f4, None) == F.FP4_ERR_INVALID_ARG
    assert d(ctypes.byref(dy), ctypes.byref(w), c, ok16, ctypes.c_void_p(66), ok16, f4, None) == F.FP4_ERR_INVALID_ARG
    wn = _t(256, 256, route=1, oc=1)
    assert d(ctypes.byref(dy), ctypes.byref(wn), c, ok16, f4, ok16, f4, None) == F.FP4_ERR_ROUTE_MISMATCH
    r = L.fp4_residual_rmsnorm_bwd_parts
    t = _t()
    # row terms missing
    assert r(0, 3, 1, ok16, None, ok16, f4, ok16, None, 128, 128, 0, 0, ok16, ctypes.byref(t), ctypes.byref(t), ok16,
             1 << 20, None) == F.FP4_ERR_INVALID_ARG
    # shape rule of the RMSNorm backward
    assert r(0, 3, 1, ok16, f4, ok16, f4, ok16, None, 100, 128, 0, 0, ok16, ctypes.byref(t), ctypes.byref(t), ok16,
             1 << 20, None) == F.FP4_ERR_UNSUPPORTED_SHAPE


def test_noalloc_checks_arguments_before_the_scratch_size():
    """fp4_quantize_noalloc fails an invalid call the way fp4_quantize does,
    even when the shape would also exceed its static scratch; undefined view
    or flag bits are rejected by the workspace query as by the quantizer."""
    L = F.load()
    f = L.fp4_quantize_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, ctypes.c_uint,
                  ctypes.c_uint, ctypes.c_uint64, ctypes.c_uint64, ctypes.POINTER(ctypes.c_int8),
                  ctypes.POINTER(F.fp4_tensor), ctypes.POINTER(F.fp4_tensor), ctypes.c_void_p]
    rows, cols = 128 * 4096, 128  # needs more amax slots than the scratch holds
    t = _t(route=F.FP4_ROUTE_NVFP4_GLOBAL, oc=1)
    # a missing row view (requested) is an invalid argument, not a workspace error
    assert f(16, rows, cols, cols, F.FP4_ROUTE_NVFP4_GLOBAL, 3, 0, 0, 0, None, None, ctypes.byref(t), None) == \
        F.FP4_ERR_INVALID_ARG
    # ld < cols, and undefined flag bits: invalid arguments too
    assert f(16, rows, cols, cols - 8, F.FP4_ROUTE_NVFP4_GLOBAL, 3, 0, 0, 0, None, ctypes.byref(t), ctypes.byref(t),
             None) == F.FP4_ERR_INVALID_ARG
    assert f(16, rows, cols, cols, F.FP4_ROUTE_NVFP4_GLOBAL, 3, 0x100, 0, 0, None, ctypes.byref(t), ctypes.byref(t),
             None) == F.FP4_ERR_INVALID_ARG
    n = ctypes.c_size_t()
    assert L.fp4_quantize_workspace_bytes(F.FP4_ROUTE_NVFP4_GLOBAL, 256, 256, 3, 0x100, ctypes.byref(n)) == \
        F.FP4_ERR_INVALID_ARG
    assert L.fp4_quantize_workspace_bytes(F.FP4_ROUTE_NVFP4_GLOBAL, 256, 256, 4, 0, ctypes.byref(n)) == \
        F.FP4_ERR_INVALID_ARG
