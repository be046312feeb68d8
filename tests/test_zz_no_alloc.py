"""fp4_quantize_noalloc: the quantizer entry point for callers that cannot
allocate device memory when they quantize (a runtime whose pool owns all
device memory, a server that reserves everything at start-up, a path that
cannot afford cudaMalloc's implicit synchronisation).  It takes its NVFP4
scratch from a fixed array in static device memory; this file checks,
through the C ABI, that it produces exactly what fp4_quantize produces with a
caller-provided workspace, on two calls in a row (the second call must not
see the first call's leftovers), and that it rejects shapes whose scratch
would not fit.  Kept in its own file so that it runs last."""
import ctypes

import numpy as np
import pytest
import torch

import fp4_quantized_linears_gb300 as F
from synthetic import normal_bf16, with_outliers_bf16


def _lib():
    L = F.load()
    f = L.fp4_quantize_noalloc
    tp = ctypes.POINTER(F.fp4_tensor)
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, ctypes.c_uint,
                  ctypes.c_uint, ctypes.c_uint64, ctypes.c_uint64, ctypes.POINTER(ctypes.c_int8), tp, tp,
                  ctypes.c_void_p]
    return L


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def _noalloc(L, x, route, views=3, flags=0, seed=0, offset=0):
    R, C = x.shape
    r = F.alloc_view(route, R, C, flags) if views & 1 else None
    c = F.alloc_view(route, C, R, flags) if views & 2 else None
    rs = r.struct() if r is not None else None
    cs = c.struct() if c is not None else None
    code = L.fp4_quantize_noalloc(ctypes.c_void_p(x.data_ptr()), R, C, x.stride(0), F.ROUTES[route], views, flags,
                                  seed, offset, None, ctypes.byref(rs) if rs else None,
                                  ctypes.byref(cs) if cs else None,
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert code == F.FP4_OK, F.status_string(code)
    for v, st in ((r, rs), (c, cs)):
        if v is not None:
            v.rows, v.cols, v.route, v.outer_count = st.rows, st.cols, st.route, st.outer_count
    return r, c


def _same(a: F.QView, b: F.QView):
    torch.cuda.synchronize()
    assert torch.equal(a.codes, b.codes)
    assert torch.equal(a.scales, b.scales)
    assert a.outer_count == b.outer_count
    if a.outer is not None:
        assert torch.equal(a.outer[:a.outer_count], b.outer[:b.outer_count])


@pytest.mark.gpu
@pytest.mark.parametrize("route,flags", [("nv_global", 0), ("nv_local", 0), ("nv_local", F.FP4_FLAG_SR_ROW),
                                         ("nv_global", F.FP4_FLAG_WEIGHT_2D), ("mx", 0)])
def test_noalloc_matches_workspace_entry_point_twice(route, flags):
    L = _lib()
    # two different tensors in a row: the second has a smaller amax, so any
    # amax left over in the shared scratch would change its scales
    xs = [with_outliers_bf16((256, 384), 1.0, 1e-3, 20.0, 41, 1), normal_bf16((256, 384), 0.01, 41, 2)]
    for i, bits in enumerate(xs):
        x = _dev(bits)
        got_r, got_c = _noalloc(L, x, route, 3, flags, seed=5, offset=i)
        ref_r, ref_c = F.fp4_quantize(x, route, 3, flags, sr_seed=5, sr_offset=i)
        _same(got_r, ref_r)
        _same(got_c, ref_c)
    assert F.fp4_status() == F.FP4_OK


@pytest.mark.gpu
def test_noalloc_rejects_shapes_beyond_the_scratch():
    L = _lib()
    t = F.fp4_tensor(16, 16, 16, 0, 0, 1, 0)
    # 1 + rows/128 + cols/128 slots of 4 bytes must fit in 16 KiB
    rows, cols = 128 * 4096, 128
    code = L.fp4_quantize_noalloc(ctypes.c_void_p(16), rows, cols, cols, F.FP4_ROUTE_NVFP4_GLOBAL, 3, 0, 0, 0, None,
                                  ctypes.byref(t), ctypes.byref(t), None)
    assert code == F.FP4_ERR_WORKSPACE
