"""GPU parity of the H16 column transform and of the operand-wise hybrid
producer and linear (Format-Aware Fusion for Fast FP4 Pretraining, Sec. 2.5
fixed-sign H16 for NVFP4 Wgrad; Sec. 3.3 operand-wise hybrid: MXFP4 Fprop and
Wgrad, CTA-local NVFP4 Dgrad with row SR, plain H16 (D = I) or fixed-sign H32
on the Wgrad pair), against the oracle run on the host inputs.  Codes, scales
and outer factors are bit-exact; the contractions are within the tolerance
(relative Frobenius <= 1e-5, per element <= 2^-18 sum_k |a_k b_k|) of the
oracle's binary64 contraction of its own views, which the GPU's equal."""
import numpy as np
import pytest
import torch

import oracle
import fp4_quantized_linears_gb300 as F
from masked import host_view as mhost
from synthetic import config_tensors, hadamard_signs, normal_bf16, with_outliers_bf16
from parity_stats import record

pytestmark = pytest.mark.gpu

ONES = np.ones(16, np.int8)
REL_FRO = 1e-5
PER_ELEM = 2.0 ** -18


def to_dev(b):
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).cuda()


def same_view(v, want, what):
    got = mhost(v)
    nc = int(np.sum(got["codes"] != want["codes"]))
    ns = int(np.sum(got["scales"] != want["scales"]))
    assert nc == 0 and ns == 0, f"{what}: {nc} code and {ns} scale mismatches"
    if want["senc"] is not None:
        assert np.array_equal(got["senc"], want["senc"]), f"{what}: outer factors"
    else:
        assert got["senc"] is None, f"{what}: unexpected outer factors"


def close(got, a, b, what):
    ref, absref = oracle.gemm(a, b), oracle.gemm_abs(a, b)
    g = got.astype(np.float64)
    fro = np.linalg.norm(g - ref) / max(np.linalg.norm(ref), 1e-300)
    record(what, fro=fro, err_over_sum_abs=(np.abs(g - ref) / np.maximum(absref, 1e-300)).max())
    assert fro <= REL_FRO, f"{what}: relative Frobenius {fro:.3e}"
    assert (np.abs(g - ref) <= PER_ELEM * absref + 1e-30).all(), what


@pytest.mark.parametrize("route", ["mx", "nv_global", "nv_local"])
@pytest.mark.parametrize("signs_seed", [None, 3])
def test_h16_column_view(route, signs_seed):
    signs = ONES if signs_seed is None else hadamard_signs(signs_seed)
    x = with_outliers_bf16((384, 256), 1.0, 1e-3, 20.0, 41, 1)
    r, c = F.fp4_quantize(to_dev(x), route, 3, F.FP4_FLAG_HADAMARD16_COL, hadamard_signs=signs)
    assert F.fp4_status() == F.FP4_OK
    same_view(r, oracle.quantize(x, route, "row"), f"{route} row")
    same_view(c, oracle.quantize(x, route, "col", hadamard16=True, signs=signs), f"{route} col H16")


@pytest.mark.parametrize("route", ["nv_global", "nv_local"])
def test_h16_with_row_sr(route):
    dy = normal_bf16((256, 512), 1e-3, 42, 1)
    signs = hadamard_signs(4)
    r, c = F.fp4_quantize(to_dev(dy), route, 3, F.FP4_FLAG_SR_ROW | F.FP4_FLAG_HADAMARD16_COL, sr_seed=9,
                          sr_offset=2, hadamard_signs=signs)
    same_view(r, oracle.quantize(dy, route, "row", sr=True, seed=9, offset=2), f"{route} row SR")
    same_view(c, oracle.quantize(dy, route, "col", hadamard16=True, signs=signs), f"{route} col H16")


@pytest.mark.parametrize("had", ["h16", "h32"])
def test_hybrid_gradient_producer(had):
    dy = normal_bf16((256, 384), 1e-3, 43, 1)
    flag = F.FP4_FLAG_HADAMARD16_COL if had == "h16" else F.FP4_FLAG_HADAMARD_COL
    signs = ONES if had == "h16" else hadamard_signs(5)
    r, c = F.fp4_quantize_hybrid(to_dev(dy), "nv_local", "mx", 3, F.FP4_FLAG_SR_ROW | flag, sr_seed=7, sr_offset=1,
                                 hadamard_signs=signs)
    assert r.route == F.FP4_ROUTE_NVFP4_LOCAL and c.route == F.FP4_ROUTE_MXFP4
    same_view(r, oracle.quantize(dy, "nv_local", "row", sr=True, seed=7, offset=1), "dY row (CTA-local, SR)")
    kw = dict(hadamard16=True) if had == "h16" else dict(hadamard=True)
    same_view(c, oracle.quantize(dy, "mx", "col", signs=signs, **kw), f"dY col (MX, {had})")


def test_hybrid_weight_producer():
    w = normal_bf16((384, 256), 0.02, 44, 1)
    r, c = F.fp4_quantize_hybrid(to_dev(w), "mx", "nv_local", 3, F.FP4_FLAG_WEIGHT_2D)
    assert r.route == F.FP4_ROUTE_MXFP4 and c.route == F.FP4_ROUTE_NVFP4_LOCAL and c.outer_count == 1
    same_view(r, oracle.quantize(w, "mx", "row", weight2d=True), "W row (MX 2D32)")
    same_view(c, oracle.quantize(w, "nv_local", "col", weight2d=True), "W col (CTA-local 2D16)")


def test_hybrid_single_view_requests():
    w = normal_bf16((256, 256), 0.02, 45, 1)
    r, c = F.fp4_quantize_hybrid(to_dev(w), "mx", "nv_local", F.FP4_VIEW_COL, F.FP4_FLAG_WEIGHT_2D)
    assert r is None
    same_view(c, oracle.quantize(w, "nv_local", "col", weight2d=True), "col only")
    r, c = F.fp4_quantize_hybrid(to_dev(w), "nv_local", "mx", F.FP4_VIEW_ROW, 0)
    assert c is None
    same_view(r, oracle.quantize(w, "nv_local", "row"), "row only")


def test_h32_on_an_nvfp4_column_view_is_rejected():
    x = normal_bf16((128, 128), 1.0, 46, 1)
    with pytest.raises(F.Fp4Error) as e:
        F.fp4_quantize_hybrid(to_dev(x), "mx", "nv_local", 3, F.FP4_FLAG_HADAMARD_COL, hadamard_signs=ONES)
    assert e.value.code == F.FP4_ERR_ROUTE_MISMATCH
    with pytest.raises(F.Fp4Error) as e:
        F.fp4_quantize(to_dev(x), "mx", 3, F.FP4_FLAG_HADAMARD_COL | F.FP4_FLAG_HADAMARD16_COL, hadamard_signs=ONES)
    assert e.value.code == F.FP4_ERR_INVALID_ARG


def run_hybrid_linear(x, w, dy, had, seed=11):
    """The operand-wise hybrid linear: MXFP4 Fprop and Wgrad (plain H16 or
    fixed-sign H32 on the pair), CTA-local NVFP4 Dgrad with row SR."""
    flag = F.FP4_FLAG_HADAMARD16_COL if had == "h16" else F.FP4_FLAG_HADAMARD_COL
    signs = ONES if had == "h16" else hadamard_signs(6)
    xr, xc = F.fp4_quantize(to_dev(x), "mx", 3, flag, hadamard_signs=signs)
    wr, wc = F.fp4_quantize_hybrid(to_dev(w), "mx", "nv_local", 3, F.FP4_FLAG_WEIGHT_2D)
    dr, dc = F.fp4_quantize_hybrid(to_dev(dy), "nv_local", "mx", 3, F.FP4_FLAG_SR_ROW | flag, sr_seed=seed,
                                   hadamard_signs=signs)
    y = F.fp4_linear_fprop(xr, wr)
    dx = F.fp4_linear_dgrad(dr, wc)
    dw = F.fp4_linear_wgrad(dc, xc)
    torch.cuda.synchronize()
    assert F.fp4_status() == F.FP4_OK
    kw = dict(hadamard16=True) if had == "h16" else dict(hadamard=True)
    ov = dict(xr=oracle.quantize(x, "mx", "row"), xc=oracle.quantize(x, "mx", "col", signs=signs, **kw),
              wr=oracle.quantize(w, "mx", "row", weight2d=True), wc=oracle.quantize(w, "nv_local", "col", weight2d=True),
              dr=oracle.quantize(dy, "nv_local", "row", sr=True, seed=seed),
              dc=oracle.quantize(dy, "mx", "col", signs=signs, **kw))
    for k, v in dict(xr=xr, xc=xc, wr=wr, wc=wc, dr=dr, dc=dc).items():
        same_view(v, ov[k], f"hybrid {had} {k}")
    return (y, dx, dw), ov


@pytest.mark.parametrize("had", ["h16", "h32"])
def test_hybrid_linear(had):
    t = config_tensors("c1_mx_small")
    (y, dx, dw), ov = run_hybrid_linear(t["x"], t["w"], t["dy"], had)
    close(y.cpu().numpy(), ov["xr"], ov["wr"], "Fprop (MX)")
    close(dx.cpu().numpy(), ov["dr"], ov["wc"], "Dgrad (CTA-local)")
    close(dw.cpu().numpy(), ov["dc"], ov["xc"], "Wgrad (MX, transformed pair)")


@pytest.mark.parametrize("route", ["nv_global", "nv_local"])
def test_nvfp4_wgrad_with_fixed_sign_h16(route):
    x = with_outliers_bf16((256, 512), 1.0, 1e-3, 20.0, 47, 1)
    dy = normal_bf16((256, 384), 1e-3, 47, 2)
    signs = hadamard_signs(8)
    _, xc = F.fp4_quantize(to_dev(x), route, F.FP4_VIEW_COL, F.FP4_FLAG_HADAMARD16_COL, hadamard_signs=signs)
    _, dc = F.fp4_quantize(to_dev(dy), route, F.FP4_VIEW_COL, F.FP4_FLAG_HADAMARD16_COL, hadamard_signs=signs)
    dw = F.fp4_linear_wgrad(dc, xc).cpu().numpy()
    ox = oracle.quantize(x, route, "col", hadamard16=True, signs=signs)
    od = oracle.quantize(dy, route, "col", hadamard16=True, signs=signs)
    same_view(xc, ox, "X col H16")
    same_view(dc, od, "dY col H16")
    close(dw, od, ox, f"{route} Wgrad with H16")
