"""GPU parity of the block-scaled tcgen05 GEMM against the oracle's binary64
contraction of the dequantized operands (Format-Aware Fusion for Fast FP4
Pretraining, Sec. 2.3 Eqs. 4-6).

The reference operands are the oracle's own quantization of the host inputs;
the GPU's views are first required to equal them bit for bit, so the GPU
contraction and the reference contract the same codes.  Tolerance: relative
Frobenius error <= 1e-5 and, per element, |err| <= 2^-18 * sum_k |a_k b_k|.
Operands with unit scales and integer-valued products are exact in FP32 and
must match bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import fp4_quantized_linears_gb300 as F
from layout import swizzle_scales
from synthetic import config_tensors, normal_bf16, with_outliers_bf16
from parity_stats import record

pytestmark = pytest.mark.gpu

REL_FRO = 1e-5
PER_ELEM = 2.0 ** -18


def to_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def host_view(v: F.QView, bs: int, fmt: int):
    from layout import expand_outer, unpack_codes, unswizzle_scales
    torch.cuda.synchronize()
    return dict(codes=unpack_codes(v.codes.cpu().numpy()),
                scales=unswizzle_scales(v.scales.cpu().numpy(), v.rows, v.cols, bs),
                senc=None if v.outer is None else expand_outer(v.outer.cpu().numpy(), v.outer_count, v.rows),
                fmt=fmt, bs=bs)


def assert_close(got: np.ndarray, ref: np.ndarray, absref: np.ndarray, what: str):
    err = np.abs(got.astype(np.float64) - ref)
    fro = np.linalg.norm(got.astype(np.float64) - ref) / max(np.linalg.norm(ref), 1e-300)
    ratio = (err / np.maximum(absref, 1e-300)).max()
    record(what, fro=fro, err_over_sum_abs=ratio)
    assert fro <= REL_FRO, f"{what}: relative Frobenius {fro:.3e}"
    assert (err <= PER_ELEM * absref + 1e-30).all(), f"{what}: max err / sum|ab| = {ratio:.3e} (> 2^-18)"


def same_view(got: dict, want: dict, what: str):
    assert np.array_equal(got["codes"], want["codes"]), f"{what}: codes differ from the oracle's"
    assert np.array_equal(got["scales"], want["scales"]), f"{what}: scales differ from the oracle's"
    if want["senc"] is not None:
        assert np.array_equal(got["senc"], want["senc"]), f"{what}: outer factors differ from the oracle's"


def oracle_views(x, w, dy, route, xflags=0, dyflags=0, signs=None, seed=0, offset=0):
    """The six operand views as the oracle quantizes the host inputs."""
    hx = bool(xflags & F.FP4_FLAG_HADAMARD_COL)
    hd = bool(dyflags & F.FP4_FLAG_HADAMARD_COL)
    sr = bool(dyflags & F.FP4_FLAG_SR_ROW)
    return dict(xr=oracle.quantize(x, route, "row"),
                xc=oracle.quantize(x, route, "col", hadamard=hx, signs=signs),
                wr=oracle.quantize(w, route, "row", weight2d=True),
                wc=oracle.quantize(w, route, "col", weight2d=True),
                dr=oracle.quantize(dy, route, "row", sr=sr, seed=seed, offset=offset),
                dc=oracle.quantize(dy, route, "col", hadamard=hd, signs=signs))


def run_linear(x, w, dy, route, xflags=0, dyflags=0, signs=None, seed=0, offset=0):
    bs, fmt = (32, 0) if route == "mx" else (16, 1)
    xr, xc = F.fp4_quantize(to_dev(x), route, 3, xflags, hadamard_signs=signs)
    wr, wc = F.fp4_quantize(to_dev(w), route, 3, F.FP4_FLAG_WEIGHT_2D)
    dr, dc = F.fp4_quantize(to_dev(dy), route, 3, dyflags, seed, offset, hadamard_signs=signs)
    y = F.fp4_linear_fprop(xr, wr)
    dx = F.fp4_linear_dgrad(dr, wc)
    dw = F.fp4_linear_wgrad(dc, xc)
    torch.cuda.synchronize()
    ov = oracle_views(x, w, dy, route, xflags, dyflags, signs, seed, offset)
    for k, v in dict(xr=xr, xc=xc, wr=wr, wc=wc, dr=dr, dc=dc).items():
        same_view(host_view(v, bs, fmt), ov[k], f"{route} {k}")
    return y.cpu().numpy(), dx.cpu().numpy(), dw.cpu().numpy(), ov


@pytest.mark.parametrize("route", ["mx", "nv_global", "nv_local"])
def test_linear_c1_shapes(route):
    t = config_tensors("c1_mx_small")
    y, dx, dw, hv = run_linear(t["x"], t["w"], t["dy"], route, dyflags=F.FP4_FLAG_SR_ROW, seed=0, offset=0)
    for name, got, a, b in (("fprop", y, "xr", "wr"), ("dgrad", dx, "dr", "wc"), ("wgrad", dw, "dc", "xc")):
        ref = oracle.gemm(hv[a], hv[b])
        absref = oracle.gemm_abs(hv[a], hv[b])
        assert_close(got, ref, absref, f"{route} {name}")
    assert F.fp4_status() == F.FP4_OK


def test_linear_c2_shape_with_hadamard_small():
    t = config_tensors("c2_mx_w1", scale_T=512, d_in=512, d_out=768)
    y, dx, dw, hv = run_linear(t["x"], t["w"], t["dy"], "mx", xflags=F.FP4_FLAG_HADAMARD_COL,
                               dyflags=F.FP4_FLAG_SR_ROW | F.FP4_FLAG_HADAMARD_COL, signs=t["signs"], seed=1)
    for name, got, a, b in (("fprop", y, "xr", "wr"), ("dgrad", dx, "dr", "wc"), ("wgrad", dw, "dc", "xc")):
        assert_close(got, oracle.gemm(hv[a], hv[b]), oracle.gemm_abs(hv[a], hv[b]), name)


@pytest.mark.parametrize("route", ["mx", "nv_global"])
def test_unit_scale_integer_gemm_is_exact(route):
    # codes with unit block scales: every product is a multiple of 1/4 and the
    # sums stay far below 2^24 quarter-units, so FP32 accumulation is exact
    rng = np.random.default_rng(1)
    M, N, K = 256, 384, 512
    bs = 32 if route == "mx" else 16
    one = 127 if route == "mx" else 0x38
    ca = rng.integers(0, 16, (M, K)).astype(np.uint8)
    cb = rng.integers(0, 16, (N, K)).astype(np.uint8)

    def make(c):
        v = F.alloc_view(route, c.shape[0], c.shape[1])
        packed = (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)
        v.codes.copy_(torch.from_numpy(packed))
        v.scales.copy_(torch.from_numpy(swizzle_scales(np.full((c.shape[0], K // bs), one, np.uint8))))
        if v.outer is not None:
            v.outer.fill_(1.0)
            v.outer_count = 1
        return v

    a, b = make(ca), make(cb)
    y = F.fp4_linear_fprop(a, b).cpu().numpy()
    ref = oracle.gemm(dict(codes=ca, scales=np.full((M, K // bs), one, np.uint8), senc=None, fmt=0 if route == "mx" else 1, bs=bs),
                      dict(codes=cb, scales=np.full((N, K // bs), one, np.uint8), senc=None, fmt=0 if route == "mx" else 1, bs=bs))
    assert np.array_equal(y.astype(np.float64), ref)


def test_bf16_output_and_beta_accumulate():
    t = config_tensors("c1_mx_small")
    xr, _ = F.fp4_quantize(to_dev(t["x"]), "mx", F.FP4_VIEW_ROW)
    wr, _ = F.fp4_quantize(to_dev(t["w"]), "mx", F.FP4_VIEW_ROW, F.FP4_FLAG_WEIGHT_2D)
    y32 = F.fp4_linear_fprop(xr, wr)
    yb = F.fp4_linear_fprop(xr, wr, out_dtype=F.FP4_OUT_BF16)
    assert torch.equal(yb, y32.to(torch.bfloat16))
    acc = y32.clone()
    F.fp4_linear_fprop(xr, wr, y=acc, beta=1.0)
    assert torch.equal(acc, 2 * y32)
    acc = y32.clone()
    F.fp4_linear_fprop(xr, wr, y=acc, beta=0.5)
    assert torch.allclose(acc, 1.5 * y32, rtol=1e-6, atol=0)
    accb = yb.clone()
    F.fp4_linear_fprop(xr, wr, y=accb, out_dtype=F.FP4_OUT_BF16, beta=1.0)
    assert torch.allclose(accb.float(), 2 * yb.float(), rtol=2 ** -7, atol=0)


def test_route_mismatch_is_rejected():
    t = config_tensors("c1_mx_small")
    xr, _ = F.fp4_quantize(to_dev(t["x"]), "mx", F.FP4_VIEW_ROW)
    wr, _ = F.fp4_quantize(to_dev(t["w"]), "nv_global", F.FP4_VIEW_ROW, F.FP4_FLAG_WEIGHT_2D)
    with pytest.raises(F.Fp4Error) as e:
        F.fp4_linear_fprop(xr, wr)
    assert e.value.code == F.FP4_ERR_ROUTE_MISMATCH


@pytest.mark.parametrize("M,N,K,route", [(384, 384, 512, "mx"), (2048, 4096, 512, "mx"), (2048, 2048, 768, "nv_local"),
                                         (640, 768, 256, "nv_global"), (1024, 640, 512, "mx"),
                                         (512, 384, 768, "nv_local"), (256, 128, 256, "nv_global")])
def test_persistent_tiles_unpaired_and_narrow(M, N, K, route):
    """Shapes that make CTAs loop over several tiles, use unpaired M blocks
    (single CTAs) and the 128-wide N tile on single CTAs and on CTA pairs
    (each CTA of a pair loads 64 rows of B); checked on sampled entries."""
    bs, fmt = (32, 0) if route == "mx" else (16, 1)
    a = normal_bf16((M, K), 1.0, M + N, 1)
    b = normal_bf16((N, K), 0.05, M + N, 2)
    ar, _ = F.fp4_quantize(to_dev(a), route, F.FP4_VIEW_ROW)
    br, _ = F.fp4_quantize(to_dev(b), route, F.FP4_VIEW_ROW)
    c = F.fp4_linear_fprop(ar, br).cpu().numpy()
    ha, hb = oracle.quantize(a, route, "row"), oracle.quantize(b, route, "row")
    same_view(host_view(ar, bs, fmt), ha, "A")
    same_view(host_view(br, bs, fmt), hb, "B")
    rng = np.random.default_rng(0)
    ms = np.concatenate([rng.integers(0, M, 4000), np.repeat(np.arange(M - 128, M), 8)])
    ns = np.concatenate([rng.integers(0, N, 4000), np.tile(rng.integers(0, N, 8), 128)])
    ref, absref = oracle.gemm_sampled(ha, hb, ms, ns)
    assert_close(c[ms, ns], ref, absref, f"{route} {M}x{N}x{K}")
    assert F.fp4_status() == F.FP4_OK
