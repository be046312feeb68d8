"""GPU parity of the quantizer producers against the CPU oracle: codes, scale
bytes and outer factors must match bit for bit (Format-Aware Fusion for Fast
FP4 Pretraining, Sec. 2.2-2.5)."""
import numpy as np
import pytest
import torch

import oracle
import fp4_quantized_linears_gb300 as F
from layout import expand_outer, unpack_codes, unswizzle_scales
from synthetic import (bf16_bits_from_f32, config_tensors, f32_from_bf16_bits, hadamard_signs, normal_bf16,
                       with_outliers_bf16)

pytestmark = pytest.mark.gpu


def to_dev(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def view_host(v: F.QView, bs: int):
    torch.cuda.synchronize()
    codes = unpack_codes(v.codes.cpu().numpy())
    scales = unswizzle_scales(v.scales.cpu().numpy(), v.rows, v.cols, bs)
    outer = None if v.outer is None else expand_outer(v.outer.cpu().numpy(), v.outer_count, v.rows)
    return codes, scales, outer


def assert_view_equal(v: F.QView, ref: dict, what: str):
    codes, scales, outer = view_host(v, ref["bs"])
    assert codes.shape == ref["codes"].shape, what
    bad = np.argwhere(codes != ref["codes"])
    assert bad.size == 0, f"{what}: {len(bad)} code mismatches, first {bad[:5].tolist()}"
    bad = np.argwhere(scales != ref["scales"])
    assert bad.size == 0, f"{what}: {len(bad)} scale mismatches, first {bad[:5].tolist()}"
    if ref["senc"] is not None:
        assert np.array_equal(outer, ref["senc"]), f"{what}: outer factors differ"


def quantize_both(x_bits, route, flags=0, seed=0, offset=0, signs=None):
    x = to_dev(x_bits)
    r, c = F.fp4_quantize(x, route, F.FP4_VIEW_ROW | F.FP4_VIEW_COL, flags, seed, offset, signs)
    return r, c


def check(x_bits, route, flags=0, seed=0, offset=0, signs=None):
    r, c = quantize_both(x_bits, route, flags, seed, offset, signs)
    w2d = bool(flags & F.FP4_FLAG_WEIGHT_2D)
    ref_r = oracle.quantize(x_bits, route, "row", sr=bool(flags & F.FP4_FLAG_SR_ROW), seed=seed, offset=offset,
                            weight2d=w2d)
    ref_c = oracle.quantize(x_bits, route, "col", hadamard=bool(flags & F.FP4_FLAG_HADAMARD_COL), signs=signs,
                            weight2d=w2d)
    assert_view_equal(r, ref_r, f"{route} row flags={flags}")
    assert_view_equal(c, ref_c, f"{route} col flags={flags}")
    assert F.fp4_status() == F.FP4_OK


def all_finite_bf16(shape=(256, 256)):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    f = f32_from_bf16_bits(bits)
    bits = np.where(np.isfinite(f), bits, 0).astype(np.uint16)
    rng = np.random.default_rng(0)
    bits = bits[rng.permutation(bits.size)]
    return bits.reshape(shape)


def probe_values():
    # every 32-block holds a 6 (exponent 0 under the upward rule) and probes at
    # the rounding thresholds, ties, zeros of both signs and subnormals
    probes = [0.0, -0.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 0.24, 0.26, 0.74, 0.76, 2.49, 2.51, 4.99, 5.01,
              1e-40, -1e-40, -0.1, 0.1, 3.0, 4.0, -6.0, 5.999, 1.5, 0.5, 1.0, -2.5, -3.5, -5.0]
    x = np.zeros((128, 128), np.float32)
    for r in range(128):
        for b in range(4):
            blk = [6.0] + probes
            x[r, b * 32:(b + 1) * 32] = np.array(blk[:32], np.float32) * (2.0 ** ((r % 9) - 4))
    return bf16_bits_from_f32(x)


@pytest.mark.parametrize("route", ["mx", "nv_global", "nv_local"])
def test_quantize_random_shapes(route):
    for shape, seed in (((256, 384), 1), ((384, 128), 2), ((128, 512), 3)):
        x = with_outliers_bf16(shape, 1.0, 1e-3, 20.0, seed, 1)
        check(x, route)


@pytest.mark.parametrize("route", ["mx", "nv_global", "nv_local"])
def test_quantize_all_bf16_values(route):
    check(all_finite_bf16(), route)


def test_quantize_rounding_probes_mx():
    check(probe_values(), "mx")
    check(probe_values(), "mx", flags=F.FP4_FLAG_SR_ROW, seed=5, offset=9)


@pytest.mark.parametrize("route", ["mx", "nv_global", "nv_local"])
def test_quantize_sr_row(route):
    x = normal_bf16((256, 256), 1e-3, 4, 1)
    check(x, route, flags=F.FP4_FLAG_SR_ROW, seed=0x1234_5678_9ABC, offset=3)
    check(x, route, flags=F.FP4_FLAG_SR_ROW, seed=7, offset=(1 << 40) + 1)


def test_quantize_hadamard_col():
    x = config_tensors("c2_mx_w1", scale_T=256, d_in=256, d_out=384)
    s = x["signs"]
    check(x["x"], "mx", flags=F.FP4_FLAG_HADAMARD_COL, signs=s)
    check(x["dy"], "mx", flags=F.FP4_FLAG_HADAMARD_COL | F.FP4_FLAG_SR_ROW, seed=11, offset=0, signs=s)


@pytest.mark.parametrize("route", ["mx", "nv_global", "nv_local"])
def test_quantize_weight_2d(route):
    w = normal_bf16((384, 256), 0.02, 6, 2)
    check(w, route, flags=F.FP4_FLAG_WEIGHT_2D)
    r, c = quantize_both(w, route, F.FP4_FLAG_WEIGHT_2D)
    # Eq. 8: the column view's codes are the bitwise transpose of the row view's
    cr, _, _ = view_host(r, 32 if route == "mx" else 16)
    cc, _, _ = view_host(c, 32 if route == "mx" else 16)
    assert np.array_equal(cr, cc.T)


def test_quantize_zero_tensor_and_single_views():
    z = np.zeros((128, 256), np.uint16)
    check(z, "mx")
    check(z, "nv_global")
    x = normal_bf16((128, 128), 1.0, 7, 1)
    r, c = F.fp4_quantize(to_dev(x), "mx", F.FP4_VIEW_ROW)
    assert c is None
    assert_view_equal(r, oracle.quantize(x, "mx", "row"), "row only")
    r, c = F.fp4_quantize(to_dev(x), "nv_local", F.FP4_VIEW_COL)
    assert r is None
    assert_view_equal(c, oracle.quantize(x, "nv_local", "col"), "col only")


def test_quantize_strided_input():
    big = normal_bf16((128, 384), 1.0, 8, 1)
    xt = to_dev(big)[:, 128:384]  # leading dimension 384, 256 columns
    r, c = F.fp4_quantize(xt, "mx")
    sub = np.ascontiguousarray(big[:, 128:384])
    assert_view_equal(r, oracle.quantize(sub, "mx", "row"), "strided row")
    assert_view_equal(c, oracle.quantize(sub, "mx", "col"), "strided col")


def test_nonfinite_input_sets_status():
    x = normal_bf16((128, 128), 1.0, 9, 1).copy()
    x[5, 7] = 0x7F80  # +inf
    F.fp4_status_reset()
    F.fp4_quantize(to_dev(x), "mx")
    assert F.fp4_status() == F.FP4_ERR_NONFINITE
    F.fp4_status_reset()
    assert F.fp4_status() == F.FP4_OK
