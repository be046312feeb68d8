"""GPU parity of the residual-RMSNorm producer (Format-Aware Fusion for Fast
FP4 Pretraining, Sec. 3.2), in two levels: the retained BF16 state and the
BF16 values it quantizes are checked against the oracle's model arithmetic,
then the FP4 views are checked bit for bit against the oracle quantizing
those same BF16 values."""
import numpy as np
import pytest
import torch

import oracle
import fp4_quantized_linears_gb300 as F
from layout import expand_outer, unpack_codes, unswizzle_scales
from synthetic import normal_bf16

pytestmark = pytest.mark.gpu


def to_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def bits(t):
    torch.cuda.synchronize()
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def ordered(b):
    b = b.astype(np.int32)
    return np.where(b & 0x8000, -(b & 0x7FFF), b)


def assert_view(v, ref, what):
    torch.cuda.synchronize()
    codes = unpack_codes(v.codes.cpu().numpy())
    scales = unswizzle_scales(v.scales.cpu().numpy(), v.rows, v.cols, ref["bs"])
    assert np.array_equal(codes, ref["codes"]), f"{what}: {np.sum(codes != ref['codes'])} code mismatches"
    assert np.array_equal(scales, ref["scales"]), f"{what}: scale mismatch"
    if ref["senc"] is not None:
        assert np.array_equal(expand_outer(v.outer.cpu().numpy(), v.outer_count, v.rows), ref["senc"]), what


@pytest.mark.parametrize("route", ["mx", "nv_global", "nv_local"])
def test_rmsnorm_forward(route):
    R, C = 256, 512
    r = normal_bf16((R, C), 1.0, 21, 1)
    b = normal_bf16((R, C), 0.5, 21, 2)
    g = normal_bf16((C,), 1.0, 21, 3)
    tap = torch.empty((R, C), dtype=torch.bfloat16, device="cuda")
    rp, rstd, yr, yc = F.fp4_residual_rmsnorm_fwd(to_dev(r), to_dev(b), to_dev(g), route, y_tap=tap)
    o_rp, o_rstd, _ = oracle.residual_rmsnorm(r, b, g, 1e-5)
    assert np.array_equal(bits(rp), o_rp), "r' must be the exact bf16 residual"
    g_rstd = rstd.cpu().numpy()
    ulps = np.abs(g_rstd.view(np.int32) - o_rstd.view(np.int32))
    assert ulps.max() <= 2, f"rstd differs by {ulps.max()} ulp"
    # y from the kernel's own row statistic is bit-exact
    _, _, y_ref = oracle.residual_rmsnorm(r, b, g, 1e-5, rstd_in=g_rstd)
    y = bits(tap)
    assert np.array_equal(y, y_ref)
    assert_view(yr, oracle.quantize(y, route, "row"), f"{route} y row")
    assert_view(yc, oracle.quantize(y, route, "col"), f"{route} y col")
    assert F.fp4_status() == F.FP4_OK


@pytest.mark.parametrize("route", ["mx", "nv_local"])
def test_rmsnorm_backward(route):
    R, C = 256, 512
    rp = normal_bf16((R, C), 1.0, 22, 1)
    g = normal_bf16((C,), 1.0, 22, 2)
    dy = normal_bf16((R, C), 1e-3, 22, 3)
    dres = normal_bf16((R, C), 1e-3, 22, 4)
    rstd = (1.0 / np.sqrt((oracle.bf16_to_f32(rp).astype(np.float64) ** 2).mean(1) + 1e-5)).astype(np.float32)
    dr, drr, drc = F.fp4_residual_rmsnorm_bwd(to_dev(dy), to_dev(rp), torch.from_numpy(rstd).cuda(), to_dev(g),
                                              to_dev(dres), route, sr=True, sr_seed=9, sr_offset=4)
    got = bits(dr)
    want = oracle.rmsnorm_bwd(dy, rp, rstd, g, dres)
    d = np.abs(ordered(got) - ordered(want))
    assert d.max() <= 1, f"dr differs by up to {d.max()} bf16 ulp"
    assert (d > 0).mean() < 0.02
    assert_view(drr, oracle.quantize(got, route, "row", sr=True, seed=9, offset=4), f"{route} dr row")
    assert_view(drc, oracle.quantize(got, route, "col"), f"{route} dr col")
    assert F.fp4_status() == F.FP4_OK
