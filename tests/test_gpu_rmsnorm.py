"""GPU parity of the residual-RMSNorm producer (Format-Aware Fusion for Fast
FP4 Pretraining, Sec. 3.2) against the oracle run on the host inputs alone.
The residual r' is exact; the FP32 row statistic may differ from the
oracle's binary64 one by an ulp (the kernel sums in a tree), so y is exact on
the rows whose statistic agrees and within one bf16 ulp elsewhere; the FP4
views are bit for bit in every scale block whose BF16 inputs agree with the
oracle's and a valid encoding of the kernel's values in the others."""
import numpy as np
import pytest
import torch

import oracle
import fp4_quantized_linears_gb300 as F
from masked import assert_view_masked, oriented
from masked import host_view as mhost
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


@pytest.mark.parametrize("route", ["mx", "nv_global", "nv_local"])
def test_rmsnorm_forward(route):
    R, C = 256, 512
    r = normal_bf16((R, C), 1.0, 21, 1)
    b = normal_bf16((R, C), 0.5, 21, 2)
    g = normal_bf16((C,), 1.0, 21, 3)
    tap = torch.empty((R, C), dtype=torch.bfloat16, device="cuda")
    rp, rstd, yr, yc = F.fp4_residual_rmsnorm_fwd(to_dev(r), to_dev(b), to_dev(g), route, y_tap=tap)
    assert F.fp4_status() == F.FP4_OK
    o_rp, o_rstd, o_y = oracle.residual_rmsnorm(r, b, g, 1e-5)
    assert np.array_equal(bits(rp), o_rp), "r' must be the exact bf16 residual"
    g_rstd = rstd.cpu().numpy()
    ulps = np.abs(g_rstd.view(np.int32) - o_rstd.view(np.int32))
    assert ulps.max() <= 2, f"rstd differs by {ulps.max()} ulp"
    # rows whose FP32 statistic equals the oracle's give the oracle's y exactly
    y = bits(tap)
    same_row = g_rstd == o_rstd
    assert np.array_equal(y[same_row], o_y[same_row])
    d = np.abs(ordered(y) - ordered(o_y))
    assert d.max() <= 1
    same = y == o_y
    assert_view_masked(mhost(yr), oracle.quantize(o_y, route, "row"), y, same, f"{route} y row")
    assert_view_masked(mhost(yc), oracle.quantize(o_y, route, "col"), oriented(y, "col"), oriented(same, "col"),
                       f"{route} y col")


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
    assert F.fp4_status() == F.FP4_OK
    got = bits(dr)
    want = oracle.rmsnorm_bwd(dy, rp, rstd, g, dres)
    d = np.abs(ordered(got) - ordered(want))
    assert d.max() <= 1, f"dr differs by up to {d.max()} bf16 ulp"
    assert (d > 0).mean() < 0.02
    same = got == want
    assert_view_masked(mhost(drr), oracle.quantize(want, route, "row", sr=True, seed=9, offset=4), got, same,
                       f"{route} dr row")
    assert_view_masked(mhost(drc), oracle.quantize(want, route, "col"), oriented(got, "col"), oriented(same, "col"),
                       f"{route} dr col")


def row_terms_host(dx_bits, rp, rstd, g):
    """The row terms' definition, per 64-column block in column order:
    sum of fl32(dx * g) * fl32(r' * rstd) (products rounded to binary32, the
    sum kept in binary64 here; the kernel's fused multiply-adds round each
    step to binary32, so the two agree to a few binary32 ulps of the sum of
    magnitudes)."""
    dx = oracle.bf16_to_f32(dx_bits)
    a = (dx * oracle.bf16_to_f32(g)[None, :]).astype(np.float32)
    b = (oracle.bf16_to_f32(rp) * rstd[:, None]).astype(np.float32)
    t = a.astype(np.float64) * b.astype(np.float64)
    R, C = t.shape
    return t.reshape(R, C // 64, 64).sum(2), np.abs(t).reshape(R, C // 64, 64).sum(2)


@pytest.mark.parametrize("route,T,K,d", [("mx", 256, 512, 512), ("nv_local", 256, 512, 512),
                                         ("mx", 384, 256, 384), ("nv_global", 384, 256, 384)])
def test_dgrad_emits_rmsnorm_row_terms(route, T, K, d):
    """fp4_linear_dgrad_rmsnorm: dx bit for bit the plain bf16 Dgrad's, and
    the per-block row terms of the adjacent RMSNorm backward (Sec. 3.2) over
    exactly those bf16 values (wide pair tiles and 128-wide single tiles)."""
    dyg = normal_bf16((T, K), 1e-2, 23, 1)
    w = normal_bf16((K, d), 0.05, 23, 2)
    rp = normal_bf16((T, d), 1.0, 23, 3)
    g = normal_bf16((d,), 1.0, 23, 4)
    rstd = (1.0 / np.sqrt((oracle.bf16_to_f32(rp).astype(np.float64) ** 2).mean(1) + 1e-5)).astype(np.float32)
    dr_, _ = F.fp4_quantize(to_dev(dyg), route, F.FP4_VIEW_ROW, F.FP4_FLAG_SR_ROW, sr_seed=5, sr_offset=1)
    _, wc = F.fp4_quantize(to_dev(w), route, F.FP4_VIEW_COL, F.FP4_FLAG_WEIGHT_2D)
    plain = F.fp4_linear_dgrad(dr_, wc, out_dtype=F.FP4_OUT_BF16)
    dx, part = F.fp4_linear_dgrad_rmsnorm(dr_, wc, to_dev(rp), torch.from_numpy(rstd).cuda(), to_dev(g))
    torch.cuda.synchronize()
    assert F.fp4_status() == F.FP4_OK
    assert torch.equal(dx, plain), "dx differs from the plain Dgrad"
    want, mag = row_terms_host(bits(dx), rp, rstd, g)
    got = part.cpu().numpy().astype(np.float64)
    assert got.shape == (T, d // 64)
    assert (np.abs(got - want) <= 64 * 2.0 ** -24 * mag + 1e-30).all()


@pytest.mark.parametrize("route", ["mx", "nv_local"])
def test_rmsnorm_backward_from_row_terms(route):
    """The RMSNorm backward fed by the Dgrad's row terms against the oracle's
    backward of the same dy, with the checks of the plain backward."""
    T, K, d = 256, 512, 512
    dyg = normal_bf16((T, K), 1e-2, 24, 1)
    w = normal_bf16((K, d), 0.05, 24, 2)
    rp = normal_bf16((T, d), 1.0, 24, 3)
    g = normal_bf16((d,), 1.0, 24, 4)
    dres = normal_bf16((T, d), 1e-3, 24, 5)
    rstd = (1.0 / np.sqrt((oracle.bf16_to_f32(rp).astype(np.float64) ** 2).mean(1) + 1e-5)).astype(np.float32)
    dr_, _ = F.fp4_quantize(to_dev(dyg), route, F.FP4_VIEW_ROW, F.FP4_FLAG_SR_ROW, sr_seed=6, sr_offset=1)
    _, wc = F.fp4_quantize(to_dev(w), route, F.FP4_VIEW_COL, F.FP4_FLAG_WEIGHT_2D)
    rs_dev = torch.from_numpy(rstd).cuda()
    dx, part = F.fp4_linear_dgrad_rmsnorm(dr_, wc, to_dev(rp), rs_dev, to_dev(g))
    dr, drr, drc = F.fp4_residual_rmsnorm_bwd_parts(dx, part, to_dev(rp), rs_dev, to_dev(g), to_dev(dres), route,
                                                    sr=True, sr_seed=9, sr_offset=4)
    assert F.fp4_status() == F.FP4_OK
    got = bits(dr)
    want = oracle.rmsnorm_bwd(bits(dx), rp, rstd, g, dres)
    d_ = np.abs(ordered(got) - ordered(want))
    assert d_.max() <= 1, f"dr differs by up to {d_.max()} bf16 ulp"
    assert (d_ > 0).mean() < 0.02
    same = got == want
    assert_view_masked(mhost(drr), oracle.quantize(want, route, "row", sr=True, seed=9, offset=4), got, same,
                       f"{route} dr row")
    assert_view_masked(mhost(drc), oracle.quantize(want, route, "col"), oriented(got, "col"), oriented(same, "col"),
                       f"{route} dr col")


def test_dgrad_rmsnorm_arguments_are_checked():
    dyg = normal_bf16((128, 256), 1e-2, 25, 1)
    w = normal_bf16((256, 256), 0.05, 25, 2)
    dr_, _ = F.fp4_quantize(to_dev(dyg), "mx", F.FP4_VIEW_ROW)
    _, wc = F.fp4_quantize(to_dev(w), "mx", F.FP4_VIEW_COL, F.FP4_FLAG_WEIGHT_2D)
    rp = to_dev(normal_bf16((128, 256), 1.0, 25, 3))
    g = to_dev(normal_bf16((256,), 1.0, 25, 4))
    rstd = torch.ones(128, device="cuda")
    with pytest.raises(F.Fp4Error) as e:  # r' one element off its 16-byte alignment
        F.fp4_linear_dgrad_rmsnorm(dr_, wc, rp.view(-1)[1:].view(-1), rstd, g)
    assert e.value.code == F.FP4_ERR_INVALID_ARG
