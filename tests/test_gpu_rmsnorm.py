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
