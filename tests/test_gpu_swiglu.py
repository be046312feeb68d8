"""GPU parity of the fused gated-FFN producers (Format-Aware Fusion for Fast
FP4 Pretraining, Sec. 3.2), against the oracle's chain computed from the host
inputs alone: the retained BF16 values (a1, a3, dh) within one bf16 ulp of
the oracle's binary64 contraction rounded to bf16 (the FP32 accumulation can
move a tie); the gate values (h, da1, da3) within one ulp of the oracle's
where their inputs agree (the device exp differs from the binary64 one); the
FP4 views bit for bit in every scale block whose BF16 inputs agree, and a
valid encoding of the kernel's values in the few blocks that do not."""
import numpy as np
import pytest
import torch

import oracle
import fp4_quantized_linears_gb300 as F
from masked import assert_view_masked, oriented
from masked import host_view as mhost
from synthetic import normal_bf16
from parity_stats import record

pytestmark = pytest.mark.gpu


def to_dev(b):
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).cuda()


def bits(t):
    torch.cuda.synchronize()
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def ordered(b):
    b = b.astype(np.int32)
    return np.where(b & 0x8000, -(b & 0x7FFF), b)


def same_views(a, b, what):
    """Two GPU views of one tensor: codes, scales and outer factors equal."""
    torch.cuda.synchronize()
    assert torch.equal(a.codes, b.codes), f"{what}: codes"
    assert torch.equal(a.scales, b.scales), f"{what}: scales"
    if a.outer is not None or b.outer is not None:
        assert torch.equal(a.outer[:a.outer_count], b.outer[:b.outer_count]), f"{what}: outer factors"


def ulp(a, b):
    return np.abs(ordered(a) - ordered(b))


def check_bf16_gemm(got_bits, ref_f64, absref, what, max_frac=4e-5):
    """A bf16-rounded FP32 contraction against the binary64 one: within one
    bf16 ulp of the reference plus the contraction tolerance 2^-18 sum|ab|
    (a cancelling sum can land on the other side of a tie, or on zero)."""
    got = oracle.bf16_to_f32(got_bits).astype(np.float64)
    ulp_ref = np.maximum(np.abs(ref_f64), 2.0 ** -126) * 2.0 ** -7
    err = np.abs(got - ref_f64)
    bound = ulp_ref + 2.0 ** -18 * absref
    d = ulp(got_bits, oracle.round_bf16(ref_f64))
    record(what, err_over_bound=(err / bound).max(), frac_not_bf16_of_ref=(d > 0).mean())
    assert (err <= bound).all(), f"{what}: max err/bound {(err / bound).max():.3f}"
    assert (d > 0).mean() <= max_frac, f"{what}: {(d > 0).mean():.3%} of values differ from bf16(reference)"


@pytest.mark.parametrize("route", ["mx", "nv_global", "nv_local"])
@pytest.mark.parametrize("T", [256, 384])
def test_swiglu_forward(route, T):
    d, f = 256, 256
    x = normal_bf16((T, d), 1.0, 31, 1)
    w13 = normal_bf16((2 * f, d), 0.05, 31, 2)
    xr, _ = F.fp4_quantize(to_dev(x), route, F.FP4_VIEW_ROW)
    wr, _ = F.fp4_quantize(to_dev(w13), route, F.FP4_VIEW_ROW, F.FP4_FLAG_WEIGHT_2D)
    tap = torch.empty((T, f), dtype=torch.bfloat16, device="cuda")
    a1, a3, hr, hc = F.fp4_swiglu_fwd(xr, wr, f, h_tap=tap)
    assert F.fp4_status() == F.FP4_OK
    # the oracle's chain from the host inputs alone
    qx = oracle.quantize(x, route, "row")
    qw = oracle.quantize(w13, route, "row", weight2d=True)
    qw1 = {k: (v[:f] if isinstance(v, np.ndarray) else v) for k, v in qw.items()}
    qw3 = {k: (v[f:] if isinstance(v, np.ndarray) else v) for k, v in qw.items()}
    c1, c3 = oracle.gemm(qx, qw1), oracle.gemm(qx, qw3)
    o_a1, o_a3 = oracle.round_bf16(c1), oracle.round_bf16(c3)
    o_h = oracle.swiglu_h(o_a1, o_a3)
    g_a1, g_a3, g_h = bits(a1), bits(a3), bits(tap)
    check_bf16_gemm(g_a1, c1, oracle.gemm_abs(qx, qw1), "a1")
    check_bf16_gemm(g_a3, c3, oracle.gemm_abs(qx, qw3), "a3")
    # where the contraction rounded alike, the gate value is the oracle's up
    # to the device exponential (<= 1 bf16 ulp, rarely)
    same_in = (g_a1 == o_a1) & (g_a3 == o_a3)
    d_h = ulp(g_h, o_h)[same_in]
    assert d_h.max() <= 1 and (d_h > 0).mean() < 0.01
    same_h = g_h == o_h
    assert_view_masked(mhost(hr), oracle.quantize(o_h, route, "row"), g_h, same_h, "Q_r(h)")
    assert_view_masked(mhost(hc), oracle.quantize(o_h, route, "col"), oriented(g_h, "col"),
                       oriented(same_h, "col"), "Q_c(h)")
    if route != "mx":
        # NVFP4: the maxima folded by the epilogue give exactly the encoding
        # of the tap by the plain producer, with or without a caller's tap
        qr, qc = F.fp4_quantize(tap, route, 3)
        same_views(hr, qr, "Q_r(h) vs the producer on the tap")
        same_views(hc, qc, "Q_c(h) vs the producer on the tap")
        _, _, hr2, hc2 = F.fp4_swiglu_fwd(xr, wr, f)
        same_views(hr2, hr, "Q_r(h) without a tap")
        same_views(hc2, hc, "Q_c(h) without a tap")


@pytest.mark.parametrize("route", ["mx", "nv_global", "nv_local"])
def test_swiglu_backward(route):
    T, d, f = 256, 256, 384
    dy2 = normal_bf16((T, d), 1e-2, 32, 1)
    w2 = normal_bf16((d, f), 0.05, 32, 2)
    a1 = normal_bf16((T, f), 2.0, 32, 3)
    a3 = normal_bf16((T, f), 2.0, 32, 4)
    dr, _ = F.fp4_quantize(to_dev(dy2), route, F.FP4_VIEW_ROW, F.FP4_FLAG_SR_ROW, sr_seed=3, sr_offset=1)
    _, wc = F.fp4_quantize(to_dev(w2), route, F.FP4_VIEW_COL, F.FP4_FLAG_WEIGHT_2D)
    dh_tap = torch.empty((T, f), dtype=torch.bfloat16, device="cuda")
    da_tap = torch.empty((T, 2 * f), dtype=torch.bfloat16, device="cuda")
    rr, cc = F.fp4_swiglu_bwd(dr, wc, f, to_dev(a1), to_dev(a3), sr_seed=77, sr_offset=5, dh_tap=dh_tap,
                              da13_tap=da_tap)
    assert F.fp4_status() == F.FP4_OK
    # the oracle's chain from the host inputs alone
    qd = oracle.quantize(dy2, route, "row", sr=True, seed=3, offset=1)
    qw = oracle.quantize(w2, route, "col", weight2d=True)
    c = oracle.gemm(qd, qw)
    o_dh = oracle.round_bf16(c)
    o1, o3 = oracle.swiglu_bwd(o_dh, a1, a3)
    o_da = np.concatenate([o1, o3], axis=1)
    g_dh, g_da = bits(dh_tap), bits(da_tap)
    check_bf16_gemm(g_dh, c, oracle.gemm_abs(qd, qw), "dh")
    same_dh = np.concatenate([g_dh == o_dh] * 2, axis=1)
    dd = ulp(g_da, o_da)[same_dh]
    assert dd.max() <= 1 and (dd > 0).mean() < 0.01, "da13"
    same_da = g_da == o_da
    assert_view_masked(mhost(rr), oracle.quantize(o_da, route, "row", sr=True, seed=77, offset=5), g_da,
                       same_da, "Q_r(da13)")
    assert_view_masked(mhost(cc), oracle.quantize(o_da, route, "col"), oriented(g_da, "col"),
                       oriented(same_da, "col"), "Q_c(da13)")
    if route != "mx":
        qr, qc = F.fp4_quantize(da_tap, route, 3, F.FP4_FLAG_SR_ROW, sr_seed=77, sr_offset=5)
        same_views(rr, qr, "Q_r(da13) vs the producer on the tap")
        same_views(cc, qc, "Q_c(da13) vs the producer on the tap")
        rr2, cc2 = F.fp4_swiglu_bwd(dr, wc, f, to_dev(a1), to_dev(a3), sr_seed=77, sr_offset=5)
        same_views(rr2, rr, "Q_r(da13) without a tap")
        same_views(cc2, cc, "Q_c(da13) without a tap")


def test_swiglu_chain_matches_unfused_path():
    # fused forward views == quantizing the fused h tap; W2 Fprop on them runs
    T, d, f = 256, 256, 256
    x = normal_bf16((T, d), 1.0, 33, 1)
    w13 = normal_bf16((2 * f, d), 0.05, 33, 2)
    w2 = normal_bf16((d, f), 0.05, 33, 3)
    xr, _ = F.fp4_quantize(to_dev(x), "mx", F.FP4_VIEW_ROW)
    wr, _ = F.fp4_quantize(to_dev(w13), "mx", F.FP4_VIEW_ROW, F.FP4_FLAG_WEIGHT_2D)
    w2r, _ = F.fp4_quantize(to_dev(w2), "mx", F.FP4_VIEW_ROW, F.FP4_FLAG_WEIGHT_2D)
    tap = torch.empty((T, f), dtype=torch.bfloat16, device="cuda")
    _, _, hr, _ = F.fp4_swiglu_fwd(xr, wr, f, h_tap=tap)
    y_fused = F.fp4_linear_fprop(hr, w2r)
    hr2, _ = F.fp4_quantize(tap, "mx", F.FP4_VIEW_ROW)
    y_unfused = F.fp4_linear_fprop(hr2, w2r)
    assert torch.equal(y_fused, y_unfused)
