"""GPU parity of the fused gated-FFN producers (Format-Aware Fusion for Fast
FP4 Pretraining, Sec. 3.2).  Two levels: the retained BF16 values (a1, a3,
dh) against the oracle's binary64 contraction rounded to bf16 (<= 1 ulp, the
FP32 accumulation can move a tie), the gate values (h, da1, da3) against the
oracle's model arithmetic on the kernel's own retained values (<= 1 ulp:
the device exp differs from the binary64 one), and the FP4 views bit for bit
against the oracle quantizing the very BF16 values the kernel quantized."""
import numpy as np
import pytest
import torch

import oracle
import fp4_quantized_linears_gb300 as F
from layout import expand_outer, unpack_codes, unswizzle_scales
from synthetic import normal_bf16

pytestmark = pytest.mark.gpu


def to_dev(b):
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).cuda()


def bits(t):
    torch.cuda.synchronize()
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def ordered(b):
    b = b.astype(np.int32)
    return np.where(b & 0x8000, -(b & 0x7FFF), b)


def ulp(a, b):
    return np.abs(ordered(a) - ordered(b))


def host_view(v, route):
    torch.cuda.synchronize()
    bs, fmt = (32, 0) if route == "mx" else (16, 1)
    return dict(codes=unpack_codes(v.codes.cpu().numpy()),
                scales=unswizzle_scales(v.scales.cpu().numpy(), v.rows, v.cols, bs),
                senc=None if v.outer is None else expand_outer(v.outer.cpu().numpy(), v.outer_count, v.rows),
                fmt=fmt, bs=bs)


def assert_view(v, ref, what):
    h = host_view(v, "mx" if ref["fmt"] == 0 else "nv")
    assert np.array_equal(h["codes"], ref["codes"]), f"{what}: {np.sum(h['codes'] != ref['codes'])} code mismatches"
    assert np.array_equal(h["scales"], ref["scales"]), f"{what}: scale mismatch"


def check_bf16_gemm(got_bits, ref_f64, absref, what, max_frac=0.02):
    """A bf16-rounded FP32 contraction against the binary64 one: within one
    bf16 ulp of the reference plus the contraction tolerance 2^-18 sum|ab|
    (a cancelling sum can land on the other side of a tie, or on zero)."""
    got = oracle.bf16_to_f32(got_bits).astype(np.float64)
    ulp_ref = np.maximum(np.abs(ref_f64), 2.0 ** -126) * 2.0 ** -7
    err = np.abs(got - ref_f64)
    bound = ulp_ref + 2.0 ** -18 * absref
    assert (err <= bound).all(), f"{what}: max err/bound {(err / bound).max():.3f}"
    d = ulp(got_bits, oracle.round_bf16(ref_f64))
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
    qx, qw = host_view(xr, route), host_view(wr, route)
    qw1 = {k: (v[:f] if isinstance(v, np.ndarray) else v) for k, v in qw.items()}
    qw3 = {k: (v[f:] if isinstance(v, np.ndarray) else v) for k, v in qw.items()}
    check_bf16_gemm(bits(a1), oracle.gemm(qx, qw1), oracle.gemm_abs(qx, qw1), "a1")
    check_bf16_gemm(bits(a3), oracle.gemm(qx, qw3), oracle.gemm_abs(qx, qw3), "a3")
    h = bits(tap)
    d_h = ulp(h, oracle.swiglu_h(bits(a1), bits(a3)))
    assert d_h.max() <= 1 and (d_h > 0).mean() < 0.01
    if route == "mx":
        assert_view(hr, oracle.quantize(h, "mx", "row"), "Q_r(h)")
        assert_view(hc, oracle.quantize(h, "mx", "col"), "Q_c(h)")
    else:
        assert hr is None and hc is None


@pytest.mark.parametrize("route", ["mx", "nv_local"])
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
    dh = bits(dh_tap)
    hd, hw = host_view(dr, route), host_view(wc, route)
    check_bf16_gemm(dh, oracle.gemm(hd, hw), oracle.gemm_abs(hd, hw), "dh")
    da = bits(da_tap)
    o1, o3 = oracle.swiglu_bwd(dh, a1, a3)
    for got, want, name in ((da[:, :f], o1, "da1"), (da[:, f:], o3, "da3")):
        dd = ulp(np.ascontiguousarray(got), want)
        assert dd.max() <= 1 and (dd > 0).mean() < 0.01, name
    if route == "mx":
        assert_view(rr, oracle.quantize(da, "mx", "row", sr=True, seed=77, offset=5), "Q_r(da13)")
        assert_view(cc, oracle.quantize(da, "mx", "col"), "Q_c(da13)")
    else:
        assert rr is None and cc is None


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
