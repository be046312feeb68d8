"""GPU parity of the QKV producer with RoPE (Format-Aware Fusion for Fast FP4
Pretraining, Sec. 3.2) against the oracle run on host inputs.

Forward: q, k (turned) and v (head-major) from the fused QKV projection are
compared with the oracle's binary64 contraction of its own operand views
turned in binary64: within two bf16 rounding steps (the contraction's
output and the turned value) plus the contraction tolerance 2^-18 sum|ab|.
Backward: the QKV-layout gradient (dq, dk turned back, dv copied) is
bit-exact against the oracle, and so are its FP4 views."""
import numpy as np
import pytest
import torch

import oracle
import fp4_quantized_linears_gb300 as F
from masked import host_view as mhost
from synthetic import normal_bf16, with_outliers_bf16

pytestmark = pytest.mark.gpu

D = 128


def to_dev(b):
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).cuda()


def bits(t):
    torch.cuda.synchronize()
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def same_view(v, want, what):
    got = mhost(v)
    assert np.array_equal(got["codes"], want["codes"]), f"{what}: codes"
    assert np.array_equal(got["scales"], want["scales"]), f"{what}: scales"
    if want["senc"] is not None:
        assert np.array_equal(got["senc"], want["senc"]), f"{what}: outer factors"


@pytest.mark.parametrize("route", ["mx", "nv_global", "nv_local"])
def test_qkv_rope_forward(route):
    T, S, d, hq, hkv = 384, 128, 256, 4, 2
    N = (hq + 2 * hkv) * D
    x = with_outliers_bf16((T, d), 1.0, 1e-3, 20.0, 91, 1)
    w = normal_bf16((N, d), 0.05, 91, 2)
    xr, _ = F.fp4_quantize(to_dev(x), route, F.FP4_VIEW_ROW)
    wr, _ = F.fp4_quantize(to_dev(w), route, F.FP4_VIEW_ROW, F.FP4_FLAG_WEIGHT_2D)
    c, s = oracle.rope_tables(S, D)
    q, k, v = F.fp4_qkv_rope_fwd(xr, wr, torch.from_numpy(c).cuda(), torch.from_numpy(s).cuda(), S, hq, hkv)
    torch.cuda.synchronize()
    assert F.fp4_status() == F.FP4_OK
    ox = oracle.quantize(x, route, "row")
    ow = oracle.quantize(w, route, "row", weight2d=True)
    ref, absref = oracle.gemm(ox, ow), oracle.gemm_abs(ox, ow)   # [T][N] binary64
    pos = np.arange(T) % S
    cp, sp = c[pos].astype(np.float64), s[pos].astype(np.float64)
    heads = [(q[h], h) for h in range(hq)] + [(k[h], hq + h) for h in range(hkv)]
    for got_t, col in heads:
        a, b = ref[:, col * D:col * D + 64], ref[:, col * D + 64:(col + 1) * D]
        aa, ab = absref[:, col * D:col * D + 64], absref[:, col * D + 64:(col + 1) * D]
        want = np.concatenate([a * cp - b * sp, b * cp + a * sp], axis=1)
        # each half's own magnitude: |a||c| + |b||s| for the first, |b||c| + |a||s| for the second
        mag = np.concatenate([np.abs(a) * np.abs(cp) + np.abs(b) * np.abs(sp),
                              np.abs(b) * np.abs(cp) + np.abs(a) * np.abs(sp)], axis=1)
        tol = np.concatenate([aa * np.abs(cp) + ab * np.abs(sp), ab * np.abs(cp) + aa * np.abs(sp)], axis=1)
        got = oracle.bf16_to_f32(bits(got_t)).astype(np.float64)
        bound = 2.0 ** -7 * mag + 2.0 ** -17 * tol + 1e-30
        assert (np.abs(got - want) <= bound).all(), f"{route} head {col}: max err/bound {(np.abs(got - want) / bound).max():.2f}"
    for h in range(hkv):
        col = hq + hkv + h
        want = ref[:, col * D:(col + 1) * D]
        got = oracle.bf16_to_f32(bits(v[h])).astype(np.float64)
        bound = 2.0 ** -8 * np.abs(want) + 2.0 ** -18 * absref[:, col * D:(col + 1) * D] + 1e-30
        assert (np.abs(got - want) <= bound).all(), f"{route} v head {h}"


@pytest.mark.parametrize("route", ["mx", "nv_global", "nv_local"])
def test_qkv_rope_backward_producer(route):
    T, S, hq, hkv = 256, 128, 4, 2
    dq = normal_bf16((hq, T, D), 1e-3, 92, 1)
    dk = normal_bf16((hkv, T, D), 1e-3, 92, 2)
    dv = normal_bf16((hkv, T, D), 1e-3, 92, 3)
    c, s = oracle.rope_tables(S, D)
    tap = torch.empty((T, (hq + 2 * hkv) * D), dtype=torch.bfloat16, device="cuda")
    rr, cc = F.fp4_qkv_rope_bwd(to_dev(dq), to_dev(dk), to_dev(dv), torch.from_numpy(c).cuda(),
                                torch.from_numpy(s).cuda(), S, route, 3, sr=True, sr_seed=13, sr_offset=2,
                                dqkv_tap=tap)
    torch.cuda.synchronize()
    assert F.fp4_status() == F.FP4_OK
    want = oracle.qkv_rope_bwd(dq, dk, dv, S, c, s)
    assert np.array_equal(bits(tap), want), "dQKV"
    same_view(rr, oracle.quantize(want, route, "row", sr=True, seed=13, offset=2), f"{route} dQKV row")
    same_view(cc, oracle.quantize(want, route, "col"), f"{route} dQKV col")


def test_qkv_rope_shapes_are_checked():
    x = normal_bf16((128, 256), 1.0, 93, 1)
    w = normal_bf16((3 * D, 256), 0.05, 93, 2)  # hq + 2 hkv = 3 heads: 384 columns, not a multiple of 256
    xr, _ = F.fp4_quantize(to_dev(x), "mx", F.FP4_VIEW_ROW)
    wr, _ = F.fp4_quantize(to_dev(w), "mx", F.FP4_VIEW_ROW, F.FP4_FLAG_WEIGHT_2D)
    c, s = oracle.rope_tables(128, D)
    with pytest.raises(F.Fp4Error) as e:
        F.fp4_qkv_rope_fwd(xr, wr, torch.from_numpy(c).cuda(), torch.from_numpy(s).cuda(), 128, 1, 1)
    assert e.value.code == F.FP4_ERR_UNSUPPORTED_SHAPE
