"""Wiring of the depth-hybrid block stack (Format-Aware Fusion for Fast FP4
Pretraining, Sec. 3.3) at small shapes: one CTA-local NVFP4 block followed by
one MXFP4 block.  Every individual producer and contraction has its own
parity test; this checks that the stack feeds each one the right operands,
using the tensors the GPU actually retained: the residual hand-off between
blocks, each producer's views, the QKV contraction, the attention stand-in
views and all four weight gradients of both blocks."""
import numpy as np
import pytest
import torch

import oracle
import fp4_quantized_linears_gb300 as F
from fp4_quantized_linears_gb300.stack import BlockShape, FP4LinearStack
from layout import expand_outer, unpack_codes, unswizzle_scales
from synthetic import normal_bf16

pytestmark = pytest.mark.gpu

REL_FRO = 1e-5


def host_view(v):
    torch.cuda.synchronize()
    bs, fmt = (32, 0) if v.route == F.FP4_ROUTE_MXFP4 else (16, 1)
    return dict(codes=unpack_codes(v.codes.cpu().numpy()),
                scales=unswizzle_scales(v.scales.cpu().numpy(), v.rows, v.cols, bs),
                senc=None if v.outer is None else expand_outer(v.outer.cpu().numpy(), v.outer_count, v.rows),
                fmt=fmt, bs=bs)


def bits(t):
    torch.cuda.synchronize()
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def rname(v):
    return "mx" if v.route == F.FP4_ROUTE_MXFP4 else "nv_local"


def same_view(v, ref, what):
    h = host_view(v)
    assert np.array_equal(h["codes"], ref["codes"]), f"{what}: codes"
    assert np.array_equal(h["scales"], ref["scales"]), f"{what}: scales"


def close_gemm(got, a, b, what):
    ref = oracle.gemm(a, b)
    absref = oracle.gemm_abs(a, b)
    err = np.abs(got.astype(np.float64) - ref)
    fro = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
    assert fro <= REL_FRO, f"{what}: rel Frobenius {fro:.2e}"
    assert (err <= 2.0 ** -18 * absref + 1e-30).all(), what


def test_two_block_hybrid_stack_wiring():
    sh = BlockShape(T=256, d=256, f=512, qkv=512)
    st = FP4LinearStack(2, 1, sh, seed=7)
    assert [b.route for b in st.blocks] == ["nv_local", "mx"]
    x = torch.from_numpy(normal_bf16((sh.T, sh.d), 1.0, 51, 1).view(np.int16)).view(torch.bfloat16).cuda()
    dy = torch.from_numpy(normal_bf16((sh.T, sh.d), 1e-2, 51, 2).view(np.int16)).view(torch.bfloat16).cuda()
    dx = st.step(x, dy, sr_seed=3)
    torch.cuda.synchronize()
    assert F.fp4_status() == F.FP4_OK
    assert torch.isfinite(dx.float()).all()
    g = bits(st.g1)
    b0, b1 = st.blocks
    # forward: the first producer sees x, the second block sees r2 + f of the first
    assert np.array_equal(bits(b0.s["r1"]), bits(x))
    want_r1 = oracle.round_bf16(oracle.bf16_to_f32(bits(b0.s["r2"])).astype(np.float64)
                                + oracle.bf16_to_f32(bits(b0.s["f"])).astype(np.float64))
    assert np.array_equal(bits(b1.s["r1"]), want_r1)
    for blk in (b0, b1):
        s, wv = blk.s, blk.wv
        route = blk.route
        # attention-side producer: y1 from r1 with the kernel's rstd
        _, _, y1 = oracle.residual_rmsnorm(bits(s["r1"]), np.zeros_like(bits(s["r1"])), g, 1e-5,
                                           rstd_in=s["rstd1"].cpu().numpy())
        same_view(s["y1"][0], oracle.quantize(y1, route, "row"), f"{route} y1 row")
        same_view(s["y1"][1], oracle.quantize(y1, route, "col"), f"{route} y1 col")
        # weights
        same_view(wv["qkv"][0], oracle.quantize(bits(blk.w["qkv"]), route, "row", weight2d=True), "Wqkv row")
        same_view(wv["w2"][1], oracle.quantize(bits(blk.w["w2"]), route, "col", weight2d=True), "W2 col")
        # QKV contraction (bf16 out) and the stand-in's views of its Q part
        qkv = oracle.bf16_to_f32(bits(s["qkv"])).astype(np.float64)
        ref = oracle.gemm(host_view(s["y1"][0]), host_view(wv["qkv"][0]))
        assert np.abs(qkv - ref).max() <= 2.0 ** -7 * np.abs(ref).max()
        q = np.ascontiguousarray(bits(s["qkv"])[:, :sh.d])
        same_view(s["attn"][0], oracle.quantize(q, route, "row"), "attn row")
        same_view(s["attn"][1], oracle.quantize(q, route, "col"), "attn col")
        # FFN-side producer: y2 from r2
        _, _, y2 = oracle.residual_rmsnorm(bits(s["r2"]), np.zeros_like(bits(s["r2"])), g, 1e-5,
                                           rstd_in=s["rstd2"].cpu().numpy())
        same_view(s["y2"][0], oracle.quantize(y2, route, "row"), f"{route} y2 row")
    # backward: weight gradients from the retained gradient views of each block
    for blk in (b0, b1):
        s, gv, dw = blk.s, st.gviews[blk.route], blk.dw
        dF = st.gviews[blk.route]["dF"]
        close_gemm(dw["w2"].cpu().numpy(), host_view(dF[1]), host_view(s["h"][1]), f"{blk.route} dW2")
        close_gemm(dw["w13"].cpu().numpy(), host_view(gv["da13"][1]), host_view(s["y2"][1]), f"{blk.route} dW13")
        close_gemm(dw["o"].cpu().numpy(), host_view(gv["dr2"][1]), host_view(s["attn"][1]), f"{blk.route} dWo")
        close_gemm(dw["qkv"].cpu().numpy(), host_view(gv["dqkv"][1]), host_view(s["y1"][1]), f"{blk.route} dWqkv")
        # the stand-in's K and V gradient columns are zero
        dq = host_view(gv["dqkv"][0])
        assert (dq["codes"][:, sh.d:] & 7 == 0).all()
