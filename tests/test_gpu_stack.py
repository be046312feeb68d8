"""Wiring of the depth-hybrid block stack (Format-Aware Fusion for Fast FP4
Pretraining, Sec. 3.3) at small shapes: one CTA-local NVFP4 block followed by
one MXFP4 block.

Every producer and contraction the stack calls has its own parity test
against the oracle.  What this test adds is that the stack feeds each call
the right operands: after one step, each boundary of each block is run again
through the same entry point on the tensors the stack retained, and its
result must equal what the stack kept, bit for bit (the kernels are
deterministic).  The residual hand-off between the blocks, the producers'
views, the QKV contraction, the attention stand-in and all four weight
gradients of both blocks are covered this way."""
import numpy as np
import pytest
import torch

import fp4_quantized_linears_gb300 as F
from fp4_quantized_linears_gb300.stack import BlockShape, FP4LinearStack
from synthetic import normal_bf16

pytestmark = pytest.mark.gpu


def same_view(a: F.QView, b: F.QView, what: str):
    torch.cuda.synchronize()
    assert torch.equal(a.codes, b.codes), f"{what}: codes"
    assert torch.equal(a.scales, b.scales), f"{what}: scales"
    if a.outer is not None:
        assert torch.equal(a.outer[:a.outer_count], b.outer[:b.outer_count]), f"{what}: outer factors"


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
    b0, b1 = st.blocks
    d, f = sh.d, sh.f
    # forward: the first producer sees x, the second block sees r2 + f of the first
    assert torch.equal(b0.s["r1"], x)
    for blk, h_in, f_in in ((b0, x, None), (b1, b0.s["r2"], b0.s["f"])):
        s, wv, r = blk.s, blk.wv, blk.route
        r1, rstd1, y1r, y1c = F.fp4_residual_rmsnorm_fwd(h_in, f_in, st.g1, r, eps=st.eps)
        assert torch.equal(r1, s["r1"]) and torch.equal(rstd1, s["rstd1"]), f"{r} r1"
        same_view(y1r, s["y1"][0], f"{r} y1 row")
        same_view(y1c, s["y1"][1], f"{r} y1 col")
        for name in ("qkv", "o", "w13", "w2"):
            wr, wc = F.fp4_quantize(blk.w[name], r, 3, F.FP4_FLAG_WEIGHT_2D)
            same_view(wr, wv[name][0], f"{r} W{name} row")
            same_view(wc, wv[name][1], f"{r} W{name} col")
        qkv = F.fp4_linear_fprop(s["y1"][0], wv["qkv"][0], out_dtype=F.FP4_OUT_BF16)
        assert torch.equal(qkv, s["qkv"]), f"{r} QKV"
        ar, ac = F.fp4_quantize(s["qkv"][:, :d].contiguous(), r, 3)
        same_view(ar, s["attn"][0], f"{r} attention stand-in row")
        same_view(ac, s["attn"][1], f"{r} attention stand-in col")
        o = F.fp4_linear_fprop(s["attn"][0], wv["o"][0], out_dtype=F.FP4_OUT_BF16)
        assert torch.equal(o, s["o"]), f"{r} O"
        r2, rstd2, y2r, y2c = F.fp4_residual_rmsnorm_fwd(s["r1"], s["o"], st.g2, r, eps=st.eps)
        assert torch.equal(r2, s["r2"]) and torch.equal(rstd2, s["rstd2"]), f"{r} r2"
        same_view(y2r, s["y2"][0], f"{r} y2 row")
        same_view(y2c, s["y2"][1], f"{r} y2 col")
        tap = torch.empty((sh.T, f), dtype=torch.bfloat16, device="cuda")
        a1, a3, _, _ = F.fp4_swiglu_fwd(s["y2"][0], wv["w13"][0], f, h_tap=tap, quantize=False)
        assert torch.equal(a1, s["a1"]) and torch.equal(a3, s["a3"]), f"{r} a1, a3"
        hr, hc = F.fp4_quantize(tap, r, 3)
        same_view(hr, s["h"][0], f"{r} h row")
        same_view(hc, s["h"][1], f"{r} h col")
        ff = F.fp4_linear_fprop(s["h"][0], wv["w2"][0], out_dtype=F.FP4_OUT_BF16)
        assert torch.equal(ff, s["f"]), f"{r} W2 Fprop"
    # backward: each weight gradient from the retained gradient views of its block
    for blk in (b0, b1):
        s, gv, dw, r = blk.s, st.gviews[blk.route], blk.dw, blk.route
        for name, a, b in (("w2", gv["dF"][1], s["h"][1]), ("w13", gv["da13"][1], s["y2"][1]),
                           ("o", gv["dr2"][1], s["attn"][1]), ("qkv", gv["dqkv"][1], s["y1"][1])):
            assert torch.equal(F.fp4_linear_wgrad(a, b), dw[name]), f"{r} dW{name}"
        # the stand-in's K and V gradient columns are zero
        torch.cuda.synchronize()
        dq = gv["dqkv"][0].codes.cpu().numpy()
        assert (dq[:, d // 2:] & 0x77 == 0).all()


def test_graph_replay_equals_eager_steps():
    """Two steps recorded into a CUDA graph and replayed give the same bits
    as the same two steps (same step indices, so the same stochastic
    rounding) launched eagerly: the graph path runs the same kernels."""
    sh = BlockShape(T=256, d=256, f=512, qkv=512)
    st = FP4LinearStack(2, 1, sh, seed=7)
    x = torch.from_numpy(normal_bf16((sh.T, sh.d), 1.0, 52, 1).view(np.int16)).view(torch.bfloat16).cuda()
    dy = torch.from_numpy(normal_bf16((sh.T, sh.d), 1e-2, 52, 2).view(np.int16)).view(torch.bfloat16).cuda()
    st.step(x, dy, sr_seed=4)  # one eager step: the library's one-time setup
    first = st.step_index
    graph = st.capture_steps(x, dy, 2, sr_seed=4)
    assert st.step_index == first + 2
    graph.replay()
    torch.cuda.synchronize()
    assert F.fp4_status() == F.FP4_OK

    def snapshot():
        torch.cuda.synchronize()
        out = [st.dr1[0].clone(), st.dr1[1].clone()]
        for blk in st.blocks:
            out += [blk.dw[n].clone() for n in ("qkv", "o", "w13", "w2")]
            out += [blk.s["a1"].clone(), blk.s["f"].clone()]
        for gv in st.gviews.values():
            out += [gv["da13"][0].codes.clone(), gv["da13"][0].scales.clone()]
        return out

    replayed = snapshot()
    st.step_index = first
    st.step(x, dy, sr_seed=4)
    st.step(x, dy, sr_seed=4)
    eager = snapshot()
    assert F.fp4_status() == F.FP4_OK
    for i, (a, b) in enumerate(zip(replayed, eager)):
        assert torch.equal(a, b), f"tensor {i} differs between the graph replay and the eager steps"
