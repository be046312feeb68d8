"""A stack of Llama-3-shaped FP4 linear blocks driven through the C ABI.

This is the "27/5 depth hybrid" of "Format-Aware Fusion for Fast FP4
Pretraining" (Sec. 3.3): blocks [0, local_blocks) run CTA-local NVFP4 and the
rest MXFP4, each with 2D weights and stochastic rounding on the row-facing
gradient only; no Hadamard.  Each block is

    r1 = bf16(h + f_prev)            residual add        \\  residual-RMSNorm
    y1 = RMSNorm(r1)                 -> Q_r(y1), Q_c(y1)  /  producer
    qkv = Q_r(y1) Wqkv^T                                     (BF16 out)
    attn = qkv[:, :d]                attention stand-in (the Q projection)
    o = Q_r(attn) Wo^T
    r2 = bf16(r1 + o), y2 = RMSNorm(r2) -> Q_r(y2), Q_c(y2)
    a1, a3, Q(h) = SwiGLU producer(Q_r(y2), [W1; W3])       (Sec. 3.2)
    f = Q_r(h) W2^T

and the backward runs the same boundaries in reverse: the residual-RMSNorm
backward producer emits the residual gradient together with its FP4 views,
which are the output-gradient operands of the preceding linear; the SwiGLU
backward producer fuses the W2 data gradient with the SiLU derivative; the
data-gradient contractions that feed an RMSNorm backward (W1/W3 and QKV)
also emit that backward's row terms, so it never re-reads their output.

Only argument marshalling happens here: every step is a call into
libfp4lin.  Buffers are allocated once by the constructor (torch device
memory) and reused by every step.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

from . import (FP4_FLAG_SR_ROW, FP4_FLAG_WEIGHT_2D, FP4_OUT_BF16, FP4_VIEW_COL, FP4_VIEW_ROW, alloc_view,
               fp4_linear_dgrad, fp4_linear_dgrad_rmsnorm, fp4_linear_fprop, fp4_linear_wgrad, fp4_quantize,
               fp4_quantize_workspace_bytes, fp4_residual_rmsnorm_bwd_parts, fp4_residual_rmsnorm_fwd,
               fp4_rmsnorm_bwd_workspace_bytes, fp4_swiglu_bwd, fp4_swiglu_fwd, fp4_swiglu_workspace_bytes)


@dataclass
class BlockShape:
    T: int = 8192
    d: int = 4096
    f: int = 14336
    qkv: int = 6144


@dataclass
class _Block:
    route: str
    w: dict                              # bf16 weights
    wv: dict = field(default_factory=dict)  # quantized weight views
    dw: dict = field(default_factory=dict)  # FP32 weight gradients
    s: dict = field(default_factory=dict)   # saved forward state


def sr_offset(step: int, block: int, k: int) -> int:
    """Philox counter offset of stochastically rounded producer k of block
    `block` in training step `step`.  Seeds and counter offsets are state
    that must never repeat across steps (Sec. 2.5; Appendix A.1 keeps them in
    the checkpoint), so the step index fills the upper 32 bits and
    (block, producer) the lower ones: no two producers of a run share draws."""
    if not (0 <= step < (1 << 32) and 0 <= block < (1 << 27) and 0 <= k < 16):
        raise ValueError("SR offset out of range")
    return (step << 32) | (16 * block + k)


def linear_flops_per_token(sh: BlockShape) -> float:
    """Fprop + Dgrad + Wgrad FLOPs of one block's linears per token."""
    per = sh.d * sh.qkv + sh.d * sh.d + 2 * sh.d * sh.f + sh.f * sh.d
    return 6.0 * per


class FP4LinearStack:
    def __init__(self, n_blocks: int, local_blocks: int, shape: BlockShape = BlockShape(), seed: int = 5,
                 device="cuda", eps: float = 1e-5, weights=None):
        self.sh = shape
        self.eps = eps
        self.dev = torch.device(device)
        T, d, f, q = shape.T, shape.d, shape.f, shape.qkv
        self.blocks = []
        for b in range(n_blocks):
            route = "nv_local" if b < local_blocks else "mx"
            if weights is not None:
                w = weights[b]
            else:
                g = torch.Generator(device=self.dev).manual_seed(seed * 1000 + b)
                w = {k: (torch.randn(shp, generator=g, device=self.dev) * 0.02).to(torch.bfloat16)
                     for k, shp in (("qkv", (q, d)), ("o", (d, d)), ("w13", (2 * f, d)), ("w2", (d, f)))}
            self.blocks.append(_Block(route, w))
        self.g1 = torch.ones(d, dtype=torch.bfloat16, device=self.dev)
        self.g2 = torch.ones(d, dtype=torch.bfloat16, device=self.dev)
        self.step_index = 0          # training steps taken: part of every SR counter offset
        self.time_standin = False    # record CUDA events around the attention stand-in's copy
        self._standin_events = []
        self._alloc()

    # ------------------------------------------------------------ buffers --
    def _alloc(self):
        T, d, f, q = self.sh.T, self.sh.d, self.sh.f, self.sh.qkv
        dev = self.dev
        bf = dict(dtype=torch.bfloat16, device=dev)
        ws_bytes = 0
        for blk in self.blocks:
            r = blk.route
            for name, (R, C) in (("qkv", (q, d)), ("o", (d, d)), ("w13", (2 * f, d)), ("w2", (d, f))):
                blk.wv[name] = (alloc_view(r, R, C, FP4_FLAG_WEIGHT_2D, dev), alloc_view(r, C, R, FP4_FLAG_WEIGHT_2D, dev))
                blk.dw[name] = torch.empty((R, C), dtype=torch.float32, device=dev)
                ws_bytes = max(ws_bytes, fp4_quantize_workspace_bytes(r, R, C))
            s = blk.s
            s["r1"], s["r2"] = torch.empty((T, d), **bf), torch.empty((T, d), **bf)
            s["rstd1"] = torch.empty(T, dtype=torch.float32, device=dev)
            s["rstd2"] = torch.empty(T, dtype=torch.float32, device=dev)
            s["y1"] = (alloc_view(r, T, d, 0, dev), alloc_view(r, d, T, 0, dev))
            s["y2"] = (alloc_view(r, T, d, 0, dev), alloc_view(r, d, T, 0, dev))
            s["qkv"] = torch.empty((T, q), **bf)
            s["attn"] = (alloc_view(r, T, d, 0, dev), alloc_view(r, d, T, 0, dev))
            s["o"] = torch.empty((T, d), **bf)
            s["a1"], s["a3"] = torch.empty((T, f), **bf), torch.empty((T, f), **bf)
            s["h"] = (alloc_view(r, T, f, 0, dev), alloc_view(r, f, T, 0, dev))
            s["f"] = torch.empty((T, d), **bf)
            ws_bytes = max(ws_bytes, fp4_quantize_workspace_bytes(r, T, q), fp4_quantize_workspace_bytes(r, T, 2 * f),
                           fp4_rmsnorm_bwd_workspace_bytes(r, T, d), fp4_swiglu_workspace_bytes(r, T, f, True, True),
                           fp4_swiglu_workspace_bytes(r, T, f, False, True))
        self.ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
        # scratch shared by all blocks (used strictly in sequence)
        self.h_tap = torch.empty((T, f), **bf)       # NVFP4 SwiGLU: the bf16 copy of h the producer encodes
        self.da13 = torch.empty((T, 2 * f), **bf)    # NVFP4 SwiGLU backward: the bf16 copy of [da1 | da3]
        self.dqkv = torch.zeros((T, q), **bf)        # attention stand-in gradient (K, V parts stay 0)
        self.dattn = torch.empty((T, d), **bf)
        self.dy = torch.empty((T, d), **bf)
        self.part = torch.empty((T, d // 64), dtype=torch.float32, device=dev)  # RMSNorm row terms
        self.dr2 = torch.empty((T, d), **bf)                            # gradient of r2
        self.dr1 = [torch.empty((T, d), **bf) for _ in range(2)]        # gradient of r1, alternating
        self.gviews = {}
        for r in {b.route for b in self.blocks}:
            self.gviews[r] = dict(
                dF=(alloc_view(r, T, d, FP4_FLAG_SR_ROW, dev), alloc_view(r, d, T, 0, dev)),
                da13=(alloc_view(r, T, 2 * f, FP4_FLAG_SR_ROW, dev), alloc_view(r, 2 * f, T, 0, dev)),
                dr2=(alloc_view(r, T, d, FP4_FLAG_SR_ROW, dev), alloc_view(r, d, T, 0, dev)),
                dqkv=(alloc_view(r, T, q, FP4_FLAG_SR_ROW, dev), alloc_view(r, q, T, 0, dev)),
            )
        self.views_in = {r: (alloc_view(r, T, d, FP4_FLAG_SR_ROW, dev), alloc_view(r, d, T, 0, dev))
                         for r in {b.route for b in self.blocks}}

    # ----------------------------------------------------------- step ------
    def quantize_weights(self):
        for blk in self.blocks:
            for name in ("qkv", "o", "w13", "w2"):
                rv, cv = blk.wv[name]
                fp4_quantize(blk.w[name], blk.route, FP4_VIEW_ROW | FP4_VIEW_COL, FP4_FLAG_WEIGHT_2D, row_out=rv,
                             col_out=cv, workspace=self.ws)

    def forward(self, x: torch.Tensor):
        d, f = self.sh.d, self.sh.f
        h_prev, f_prev = x, None
        for blk in self.blocks:
            r, s, wv = blk.route, blk.s, blk.wv
            fp4_residual_rmsnorm_fwd(h_prev, f_prev, self.g1, r, 3, self.eps, r_out=s["r1"], rstd=s["rstd1"],
                                     y_row=s["y1"][0], y_col=s["y1"][1], workspace=self.ws)
            fp4_linear_fprop(s["y1"][0], wv["qkv"][0], s["qkv"], FP4_OUT_BF16)
            fp4_quantize(s["qkv"][:, :d], r, 3, 0, row_out=s["attn"][0], col_out=s["attn"][1], workspace=self.ws)
            fp4_linear_fprop(s["attn"][0], wv["o"][0], s["o"], FP4_OUT_BF16)
            fp4_residual_rmsnorm_fwd(s["r1"], s["o"], self.g2, r, 3, self.eps, r_out=s["r2"], rstd=s["rstd2"],
                                     y_row=s["y2"][0], y_col=s["y2"][1], workspace=self.ws)
            # the views of h come from the producer for both routes (NVFP4
            # through one bf16 copy of h whose maxima the epilogue folds)
            fp4_swiglu_fwd(s["y2"][0], wv["w13"][0], f, a1=s["a1"], a3=s["a3"], h_row=s["h"][0], h_col=s["h"][1],
                           h_tap=None if r == "mx" else self.h_tap, workspace=self.ws)
            fp4_linear_fprop(s["h"][0], wv["w2"][0], s["f"], FP4_OUT_BF16)
            h_prev, f_prev = s["r2"], s["f"]
        return h_prev, f_prev

    def backward(self, dy: torch.Tensor, sr_seed: int = 1, step: int | None = None):
        d, f = self.sh.d, self.sh.f
        st = self.step_index if step is None else step
        nb = len(self.blocks)
        top = self.blocks[-1]
        dF = self.gviews[top.route]["dF"]
        fp4_quantize(dy, top.route, 3, FP4_FLAG_SR_ROW, sr_seed=sr_seed, sr_offset=sr_offset(st, nb, 0), row_out=dF[0],
                     col_out=dF[1], workspace=self.ws)
        dh_out = dy
        for i in range(nb - 1, -1, -1):
            blk = self.blocks[i]
            r, s, wv, dw, gv = blk.route, blk.s, blk.wv, blk.dw, self.gviews[blk.route]
            off1, off2, off3, off4 = (sr_offset(st, i, k) for k in (1, 2, 3, 4))
            # FFN: W2 Wgrad, fused W2 Dgrad + SiLU derivative, W1/W3 Dgrad and Wgrad
            fp4_linear_wgrad(dF[1], s["h"][1], dw["w2"])
            fp4_swiglu_bwd(dF[0], wv["w2"][1], f, s["a1"], s["a3"], sr_seed, off1, da13_row=gv["da13"][0],
                           da13_col=gv["da13"][1], da13_tap=None if r == "mx" else self.da13, workspace=self.ws)
            fp4_linear_dgrad_rmsnorm(gv["da13"][0], wv["w13"][1], s["r2"], s["rstd2"], self.g2, dx=self.dy,
                                     part=self.part)
            fp4_linear_wgrad(gv["da13"][1], s["y2"][1], dw["w13"])
            # residual-RMSNorm backward -> gradient of r2 and its views (the O projection's dY)
            dr2 = self.dr2
            fp4_residual_rmsnorm_bwd_parts(self.dy, self.part, s["r2"], s["rstd2"], self.g2, dh_out, r, 3, True,
                                           sr_seed, off2, dr=dr2, dr_row=gv["dr2"][0], dr_col=gv["dr2"][1],
                                           workspace=self.ws)
            fp4_linear_wgrad(gv["dr2"][1], s["attn"][1], dw["o"])
            fp4_linear_dgrad(gv["dr2"][0], wv["o"][1], self.dattn, FP4_OUT_BF16)
            # attention stand-in backward: dQKV = [dattn | 0 | 0] (a copy that
            # stands in for the attention core, which is not part of the FP4
            # boundary; its time can be recorded and taken out)
            if self.time_standin:
                ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                ev[0].record()
            self.dqkv[:, :d].copy_(self.dattn)
            if self.time_standin:
                ev[1].record()
                self._standin_events.append(ev)
            fp4_quantize(self.dqkv, r, 3, FP4_FLAG_SR_ROW, sr_seed=sr_seed, sr_offset=off3, row_out=gv["dqkv"][0],
                         col_out=gv["dqkv"][1], workspace=self.ws)
            fp4_linear_wgrad(gv["dqkv"][1], s["y1"][1], dw["qkv"])
            fp4_linear_dgrad_rmsnorm(gv["dqkv"][0], wv["qkv"][1], s["r1"], s["rstd1"], self.g1, dx=self.dy,
                                     part=self.part)
            # residual-RMSNorm backward -> gradient of the block input, quantized
            # for the preceding block's FFN (in that block's route)
            prev_route = self.blocks[i - 1].route if i > 0 else r
            dF = self.gviews[prev_route]["dF"] if i > 0 else self.views_in[r]
            dr1 = self.dr1[i % 2]  # never the buffer that holds dh_out (block i + 1's)
            fp4_residual_rmsnorm_bwd_parts(self.dy, self.part, s["r1"], s["rstd1"], self.g1, dr2, prev_route,
                                           3 if i > 0 else FP4_VIEW_ROW, True, sr_seed, off4, dr=dr1,
                                           dr_row=dF[0], dr_col=dF[1] if i > 0 else None, workspace=self.ws)
            dh_out = dr1
        return dh_out

    def step(self, x: torch.Tensor, dy: torch.Tensor, sr_seed: int = 1):
        """One forward + backward; the step index advances, so the next
        step's stochastic rounding draws fresh random numbers."""
        self.quantize_weights()
        self.forward(x)
        out = self.backward(dy, sr_seed, self.step_index)
        self.step_index += 1
        return out

    def capture_steps(self, x: torch.Tensor, dy: torch.Tensor, steps: int, sr_seed: int = 1):
        """Record `steps` consecutive training steps (each with its own step
        index, hence its own stochastic-rounding draws) into one CUDA graph
        and return it; replaying it runs exactly those launches with no host
        work between them.  Every buffer the steps touch is allocated
        beforehand, so nothing allocates while recording; run one eager step
        first, so that the library's one-time per-device setup is done."""
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        timing, self.time_standin = self.time_standin, False
        try:
            with torch.cuda.graph(graph, stream=side):
                for _ in range(steps):
                    self.step(x, dy, sr_seed)
        finally:
            self.time_standin = timing
        torch.cuda.current_stream().wait_stream(side)
        return graph

    def standin_ms(self) -> float:
        """Device milliseconds of the attention stand-in's copies recorded
        since the last call (time_standin must be set); synchronises."""
        torch.cuda.synchronize()
        ms = sum(a.elapsed_time(b) for a, b in self._standin_events)
        self._standin_events = []
        return ms
