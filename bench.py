"""Benchmark of the FP4 linear boundary on one GB300.

One step = one pass of the whole boundary over one batch of seeded synthetic
input at the Llama-3-8B W1 shape ("MXFP4 Llama-3-8B W1-shaped linear"):
    producers  X [8192 x 4096]  -> Q_r(X), Q_c(X) with fixed-sign H32
               W [14336 x 4096] -> 2D32 Q_r(W), Q_c(W)
               dY [8192 x 14336]-> Q_r(dY) with Philox SR, Q_c(dY) with H32
    GEMMs      Fprop Y = X W^T, Dgrad dX = dY W, Wgrad dW = dY^T X (FP32 out)
value = 3 * 2*M*N*K FP4 FLOPs / step time (TFLOP/s), with tokens/s and the
producers' algorithmic GB/s alongside.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun (N > 1) every rank runs its own replica of the step (weak
scaling, no data-path collective); rank 0 prints the JSON line.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "Fprop+Dgrad+Wgrad FP4 TFLOPS and tokens/s at Llama-3-8B shapes; quant GB/s"
WORKLOAD = "mxfp4_llama3_8b_w1_linear"
T, D_IN, D_OUT = 8192, 4096, 14336
FP4_NOMINAL_OVER_BF16 = 13.5 / 2.25  # dense FP4 / dense BF16 nominal ratio on GB300


def flops_per_step() -> float:
    return 3 * 2.0 * T * D_IN * D_OUT


def producer_bytes() -> dict:
    # algorithmic bytes: 2 B/elem read + per view 0.5 B codes + 1/32 B E8M0 scales
    mx_both = 2 + 2 * (0.5 + 1 / 32)
    return dict(x=T * D_IN * mx_both, w=D_OUT * D_IN * mx_both, dy=T * D_OUT * mx_both)


def gemm_bytes_min() -> float:
    return 0.0


KERNEL_SOURCES = {
    "gemm": ("gemm.cu", "common.cuh", "internal.h"),
    "quant": ("quantize.cu", "common.cuh", "internal.h"),
}


def _sources_digest(kind: str) -> str:
    import hashlib
    m = hashlib.sha256()
    for f in KERNEL_SOURCES[kind]:
        with open(os.path.join(ROOT, "fp4_quantized_linears_gb300", "csrc", f), "rb") as fh:
            m.update(fh.read())
    return m.hexdigest()[:16]


def profiled_traffic(kernel: str):
    """DRAM bytes (read + write) per launch of `kernel` from the ncu summaries
    under profiles/, or None when none was taken of the current sources."""
    import glob
    want = _sources_digest("quant" if kernel.startswith("quant") else "gemm")
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        with open(path) as f:
            for line in f:
                if not line.startswith("traffic-record "):
                    continue
                kv = dict(tok.split("=", 1) for tok in line.split()[1:])
                if kv.get("kernel") == kernel and kv.get("sources") == want:
                    return int(kv["bytes"])
    return None


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sus=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


# ------------------------------------------------------------------ clocks --
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------- distributed ----
def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if os.environ.get("FP4_BENCH_BACKEND", "nccl") == "nccl" else "gloo"
        dist.init_process_group(backend=backend)
        pg = dist
    return rank, local, world, pg


def barrier(pg, device=None):
    if pg is not None:
        if device is not None and pg.get_backend() == "nccl":
            pg.barrier(device_ids=[device])
        else:
            pg.barrier()


def max_over_ranks(pg, v: float) -> float:
    if pg is None:
        return v
    import torch
    dev = "cuda" if pg.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------- our arm ----
def run_ours(args):
    import torch
    import fp4_quantized_linears_gb300 as F
    from synthetic import config_tensors

    rank, local, world, pg = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    F.load()
    t0 = time.time()
    host = config_tensors("c2_mx_w1", scale_T=T)
    signs = [int(s) for s in host["signs"]]

    def to_dev(b):
        return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).to(dev)

    X, W, DY = to_dev(host["x"]), to_dev(host["w"]), to_dev(host["dy"])
    gen_s = time.time() - t0
    # persistent outputs (allocated once, outside the timed region)
    xr, xc = F.alloc_view("mx", T, D_IN), F.alloc_view("mx", D_IN, T)
    wr, wc = F.alloc_view("mx", D_OUT, D_IN), F.alloc_view("mx", D_IN, D_OUT)
    dr, dc = F.alloc_view("mx", T, D_OUT), F.alloc_view("mx", D_OUT, T)
    Y = torch.empty((T, D_OUT), dtype=torch.float32, device=dev)
    DX = torch.empty((T, D_IN), dtype=torch.float32, device=dev)
    DW = torch.empty((D_OUT, D_IN), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    names = ["quant_x", "quant_w", "quant_dy", "fprop", "dgrad", "wgrad"]

    def step(ev=None, seed_offset=0, x=X, w=W, dy=DY):
        def mark(i):
            if ev is not None:
                ev[i].record(stream)
        mark(0)
        F.fp4_quantize(x, "mx", 3, F.FP4_FLAG_HADAMARD_COL, hadamard_signs=signs, row_out=xr, col_out=xc)
        mark(1)
        F.fp4_quantize(w, "mx", 3, F.FP4_FLAG_WEIGHT_2D, row_out=wr, col_out=wc)
        mark(2)
        F.fp4_quantize(dy, "mx", 3, F.FP4_FLAG_SR_ROW | F.FP4_FLAG_HADAMARD_COL, sr_seed=1, sr_offset=seed_offset,
                       hadamard_signs=signs, row_out=dr, col_out=dc)
        mark(3)
        F.fp4_linear_fprop(xr, wr, Y)
        mark(4)
        F.fp4_linear_dgrad(dr, wc, DX)
        mark(5)
        F.fp4_linear_wgrad(dc, xc, DW)
        mark(6)

    for i in range(args.warmup):
        step(seed_offset=i)
    torch.cuda.synchronize()
    if F.fp4_status() != F.FP4_OK:
        raise RuntimeError("device status set during warm-up")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(7)] for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier(pg, local)
    torch.cuda.synchronize()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(args.steps):
        step(evs[i], seed_offset=1000 + i)
    stop.record(stream)
    torch.cuda.synchronize()
    barrier(pg, local)
    clk = clocks.stop()
    total_ms = start.elapsed_time(stop)
    total_ms = max_over_ranks(pg, total_ms)
    per_kernel = {n: statistics.mean(evs[i][k].elapsed_time(evs[i][k + 1]) for i in range(args.steps))
                  for k, n in enumerate(names)}
    if F.fp4_status() != F.FP4_OK:
        raise RuntimeError("device status set during the timed region")

    # end to end through the public API with pinned host buffers
    pin = (lambda t: t) if args.no_e2e else (lambda t: t.pin_memory())
    hx = pin(torch.from_numpy(host["x"].view(np.int16)).view(torch.bfloat16))
    hw = pin(torch.from_numpy(host["w"].view(np.int16)).view(torch.bfloat16))
    hdy = pin(torch.from_numpy(host["dy"].view(np.int16)).view(torch.bfloat16))
    hY = pin(torch.empty(Y.shape, dtype=torch.float32))
    hDX = pin(torch.empty(DX.shape, dtype=torch.float32))
    hDW = pin(torch.empty(DW.shape, dtype=torch.float32))
    e2e_steps = max(3, min(args.steps, 10))
    e2e_ms = float("nan")
    if not args.no_e2e:
        # Pipelined across three streams, as a caller of the C ABI runs it:
        # step i's inputs are copied in on one stream while step i-1 computes
        # on another and step i-2's outputs are copied out on a third.  The
        # device inputs and outputs are double-buffered; events order every
        # use of a buffer after the copy that fills it and before the next
        # copy that overwrites it.
        s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
        din = [(torch.empty_like(X), torch.empty_like(W), torch.empty_like(DY)) for _ in range(2)]
        dout = [(Y, DX, DW), (torch.empty_like(Y), torch.empty_like(DX), torch.empty_like(DW))]
        ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in", "cmp", "out")}
        for k in ev:
            for e in ev[k]:
                e.record(stream)  # all buffers start free

        def e2e_step(i):
            b = i % 2
            xb, wb, db = din[b]
            yb, dxb, dwb = dout[b]
            with torch.cuda.stream(s_in):
                s_in.wait_event(ev["cmp"][b])           # the step that last read these inputs is done
                xb.copy_(hx, non_blocking=True)
                wb.copy_(hw, non_blocking=True)
                db.copy_(hdy, non_blocking=True)
                ev["in"][b].record(s_in)
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(ev["in"][b])
                s_cmp.wait_event(ev["out"][b])          # these outputs were copied out
                F.fp4_quantize(xb, "mx", 3, F.FP4_FLAG_HADAMARD_COL, hadamard_signs=signs, row_out=xr, col_out=xc)
                F.fp4_quantize(wb, "mx", 3, F.FP4_FLAG_WEIGHT_2D, row_out=wr, col_out=wc)
                F.fp4_quantize(db, "mx", 3, F.FP4_FLAG_SR_ROW | F.FP4_FLAG_HADAMARD_COL, sr_seed=1,
                               sr_offset=5000 + i, hadamard_signs=signs, row_out=dr, col_out=dc)
                F.fp4_linear_fprop(xr, wr, yb)
                F.fp4_linear_dgrad(dr, wc, dxb)
                F.fp4_linear_wgrad(dc, xc, dwb)
                ev["cmp"][b].record(s_cmp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev["cmp"][b])
                hY.copy_(yb, non_blocking=True)
                hDX.copy_(dxb, non_blocking=True)
                hDW.copy_(dwb, non_blocking=True)
                ev["out"][b].record(s_out)

        e2e_step(0)
        e2e_step(1)
        torch.cuda.synchronize()
        barrier(pg, local)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s_in)
        for i in range(e2e_steps):
            e2e_step(i + 2)
        e1.record(s_out)  # after the last step's outputs reached the host
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(pg, e0.elapsed_time(e1) / e2e_steps)
        if F.fp4_status() != F.FP4_OK:
            raise RuntimeError("device status set in the end-to-end leg")
        del din, dout
    h2d = (hx.numel() + hw.numel() + hdy.numel()) * 2
    d2h = (hY.numel() + hDX.numel() + hDW.numel()) * 4

    if rank != 0:
        if pg is not None:
            pg.destroy_process_group()
        return

    ms = total_ms / args.steps
    tflops = flops_per_step() / (ms * 1e-3) / 1e12 * world
    pb = producer_bytes()
    quant_ms = per_kernel["quant_x"] + per_kernel["quant_w"] + per_kernel["quant_dy"]
    quant_gbs = (pb["x"] + pb["w"] + pb["dy"]) / (quant_ms * 1e-3) / 1e9
    peaks = load_peaks()
    fp4_peak = peaks["bf16"] * FP4_NOMINAL_OVER_BF16
    gemm_flops = 2.0 * T * D_IN * D_OUT
    # dominant kernel by time share
    dom = max(per_kernel, key=per_kernel.get)
    if dom in ("fprop", "dgrad", "wgrad"):
        ach = gemm_flops / (per_kernel[dom] * 1e-3) / 1e12
        roof = {"kernel": dom, "bound": "tensor", "achieved": round(ach, 1), "peak": round(fp4_peak, 1),
                "unit": "TFLOP/s", "frac": round(ach / fp4_peak, 4), "traffic": profiled_traffic(dom),
                "peak_note": f"{peaks['src']} bf16 burst {peaks['bf16']} x nominal fp4/bf16 ratio 6"}
    else:
        b = pb[dom.split("_")[1]]
        ach = b / (per_kernel[dom] * 1e-3) / 1e9
        roof = {"kernel": dom, "bound": "hbm", "achieved": round(ach, 1), "peak": peaks["hbm"], "unit": "GB/s",
                "frac": round(ach / peaks["hbm"], 4), "traffic": profiled_traffic(dom), "peak_note": f"{peaks['src']} hbm_gbs"}
    kernels = {}
    for n, v in per_kernel.items():
        if n.startswith("quant"):
            b = pb[n.split("_")[1]]
            kernels[n] = {"ms": round(v, 4), "GB/s": round(b / (v * 1e-3) / 1e9, 1),
                          "hbm_frac": round(b / (v * 1e-3) / 1e9 / peaks["hbm"], 4)}
        else:
            tf = gemm_flops / (v * 1e-3) / 1e12
            kernels[n] = {"ms": round(v, 4), "TFLOP/s": round(tf, 1), "fp4_frac": round(tf / fp4_peak, 4)}

    # the operand-wise hybrid on the same tensors (MXFP4 Fprop and Wgrad with
    # plain H16 on the pair, CTA-local NVFP4 Dgrad with row SR)
    hybrid = None if args.no_legs else run_hybrid_leg(X, W, DY, peaks)
    # free the main workload's buffers before the other legs
    del X, W, DY, Y, DX, DW, xr, xc, wr, wc, dr, dc
    torch.cuda.empty_cache()
    legs = {} if args.no_legs else run_legs(args, peaks)
    if hybrid is not None:
        legs = {"operand_hybrid_h16_w1": hybrid, **legs}
    cpu = cpu_baseline_sample(seconds_target=args.cpu_seconds) if args.cpu_seconds > 0 else None
    line = {
        "metric": METRIC, "value": round(tflops, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e2m1", "data": "synthetic (seeded: X Student-t4 unit var, W N(0,0.02), dY N(0,1e-4))",
        "config": main_config(world),
        "tokens_per_s": round(T / (ms * 1e-3) * world, 1),
        "quant_gbs": round(quant_gbs, 1),
        "kernels": kernels,
        "roofline": roof,
        "e2e": None if args.no_e2e else {
            "value": round(flops_per_step() / (e2e_ms * 1e-3) / 1e12 * world, 2), "unit": "TFLOP/s",
            "ms_per_step": round(e2e_ms, 3), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps * 6,
        "clocks": clk,
        "cpu_baseline": cpu,
        "legs": legs,
        "input_gen_s": round(gen_s, 1),
    }
    print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


# ------------------------------------------------------------ other legs ----
def run_hybrid_leg(X, W, DY, peaks, steps: int = 10, warmup: int = 3) -> dict:
    """One pass of the operand-wise hybrid boundary over the W1-shaped tensors:
    the three producers (X: MXFP4 both views, plain H16 on the column view;
    W: MXFP4 2D32 row view + CTA-local 2D16 column view; dY: CTA-local row
    view with SR + MXFP4 column view with plain H16) and the three GEMMs."""
    import torch
    import fp4_quantized_linears_gb300 as F
    T_, di = X.shape
    do = W.shape[0]
    ones = [1] * 16
    h16 = F.FP4_FLAG_HADAMARD16_COL
    xr, xc = F.alloc_view("mx", T_, di), F.alloc_view("mx", di, T_)
    wr, wc = F.alloc_view("mx", do, di, F.FP4_FLAG_WEIGHT_2D), F.alloc_view("nv_local", di, do, F.FP4_FLAG_WEIGHT_2D)
    dr, dc = F.alloc_view("nv_local", T_, do), F.alloc_view("mx", do, T_)
    ws = torch.empty(max(F.fp4_quantize_hybrid_workspace_bytes("nv_local", "mx", T_, do, 3, h16),
                         F.fp4_quantize_hybrid_workspace_bytes("mx", "nv_local", do, di, 3, F.FP4_FLAG_WEIGHT_2D), 16),
                     dtype=torch.uint8, device=X.device)
    Y = torch.empty((T_, do), dtype=torch.float32, device=X.device)
    DX = torch.empty((T_, di), dtype=torch.float32, device=X.device)
    DW = torch.empty((do, di), dtype=torch.float32, device=X.device)
    names = ["quant_x", "quant_w", "quant_dy", "fprop", "dgrad", "wgrad"]

    def step(ev=None, i=0):
        def mark(k):
            if ev is not None:
                ev[k].record()
        mark(0)
        F.fp4_quantize(X, "mx", 3, h16, hadamard_signs=ones, row_out=xr, col_out=xc)
        mark(1)
        F.fp4_quantize_hybrid(W, "mx", "nv_local", 3, F.FP4_FLAG_WEIGHT_2D, row_out=wr, col_out=wc, workspace=ws)
        mark(2)
        F.fp4_quantize_hybrid(DY, "nv_local", "mx", 3, F.FP4_FLAG_SR_ROW | h16, sr_seed=4, sr_offset=i,
                              hadamard_signs=ones, row_out=dr, col_out=dc, workspace=ws)
        mark(3)
        F.fp4_linear_fprop(xr, wr, Y)
        mark(4)
        F.fp4_linear_dgrad(dr, wc, DX)
        mark(5)
        F.fp4_linear_wgrad(dc, xc, DW)
        mark(6)

    for i in range(warmup):
        step(i=i)
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(7)] for _ in range(steps)]
    for i in range(steps):
        step(evs[i], 100 + i)
    torch.cuda.synchronize()
    if F.fp4_status() != F.FP4_OK:
        raise RuntimeError("device status set in the hybrid leg")
    per = {n: statistics.mean(evs[i][k].elapsed_time(evs[i][k + 1]) for i in range(steps))
           for k, n in enumerate(names)}
    ms = sum(per.values())
    fl = 3 * 2.0 * T_ * di * do
    return {"ms_per_step": round(ms, 4), "TFLOP/s": round(fl / ms / 1e9, 1),
            "kernels_ms": {k: round(v, 4) for k, v in per.items()}}


def _timed(fn, steps: int, warmup: int) -> float:
    """Mean device milliseconds of fn() over `steps` calls after `warmup`."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def run_legs(args, peaks, only=None) -> dict:
    """The other workloads of the boundary, each one pass per step:
    NVFP4 (global and CTA-local) on attention-projection shapes, the fused
    SwiGLU FFN forward + backward, and the 32-block 27/5 depth-hybrid stack."""
    import torch
    import fp4_quantized_linears_gb300 as F
    from fp4_quantized_linears_gb300.stack import BlockShape, FP4LinearStack, linear_flops_per_token
    from synthetic import config_tensors
    fp4_peak = peaks["bf16"] * FP4_NOMINAL_OVER_BF16
    out = {}

    def dev(b):
        return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).cuda()

    def frac(tf):
        return round(tf / fp4_peak, 4)

    # NVFP4 attention projections: X 8192x4096, W 4096x4096 and 6144x4096
    if only not in (None, "nvfp4"):
        t3 = None
    else:
        t3 = config_tensors("c3_nv_attn", scale_T=args.tokens)
    X3 = dev(t3["x"]) if t3 is not None else None
    for route in (("nv_global", "nv_local") if t3 is not None else ()):
        for wname, dyname in (("w", "dy"), ("w_qkv", "dy_qkv")):
            Wt, DYt = dev(t3[wname]), dev(t3[dyname])
            n_out, n_in = Wt.shape
            T3 = X3.shape[0]
            ws = torch.empty(max(F.fp4_quantize_workspace_bytes(route, T3, n_out), F.fp4_quantize_workspace_bytes(route, n_out, n_in), 16), dtype=torch.uint8, device="cuda")
            xr, xc = F.alloc_view(route, T3, n_in), F.alloc_view(route, n_in, T3)
            wr, wc = F.alloc_view(route, n_out, n_in, F.FP4_FLAG_WEIGHT_2D), F.alloc_view(route, n_in, n_out, F.FP4_FLAG_WEIGHT_2D)
            dr, dc = F.alloc_view(route, T3, n_out), F.alloc_view(route, n_out, T3)
            Y = torch.empty((T3, n_out), device="cuda")
            DXo = torch.empty((T3, n_in), device="cuda")
            DWo = torch.empty((n_out, n_in), device="cuda")

            def step3():
                F.fp4_quantize(X3, route, 3, 0, row_out=xr, col_out=xc, workspace=ws)
                F.fp4_quantize(Wt, route, 3, F.FP4_FLAG_WEIGHT_2D, row_out=wr, col_out=wc, workspace=ws)
                F.fp4_quantize(DYt, route, 3, F.FP4_FLAG_SR_ROW, sr_seed=2, row_out=dr, col_out=dc, workspace=ws)
                F.fp4_linear_fprop(xr, wr, Y)
                F.fp4_linear_dgrad(dr, wc, DXo)
                F.fp4_linear_wgrad(dc, xc, DWo)

            ms = _timed(step3, 5, 3)
            gemm_ms = _timed(lambda: (F.fp4_linear_fprop(xr, wr, Y), F.fp4_linear_dgrad(dr, wc, DXo),
                                      F.fp4_linear_wgrad(dc, xc, DWo)), 5, 2)
            fl = 3 * 2.0 * T3 * n_in * n_out
            out[f"nvfp4_{route.split('_')[1]}_{n_out}x{n_in}"] = {
                "ms_per_step": round(ms, 4), "TFLOP/s": round(fl / ms / 1e9, 1),
                "gemm_TFLOP/s": round(fl / gemm_ms / 1e9, 1), "gemm_fp4_frac": frac(fl / gemm_ms / 1e9)}
            del Wt, DYt, xr, xc, wr, wc, dr, dc, Y, DXo, DWo, ws
    del X3, t3
    torch.cuda.empty_cache()

    if only in (None, "qkv"):
        out["qkv_rope_T8192"] = run_qkv_rope_leg()
        if only == "qkv":
            return out
    if only in (None, "diagnostic"):
        # the Dgrad-error diagnostic: E_MX / E_localCTA over 32 blocks x 3
        # batches of 2048 tokens x 4 components (an accuracy figure, not a rate)
        from fp4_quantized_linears_gb300.diagnostic import dgrad_diagnostic
        t0 = time.time()
        d = dgrad_diagnostic(blocks=32, batches=3, T=2048)
        out["dgrad_error_diagnostic"] = {
            "pairs": d["pairs"], "geomean_EMX_over_ElocalCTA": round(d["geomean"], 4),
            "pairs_lower_for_localCTA": d["favour_local"],
            "per_component": {k: round(v, 4) for k, v in d["per_component"].items()},
            "pages_value_on_captured_tensors": 1.292, "wall_s": round(time.time() - t0, 1)}
        torch.cuda.empty_cache()
        if only == "diagnostic":
            return out
    if only not in (None, "swiglu", "stack"):
        return out
    # fused SwiGLU FFN, MXFP4, T 16384, d 4096, f 14336
    if only == "stack":
        return run_stack_leg(args, out, peaks)
    t4 = config_tensors("c4_swiglu", scale_T=args.tokens)
    X4, W13, W2, DY2 = dev(t4["x"]), dev(t4["w13"]), dev(t4["w2"]), dev(t4["dy2"])
    del t4
    T4, d4 = X4.shape
    f4 = W2.shape[1]
    xr, xc = F.alloc_view("mx", T4, d4), F.alloc_view("mx", d4, T4)
    w13r, w13c = F.alloc_view("mx", 2 * f4, d4), F.alloc_view("mx", d4, 2 * f4)
    w2r, w2c = F.alloc_view("mx", d4, f4), F.alloc_view("mx", f4, d4)
    dyr, dyc = F.alloc_view("mx", T4, d4), F.alloc_view("mx", d4, T4)
    a1 = torch.empty((T4, f4), dtype=torch.bfloat16, device="cuda")
    a3 = torch.empty_like(a1)
    hr, hc = F.alloc_view("mx", T4, f4), F.alloc_view("mx", f4, T4)
    dar, dac = F.alloc_view("mx", T4, 2 * f4), F.alloc_view("mx", 2 * f4, T4)
    Y2 = torch.empty((T4, d4), dtype=torch.bfloat16, device="cuda")
    DX4 = torch.empty((T4, d4), dtype=torch.bfloat16, device="cuda")
    DW13 = torch.empty((2 * f4, d4), device="cuda")
    DW2 = torch.empty((d4, f4), device="cuda")

    def step4():
        F.fp4_quantize(X4, "mx", 3, 0, row_out=xr, col_out=xc)
        F.fp4_quantize(W13, "mx", 3, F.FP4_FLAG_WEIGHT_2D, row_out=w13r, col_out=w13c)
        F.fp4_quantize(W2, "mx", 3, F.FP4_FLAG_WEIGHT_2D, row_out=w2r, col_out=w2c)
        F.fp4_swiglu_fwd(xr, w13r, f4, a1=a1, a3=a3, h_row=hr, h_col=hc)
        F.fp4_linear_fprop(hr, w2r, Y2, F.FP4_OUT_BF16)
        F.fp4_quantize(DY2, "mx", 3, F.FP4_FLAG_SR_ROW, sr_seed=3, row_out=dyr, col_out=dyc)
        F.fp4_swiglu_bwd(dyr, w2c, f4, a1, a3, sr_seed=3, sr_offset=1, da13_row=dar, da13_col=dac)
        F.fp4_linear_dgrad(dar, w13c, DX4, F.FP4_OUT_BF16)
        F.fp4_linear_wgrad(dac, xc, DW13)
        F.fp4_linear_wgrad(dyc, hc, DW2)

    ms = _timed(step4, 3, 2)
    fl4 = 18.0 * T4 * d4 * f4
    ms_fwd = _timed(lambda: F.fp4_swiglu_fwd(xr, w13r, f4, a1=a1, a3=a3, h_row=hr, h_col=hc), 3, 1)
    ms_bwd = _timed(lambda: F.fp4_swiglu_bwd(dyr, w2c, f4, a1, a3, sr_seed=3, sr_offset=1, da13_row=dar,
                                             da13_col=dac), 3, 1)
    out["swiglu_ffn_mxfp4_T16384"] = {
        "ms_per_step": round(ms, 3), "TFLOP/s": round(fl4 / ms / 1e9, 1), "tokens_per_s": round(T4 / ms * 1e3, 1),
        "fused_fwd_ms": round(ms_fwd, 4), "fused_fwd_TFLOP/s": round(4.0 * T4 * d4 * f4 / ms_fwd / 1e9, 1),
        "fused_bwd_ms": round(ms_bwd, 4), "fused_bwd_TFLOP/s": round(2.0 * T4 * d4 * f4 / ms_bwd / 1e9, 1)}
    del X4, W13, W2, DY2, xr, xc, w13r, w13c, w2r, w2c, dyr, dyc, a1, a3, hr, hc, dar, dac, Y2, DX4, DW13, DW2
    torch.cuda.empty_cache()

    if not args.no_stack and only is None:
        run_stack_leg(args, out, peaks)
    return out


def run_qkv_rope_leg(T: int = 8192, d: int = 4096, hq: int = 32, hkv: int = 8, S: int = 4096,
                     route: str = "nv_local") -> dict:
    """The QKV boundary with RoPE at Llama-3-8B shapes: the fused projection +
    RoPE + head-major layout against the plain projection, and the fused
    backward producer (inverse layout and RoPE + quantization of dQKV) against
    quantizing an already-assembled dQKV."""
    import torch
    import fp4_quantized_linears_gb300 as F
    N = (hq + 2 * hkv) * 128
    g = torch.Generator(device="cuda").manual_seed(7)
    X = torch.randn((T, d), generator=g, device="cuda").to(torch.bfloat16)
    W = (torch.randn((N, d), generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    xr, _ = F.fp4_quantize(X, route, F.FP4_VIEW_ROW)
    wr, _ = F.fp4_quantize(W, route, F.FP4_VIEW_ROW, F.FP4_FLAG_WEIGHT_2D)
    pos = torch.arange(S, device="cuda", dtype=torch.float64)[:, None]
    inv = torch.tensor(500000.0, dtype=torch.float64) ** (-torch.arange(64, dtype=torch.float64) / 64.0)
    ang = pos * inv.cuda()[None, :]
    cs, sn = torch.cos(ang).float().contiguous(), torch.sin(ang).float().contiguous()
    q = torch.empty((hq, T, 128), dtype=torch.bfloat16, device="cuda")
    k = torch.empty((hkv, T, 128), dtype=torch.bfloat16, device="cuda")
    v = torch.empty_like(k)
    Y = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
    fwd = _timed(lambda: F.fp4_qkv_rope_fwd(xr, wr, cs, sn, S, hq, hkv, q, k, v), 10, 3)
    plain = _timed(lambda: F.fp4_linear_fprop(xr, wr, Y, F.FP4_OUT_BF16), 10, 3)
    dq, dk, dv = (t.mul(1e-3) for t in (q, k, v))
    rv, cv = F.alloc_view(route, T, N, F.FP4_FLAG_SR_ROW), F.alloc_view(route, N, T)
    ws = torch.empty(max(F.fp4_quantize_workspace_bytes(route, T, N), 16), dtype=torch.uint8, device="cuda")
    bwd = _timed(lambda: F.fp4_qkv_rope_bwd(dq, dk, dv, cs, sn, S, route, 3, True, 8, 0, None, rv, cv, ws), 10, 3)
    dY = Y.mul(1e-3)
    qplain = _timed(lambda: F.fp4_quantize(dY, route, 3, F.FP4_FLAG_SR_ROW, sr_seed=8, row_out=rv, col_out=cv,
                                           workspace=ws), 10, 3)
    if F.fp4_status() != F.FP4_OK:
        raise RuntimeError("device status set in the QKV leg")
    fl = 2.0 * T * N * d
    return {"route": route, "fused_fwd_ms": round(fwd, 4), "fused_fwd_TFLOP/s": round(fl / fwd / 1e9, 1),
            "plain_fprop_ms": round(plain, 4), "fused_bwd_producer_ms": round(bwd, 4),
            "plain_quantize_ms": round(qplain, 4)}


def stack_producer_bytes(sh, n_blocks: int, local_blocks: int) -> float:
    """Algorithmic bytes of every producer of one stack step (forward +
    backward): BF16 inputs read once (twice for NVFP4, whose outer factors
    need a maximum before the encode), the retained BF16 values written once,
    and per FP4 view 0.5 B of codes + 1 / block size B of scales per element.
    The contractions' own operand reads and outputs are not counted: they are
    inside the FLOP term of the composite roofline."""
    T, d, f, q = sh.T, sh.d, sh.f, sh.qkv
    total = 0.0
    for b in range(n_blocks):
        nv = b < local_blocks
        nvx = 2.0 if nv else 0.0                        # the NVFP4 maximum pass
        v2 = 2 * (0.5 + (1 / 16 if nv else 1 / 32))     # both views
        W = q * d + d * d + 2 * f * d + d * f
        total += W * (2 + nvx + v2)                     # 2D weight producers
        total += 2 * (T * d * (2 + 2 + 2 + nvx + v2) + 4 * T)  # residual-RMSNorm fwd: r, b in; r', views, rstd out
        total += T * d * (2 + nvx + v2)                 # attention output producer
        total += T * f * (4 + v2)                       # SwiGLU fwd epilogue: a1, a3 out, views of h
        total += T * f * 4 + 2 * T * f * v2             # SwiGLU bwd epilogue: a1, a3 in, views of [da1 | da3]
        total += 2 * T * d * (2 + 2 + 2 + 2 + nvx + v2)  # residual-RMSNorm bwd: dx, r', dres in; dr, views out
        total += T * q * (2 + nvx + v2)                 # dQKV producer
    top_nv = n_blocks - 1 < local_blocks
    total += T * d * (2 + (2.0 if top_nv else 0.0) + 2 * (0.5 + (1 / 16 if top_nv else 1 / 32)))
    return total


def run_stack_leg(args, out: dict, peaks=None) -> dict:
    """The depth-hybrid block stack at T 8192 (blocks 1-27 CTA-local NVFP4,
    28-32 MXFP4); --stack-blocks keeps the same 27/32 split on fewer blocks.
    Ten timed steps; the attention stand-in's gradient copy (not part of the
    FP4 boundary) is timed by events and taken out of the step time."""
    import torch
    import fp4_quantized_linears_gb300 as F
    from fp4_quantized_linears_gb300.stack import BlockShape, FP4LinearStack, linear_flops_per_token
    peaks = peaks or load_peaks()
    nb = args.stack_blocks
    local = (27 * nb) // 32 if nb != 32 else 27
    sh = BlockShape()
    st = FP4LinearStack(nb, local, sh, seed=5)
    g = torch.Generator(device="cuda").manual_seed(5)
    x5 = torch.randn((sh.T, sh.d), generator=g, device="cuda").to(torch.bfloat16)
    dy5 = (torch.randn((sh.T, sh.d), generator=g, device="cuda") * 1e-4).to(torch.bfloat16)
    steps = args.stack_steps
    for _ in range(2):
        st.step(x5, dy5, sr_seed=5)
    torch.cuda.synchronize()
    st.time_standin = True
    st.standin_ms()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        st.step(x5, dy5, sr_seed=5)
    e1.record()
    torch.cuda.synchronize()
    standin = st.standin_ms() / steps
    ms_eager_all = e0.elapsed_time(e1) / steps
    # the same number of steps recorded into one CUDA graph and replayed: the
    # launches without the host between them (the stand-in's copies are in
    # the graph too and are taken out as above)
    graph_note = "cuda graph of the timed steps, replayed"
    try:
        if args.stack_eager:
            raise RuntimeError("--stack-eager")
        graph = st.capture_steps(x5, dy5, steps, sr_seed=5)
        graph.replay()
        torch.cuda.synchronize()
        e0.record()
        graph.replay()
        e1.record()
        torch.cuda.synchronize()
        ms_all = e0.elapsed_time(e1) / steps
        del graph
    except RuntimeError as exc:  # capture refused: report the eager launches
        graph_note = ("eager launches" if args.stack_eager else
                      f"eager launches (graph capture failed: {str(exc).splitlines()[0][:120]})")
        ms_all = ms_eager_all
    if F.fp4_status() != F.FP4_OK:
        raise RuntimeError("device status set in the stack leg")
    ms = ms_all - standin
    fl5 = linear_flops_per_token(sh) * nb * sh.T
    pb = stack_producer_bytes(sh, nb, local)
    p_fp4 = peaks["bf16_sus"] * FP4_NOMINAL_OVER_BF16  # a long step: the sustained figure
    t_roof = fl5 / (p_fp4 * 1e12) + pb / (peaks["hbm"] * 1e9)
    out[f"stack{nb}_hybrid_{local}nv_{nb - local}mx_T8192"] = {
        "ms_per_step": round(ms, 2), "tokens_per_s": round(sh.T / ms * 1e3, 1),
        "linear_TFLOP/s": round(fl5 / ms / 1e9, 1), "linear_tflop_per_step": round(fl5 / 1e12, 2),
        "steps": steps, "launch": graph_note, "ms_per_step_eager": round(ms_eager_all - standin, 2),
        "standin_copy_ms_excluded": round(standin, 3), "ms_per_step_with_standin": round(ms_all, 2),
        "producer_GB_per_step": round(pb / 1e9, 2),
        "roofline": {"composite_ms": round(t_roof * 1e3, 2), "frac": round(t_roof * 1e3 / ms, 4),
                     "peak_fp4_TFLOP/s": round(p_fp4, 1), "peak_hbm_GB/s": peaks["hbm"],
                     "peak_note": f"{peaks['src']} bf16 sustained x 6; {peaks['src']} hbm_gbs"}}
    del st, x5, dy5
    torch.cuda.empty_cache()
    return out


# ------------------------------------------------------------ CPU oracle ----
_CPU_T = {}


def _cpu_tensors():
    if not _CPU_T:
        from synthetic import config_tensors
        _CPU_T.update(config_tensors("c2_mx_w1"))
    return _CPU_T


def cpu_sample_slices(seed: int) -> dict:
    """The operand slices that one 128 x 128 output tile of each contraction
    needs (rows of X, W and dY for Fprop / Dgrad, columns of dY and X for
    Wgrad, full K), chosen by the seed."""
    t = _cpu_tensors()
    x, w, dy = t["x"], t["w"], t["dy"]
    rng = np.random.default_rng(seed)
    mt = int(rng.integers(0, T // 128)) * 128
    ot = int(rng.integers(0, D_OUT // 128)) * 128
    it = int(rng.integers(0, D_IN // 128)) * 128
    c = np.ascontiguousarray
    return dict(x_rows=c(x[mt:mt + 128]), w_rows=c(w[ot:ot + 128]), dy_rows=c(dy[mt:mt + 128]),
                w_cols=c(w[:, it:it + 128]), dy_cols=c(dy[:, ot:ot + 128]), x_cols=c(x[:, it:it + 128]),
                signs=t["signs"])


def cpu_sample_task(sl: dict):
    """One bounded sample on the CPU oracle, as it stands: quantize the
    slices and contract them.  Returns (FLOPs counted, seconds)."""
    import oracle
    t0 = time.perf_counter()
    a = oracle.quantize(sl["x_rows"], "mx", "row")
    b = oracle.quantize(sl["w_rows"], "mx", "row", weight2d=True)
    oracle.gemm(a, b)
    a = oracle.quantize(sl["dy_rows"], "mx", "row", sr=True, seed=1)
    b = oracle.quantize(sl["w_cols"], "mx", "col", weight2d=True)
    oracle.gemm(a, b)
    a = oracle.quantize(sl["dy_cols"], "mx", "col", hadamard=True, signs=sl["signs"])
    b = oracle.quantize(sl["x_cols"], "mx", "col", hadamard=True, signs=sl["signs"])
    oracle.gemm(a, b)
    return 2.0 * 128 * 128 * (D_IN + D_OUT + T), time.perf_counter() - t0


class CpuPool:
    """The oracle on every host core: one spawned worker process per core
    (spawned, so no worker inherits a CUDA context), each running one sample
    at a time."""

    def __init__(self, cores: int | None = None):
        import multiprocessing as mp
        import oracle
        oracle.build()
        self.cores = max(1, cores or os.cpu_count() or 1)
        self.pool = mp.get_context("spawn").Pool(self.cores)

    def round(self, seed0: int):
        """One sample per core; returns (FLOPs, wall seconds)."""
        tasks = [cpu_sample_slices(seed0 + i) for i in range(self.cores)]
        t0 = time.perf_counter()
        res = self.pool.map(cpu_sample_task, tasks)
        return sum(r[0] for r in res), time.perf_counter() - t0

    def close(self):
        self.pool.close()
        self.pool.join()


CPU_SAMPLE = ("one 128x128 output tile of each of Fprop, Dgrad, Wgrad at the full K, with the quantization "
              "of the operand slices it needs, per core, on the C oracle")


def cpu_baseline_sample(seconds_target: float = 10.0) -> dict:
    pool = CpuPool()
    try:
        pool.round(0)  # workers start and load the oracle
        flops, secs, n = 0.0, 0.0, 0
        while secs < seconds_target or n == 0:
            f, s_ = pool.round(100 + n * pool.cores)
            flops += f
            secs += s_
            n += 1
    finally:
        pool.close()
    return {"value": round(flops / secs / 1e12, 6), "unit": "TFLOP/s", "cores": pool.cores, "kind": "oracle",
            "sample": f"{n} rounds x {pool.cores} cores x ({CPU_SAMPLE}), {secs:.1f} s wall"}


def main_config(world: int) -> dict:
    return {"workload": WORKLOAD, "tokens": T, "d_in": D_IN, "d_out": D_OUT, "route": "mxfp4",
            "flags": "X col H32, W 2D32, dY row SR + col H32", "out_dtype": "f32",
            "l2": "inputs larger than L2 (419 MB bf16 per step)", "parallelism": f"replicas{world}"}


def run_reference(args):
    """The reference arm: the CPU oracle, as it stands, on every host core;
    each step is one bounded sample per core of the same workload."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    pool = CpuPool()
    try:
        for i in range(args.warmup):
            pool.round(i * pool.cores)
        flops, secs = 0.0, 0.0
        for i in range(args.steps):
            f, s_ = pool.round(1000 + i * pool.cores)
            flops += f
            secs += s_
    finally:
        pool.close()
    v = flops / secs / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": "TFLOP/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(secs / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (same seeded tensors as the GPU arm)",
        "config": main_config(1),
        "cpu_baseline": {"value": round(v, 6), "unit": "TFLOP/s", "cores": pool.cores, "kind": "oracle",
                         "sample": f"per step: {CPU_SAMPLE}"},
        "e2e": {"value": round(v, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--stack-eager", action="store_true",
                    help="stack leg: time the eager launches only (no CUDA graph of the timed steps)")
    ap.add_argument("--no-legs", action="store_true", help="only the main workload")
    ap.add_argument("--no-stack", action="store_true", help="skip the 32-block stack leg")
    ap.add_argument("--stack-blocks", type=int, default=32, help="blocks of the stack leg (profiling-sized runs)")
    ap.add_argument("--stack-steps", type=int, default=10, help="timed steps of the stack leg")
    ap.add_argument("--only", choices=["nvfp4", "swiglu", "stack", "diagnostic", "qkv"], default=None,
                    help="run just one of the other legs (sized by --tokens) and print its numbers")
    ap.add_argument("--tokens", type=int, default=None,
                    help="token count (default 8192); smaller values make a profiling-sized case")
    args = ap.parse_args()
    if args.tokens:
        global T
        T = int(args.tokens)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.only:
        import torch
        torch.cuda.set_device(0)
        print(json.dumps({"only": args.only, "legs": run_legs(args, load_peaks(), args.only)}), flush=True)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
