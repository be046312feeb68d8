"""Controlled Dgrad-error diagnostic of "Format-Aware Fusion for Fast FP4
Pretraining" (Sec. 3.3 and Sec. 5.2, Appendix C.4): on identical BF16
tensors, recompute the input gradient dX = dY . W with MXFP4 and with
CTA-local NVFP4, measure each one's error energy against the unquantized
product, and compare them as the ratio E_MX / E_localCTA (the pages report a
geometric mean of 1.292 over 288 captured layer-component pairs; the captured
tensors are not available, so the diagnostic runs on seeded synthetic ones).

Each Dgrad follows its route's contract: the row-facing dY with stochastic
rounding (MXFP4 E8M0 32-blocks, or CTA-local NVFP4 E4M3 16-blocks under the
128-row strip factors) against the column-facing 2D weight (2D32 MXFP4, or
2D16 NVFP4 under the tensor factor).  The reference is the plain product of
the BF16 operands accumulated in FP32 (a library GEMM; it is the yardstick,
not part of the FP4 path).  Error energy E = sum((dX_q - dX_ref)^2)."""
from __future__ import annotations

import math

import torch

from . import (FP4_FLAG_SR_ROW, FP4_FLAG_WEIGHT_2D, FP4_VIEW_COL, FP4_VIEW_ROW, fp4_linear_dgrad, fp4_quantize)

COMPONENTS = {  # name: (rows of W = width of dY, cols of W = width of dX), Llama-3-8B shapes
    "qkv": (6144, 4096),
    "o": (4096, 4096),
    "w13": (2 * 14336, 4096),
    "w2": (4096, 14336),
}


def dgrad_error_energy(dy: torch.Tensor, w: torch.Tensor, sr_seed: int = 1) -> dict:
    """dy [T, n_out] and w [n_out, n_in] bf16 CUDA tensors -> error energies
    of the MXFP4 and CTA-local NVFP4 Dgrads and their ratio."""
    ref = torch.matmul(dy.float(), w.float())
    out = {}
    for route in ("mx", "nv_local"):
        dr, _ = fp4_quantize(dy, route, FP4_VIEW_ROW, FP4_FLAG_SR_ROW, sr_seed=sr_seed)
        _, wc = fp4_quantize(w, route, FP4_VIEW_COL, FP4_FLAG_WEIGHT_2D)
        dx = fp4_linear_dgrad(dr, wc)
        out[route] = float(((dx.double() - ref.double()) ** 2).sum())
    return dict(E_mx=out["mx"], E_local=out["nv_local"], ratio=out["mx"] / out["nv_local"],
                E_ref=float((ref.double() ** 2).sum()))


def synthetic_pair(comp: str, T: int, block: int, batch: int, seed: int = 5, device="cuda"):
    """Seeded synthetic (dY, W) of one component: W ~ N(0, 0.02) per block;
    dY heavy-tailed (Student-t with 4 degrees of freedom, unit variance,
    scaled by 1e-4) per block and batch."""
    n_out, n_in = COMPONENTS[comp]
    ci = list(COMPONENTS).index(comp)
    gw = torch.Generator(device=device).manual_seed(seed * 100003 + block * 97 + ci)
    w = (torch.randn((n_out, n_in), generator=gw, device=device) * 0.02).to(torch.bfloat16)
    gd = torch.Generator(device=device).manual_seed(seed * 100003 + block * 97 + batch * 7919 + 1000 + ci)
    z = torch.randn((T, n_out), generator=gd, device=device)
    chi = torch.randn((4, T, n_out), generator=gd, device=device).pow(2).sum(0) / 4.0
    dy = (z / chi.sqrt() / math.sqrt(2.0) * 1e-4).to(torch.bfloat16)
    return dy, w


def dgrad_diagnostic(blocks: int = 32, batches: int = 3, T: int = 2048, comps=tuple(COMPONENTS), seed: int = 5):
    """Every (block, batch, component) pair: per-pair ratios, the geometric
    mean overall and per component, and how many pairs favour CTA-local."""
    ratios = {c: [] for c in comps}
    for b in range(blocks):
        for k in range(batches):
            for c in comps:
                dy, w = synthetic_pair(c, T, b, k, seed)
                ratios[c].append(dgrad_error_energy(dy, w, sr_seed=seed + b * 16 + k)["ratio"])
    allr = [r for c in comps for r in ratios[c]]

    def gmean(v):
        return math.exp(sum(math.log(x) for x in v) / len(v))

    return dict(pairs=len(allr), geomean=gmean(allr), favour_local=sum(r > 1.0 for r in allr),
                per_component={c: gmean(v) for c, v in ratios.items()})
