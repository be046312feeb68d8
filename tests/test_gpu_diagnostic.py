"""The Dgrad-error diagnostic (Format-Aware Fusion for Fast FP4 Pretraining,
Sec. 5.2 and Appendix C.4) against the oracle: the error energies of the
MXFP4 and CTA-local NVFP4 Dgrads measured through the C ABI equal the ones
the oracle computes from its own views and the exact binary64 product, up to
the FP32 accumulation of the contraction and of the reference."""
import numpy as np
import pytest
import torch

import oracle
from fp4_quantized_linears_gb300.diagnostic import dgrad_diagnostic, dgrad_error_energy
from synthetic import normal_bf16, student_t_unitvar_bf16

pytestmark = pytest.mark.gpu


def to_dev(b):
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).cuda()


def test_error_energies_match_the_oracle():
    dy = student_t_unitvar_bf16((256, 512), 4.0, 71, 1)
    w = normal_bf16((512, 384), 0.02, 71, 2)
    got = dgrad_error_energy(to_dev(dy), to_dev(w), sr_seed=3)
    ref = oracle.bf16_to_f32(dy).astype(np.float64) @ oracle.bf16_to_f32(w).astype(np.float64)
    want = {}
    for route in ("mx", "nv_local"):
        a = oracle.quantize(dy, route, "row", sr=True, seed=3)
        b = oracle.quantize(w, route, "col", weight2d=True)
        want[route] = float(((oracle.gemm(a, b) - ref) ** 2).sum())
    assert abs(got["E_mx"] / want["mx"] - 1) < 1e-4
    assert abs(got["E_local"] / want["nv_local"] - 1) < 1e-4
    assert abs(got["ratio"] / (want["mx"] / want["nv_local"]) - 1) < 2e-4


def test_small_diagnostic_runs_and_is_deterministic():
    a = dgrad_diagnostic(blocks=2, batches=1, T=256, comps=("qkv", "o"))
    b = dgrad_diagnostic(blocks=2, batches=1, T=256, comps=("qkv", "o"))
    assert a == b and a["pairs"] == 4 and a["geomean"] > 0
