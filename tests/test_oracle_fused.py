"""Pins of the fused-producer model arithmetic (Format-Aware Fusion for Fast
FP4 Pretraining, Sec. 3.2) against torch's float64 SiLU / RMSNorm and their
autograd gradients (library routines)."""
import numpy as np
import torch

import oracle
from synthetic import f32_from_bf16_bits, normal_bf16


def _bf(bits):
    return torch.from_numpy(f32_from_bf16_bits(bits).astype(np.float64))


def _ulp_diff(a_bits, b_bits):
    a = a_bits.astype(np.int32)
    b = b_bits.astype(np.int32)
    # map sign-magnitude to ordered ints
    a = np.where(a & 0x8000, -(a & 0x7FFF), a)
    b = np.where(b & 0x8000, -(b & 0x7FFF), b)
    return np.abs(a - b)


def test_swiglu_forward_and_backward_vs_torch():
    a1 = normal_bf16((64, 128), 2.0, 1, 1)
    a3 = normal_bf16((64, 128), 2.0, 1, 2)
    dh = normal_bf16((64, 128), 1e-3, 1, 3)
    h = oracle.swiglu_h(a1, a3)
    t1, t3 = _bf(a1).requires_grad_(), _bf(a3).requires_grad_()
    ref = torch.nn.functional.silu(t1) * t3
    ref_bits = ref.detach().to(torch.float32).to(torch.bfloat16).view(torch.uint16).numpy().astype(np.uint16)
    assert _ulp_diff(h, ref_bits).max() <= 1
    ref.backward(_bf(dh))
    da1, da3 = oracle.swiglu_bwd(dh, a1, a3)
    g1 = t1.grad.to(torch.float32).to(torch.bfloat16).view(torch.uint16).numpy().astype(np.uint16)
    g3 = t3.grad.to(torch.float32).to(torch.bfloat16).view(torch.uint16).numpy().astype(np.uint16)
    assert _ulp_diff(da1, g1).max() <= 1 and _ulp_diff(da3, g3).max() <= 1


def test_residual_rmsnorm_forward_and_backward_vs_torch():
    R, C = 32, 256
    r = normal_bf16((R, C), 1.0, 2, 1)
    b = normal_bf16((R, C), 1.0, 2, 2)
    g = normal_bf16((C,), 1.0, 2, 3)
    rp, rstd, y = oracle.residual_rmsnorm(r, b, g, 1e-5)
    # r' is a single bf16 rounding of the exact sum
    s = (_bf(r) + _bf(b)).to(torch.float32).to(torch.bfloat16).view(torch.uint16).numpy().astype(np.uint16)
    assert np.array_equal(rp, s)
    t = _bf(rp).requires_grad_()
    ref = torch.nn.functional.rms_norm(t, (C,), weight=_bf(g), eps=1e-5)
    ref_rstd = torch.rsqrt((_bf(rp) ** 2).mean(-1) + 1e-5).to(torch.float32).numpy()
    assert np.array_equal(rstd, ref_rstd)
    yb = ref.detach().to(torch.float32).to(torch.bfloat16).view(torch.uint16).numpy().astype(np.uint16)
    assert _ulp_diff(y, yb).max() <= 1
    dy = normal_bf16((R, C), 1.0, 2, 4)
    dres = normal_bf16((R, C), 1.0, 2, 5)
    ref.backward(_bf(dy))
    want = (t.grad + _bf(dres)).to(torch.float32).to(torch.bfloat16).view(torch.uint16).numpy().astype(np.uint16)
    got = oracle.rmsnorm_bwd(dy, rp, rstd, g, dres)
    # the oracle uses the binary32 rstd; torch recomputes it in float64
    assert _ulp_diff(got, want).max() <= 1
