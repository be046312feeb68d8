"""Seeded synthetic inputs for the FP4 linear boundary.

This module only draws random tensors.  It holds none of the quantization,
rounding or contraction arithmetic: both the CUDA path and the CPU oracle take
the bytes produced here as their input, and nothing here imports either side.

Distributions follow the workloads of "Format-Aware Fusion for Fast FP4
Pretraining" (Llama-3-8B linear shapes, Sec. 4.1): normal weights with standard
deviation 0.02, activations with unit variance (optionally heavy-tailed or with
sparse x20 outliers), and small-magnitude gradients.  N(mu, s) below means
standard deviation s.

BF16 tensors are returned as numpy ``uint16`` bit patterns (row-major), made by
round-to-nearest-even from float32 samples.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "bf16_bits_from_f32",
    "f32_from_bf16_bits",
    "normal_bf16",
    "student_t_unitvar_bf16",
    "with_outliers_bf16",
    "hadamard_signs",
    "config_tensors",
    "CONFIGS",
]


def bf16_bits_from_f32(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); return uint16 bits."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    bias = ((u >> 16) & 1) + 0x7FFF
    return ((u + bias) >> 16).astype(np.uint16)


def f32_from_bf16_bits(b: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns to float32 (exact)."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([int(seed), int(stream)]))


def normal_bf16(shape, std: float, seed: int, stream: int) -> np.ndarray:
    g = _rng(seed, stream)
    a = g.standard_normal(size=shape, dtype=np.float32)
    a *= np.float32(std)
    return bf16_bits_from_f32(a)


def student_t_unitvar_bf16(shape, nu: float, seed: int, stream: int) -> np.ndarray:
    """Student-t(nu) samples divided by sqrt(nu/(nu-2)), i.e. unit variance."""
    g = _rng(seed, stream)
    a = g.standard_t(nu, size=shape) / np.sqrt(nu / (nu - 2.0))
    return bf16_bits_from_f32(a.astype(np.float32))


def with_outliers_bf16(shape, std: float, frac: float, mult: float, seed: int,
                       stream: int) -> np.ndarray:
    """N(0, std) samples with round(frac * n) positions (drawn by the seed) scaled by mult."""
    g = _rng(seed, stream)
    a = g.standard_normal(size=shape, dtype=np.float32) * np.float32(std)
    n = a.size
    k = int(round(frac * n))
    if k:
        pos = g.choice(n, size=k, replace=False)
        a.reshape(-1)[pos] *= np.float32(mult)
    return bf16_bits_from_f32(a)


def hadamard_signs(seed: int) -> np.ndarray:
    """A fixed 16-entry +-1 sign vector drawn from the seed (int8)."""
    g = _rng(seed, 0x5167)
    return np.where(g.integers(0, 2, size=16) == 1, -1, 1).astype(np.int8)


# Shapes of the five workloads (tokens, d, f or out) and their seeds.
CONFIGS = {
    "c1_mx_small": dict(seed=0, T=256, d_in=512, d_out=512),
    "c2_mx_w1": dict(seed=1, T=8192, d_in=4096, d_out=14336),
    "c3_nv_attn": dict(seed=2, T=8192, d_in=4096, d_out=4096, d_out_qkv=6144),
    "c4_swiglu": dict(seed=3, T=16384, d=4096, f=14336),
    "c5_stack": dict(seed=5, T=8192, d=4096, f=14336, qkv=6144, blocks=32, local_blocks=27),
}


def config_tensors(name: str, scale_T: int | None = None, **over):
    """Draw the input tensors of one workload.

    ``scale_T`` replaces the token count (and, for square shapes, nothing else),
    so that the same distributions can be drawn at a reduced size.
    Returns a dict of uint16 bf16 arrays (plus ``signs`` for the H32 workload).
    """
    cfg = dict(CONFIGS[name])
    cfg.update(over)
    s = cfg["seed"]
    T = scale_T if scale_T is not None else cfg["T"]
    if name == "c1_mx_small":
        di, do = cfg["d_in"], cfg["d_out"]
        return dict(
            x=with_outliers_bf16((T, di), 1.0, 1e-3, 20.0, s, 1),
            w=normal_bf16((do, di), 0.02, s, 2),
            dy=normal_bf16((T, do), 1e-3, s, 3),
        )
    if name == "c2_mx_w1":
        di, do = cfg["d_in"], cfg["d_out"]
        return dict(
            x=student_t_unitvar_bf16((T, di), 4.0, s, 1),
            w=normal_bf16((do, di), 0.02, s, 2),
            dy=normal_bf16((T, do), 1e-4, s, 3),
            signs=hadamard_signs(s),
        )
    if name == "c3_nv_attn":
        di, do, dq = cfg["d_in"], cfg["d_out"], cfg["d_out_qkv"]
        return dict(
            x=with_outliers_bf16((T, di), 1.0, 1e-3, 20.0, s, 1),
            w=normal_bf16((do, di), 0.02, s, 2),
            w_qkv=normal_bf16((dq, di), 0.02, s, 4),
            dy=normal_bf16((T, do), 1e-3, s, 3),
            dy_qkv=normal_bf16((T, dq), 1e-3, s, 5),
        )
    if name == "c4_swiglu":
        d, f = cfg["d"], cfg["f"]
        return dict(
            x=normal_bf16((T, d), 1.0, s, 1),
            w13=normal_bf16((2 * f, d), 0.02, s, 2),  # rows [0,f) = W1, [f,2f) = W3
            w2=normal_bf16((d, f), 0.02, s, 3),
            dy2=normal_bf16((T, d), 1e-4, s, 4),
        )
    if name == "c5_stack":
        d = cfg["d"]
        return dict(
            x=normal_bf16((T, d), 1.0, s, 1),
            dy=normal_bf16((T, d), 1e-4, s, 2),
        )
    raise KeyError(name)


def c5_block_weights(block: int, d: int, f: int, qkv: int, seed: int = 5):
    """Weights of one block of the stacked workload: per-block substreams of the seed."""
    base = 1000 + 10 * block
    return dict(
        w_qkv=normal_bf16((qkv, d), 0.02, seed, base + 1),
        w_o=normal_bf16((d, d), 0.02, seed, base + 2),
        w13=normal_bf16((2 * f, d), 0.02, seed, base + 3),
        w2=normal_bf16((d, f), 0.02, seed, base + 4),
    )
