"""Pins of the oracle's scalar formats against facts fixed by the pages and by
the format definitions (closed forms, brute force, library conversions).

Format-Aware Fusion for Fast FP4 Pretraining, Sec. 2.2 / 2.2.1 / 2.2.2.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from synthetic import bf16_bits_from_f32, f32_from_bf16_bits


# ---------------------------------------------------------------- E2M1 -----

def _e2m1_closed_form(code: int) -> float:
    # 1 sign, 2 exponent (bias 1), 1 fraction bit; exponent 0 is subnormal.
    s, e, m = code >> 3, (code >> 1) & 3, code & 1
    mag = (m * 0.5) if e == 0 else (1.0 + 0.5 * m) * 2.0 ** (e - 1)
    return -mag if s else mag


def test_e2m1_grid_matches_bit_layout_and_max(paper_facts):
    bits = paper_facts["e2m1_bits"]
    assert (bits["sign"], bits["exponent"], bits["fraction"]) == (1, 2, 1)
    vals = [oracle.e2m1_value(c) for c in range(16)]
    assert vals == [_e2m1_closed_form(c) for c in range(16)]
    assert max(vals) == paper_facts["e2m1_max"]
    assert sorted(set(abs(v) for v in vals)) == [0, 0.5, 1, 1.5, 2, 3, 4, 6]


# Rounding boundaries: midpoints between neighbouring magnitudes; a midpoint
# goes to the neighbour whose fraction bit is 0 (even code).
_MAG = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _e2m1_by_thresholds(v: float) -> int:
    a = abs(v)
    idx = 7
    for k in range(7):
        mid = (_MAG[k] + _MAG[k + 1]) / 2
        if a < mid or (a == mid and k % 2 == 0):
            idx = k
            break
    return (8 if math.copysign(1.0, v) < 0 else 0) | idx


def test_e2m1_rn_ties_and_saturation():
    expect = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6,
              6.0: 7, 7.0: 7, 1e30: 7, 0.0: 0, 0.2: 0, 0.3: 1, 5.01: 7}
    for v, c in expect.items():
        assert oracle.e2m1_rn(v) == c, v
        assert oracle.e2m1_rn(-v) == 8 | c, -v
    # the sign of a value that rounds to zero is kept
    assert oracle.e2m1_rn(-0.1) == 8
    assert oracle.e2m1_rn(-0.0) == 8


def test_e2m1_rn_every_bf16_value_unscaled():
    # Every finite bf16 value below 1e3 as it stands (scale 1), against the
    # threshold rule; the sweep over every landing exponent is in
    # test_oracle_bruteforce.py.
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    f = f32_from_bf16_bits(bits)
    f = f[np.isfinite(f)].astype(np.float64)
    f = f[np.abs(f) < 1e3]
    for v in f:
        assert oracle.e2m1_rn(float(v)) == _e2m1_by_thresholds(float(v))


def test_e2m1_sr_grid_values_fixed_and_bins():
    for c in range(8):
        v = _MAG[c]
        for u in (0, 1, 12345, 65535):
            assert oracle.e2m1_sr(v, u) == c
            assert oracle.e2m1_sr(-v, u) == 8 | c
    # p = 1/4 inside (1, 1.5): up iff u/65536 < 0.25
    assert oracle.e2m1_sr(1.125, 16383) == 3
    assert oracle.e2m1_sr(1.125, 16384) == 2
    # saturation
    assert oracle.e2m1_sr(6.5, 0) == 7 and oracle.e2m1_sr(100.0, 65535) == 7


# ---------------------------------------------------------------- E8M0 -----

def test_e8m0_upward_exponent_is_minimal_no_clip():
    rng = np.random.default_rng(7)
    vals = list(np.exp(rng.uniform(-80, 80, 4000))) + [6.0, 6.0000001, 3.0, 12.0, 1.0, 1.5, 0.75]
    for a in vals:
        e = oracle.e8m0_exponent_up(float(a))
        assert Fraction(6) * Fraction(2) ** e >= Fraction(float(a))
        if e > -127:
            assert Fraction(6) * Fraction(2) ** (e - 1) < Fraction(float(a))
        # closed form ceil(log2(a / 6)) (exact with Fractions)
        fa = Fraction(float(a)) / 6
        k = math.floor(math.log2(float(fa)))
        while Fraction(2) ** k < fa:
            k += 1
        while k - 1 >= -300 and Fraction(2) ** (k - 1) >= fa:
            k -= 1
        assert e == max(-127, min(127, k))
    assert oracle.e8m0_exponent_up(0.0) == -127


def test_e8m0_byte_decodes_like_torch_e8m0():
    # dequantize a block whose codes are all 1.0 under every scale byte 0..254
    sc = np.arange(0, 255, dtype=np.uint8).reshape(-1, 1)
    q = dict(codes=np.full((255, 32), 2, np.uint8), scales=sc, senc=None, fmt=0, bs=32)
    deq = oracle.dequantize(q)[:, 0]
    ref = torch.from_numpy(sc[:, 0].copy()).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    assert np.array_equal(deq, ref)


def test_weight2d_fine_rule(paper_facts):
    c = paper_facts["weight2d_fine_ratio"]
    rng = np.random.default_rng(3)
    for a in list(np.exp(rng.uniform(-40, 40, 3000))) + [6.0, 5.22, 5.25, 5.1875, 3.0]:
        # tile amax values of bf16 weights are bf16 numbers
        a = float(f32_from_bf16_bits(bf16_bits_from_f32(np.array([a], np.float32)))[0])
        e = oracle.e8m0_exponent_up(a)
        ef = oracle.mx_weight_tile_exponent(a)
        ratio = a / (6.0 * 2.0 ** e)
        if ratio < c:
            assert ef == max(e - 1, -127)
            # bounded upper-tail clipping: the finer span is at most 2 * 0.87 short
            assert a / (6.0 * 2.0 ** ef) < 2 * c + 1e-6
        else:
            assert ef == e


# ---------------------------------------------------------------- E4M3 -----

def test_e4m3_decode_matches_torch(paper_facts):
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = np.array([oracle.e4m3_value(int(c)) for c in codes])
    fin = np.isfinite(ref)
    assert np.array_equal(mine[fin], ref[fin])
    assert np.isnan(mine[~fin]).all()
    assert max(mine[fin]) == paper_facts["e4m3_max"]


def test_e4m3_encode_exhaustive_midpoints_vs_torch():
    vals = sorted(oracle.e4m3_value(c) for c in range(0x7F))
    probes = set(vals)
    for a, b in zip(vals, vals[1:]):
        mid = (a + b) / 2
        probes.update([mid, np.nextafter(mid, 0), np.nextafter(mid, 1e9), (a + mid) / 2])
    probes = np.array(sorted(probes), dtype=np.float64)
    probes = probes[probes <= 448.0]
    probes32 = probes.astype(np.float32).astype(np.float64)
    ref = torch.from_numpy(probes32.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    mine = np.array([oracle.e4m3_rn_satfinite(float(p)) for p in probes32], dtype=np.uint8)
    assert np.array_equal(mine, ref)
    # saturation instead of NaN above the largest finite value
    for s in (448.0, 460.0, 464.0, 500.0, 1e9, 3.4e38):
        assert oracle.e4m3_rn_satfinite(s) == 0x7E


def test_e4m3_scale_underflows_to_zero(paper_facts):
    assert paper_facts["e4m3_scale_can_underflow"]
    # a block amax tiny against the outer factor gets the zero scale and m = 0
    d, m = oracle.nv_block_scale(1e-6, 1.0)
    assert d == 0 and m == 0.0


def test_nv_senc():
    assert oracle.nv_senc(0.0) == 1.0
    assert oracle.nv_senc(2688.0) == 1.0
    assert oracle.nv_senc(1.0) == np.float32(2688.0)
    assert oracle.nv_senc(1e-40) == np.finfo(np.float32).max
    a = np.float32(3.3)
    assert oracle.nv_senc(float(a)) == np.float32(np.float32(2688.0) / a)


# ---------------------------------------------------------------- bf16 -----

def test_bf16_round_matches_torch():
    rng = np.random.default_rng(11)
    v = np.concatenate([rng.standard_normal(20000) * np.exp(rng.uniform(-30, 30, 20000)),
                        [1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8), 1e-40, 2 ** -133, 0.0]])
    v = v.astype(np.float32).astype(np.float64)  # single rounding on both sides
    ref = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).view(torch.uint16).numpy().astype(np.uint16)
    mine = oracle.round_bf16(v)
    assert np.array_equal(mine, ref)
