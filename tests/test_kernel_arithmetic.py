"""Host checks of the two exact-arithmetic shortcuts the kernels take instead
of the plain rules, restated here in Python from the kernels' comments (the
GPU parity tests then compare the kernels themselves with the oracle):

* stochastic rounding (Format-Aware Fusion for Fast FP4 Pretraining, Sec. 2.5,
  Eq. 9) by a carry into the grid bit: b = max(|v|, fl_up((|v| + 1) / 2)),
  code = (bits(b) + 2^22 - 1 - u * 2^6 - 0x3F000000) >> 22, saturated at 7;
  compared with the oracle's rule (round up iff u / 2^16 < p) on values at,
  next to and between every 2^-16 step of every grid interval; the kernels
  form the addend as the 32-bit multiply-add u * (2^32 - 64) + K and gather
  the 8 sign bits of a code word with byte permutes, both checked here
  against the plain forms;
* fl32(a / 6) of a bf16 block maximum (the NVFP4 scale, Sec. 2.2.2) as
  RN(q + RN(a - 6 q) * c), q = RN(a * c), c = RN(1 / 6), compared with the
  correctly rounded quotient for every finite positive bf16 value.
"""
import struct
from fractions import Fraction

import numpy as np

import oracle

MAG = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def f2b(f: float) -> int:
    return struct.unpack("<I", struct.pack("<f", f))[0]


def b2f(b: int) -> float:
    return struct.unpack("<f", struct.pack("<I", b))[0]


def rn32(x: Fraction) -> Fraction:
    """Correct rounding of a rational to binary32 (subnormals included)."""
    if x == 0:
        return Fraction(0)
    s = -1 if x < 0 else 1
    x = abs(x)
    e = x.numerator.bit_length() - x.denominator.bit_length()
    if Fraction(2) ** e > x:
        e -= 1
    if Fraction(2) ** (e + 1) <= x:
        e += 1
    q = Fraction(2) ** (max(e, -126) - 23)
    n = x / q
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return s * fl * q


def up32(x: Fraction) -> float:
    """Round a positive rational up to binary32 (normal range)."""
    r = rn32(x)
    if r < x:
        r = Fraction(b2f(f2b(float(r)) + 1))
    return float(r)


def carry_code(a: float, u: int) -> int:
    b = max(f2b(a), f2b(up32(Fraction(a) / 2 + Fraction(1, 2))))
    r = ((u << 6) & 0x3FFFC0) ^ 0x3FFFFF
    return min(((b + r - 0x3F000000) & 0xFFFFFFFF) >> 22, 7)


def test_sr_carry_rule_equals_the_oracle_rule():
    rng = np.random.default_rng(2)
    vals = [0.0, 1e-45, 2.0 ** -126, 0.25, 0.75, 1.0, 5.999, 6.0, 7.0, 1e30]
    for k in range(7):
        lo, hi = MAG[k], MAG[k + 1]
        for t in list(range(0, 65536, 211)) + [0, 1, 32767, 32768, 65535]:
            v = float(Fraction(lo) + Fraction(hi - lo) * Fraction(t, 65536))
            vals += [v] + ([b2f(f2b(v) - 1)] if v > 0 else []) + [b2f(f2b(v) + 1)]
    vals += [b2f(int(b)) for b in rng.integers(0, 0x40E00000, 4000)]
    n = 0
    for v in vals:
        q = Fraction(v)
        us = [0, 1, 32767, 32768, 65535] + [int(x) for x in rng.integers(0, 65536, 2)]
        lo = max(k for k in range(8) if Fraction(MAG[k]) <= q)
        if lo < 7:  # the uniforms either side of the threshold p * 2^16
            th = int((q - Fraction(MAG[lo])) / (Fraction(MAG[lo + 1]) - Fraction(MAG[lo])) * 65536)
            us += [max(0, th - 1), th, min(65535, th + 1)]
        for u in us:
            assert carry_code(v, u) == oracle.e2m1_sr(v, u), (v, u)
            n += 1
    assert n > 100000


def test_division_by_six_is_correctly_rounded_for_every_bf16():
    c = rn32(Fraction(1, 6))
    for b in range(1, 0x7F80):
        a = Fraction(b2f(b << 16))
        q = rn32(a * c)
        r = rn32(a - 6 * q)
        assert rn32(q + r * c) == rn32(a / 6), hex(b)


def prmt(a: int, b: int, sel: int) -> int:
    """prmt.b32 in its default mode: byte n of d is byte (sel_n & 7) of the
    8 bytes {b, a}, or that byte's sign replicated when sel_n & 8."""
    src = [(a >> (8 * i)) & 0xFF for i in range(4)] + [(b >> (8 * i)) & 0xFF for i in range(4)]
    d = 0
    for n in range(4):
        s = (sel >> (4 * n)) & 0xF
        byte = src[s & 7]
        if s & 8:
            byte = 0xFF if byte & 0x80 else 0
        d |= byte << (8 * n)
    return d


def test_sr_addend_multiply_add_form():
    rng = np.random.default_rng(3)
    k = (0x3FFFFF - 0x3F000000) & 0xFFFFFFFF
    words = [0, 0xFFFFFFFF, 0xFFFF, 0xFFFF0000] + [int(x) for x in rng.integers(0, 2**32, 20000, dtype=np.uint64)]
    for rw in words:
        for u in (rw & 0xFFFF, rw >> 16):
            plain = ((((u << 6) & 0x3FFFC0) ^ 0x3FFFFF) - 0x3F000000) & 0xFFFFFFFF
            assert (u * 0xFFFFFFC0 + k) & 0xFFFFFFFF == plain, hex(rw)


def test_sign_gather_by_byte_permutes():
    rng = np.random.default_rng(4)
    for _ in range(20000):
        w = [int(x) for x in rng.integers(0, 2**32, 4, dtype=np.uint64)]
        p01, p23 = prmt(w[0], w[1], 0x7351), prmt(w[2], w[3], 0x7351)
        even, odd = prmt(p01, p23, 0xDC98), prmt(p01, p23, 0xFEBA)
        got = ((even & 0x0F0F0F0F) | (odd & 0xF0F0F0F0)) & 0x88888888
        want = 0
        for b in range(4):  # value 2b: bit 15 of word b -> bit 8b + 3; value 2b + 1: bit 31 -> 8b + 7
            want |= ((w[b] >> 15) & 1) << (8 * b + 3)
            want |= ((w[b] >> 31) & 1) << (8 * b + 7)
        assert got == want
