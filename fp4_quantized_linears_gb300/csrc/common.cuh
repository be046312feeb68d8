// common.cuh -- device helpers shared by the fp4lin kernels (sm_103a).
//
// Number formats of "Format-Aware Fusion for Fast FP4 Pretraining", Sec. 2.2:
// E2M1 values, E8M0 and E4M3 block scales; Philox4x32-10 (Salmon et al.,
// SC'11) for the stochastic rounding of Sec. 2.5.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/fp4lin.h"

#define FP4_DEV __device__ __forceinline__

namespace fp4 {

// ---------------------------------------------------------------- status ---
// Each translation unit keeps its own sticky status word; the API reads all.
// The first error code wins.
FP4_DEV void set_status(unsigned int* word, int code) { atomicCAS(word, 0u, (unsigned int)code); }

// ----------------------------------------------------------------- bf16 ----
FP4_DEV float bf16_lo(uint32_t pair) { return __uint_as_float(pair << 16); }
FP4_DEV float bf16_hi(uint32_t pair) { return __uint_as_float(pair & 0xFFFF0000u); }
FP4_DEV float bf16_to_f32(uint16_t h) { return __uint_as_float(((uint32_t)h) << 16); }

// Round-to-nearest-even binary32 -> bf16 bits (finite inputs).
FP4_DEV uint16_t f32_to_bf16_rn(float f) {
    uint32_t u = __float_as_uint(f);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

// --------------------------------------------------------------- E2M1 RN ---
// Two binary32 values -> one byte of two E2M1 codes, `lo` in the low nibble,
// round to nearest even with saturation at 6 (the hardware conversion).  The
// conversion keeps the sign of a value that rounds to zero (code 8 for -0.1),
// which the exhaustive quantizer parity tests check against the oracle.
FP4_DEV uint32_t e2m1x2_rn(float lo, float hi) {
    uint32_t r;
    asm("{\n\t.reg .b8 t;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
        "cvt.u32.u8 %0, t;\n\t}"
        : "=r"(r)
        : "f"(hi), "f"(lo));
    return r;
}

// Eight binary32 values -> one word of eight E2M1 codes (value 2k in the low
// nibble of byte k), four conversions assembled into the word by one vector
// move; the same rounding as e2m1x2_rn.
FP4_DEV uint32_t e2m1x8_rn(float a0, float a1, float a2, float a3, float a4, float a5, float a6, float a7) {
    uint32_t r;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(r)
        : "f"(a0), "f"(a1), "f"(a2), "f"(a3), "f"(a4), "f"(a5), "f"(a6), "f"(a7));
    return r;
}

// ----------------------------------------------------- packed binary32 ----
// Two binary32 lanes per instruction (f32x2 arithmetic of sm_100 and later):
// each lane is the correctly rounded result of the scalar operation on
// that lane (to nearest even, or upward for fma_rp), so a pair op and two
// scalar ops give the same bits.
FP4_DEV void f32x2_add(float& x, float& y, float a0, float a1, float b0, float b1) {
    asm("{\n\t.reg .b64 a, b, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
        "add.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(x), "=f"(y) : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
FP4_DEV void f32x2_sub(float& x, float& y, float a0, float a1, float b0, float b1) {
    asm("{\n\t.reg .b64 a, b, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
        "sub.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(x), "=f"(y) : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
FP4_DEV void f32x2_fma(float& x, float& y, float a0, float a1, float b0, float b1, float c0, float c1) {
    asm("{\n\t.reg .b64 a, b, c, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\tmov.b64 c, {%6, %7};\n\t"
        "fma.rn.f32x2 d, a, b, c;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(x), "=f"(y) : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}
FP4_DEV void f32x2_fma_rp(float& x, float& y, float a0, float a1, float b0, float b1, float c0, float c1) {
    asm("{\n\t.reg .b64 a, b, c, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\tmov.b64 c, {%6, %7};\n\t"
        "fma.rp.f32x2 d, a, b, c;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(x), "=f"(y) : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}
FP4_DEV void f32x2_mul(float& x, float& y, float a0, float a1, float b0, float b1) {
    asm("{\n\t.reg .b64 a, b, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
        "mul.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(x), "=f"(y) : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
// max(m, |a|, |b|), NaN if any operand is NaN (so a NaN input still reaches
// the non-finite check through the block maximum).
FP4_DEV float max3_abs_nan(float m, float a, float b) {
    float d;
    asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(m), "f"(fabsf(a)), "f"(fabsf(b)));
    return d;
}

// --------------------------------------------------------------- E2M1 SR ---
// Adjacent-bin stochastic rounding (Sec. 2.5, Eq. 9): with q- <= |v| < q+
// neighbouring grid values, round up iff u * 2^-16 < p = (|v| - q-) / (q+ - q-)
// for a 16-bit uniform u; |v| >= 6 saturates.  Evaluated exactly on the bits:
//   |v| >= 1: the grid has one fraction bit, q- is |v| truncated to it (code
//     (bits - 0x3F000000) >> 22) and p = low22 / 2^22 (the 22 fraction bits
//     below it).  Adding r = 2^22 - 1 - u * 2^6 to the bits carries into the
//     grid bit exactly when u * 2^6 < low22, i.e. when the value rounds up;
//   |v| < 1: the grid 0, 0.5, 1 has step 0.5 = the grid step of [1, 2), so
//     |v| is first mapped to b = (|v| + 1) / 2 in [0.5, 1], rounded upward to
//     binary32; b has the same fraction of a grid step (rounded up to a
//     multiple of 2^-22 of the step, which leaves the comparison with u * 2^-16
//     unchanged), and the same carry rule gives codes 0, 1, 2.  Because
//     (|v| + 1) / 2 > |v| exactly when |v| < 1, b = max(|v|, that) selects the
//     right form without a branch (integer max on the bit patterns).
// sr_code_pair takes the two scaled magnitudes and returns their two 3-bit
// magnitude codes (x in the low nibble); rw holds u_x in its low and u_y in
// its high 16 bits.
// SAT: saturate at code 7 (|v| >= 6).  Without it the caller guarantees
// |v| <= 6, as an MXFP4 block under its upward scale does (6 * 2^e >= amax,
// and scaling by 2^-e is exact); then b <= 6 and the code is at most 7.
//
// The encoders are bound by the integer ALU pipe, so the addends
// 2^22 - 1 - u * 2^6 - 0x3F000000 (mod 2^32) are formed as u * -64 + K by
// the integer multiply-add, which issues to the multiply-add pipe instead,
// and the sign bits of 8 values are gathered once per code word by byte
// permutes (prmt with the sign-replicating selector nibbles 8-15).
FP4_DEV uint32_t mad_lo_u32(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("mad.lo.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
FP4_DEV uint32_t prmt_b32(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}
template <bool SAT = true>
FP4_DEV uint32_t sr_code_pair(float ax, float ay, uint32_t rw) {
    constexpr uint32_t K = 0x3FFFFFu - 0x3F000000u;
    float cx, cy;
    f32x2_fma_rp(cx, cy, ax, ay, 0.5f, 0.5f, 0.5f, 0.5f);  // fl_up((|v| + 1) / 2)
    const uint32_t tx = max(__float_as_uint(ax), __float_as_uint(cx));
    const uint32_t ty = max(__float_as_uint(ay), __float_as_uint(cy));
    uint32_t hx = (tx + mad_lo_u32(rw & 0xFFFFu, 0xFFFFFFC0u, K)) >> 22;
    uint32_t hy = (ty + mad_lo_u32(rw >> 16, 0xFFFFFFC0u, K)) >> 22;
    if (SAT) {
        hx = min(hx, 7u);
        hy = min(hy, 7u);
    }
    return hx | (hy << 4);
}
// The sign bits of the 8 bf16 values of 4 words (word b: values 2b low half,
// 2b + 1 high half) at the sign positions 4k + 3 of a word of 8 codes: the
// high bytes of the halves (bytes 1 and 3 of each word) are collected, the
// even values' bytes and the odd values' bytes each sign-replicated into one
// word, and nibble k takes its sign from the matching one.
FP4_DEV uint32_t e2m1x8_signs(const uint32_t* w) {
    const uint32_t p01 = prmt_b32(w[0], w[1], 0x7351u), p23 = prmt_b32(w[2], w[3], 0x7351u);
    const uint32_t even = prmt_b32(p01, p23, 0xDC98u), odd = prmt_b32(p01, p23, 0xFEBAu);
    return ((even & 0x0F0F0F0Fu) | (odd & 0xF0F0F0F0u)) & 0x88888888u;
}
// The 8 bf16 values of 4 words scaled by a non-negative multiplier
// (fl32(x * mult), as the RN path) and rounded stochastically with the 16-bit
// uniforms of rb (word b: value 2b low half, 2b + 1 high half); the codes keep
// the inputs' sign bits.
template <bool SAT = true>
FP4_DEV uint32_t e2m1x8_sr_bf16(const uint32_t* w, float mult, uint4 rb) {
    const uint32_t rw[4] = {rb.x, rb.y, rb.z, rb.w};
    uint32_t word = e2m1x8_signs(w);
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        const uint32_t wa = w[b] & 0x7FFF7FFFu;
        float ax, ay;
        f32x2_mul(ax, ay, __uint_as_float(wa << 16), __uint_as_float(wa & 0xFFFF0000u), mult, mult);
        word |= sr_code_pair<SAT>(ax, ay, rw[b]) << (8 * b);
    }
    return word;
}

// --------------------------------------------------------------- E4M3 ------
// binary32 -> OCP E4M3 byte, round to nearest even, saturating at 448.
FP4_DEV uint32_t e4m3_rn_satfinite(float s) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(s));
    return (uint32_t)(r & 0xFFu);
}

// E4M3 byte (sign 0) -> binary32, exact.
FP4_DEV float e4m3_value(uint32_t c) {
    uint32_t E = (c >> 3) & 15u, m = c & 7u;
    if (E == 0) return (float)m * 0.001953125f;  // m * 2^-9
    return __uint_as_float(((E + 120u) << 23) | (m << 20));
}

// ------------------------------------------------------------ E8M0 (MX) ----
// Upward E8M0 exponent of a block from the bit pattern of its amax (sign
// cleared): the smallest e with 6 * 2^e >= amax, clamped to [-127, 127].
// amax = f * 2^E with f in [1, 2): e = E - 2 if f <= 1.5 else E - 1.
FP4_DEV int e8m0_exponent_up(uint32_t amax_bits) {
    int field = (int)(amax_bits >> 23);
    if (field == 0) return -127;  // zero or subnormal amax
    int E = field - 127;
    int e = (amax_bits & 0x7FFFFFu) <= 0x400000u ? E - 2 : E - 1;
    return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// 2^-e as binary32 for e in [-126, 127] ... callers keep e <= 126.
FP4_DEV float exp2_neg(int e) { return __uint_as_float((uint32_t)(127 - e) << 23); }

// --------------------------------------------------------------- NVFP4 -----
// Outer encode factor S_enc = fl32(2688 / amax) (Sec. 2.2.2); 1 for amax 0;
// an overflow clamps to the largest finite binary32.
FP4_DEV float nv_senc(float amax) {
    if (amax == 0.0f) return 1.0f;
    float s = __fdiv_rn(2688.0f, amax);
    return isinf(s) ? 3.402823466e38f : s;
}

// fl32(a / 6) for a block maximum that is a bf16 value (held as binary32):
// the product with fl32(1/6), then one FMA correction with the exact
// remainder (division by a constant known in advance, after Markstein;
// Brisebarre, Muller and Raina, IEEE Trans. Computers 53(8), 2004).  Checked
// equal to the correctly rounded quotient for every finite positive bf16
// value, subnormals included; binary32 maxima of other origin take __fdiv_rn.
FP4_DEV float div6_bf16(float a) {
    const float c = __uint_as_float(0x3E2AAAABu);  // fl32(1/6)
    const float q = __fmul_rn(a, c);
    const float r = __fmaf_rn(-q, 6.0f, a);
    return __fmaf_rn(r, c, q);
}

// The multipliers m[d] = fl32(S_enc / E4M3(d)) (0 for d = 0) of one outer
// factor, computed once per tile into a 128-entry table (d <= 126: the
// saturating encoder never returns the NaN code 127).
FP4_DEV float nv_mult_entry(float senc, uint32_t d) { return d == 0 ? 0.0f : __fdiv_rn(senc, e4m3_value(d)); }

// Block scale byte and multiplier of a 16-value block whose maximum is a bf16
// value, with the multiplier read from a table of nv_mult_entry; the same
// results as nv_block_scale.
FP4_DEV uint32_t nv_block_scale_bf16(float block_amax, float senc, const float* mtab, float& mult) {
    const uint32_t d = e4m3_rn_satfinite(__fmul_rn(div6_bf16(block_amax), senc));
    mult = mtab[d];
    return d;
}

// Block scale byte and binary32 multiplier of one 16-value block:
// s_raw = fl32(fl32(a_b / 6) * S_enc), delta = E4M3(s_raw),
// m_b = delta == 0 ? 0 : fl32(S_enc / delta).
FP4_DEV uint32_t nv_block_scale(float block_amax, float senc, float& mult) {
    float s_raw = __fmul_rn(__fdiv_rn(block_amax, 6.0f), senc);
    uint32_t d = e4m3_rn_satfinite(s_raw);
    mult = d == 0 ? 0.0f : __fdiv_rn(senc, e4m3_value(d));
    return d;
}

// -------------------------------------------------------------- Philox ----
// Philox4x32-10: ten rounds of the 4x32 S-box with key increments.  Each
// round's two 32x32 -> 64-bit products are single widening multiplies.  The
// ten round keys depend only on the seed: the host computes them once per
// launch (sr_round_keys) and the kernels read them from their parameters.
constexpr int SR_ROUND_KEYS = 20;
__host__ __device__ inline void sr_round_keys(uint64_t seed, uint32_t* rk) {
    uint32_t kx = (uint32_t)seed, ky = (uint32_t)(seed >> 32);
    for (int r = 0; r < 10; ++r) {
        rk[2 * r] = kx;
        rk[2 * r + 1] = ky;
        kx += 0x9E3779B9u;
        ky += 0xBB67AE85u;
    }
}
FP4_DEV uint4 philox4x32_10(uint4 c, const uint32_t* rk) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint64_t p0 = (uint64_t)0xD2511F53u * c.x;
        const uint64_t p1 = (uint64_t)0xCD9E8D57u * c.z;
        c = make_uint4((uint32_t)(p1 >> 32) ^ c.y ^ rk[2 * r], (uint32_t)p1, (uint32_t)(p0 >> 32) ^ c.w ^ rk[2 * r + 1],
                       (uint32_t)p0);
    }
    return c;
}

// The eight 16-bit uniforms of elements 8g .. 8g+7 under (seed, offset); rk
// holds the seed's round keys.
FP4_DEV uint4 sr_bits8(uint64_t g, const uint32_t* rk, uint64_t offset) {
    return philox4x32_10(make_uint4((uint32_t)g, (uint32_t)(g >> 32), (uint32_t)offset, (uint32_t)(offset >> 32)), rk);
}

// ----------------------------------------------------------- scale layout --
// Byte offset of block j of stored row r in the 128x4 atom layout, for a
// view whose stored rows hold `nblk` blocks.
__host__ __device__ inline int64_t scale_offset(int64_t r, int64_t j, int64_t nblk) {
    return ((r >> 7) * (nblk >> 2) + (j >> 2)) * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4 + (j & 3);
}

}  // namespace fp4
