// quantize.cu -- FP4 quantizer producers for sm_103a.
//
// One kernel emits, from a single read of each 128 x 128 BF16 tile, every view
// the next contractions need ("Format-Aware Fusion for Fast FP4 Pretraining",
// Sec. 3.1 boundary contract): the row-facing view Q_r (blocks along the row,
// optionally stochastically rounded, Sec. 2.5 Eq. 9) and the column-facing view
// Q_c (blocks along the column, optionally through the fixed-sign H32 of
// Sec. 2.5 Eq. 10), with
//   MXFP4         upward E8M0 scale per 32 values (Sec. 2.2.1),
//   2D32 weights  one adaptive E8M0 per 32x32 tile, finer when a/s < 0.87,
//   NVFP4         E4M3 scale per 16 values under the S_enc outer factor of
//                 the tensor (global) or of the 128-strip (CTA-local),
//                 (Sec. 2.2.2),
//   2D16 weights  one E4M3 per 16x16 tile under the tensor factor (Sec. 2.4).
// NVFP4 first runs a tile-amax pre-pass (the tensor-wide / strip-wide maximum
// that the outer factors need), so its algorithmic traffic is two reads.
//
// Memory behaviour: persistent CTAs, four per SM (64 registers, one tile slot
// of 16-byte cp.async copies each: the other CTAs' encoding hides a CTA's
// load) or, for the MXFP4 row view with stochastic rounding, three per SM (80
// registers, two slots: the next tile lands while one is encoded);
// per-thread 32-value segments for both orientations read from shared memory
// (unpadded tiles, 16-byte chunks XOR-swizzled by row); codes stored from
// registers as 16-byte pieces whose sector halves come from neighbouring
// warps and merge in L2 (row view: the four pieces of a row's 64 bytes from
// the four warps of its block indices; column view likewise down the stored
// rows); scale atoms staged in shared memory and
// written with coalesced 16-byte stores (each tile's scale bytes form whole
// 512-byte atoms).
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace fp4 {

__device__ unsigned int g_status_quant;

namespace {

constexpr int TILE = 128;
constexpr int THREADS = 256;

// CTAs per SM of an encoder launch: three at 80 registers with two tile
// slots each (the tile being encoded and the next one landing), or four at
// 64 registers with one slot (the other CTAs' work hides each one's load).
// Four are 1-6 % faster on every route but the MXFP4 row view with
// stochastic rounding, which is 2 % slower with four and takes three.
template <int CTAS>
constexpr int slots_of() { return CTAS == 4 ? 1 : 2; }

// Shared tiles are unpadded (256-byte rows) with the 16-byte chunks of row r
// XOR-ed by r & 7: element (r, c) sits at r * 128 + ((c / 8) ^ (r & 7)) * 8 +
// c % 8.  Every access pattern of the kernels then touches each bank once
// per phase: the 16-byte copies and loads of a row's chunks, the 16-byte
// loads of one chunk index over 8 consecutive rows (row segments), and the
// 32-bit loads of 32 consecutive column pairs of one row (column view).
FP4_DEV int tile_off(int r, int c) { return r * TILE + ((((c >> 3) ^ r) & 7) | ((c >> 3) & ~7)) * 8 + (c & 7); }

template <int SLOTS>
struct SmemQ {
    uint16_t tile[SLOTS][TILE * TILE];  // SLOTS x 32 KB
    uint8_t row_sc[1024];            // staged scale atoms (1 MX / 2 NV)
    uint8_t col_sc[1024];
    int tile_e[16];                  // 2D32: per 32x32 tile exponent
    float tile_m[64];                // 2D16: per 16x16 tile multiplier
    uint32_t tile_d[64];             // 2D16: per 16x16 tile E4M3 byte
    float mtab[2][128];              // NVFP4: S_enc / E4M3(d) of the row / column view's factor
    float signf[16];                 // the Hadamard's fixed signs as +-1 (set once per CTA)
    uint32_t red[THREADS / 32];
};


// Byte offset of local block j (0..nb-1) of local row r in staged atoms.
// Row segments: work item idx (0 .. 511) is 32-value segment j of local row
// r, numbered so that each warp holds 32 consecutive rows at one j: a 32x32
// block of the tile is one warp's segments (2D weight maxima by shuffles),
// and the 8 lanes of each 16-byte shared-load phase read 8 consecutive rows
// at one chunk index, which the tile swizzle spreads over all 32 banks.
FP4_DEV int seg_row(int idx) { return (idx & 31) + 32 * (idx >> 7); }
FP4_DEV int seg_j(int idx) { return (idx >> 5) & 3; }

FP4_DEV int atom_off(int r, int j) { return (j >> 2) * 512 + (r & 31) * 16 + (r >> 5) * 4 + (j & 3); }

// fp32 bits of max |v[i]| over n values (non-negative, so the float and the
// bit order agree; a NaN anywhere gives a NaN, caught by check_finite).
template <int N>
FP4_DEV uint32_t amax_bits(const float* v) {
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < N; i += 2) m = max3_abs_nan(m, v[i], v[i + 1]);
    return __float_as_uint(m);
}
FP4_DEV uint32_t amax_bits32(const float* v) { return amax_bits<32>(v); }
FP4_DEV uint32_t amax_bits16(const float* v) { return amax_bits<16>(v); }
// Packed per-half maximum of |bf16| over n bf16x2 words (bits of the low and
// high halves' maxima in the two 16-bit lanes).
template <int N>
FP4_DEV uint32_t amax_words(const uint32_t* w) {
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < N; i += 2) m = __vimax3_u16x2(m, w[i] & 0x7FFF7FFFu, w[i + 1] & 0x7FFF7FFFu);
    return m;
}
// fp32 bit pattern of a bf16 magnitude held in a 16-bit lane.
FP4_DEV uint32_t lane_lo_f32bits(uint32_t m2) { return m2 << 16; }
FP4_DEV uint32_t lane_hi_f32bits(uint32_t m2) { return m2 & 0xFFFF0000u; }

// Pack 32 E2M1 codes (RN) of v * m (m0 for values 0..15, m1 for 16..31).
FP4_DEV uint4 pack_rn32(const float* v, float m0, float m1) {
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float mult = q < 2 ? m0 : m1;
        float s[8];
#pragma unroll
        for (int b = 0; b < 8; b += 2) f32x2_mul(s[b], s[b + 1], v[q * 8 + b], v[q * 8 + b + 1], mult, mult);
        w[q] = e2m1x8_rn(s[0], s[1], s[2], s[3], s[4], s[5], s[6], s[7]);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Stochastic rounding of the 32 bf16 values of 16 words (logical indices
// 8*g0 .. 8*g0+31), scaled by m0 (values 0..15) and m1 (16..31); SAT for
// NVFP4 blocks, whose scaled values can pass 6 by the E4M3 scale rounding.
template <bool SAT>
FP4_DEV uint4 pack_sr32(const uint32_t* w, float m0, float m1, uint64_t g0, const uint32_t* rk, uint64_t offset) {
    uint32_t out[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) out[q] = e2m1x8_sr_bf16<SAT>(w + 4 * q, q < 2 ? m0 : m1, sr_bits8(g0 + q, rk, offset));
    return make_uint4(out[0], out[1], out[2], out[3]);
}

// Butterfly stages of strides 1 .. H/2 on each H-value group of 32
// registers, after the fixed signs sg[i mod 16] (+-1) of Sec. 2.5.  Stride 1
// pairs the two lanes of a register pair (v[2i], v[2i + 1]) and runs scalar,
// with the signs folded in: u = s v is exact, so fl(u0 + u1) =
// fma(s1, v1, s0 v0) and fl(u0 - u1) = fma(-s1, v1, s0 v0) give the bits of
// flipping first (the flips then cost no integer instructions); every wider
// stride pairs whole register pairs and runs on f32x2 lanes.
template <int H>
FP4_DEV void butterflies(float* v, const float* sg) {
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
        const float t = __fmul_rn(v[j], sg[j & 15]), s1 = sg[(j + 1) & 15], b = v[j + 1];
        v[j] = __fmaf_rn(s1, b, t);
        v[j + 1] = __fmaf_rn(-s1, b, t);
    }
#pragma unroll
    for (int h = 2; h < H; h <<= 1) {
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
            if ((j & h) == 0) {
                const float a0 = v[j], a1 = v[j + 1], b0 = v[j + h], b1 = v[j + h + 1];
                f32x2_add(v[j], v[j + 1], a0, a1, b0, b1);
                f32x2_sub(v[j + h], v[j + h + 1], a0, a1, b0, b1);
            }
        }
    }
}
FP4_DEV void scale_all(float* v, float s) {
#pragma unroll
    for (int i = 0; i < 32; i += 2) f32x2_mul(v[i], v[i + 1], v[i], v[i + 1], s, s);
}

__device__ const float kUnitSigns[16] = {1.f, 1.f, 1.f, 1.f, 1.f, 1.f, 1.f, 1.f,
                                         1.f, 1.f, 1.f, 1.f, 1.f, 1.f, 1.f, 1.f};

// Fixed-sign H32 on 32 registers (signs sg): stages of stride 1, 2, 4, 8
// within each 16-value half, then the cross-half stage of stride 16, then the
// binary32 multiply by fl32(1/sqrt(32)).
FP4_DEV void hadamard32(float* v, const float* sg) {
    butterflies<32>(v, sg);
    scale_all(v, __uint_as_float(0x3E3504F3u));  // fl32(1 / sqrt(32))
}

// Fixed-sign H16 on each 16-value half of 32 registers (signs sg): stages
// of stride 1, 2, 4, 8, then the multiply by 1/sqrt(16) = 0.25 (exact).
FP4_DEV void hadamard16x2(float* v, const float* sg) {
    butterflies<16>(v, sg);
    scale_all(v, 0.25f);
}

// Load the 128x128 tile at (r0, c0) into shared memory (tile_off layout),
// applying the pre-op; with write_tap the pre-op results are also stored.
FP4_DEV void load_tile(const QuantParams& p, int64_t r0, int64_t c0, uint16_t* tile, bool write_tap) {
    const int t = threadIdx.x;
    if (p.pre == PRE_NONE) {
        // all eight 16-byte loads of this thread in flight before any store
        uint4 d[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int q = t + i * THREADS;
            d[i] = *reinterpret_cast<const uint4*>(p.x + (r0 + (q >> 4)) * p.ld + c0 + (q & 15) * 8);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int q = t + i * THREADS;
            *reinterpret_cast<uint4*>(&tile[tile_off(q >> 4, (q & 15) * 8)]) = d[i];
        }
        return;
    }
    if (p.pre == PRE_ROPE_BWD) {
        // the tile's 128 columns are one head (c0 / 128); each thread takes
        // 8 values of the low half and their rotate-half partners
        const int head = (int)(c0 >> 7), hqk = p.heads_q + p.heads_kv;
        const uint16_t* src = head < p.heads_q ? p.rope_src[0] + (int64_t)head * p.R * 128
                              : head < hqk     ? p.rope_src[1] + (int64_t)(head - p.heads_q) * p.R * 128
                                               : p.rope_src[2] + (int64_t)(head - hqk) * p.R * 128;
#pragma unroll 2
        for (int i = 0; i < 4; ++i) {
            const int q = t + i * THREADS, rr = q >> 3, g = q & 7;
            const int64_t tok = r0 + rr;
            uint4 lo = *reinterpret_cast<const uint4*>(src + tok * 128 + 8 * g);
            uint4 hi = *reinterpret_cast<const uint4*>(src + tok * 128 + 64 + 8 * g);
            if (head < hqk) {
                const int64_t pos = tok % p.seq_len;
                const float* cs = p.rope_cos + pos * 64 + 8 * g;
                const float* sn = p.rope_sin + pos * 64 + 8 * g;
                uint32_t la[4] = {lo.x, lo.y, lo.z, lo.w}, ha[4] = {hi.x, hi.y, hi.z, hi.w}, lo_o[4], hi_o[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float l[2], h[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const float a = e ? bf16_hi(la[j]) : bf16_lo(la[j]);
                        const float b = e ? bf16_hi(ha[j]) : bf16_lo(ha[j]);
                        const float c = cs[2 * j + e], sv = sn[2 * j + e];
                        l[e] = __fadd_rn(__fmul_rn(a, c), __fmul_rn(b, sv));
                        h[e] = __fsub_rn(__fmul_rn(b, c), __fmul_rn(a, sv));
                    }
                    lo_o[j] = (uint32_t)f32_to_bf16_rn(l[0]) | ((uint32_t)f32_to_bf16_rn(l[1]) << 16);
                    hi_o[j] = (uint32_t)f32_to_bf16_rn(h[0]) | ((uint32_t)f32_to_bf16_rn(h[1]) << 16);
                }
                lo = make_uint4(lo_o[0], lo_o[1], lo_o[2], lo_o[3]);
                hi = make_uint4(hi_o[0], hi_o[1], hi_o[2], hi_o[3]);
            }
            if (write_tap && p.tap) {
                *reinterpret_cast<uint4*>(p.tap + tok * p.C + c0 + 8 * g) = lo;
                *reinterpret_cast<uint4*>(p.tap + tok * p.C + c0 + 64 + 8 * g) = hi;
            }
            *reinterpret_cast<uint4*>(&tile[tile_off(rr, 8 * g)]) = lo;
            *reinterpret_cast<uint4*>(&tile[tile_off(rr, 64 + 8 * g)]) = hi;
        }
        return;
    }
#pragma unroll 2
    for (int i = 0; i < 8; ++i) {
        int q = t + i * THREADS;
        int rr = q >> 4, cc = (q & 15) * 8;
        const int64_t gr = r0 + rr, gc = c0 + cc;
        uint4 d = *reinterpret_cast<const uint4*>(p.x + gr * p.ld + gc);
        if (p.pre != PRE_NONE) {
            uint4 gv = *reinterpret_cast<const uint4*>(p.g + gc);
            uint32_t xs[4] = {d.x, d.y, d.z, d.w}, gs[4] = {gv.x, gv.y, gv.z, gv.w}, os[4];
            const float rs = p.rstd[gr];
            if (p.pre == PRE_RMSNORM_FWD) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    float y0 = __fmul_rn(__fmul_rn(bf16_lo(xs[k]), rs), bf16_lo(gs[k]));
                    float y1 = __fmul_rn(__fmul_rn(bf16_hi(xs[k]), rs), bf16_hi(gs[k]));
                    os[k] = (uint32_t)f32_to_bf16_rn(y0) | ((uint32_t)f32_to_bf16_rn(y1) << 16);
                }
            } else {
                const float mg = p.mean_g[gr];
                uint4 xv = *reinterpret_cast<const uint4*>(p.rp + gr * p.C + gc);
                uint4 dv = p.dres ? *reinterpret_cast<const uint4*>(p.dres + gr * p.C + gc) : make_uint4(0, 0, 0, 0);
                uint32_t rps[4] = {xv.x, xv.y, xv.z, xv.w}, drs[4] = {dv.x, dv.y, dv.z, dv.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    float o[2];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        float dyv = h ? bf16_hi(xs[k]) : bf16_lo(xs[k]);
                        float gg = h ? bf16_hi(gs[k]) : bf16_lo(gs[k]);
                        float xr = h ? bf16_hi(rps[k]) : bf16_lo(rps[k]);
                        float dr = h ? bf16_hi(drs[k]) : bf16_lo(drs[k]);
                        float xh = __fmul_rn(xr, rs);
                        float gy = __fmul_rn(dyv, gg);
                        float u = __fsub_rn(gy, __fmul_rn(xh, mg));
                        o[h] = __fadd_rn(__fmul_rn(rs, u), dr);
                    }
                    os[k] = (uint32_t)f32_to_bf16_rn(o[0]) | ((uint32_t)f32_to_bf16_rn(o[1]) << 16);
                }
            }
            d = make_uint4(os[0], os[1], os[2], os[3]);
            if (write_tap && p.tap) *reinterpret_cast<uint4*>(p.tap + gr * p.C + gc) = d;
        }
        *reinterpret_cast<uint4*>(&tile[tile_off(rr, cc)]) = d;
    }
}

FP4_DEV void check_finite(uint32_t amax_bits) {
    if (amax_bits >= 0x7F800000u) set_status(&g_status_quant, FP4_ERR_NONFINITE);
}

// Scale choice of one 32-value segment (MX: one block; NV: two blocks of 16)
// from the fp32 bit patterns of the blocks' amax; stages the scale bytes and
// returns the two multipliers.
// NVFP4: with mtab the block maxima are bf16 values and the multipliers come
// from the tile's table; without it (H16-transformed binary32 values) both
// quotients are divided out.
template <bool NV>
FP4_DEV void segment_scale(uint32_t am0, uint32_t am1, float senc, uint8_t* sc_base, int lr, int lj, float& m0,
                           float& m1, const float* mtab = nullptr) {
    if (!NV) {
        check_finite(am0);
        const int e = e8m0_exponent_up(am0);
        m0 = m1 = exp2_neg(e);
        sc_base[atom_off(lr, lj)] = (uint8_t)(e + 127);
    } else if (mtab) {
        check_finite(max(am0, am1));
        sc_base[atom_off(lr, 2 * lj)] = (uint8_t)nv_block_scale_bf16(__uint_as_float(am0), senc, mtab, m0);
        sc_base[atom_off(lr, 2 * lj + 1)] = (uint8_t)nv_block_scale_bf16(__uint_as_float(am1), senc, mtab, m1);
    } else {
        check_finite(max(am0, am1));
        sc_base[atom_off(lr, 2 * lj)] = (uint8_t)nv_block_scale(__uint_as_float(am0), senc, m0);
        sc_base[atom_off(lr, 2 * lj + 1)] = (uint8_t)nv_block_scale(__uint_as_float(am1), senc, m1);
    }
}

// Encode the 128x128 tile (ty, tx), already in shared memory at `tbuf`, into
// both views: steps 2-5 below.  NVR / NVC: the row / column view is NVFP4
// (else MXFP4); the two differ in the operand-wise hybrid producer.  Called
// by all threads of the CTA with the tile visible to every thread.
template <bool NVR, bool NVC, class SmemT>
FP4_DEV void encode_tile(const QuantParams& p, SmemT& s, const uint16_t* tbuf, int64_t ty, int64_t tx) {
    const int t = threadIdx.x;
    const int64_t r0 = ty * TILE, c0 = tx * TILE;
    const bool w2d = (p.flags & FP4_FLAG_WEIGHT_2D) != 0;
    const bool h16 = (p.flags & FP4_FLAG_HADAMARD16_COL) != 0;
    const bool do_row = (p.views & FP4_VIEW_ROW) != 0, do_col = (p.views & FP4_VIEW_COL) != 0;

    // outer factors of this tile's row strip / column strip, per view route:
    // the tensor factor (ws[0]) for 2D weights and global NVFP4, the strip
    // factor for CTA-local NVFP4; an H16 column view takes the factors of
    // the transformed values (column strips, and the last slot for global)
    float senc_row = 1.0f, senc_col = 1.0f, senc_w = 1.0f;
    if (NVR || NVC) {
        const uint32_t* ws = p.amax_ws;
        senc_w = nv_senc(__uint_as_float(ws[0]));
        if (NVR)
            senc_row = (w2d || p.row_route == FP4_ROUTE_NVFP4_GLOBAL) ? senc_w : nv_senc(__uint_as_float(ws[1 + ty]));
        if (NVC) {
            if (w2d)
                senc_col = senc_w;
            else if (p.col_route == FP4_ROUTE_NVFP4_GLOBAL)
                senc_col = h16 ? nv_senc(__uint_as_float(ws[1 + (p.R >> 7) + (p.C >> 7)])) : senc_w;
            else
                senc_col = nv_senc(__uint_as_float(ws[1 + (p.R >> 7) + tx]));
        }
        // the multipliers S_enc / E4M3(d) of both views' factors, one
        // division per thread (visible after the barrier below)
        if (t < 128) {
            if (NVR) s.mtab[0][t] = nv_mult_entry(senc_row, (uint32_t)t);
        } else {
            if (NVC) s.mtab[1][t - 128] = nv_mult_entry(w2d ? senc_w : senc_col, (uint32_t)(t - 128));
        }
        if (t == 0) {
            if (NVR && do_row) {
                if (p.row_route == FP4_ROUTE_NVFP4_LOCAL && !w2d) {
                    if (tx == 0) p.row_outer[ty] = senc_row;
                } else if (tx == 0 && ty == 0) {
                    p.row_outer[0] = senc_row;
                }
            }
            if (NVC && do_col) {
                if (p.col_route == FP4_ROUTE_NVFP4_LOCAL && !w2d) {
                    if (ty == 0) p.col_outer[tx] = senc_col;
                } else if (tx == 0 && ty == 0) {
                    p.col_outer[0] = senc_col;
                }
            }
        }
        __syncthreads();  // the multiplier tables
    }

    // 16-byte shared loads of this thread's row segment k (steps 2 and 3)
    auto load_segment = [&](int k, uint32_t* w) {
        const int idx = t + k * THREADS, r = seg_row(idx), j = seg_j(idx);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint4 d = *reinterpret_cast<const uint4*>(&tbuf[tile_off(r, 32 * j + 8 * q)]);
            w[4 * q] = d.x; w[4 * q + 1] = d.y; w[4 * q + 2] = d.z; w[4 * q + 3] = d.w;
        }
    };

    // 2-3. row-facing view: segment (r, j) = 32 values of local row r
    //      starting at 32 j; 2D weights first take their shared tile scales
    //      from the same registers
    {
        const bool sr = (p.flags & FP4_FLAG_SR_ROW) != 0;
        auto row_segment = [&](int k, const uint32_t* w) {
            const int idx = t + k * THREADS, r = seg_row(idx), j = seg_j(idx);
            float m0, m1;
            if (w2d) {
                if (!NVR) {
                    const int e = s.tile_e[(r >> 5) * 4 + j];
                    m0 = m1 = exp2_neg(e);
                    s.row_sc[atom_off(r, j)] = (uint8_t)(e + 127);
                } else {
                    const int tl = (r >> 4) * 8 + 2 * j;
                    m0 = s.tile_m[tl];
                    m1 = s.tile_m[tl + 1];
                    s.row_sc[atom_off(r, 2 * j)] = (uint8_t)s.tile_d[tl];
                    s.row_sc[atom_off(r, 2 * j + 1)] = (uint8_t)s.tile_d[tl + 1];
                }
            } else if (!NVR) {
                const uint32_t a2 = amax_words<16>(w);
                segment_scale<false>(max(lane_lo_f32bits(a2), lane_hi_f32bits(a2)), 0, 0.f, s.row_sc, r, j, m0, m1);
            } else {
                const uint32_t a0 = amax_words<8>(w), a1 = amax_words<8>(w + 8);
                segment_scale<true>(max(lane_lo_f32bits(a0), lane_hi_f32bits(a0)),
                                    max(lane_lo_f32bits(a1), lane_hi_f32bits(a1)), senc_row, s.row_sc, r, j, m0, m1,
                                    s.mtab[0]);
            }
            uint4 packed;
            if (sr) {
                const uint64_t g0 = (uint64_t)(((r0 + r) * p.C + c0 + 32 * j) >> 3);
                packed = pack_sr32<NVR>(w, m0, m1, g0, p.sr_keys, p.offset);
            } else {
                float v[32];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    v[2 * i] = bf16_lo(w[i]);
                    v[2 * i + 1] = bf16_hi(w[i]);
                }
                packed = pack_rn32(v, m0, m1);
            }
            *reinterpret_cast<uint4*>(p.row_codes + (r0 + r) * (p.C >> 1) + (c0 >> 1) + j * 16) = packed;
        };
        if (w2d) {
            // The warp's segments are the 32x32 block (rows 32 (r / 32) ..,
            // columns 32 j ..): its maximum by shuffles over the 32 lanes; a
            // 16x16 block is one half-warp's 16-value pieces.  The scales go
            // to shared memory for the column view (after the barrier below)
            // and for this warp's own row segments (after __syncwarp).
            const int lane = t & 31;
#pragma unroll 1
            for (int k = 0; k < 2; ++k) {
                const int idx = t + k * THREADS, r = seg_row(idx), j = seg_j(idx);
                uint32_t w[16];
                load_segment(k, w);
                const uint32_t a0 = amax_words<8>(w), a1 = amax_words<8>(w + 8);
                uint32_t ma = max(lane_lo_f32bits(a0), lane_hi_f32bits(a0));
                uint32_t mb = max(lane_lo_f32bits(a1), lane_hi_f32bits(a1));
                if (!NVR || !NVC) {
                    uint32_t m = max(ma, mb);
#pragma unroll
                    for (int o = 16; o; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
                    if (lane == 0) {
                        check_finite(m);
                        int e = e8m0_exponent_up(m);
                        // adaptive rule: finer exponent when a_T * 2^-e < fl32(5.22)
                        if (__fmul_rn(__uint_as_float(m), exp2_neg(e)) < 5.22f && e > -127) e -= 1;
                        s.tile_e[(r >> 5) * 4 + j] = e;
                    }
                }
                if (NVR || NVC) {
#pragma unroll
                    for (int o = 8; o; o >>= 1) {
                        ma = max(ma, __shfl_xor_sync(0xFFFFFFFFu, ma, o));
                        mb = max(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, o));
                    }
                    if ((lane & 15) == 0) {
                        check_finite(max(ma, mb));
                        const int tl = (r >> 4) * 8 + 2 * j;
                        const float* mt = s.mtab[NVR ? 0 : 1];
                        float mm;
                        s.tile_d[tl] = nv_block_scale_bf16(__uint_as_float(ma), senc_w, mt, mm);
                        s.tile_m[tl] = mm;
                        s.tile_d[tl + 1] = nv_block_scale_bf16(__uint_as_float(mb), senc_w, mt, mm);
                        s.tile_m[tl + 1] = mm;
                    }
                }
                __syncwarp();
                if (do_row) row_segment(k, w);
            }
            __syncthreads();  // every tile scale, for the column view
        } else if (do_row) {
#pragma unroll 1
            for (int k = 0; k < 2; ++k) {
                uint32_t w[16];
                load_segment(k, w);
                row_segment(k, w);
            }
        }
    }

    // 4. column-facing view: thread = (column pair cp, row block j); each
    //    column of the pair (2 cp, then 2 cp + 1) is one 32-value segment of
    //    its stored row (blocks along the rows), read down the tile with
    //    16-bit loads (one column at a time keeps the register count low)
    if (do_col) {
        const bool had = (p.flags & FP4_FLAG_HADAMARD_COL) != 0;  // H32 (MXFP4)
        const int cp = t & 63, j = t >> 6;
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
            const int c = 2 * cp + h;
            // column c of rows j * 32 + i: the swizzle depends on i & 7 only,
            // so eight element offsets serve all 32 loads
            const uint16_t* col = tbuf + j * 32 * TILE;
            int off[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) off[k] = tile_off(k, c) - k * TILE;
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __uint_as_float((uint32_t)col[i * TILE + off[i & 7]] << 16);
            float m0, m1;
            if (w2d) {
                if (!NVC) {
                    const int e = s.tile_e[j * 4 + (c >> 5)];
                    m0 = m1 = exp2_neg(e);
                    s.col_sc[atom_off(c, j)] = (uint8_t)(e + 127);
                } else {
                    const int tl = (2 * j) * 8 + (c >> 4);
                    m0 = s.tile_m[tl];
                    m1 = s.tile_m[tl + 8];
                    s.col_sc[atom_off(c, 2 * j)] = (uint8_t)s.tile_d[tl];
                    s.col_sc[atom_off(c, 2 * j + 1)] = (uint8_t)s.tile_d[tl + 8];
                }
            } else if (had) {
                hadamard32(v, s.signf);
                segment_scale<NVC>(amax_bits32(v), 0, senc_col, s.col_sc, c, j, m0, m1);
            } else if (h16) {
                hadamard16x2(v, s.signf);
                if (NVC)
                    segment_scale<true>(amax_bits16(v), amax_bits16(v + 16), senc_col, s.col_sc, c, j, m0, m1);
                else
                    segment_scale<false>(amax_bits32(v), 0, senc_col, s.col_sc, c, j, m0, m1);
            } else if (!NVC) {
                segment_scale<false>(amax_bits32(v), 0, senc_col, s.col_sc, c, j, m0, m1);
            } else {
                segment_scale<true>(amax_bits16(v), amax_bits16(v + 16), senc_col, s.col_sc, c, j, m0, m1, s.mtab[1]);
            }
            *reinterpret_cast<uint4*>(p.col_codes + (c0 + c) * (p.R >> 1) + (r0 >> 1) + j * 16) = pack_rn32(v, m0, m1);
        }
    }
    __syncthreads();

    // 5. coalesced write-out of the staged scale atoms
    if (do_row) {
        const int nat = NVR ? 2 : 1;
        if (t < nat * 32) {
            int64_t atoms_per_rowblock = NVR ? (p.C >> 6) : (p.C >> 7);
            int64_t a0 = (r0 >> 7) * atoms_per_rowblock + (NVR ? (c0 >> 6) : (c0 >> 7));
            *reinterpret_cast<uint4*>(p.row_scales + a0 * 512 + t * 16) =
                *reinterpret_cast<const uint4*>(&s.row_sc[t * 16]);
        }
    }
    if (do_col) {
        const int nat = NVC ? 2 : 1;
        if (t < nat * 32) {
            int64_t atoms_per_rowblock = NVC ? (p.R >> 6) : (p.R >> 7);
            int64_t a0 = (c0 >> 7) * atoms_per_rowblock + (NVC ? (r0 >> 6) : (r0 >> 7));
            *reinterpret_cast<uint4*>(p.col_scales + a0 * 512 + t * 16) =
                *reinterpret_cast<const uint4*>(&s.col_sc[t * 16]);
        }
    }
}

// Asynchronous 16-byte global -> shared copies (bypassing L1).
FP4_DEV void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
                 "l"(src)
                 : "memory");
}
FP4_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// all but the newest N groups of this thread's copies have landed
template <int N>
FP4_DEV void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Start loading the 128x128 tile at (r0, c0) into `tile` (tile_off layout).
FP4_DEV void prefetch_tile(const QuantParams& p, int64_t r0, int64_t c0, uint16_t* tile) {
    const int t = threadIdx.x;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int q = t + i * THREADS;
        cp_async16(&tile[tile_off(q >> 4, (q & 15) * 8)], p.x + (r0 + (q >> 4)) * p.ld + c0 + (q & 15) * 8);
    }
}

// Each CTA walks tiles blockIdx.x, blockIdx.x + gridDim.x, ... (row-strip-major
// order) through a ring of SLOTS tile slots: while one tile is encoded the
// next SLOTS - 1 are in flight (one commit group per tile, possibly empty).
// The slot of tile it + SLOTS - 1 is refilled only after the barrier that
// ends tile it - 1, its last reader.
// With an RMSNorm pre-op the tile is loaded (and transformed) synchronously.
template <bool NVR, bool NVC, int CTAS>
__global__ void __launch_bounds__(THREADS, CTAS) quantize_tile_kernel(const __grid_constant__ QuantParams p) {
    constexpr int SLOTS = slots_of<CTAS>();
    extern __shared__ __align__(16) uint8_t smem_raw[];
    SmemQ<SLOTS>& s = *reinterpret_cast<SmemQ<SLOTS>*>(smem_raw);
    const int64_t tiles_x = p.C / TILE, n_tiles = tiles_x * (p.R / TILE);
    const bool async = p.pre == PRE_NONE;
    int64_t tile = blockIdx.x;
    if (tile >= n_tiles) return;
    // the Hadamard's fixed signs (read after the first tile's barrier)
    if (threadIdx.x < 16) s.signf[threadIdx.x] = ((p.sign_mask >> threadIdx.x) & 1u) ? -1.0f : 1.0f;
    if (async) {
#pragma unroll
        for (int i = 0; i < SLOTS - 1; ++i) {
            const int64_t t2 = tile + i * (int64_t)gridDim.x;
            if (t2 < n_tiles) prefetch_tile(p, (t2 / tiles_x) * TILE, (t2 % tiles_x) * TILE, s.tile[i]);
            cp_async_commit();
        }
    }
    for (int slot = 0; tile < n_tiles; tile += gridDim.x, slot = slot == SLOTS - 1 ? 0 : slot + 1) {
        uint16_t* cur = s.tile[slot];
        const int64_t ty = tile / tiles_x, tx = tile % tiles_x;
        if (async) {
            const int64_t ahead = tile + (SLOTS - 1) * (int64_t)gridDim.x;
            const int fill = slot == 0 ? SLOTS - 1 : slot - 1;  // the slot of tile it - 1 (ring order)
            if (ahead < n_tiles) prefetch_tile(p, (ahead / tiles_x) * TILE, (ahead % tiles_x) * TILE, s.tile[fill]);
            cp_async_commit();                 // one group per iteration (possibly empty)
            cp_async_wait<SLOTS - 1>();        // this thread's copies of the current tile have landed
        } else {
            load_tile(p, ty * TILE, tx * TILE, cur, true);
        }
        __syncthreads();
        encode_tile<NVR, NVC>(p, s, cur, ty, tx);
        __syncthreads();  // the scale staging and `cur` are free again
    }
}

// Tile-amax pre-pass for NVFP4: max |x| of each 128x128 tile folded into the
// tensor slot ws[0], the tile's row-strip slot and its column-strip slot.
// When the column view is NVFP4 through H16, its factors are those of the
// transformed values: the column-strip slots and the last slot (the global
// column factor) then take the maxima of the H16 output of each 16-row block.
__global__ void __launch_bounds__(THREADS) nv_amax_kernel(const __grid_constant__ QuantParams p) {
    __shared__ uint32_t red[2][THREADS / 32];
    extern __shared__ __align__(16) uint8_t amax_smem[];
    uint16_t* tile = reinterpret_cast<uint16_t*>(amax_smem);
    uint32_t* ws = p.amax_ws;
    const int64_t n_row_strips = p.R / TILE, n_col_strips = p.C / TILE;
    const int t = threadIdx.x;
    const int64_t r0 = (int64_t)blockIdx.y * TILE, c0 = (int64_t)blockIdx.x * TILE;
    const bool col_h16 = (p.flags & FP4_FLAG_HADAMARD16_COL) && (p.views & FP4_VIEW_COL) &&
                         p.col_route != FP4_ROUTE_MXFP4;
    const bool staged = p.pre != PRE_NONE || col_h16;
    uint32_t m = 0, mc = 0;
    if (staged) {
        load_tile(p, r0, c0, tile, false);
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        int q = t + i * THREADS;
        int rr = q >> 4, cc = (q & 15) * 8;
        uint4 d = staged ? *reinterpret_cast<const uint4*>(&tile[tile_off(rr, cc)])
                         : *reinterpret_cast<const uint4*>(p.x + (r0 + rr) * p.ld + c0 + cc);
        uint32_t w[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            m = max(m, (w[b] << 16) & 0x7FFFFFFFu);
            m = max(m, w[b] & 0x7FFF0000u);
        }
    }
    if (col_h16) {
        // (column pair, 16-row block) tasks: signs, H16 down the column, max
#pragma unroll 1
        for (int k = 0; k < 2; ++k) {
            const int task = t + k * THREADS, cp = task & 63, jb = task >> 6;
            float v[32];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                uint32_t w = *reinterpret_cast<const uint32_t*>(&tile[tile_off(jb * 16 + i, 2 * cp)]);
                w ^= ((p.sign_mask >> i) & 1u) * 0x80008000u;
                v[i] = bf16_lo(w);
                v[16 + i] = bf16_hi(w);
            }
            hadamard16x2(v, kUnitSigns);  // the signs are already applied to the words
            mc = max(mc, max(amax_bits16(v), amax_bits16(v + 16)));
        }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        mc = max(mc, __shfl_xor_sync(0xFFFFFFFFu, mc, o));
    }
    if ((t & 31) == 0) {
        red[0][t >> 5] = m;
        red[1][t >> 5] = mc;
    }
    __syncthreads();
    if (t == 0) {
        for (int i = 1; i < THREADS / 32; ++i) {
            m = max(m, red[0][i]);
            mc = max(mc, red[1][i]);
        }
        check_finite(m);
        atomicMax(&ws[0], m);
        atomicMax(&ws[1 + blockIdx.y], m);
        if (col_h16) {
            atomicMax(&ws[1 + n_row_strips + blockIdx.x], mc);
            atomicMax(&ws[1 + n_row_strips + n_col_strips], mc);
        } else {
            atomicMax(&ws[1 + n_row_strips + blockIdx.x], m);
        }
    }
}

// The same maxima streamed without a pre-op or H16 (the common case): each
// CTA of a grid sized to the resident slots walks tiles blockIdx.x,
// blockIdx.x + gridDim.x, ... (row-strip-major), issuing the next tile's eight
// 16-byte loads per thread before it reduces the current tile, so every
// thread keeps a tile's loads in flight; one atomic per tile for its row strip
// and its column strip, one per CTA for the tensor.
__global__ void __launch_bounds__(THREADS) nv_amax_stream_kernel(const __grid_constant__ QuantParams p) {
    __shared__ uint32_t red[THREADS / 32];
    uint32_t* ws = p.amax_ws;
    const int t = threadIdx.x;
    const int64_t tiles_x = p.C / TILE, n_tiles = tiles_x * (p.R / TILE), n_row_strips = p.R / TILE;
    uint4 d[8];
    auto load = [&](int64_t tl) {
        const int64_t r0 = (tl / tiles_x) * TILE, c0 = (tl % tiles_x) * TILE;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int q = t + i * THREADS;
            d[i] = *reinterpret_cast<const uint4*>(p.x + (r0 + (q >> 4)) * p.ld + c0 + (q & 15) * 8);
        }
    };
    uint32_t mt = 0;  // this CTA's running tensor maximum (fp32 bits)
    int64_t tile = blockIdx.x;
    if (tile < n_tiles) load(tile);
    for (; tile < n_tiles; tile += gridDim.x) {
        uint32_t m2 = 0;  // per 16-bit lane maxima of |bf16|
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            m2 = __vimax3_u16x2(m2, d[i].x & 0x7FFF7FFFu, d[i].y & 0x7FFF7FFFu);
            m2 = __vimax3_u16x2(m2, d[i].z & 0x7FFF7FFFu, d[i].w & 0x7FFF7FFFu);
        }
        if (tile + gridDim.x < n_tiles) load(tile + gridDim.x);
        uint32_t m = max(m2 << 16, m2 & 0xFFFF0000u);
#pragma unroll
        for (int o = 16; o; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        if ((t & 31) == 0) red[t >> 5] = m;
        __syncthreads();
        if (t == 0) {
            for (int i = 1; i < THREADS / 32; ++i) m = max(m, red[i]);
            atomicMax(&ws[1 + tile / tiles_x], m);
            atomicMax(&ws[1 + n_row_strips + tile % tiles_x], m);
            mt = max(mt, m);
        }
        __syncthreads();  // red is reused by the next tile
    }
    if (t == 0 && mt) {
        check_finite(mt);
        atomicMax(&ws[0], mt);
    }
}

int quant_sm_count() {
    static int cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
    if (!cached[dev]) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cached[dev] = n > 0 ? n : 1;
    }
    return cached[dev];
}

// CTAs of the encoder: one per resident slot (CTAS per SM), each looping
// over its tiles through its ring.  (Measured: two CTAs of 128 registers
// with a three-slot ring, or two tiles per CTA, were slower: the encoders
// are latency-bound at four warps per scheduler.)
unsigned encoder_grid(int64_t n_tiles, int ctas) {
    const int64_t slots = ctas * (int64_t)quant_sm_count();
    return (unsigned)(n_tiles < slots ? n_tiles : slots);
}

// The encoder's shared memory (about 72 or 40 KB) is above the 48 KB default
// (or close to it), so each instantiation's limit is raised once per device,
// under a lock.
template <bool NVR, bool NVC, int CTAS>
int launch_encoder_n(const QuantParams& p, cudaStream_t stream) {
    const size_t smem = sizeof(SmemQ<slots_of<CTAS>()>);
    static std::mutex mu;
    static bool attr_done[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FP4_ERR_CUDA;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!attr_done[dev]) {
            if (cudaFuncSetAttribute(quantize_tile_kernel<NVR, NVC, CTAS>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess ||
                cudaFuncSetAttribute(quantize_tile_kernel<NVR, NVC, CTAS>,
                                     cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess)
                return FP4_ERR_CUDA;
            attr_done[dev] = true;
        }
    }
    const int64_t n_tiles = (p.C / TILE) * (p.R / TILE);
    quantize_tile_kernel<NVR, NVC, CTAS><<<encoder_grid(n_tiles, CTAS), THREADS, smem, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? FP4_OK : FP4_ERR_CUDA;
}
template <bool NVR, bool NVC>
int launch_encoder(const QuantParams& p, cudaStream_t stream) {
    if constexpr (!NVR) {
        if ((p.views & FP4_VIEW_ROW) && (p.flags & FP4_FLAG_SR_ROW)) return launch_encoder_n<NVR, NVC, 3>(p, stream);
    }
    return launch_encoder_n<NVR, NVC, 4>(p, stream);
}

}  // namespace

size_t quant_workspace_slots(int64_t R, int64_t C, int row_route, int col_route, unsigned views, unsigned flags) {
    const bool nv_row = (views & FP4_VIEW_ROW) && row_route != FP4_ROUTE_MXFP4;
    const bool nv_col = (views & FP4_VIEW_COL) && col_route != FP4_ROUTE_MXFP4;
    if (!nv_row && !nv_col) return 0;
    return (size_t)(1 + R / TILE + C / TILE) + ((nv_col && (flags & FP4_FLAG_HADAMARD16_COL)) ? 1 : 0);
}

int launch_quantize(const QuantParams& p, cudaStream_t stream) {
    const bool do_row = (p.views & FP4_VIEW_ROW) != 0, do_col = (p.views & FP4_VIEW_COL) != 0;
    // a view that is not produced takes the other view's format
    const bool nvr = (do_row ? p.row_route : p.col_route) != FP4_ROUTE_MXFP4;
    const bool nvc = (do_col ? p.col_route : p.row_route) != FP4_ROUTE_MXFP4;
    const size_t slots = quant_workspace_slots(p.R, p.C, p.row_route, p.col_route, p.views, p.flags);
    if (slots && !p.amax_ready) {
        if (cudaMemsetAsync(p.amax_ws, 0, slots * 4, stream) != cudaSuccess) return FP4_ERR_CUDA;
        const bool col_h16 = (p.flags & FP4_FLAG_HADAMARD16_COL) && do_col && p.col_route != FP4_ROUTE_MXFP4;
        if (p.pre != PRE_NONE || col_h16) {
            const size_t amax_smem = sizeof(uint16_t) * TILE * TILE;
            dim3 grid((unsigned)(p.C / TILE), (unsigned)(p.R / TILE));
            nv_amax_kernel<<<grid, THREADS, amax_smem, stream>>>(p);
        } else {
            const int64_t n_tiles = (p.C / TILE) * (p.R / TILE);
            const int64_t slots = (int64_t)quant_sm_count() * 4;  // 256 threads x 64 registers: four CTAs per SM
            nv_amax_stream_kernel<<<(unsigned)(n_tiles < slots ? n_tiles : slots), THREADS, 0, stream>>>(p);
        }
        if (cudaGetLastError() != cudaSuccess) return FP4_ERR_CUDA;
    }
    if (nvr && nvc) return launch_encoder<true, true>(p, stream);
    if (nvr) return launch_encoder<true, false>(p, stream);
    if (nvc) return launch_encoder<false, true>(p, stream);
    return launch_encoder<false, false>(p, stream);
}

int quant_status(cudaStream_t stream, int* code, bool reset) {
    unsigned int v = 0;
    if (reset) {
        return cudaMemcpyToSymbolAsync(g_status_quant, &v, sizeof v, 0, cudaMemcpyHostToDevice, stream) == cudaSuccess
                   ? FP4_OK
                   : FP4_ERR_CUDA;
    }
    if (cudaMemcpyFromSymbolAsync(&v, g_status_quant, sizeof v, 0, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
        return FP4_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return FP4_ERR_CUDA;
    *code = (int)v;
    return FP4_OK;
}

}  // namespace fp4
