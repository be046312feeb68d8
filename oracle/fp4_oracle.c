/*
 * fp4_oracle.c -- plain, slow CPU reference of the format-aware FP4 linear
 * boundary described in "Format-Aware Fusion for Fast FP4 Pretraining".
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test-suite, the smoke check and the
 * benchmark's CPU-baseline leg load this library.  It shares no code, header,
 * table or constant generator with the CUDA library, and it does not include
 * or link anything from it.
 *
 * Conventions
 *  - Every function follows one passage of the paper (cited by section /
 *    equation).  Where the page's equation did not survive, the reading taken
 *    is stated next to the function.
 *  - Steps marked fl32 are IEEE binary32 operations with round-to-nearest-even
 *    (compile with -ffp-contract=off so that no multiply-add is fused).  They
 *    are the steps where a floating-point value decides an integer code, so
 *    the oracle takes that decision in the precision of the kernel (binary32).
 *  - Contractions are evaluated in binary64 over the decoded operands.
 *  - No blocking, fusion or reordering: each function is a direct loop.
 *
 * Parity pins (all in tests/test_oracle_*.py, run without a GPU):
 *  E2M1 RN / SR, E8M0 upward exponent, adaptive 2D32 rule, E4M3 RN-satfinite,
 *  global / CTA-local NVFP4, Sylvester H32, SR statistics, dequantized GEMM.
 *  Philox4x32-10 has no printed test vector in the paper; it is pinned by
 *  its bijectivity and output statistics and cross-checked against the
 *  independent CUDA implementation.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#include <float.h>

/* ------------------------------------------------------------------------ */
/* bfloat16 helpers                                                          */
/* ------------------------------------------------------------------------ */

static float bf16_value(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round a binary64 value to bfloat16, nearest, ties to even (finite inputs). */
uint16_t orc_bf16_round(double v)
{
    /* bfloat16 keeps 8 significant bits and the binary32 exponent range:
     * scale |v| so that the last kept bit has weight 1, round half to even,
     * scale back. */
    if (v == 0.0) return signbit(v) ? 0x8000u : 0u;
    int ex;
    (void)frexp(fabs(v), &ex);               /* |v| = m * 2^ex, m in [0.5, 1) */
    int sig_bits = 8;
    /* bfloat16 subnormals: exponent floor of 2^-133 for the last bit */
    int lsb_exp = ex - sig_bits;             /* weight of the last kept bit */
    if (lsb_exp < -133) lsb_exp = -133;
    double q = ldexp(fabs(v), -lsb_exp);     /* exact scaling */
    double fl = floor(q);
    double rem = q - fl;
    double r;
    if (rem > 0.5) r = fl + 1.0;
    else if (rem < 0.5) r = fl;
    else r = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
    double mag = ldexp(r, lsb_exp);
    float f = (float)mag;                    /* exact: mag has <= 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint16_t h = (uint16_t)(u >> 16);
    if (v < 0) h |= 0x8000u;
    return h;
}

double orc_bf16_value(uint16_t h) { return (double)bf16_value(h); }

/* ------------------------------------------------------------------------ */
/* E2M1 (Sec. 2.2, the common scalar notation, Eq. 1)                       */
/* One sign, two exponent and one fraction bit; magnitudes                   */
/* {0, 0.5, 1, 1.5, 2, 3, 4, 6}; Q_E2M1 rounds and saturates.                */
/* Code = sign << 3 | index into the magnitude list.                         */
/* ------------------------------------------------------------------------ */

static const double E2M1_MAG[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double orc_e2m1_value(uint8_t code)
{
    double m = E2M1_MAG[code & 7];
    return (code & 8) ? -m : m;
}

/* Round-to-nearest onto the E2M1 grid.  Reading: "rounds" is nearest with
 * ties to the even code (fraction bit 0); values beyond 6 saturate to 6; the
 * sign bit of the input is kept, also for results of magnitude 0. */
uint8_t orc_e2m1_rn(double v)
{
    double a = fabs(v);
    if (a >= 6.0) return (uint8_t)((signbit(v) ? 8 : 0) | 7); /* saturate */
    int best = 0;
    double bestd = a;
    for (int k = 1; k < 8; ++k) {
        double d = fabs(a - E2M1_MAG[k]);
        if (d < bestd || (d == bestd && (k % 2) == 0)) {
            best = k;
            bestd = d;
        }
    }
    return (uint8_t)((signbit(v) ? 8 : 0) | best);
}

/* Stochastic rounding between adjacent grid values (Sec. 2.5, Eq. 9):
 * P(round up to q+) = (|v| - q-) / (q+ - q-), saturating at 6.
 * u16 is a uniform 16-bit integer; the value rounds up iff u16 * 2^-16 < p. */
uint8_t orc_e2m1_sr(double v, uint32_t u16)
{
    double a = fabs(v);
    int sign = signbit(v) ? 8 : 0;
    if (a >= 6.0) return (uint8_t)(sign | 7);
    int lo = 0;
    for (int k = 1; k < 8; ++k)
        if (E2M1_MAG[k] <= a) lo = k;
    double qm = E2M1_MAG[lo], qp = E2M1_MAG[lo + 1];
    double p = (a - qm) / (qp - qm);
    int up = ((double)u16 / 65536.0) < p;
    return (uint8_t)(sign | (lo + up));
}

/* ------------------------------------------------------------------------ */
/* E8M0 encode-centric scale (Sec. 2.2.1)                                    */
/* Activation and gradient block scales are rounded upward: the exponent is  */
/* the smallest e with 6 * 2^e >= amax, clamped to the E8M0 range            */
/* [-127, 127]; the stored byte is e + 127.                                   */
/* ------------------------------------------------------------------------ */

int orc_e8m0_exponent_up(double amax)
{
    for (int e = -127; e <= 127; ++e)
        if (ldexp(6.0, e) >= amax) return e;
    return 127;
}

/* Adaptive 2D32 weight rule (Sec. 2.2.1, Figure 1): with s_T = 6 * 2^e the
 * upward span of the tile, take the finer exponent e - 1 when
 * a_T / s_T < 0.87, i.e. a_T * 2^-e < 5.22 (the binary32 value of 5.22).
 * Floored at -127. */
int orc_mx_weight_tile_exponent(double tile_amax)
{
    int e = orc_e8m0_exponent_up(tile_amax);
    const double c = (double)5.22f;
    if (tile_amax * ldexp(1.0, -e) < c && e > -127) e -= 1;
    return e;
}

/* ------------------------------------------------------------------------ */
/* E4M3 block scale (Sec. 2.2, NVFP4): OCP FP8 E4M3, bias 7, largest finite  */
/* 448, subnormals down to 2^-9.  Encoding is nearest, ties to even, with    */
/* saturation to 448 (the repaired "saturating E4M3 scale encoder").          */
/* ------------------------------------------------------------------------ */

double orc_e4m3_value(uint8_t c)
{
    int s = c >> 7, E = (c >> 3) & 15, m = c & 7;
    if (E == 15 && m == 7) return NAN;
    double v = (E == 0) ? ldexp((double)m, -9) : ldexp((double)(8 + m), E - 10);
    return s ? -v : v;
}

uint8_t orc_e4m3_rn_satfinite(double s)
{
    /* s >= 0 (scales are unsigned). Nearest of the codes 0x00..0x7E. */
    if (s >= 448.0) return 0x7E;
    int best = 0;
    double bestd = fabs(s);
    for (int c = 1; c <= 0x7E; ++c) {
        double d = fabs(s - orc_e4m3_value((uint8_t)c));
        if (d < bestd || (d == bestd && (c % 2) == 0)) {
            best = c;
            bestd = d;
        }
    }
    return (uint8_t)best;
}

/* NVFP4 outer encode factor (Sec. 2.2.2): the tensor amax A maps to the
 * largest code x block-scale product 6 * 448 = 2688.  fl32(2688 / A);
 * A = 0 gives 1; an overflow is clamped to the largest finite binary32. */
float orc_nv_senc(float amax)
{
    if (amax == 0.0f) return 1.0f;
    float s = 2688.0f / amax;
    if (isinf(s)) s = FLT_MAX;
    return s;
}

/* One NVFP4 block: returns the E4M3 block-scale byte and the binary32
 * multiplier m_b that maps the block's values onto the E2M1 grid.
 *   s_raw = fl32(fl32(a_b / 6) * S_enc), delta = E4M3(s_raw),
 *   m_b   = delta == 0 ? 0 : fl32(S_enc / delta). */
uint8_t orc_nv_block_scale(float block_amax, float senc, float* mult)
{
    float t = block_amax / 6.0f;
    float s_raw = t * senc;
    uint8_t d = orc_e4m3_rn_satfinite((double)s_raw);
    float dv = (float)orc_e4m3_value(d);
    *mult = (d == 0) ? 0.0f : senc / dv;
    return d;
}

/* ------------------------------------------------------------------------ */
/* Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as   */
/* easy as 1, 2, 3", SC'11).  Ten rounds of the 4x32 S-box with multipliers   */
/* 0xD2511F53 / 0xCD9E8D57 and the Weyl key increments 0x9E3779B9 (golden     */
/* ratio) / 0xBB67AE85 (sqrt(3) - 1).                                          */
/* ------------------------------------------------------------------------ */

void orc_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4])
{
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int r = 0; r < 10; ++r) {
        uint64_t p0 = (uint64_t)0xD2511F53u * (uint64_t)c0;
        uint64_t p1 = (uint64_t)0xCD9E8D57u * (uint64_t)c2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n1 = lo1;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        uint32_t n3 = lo0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* The 16-bit uniform used for SR of logical element i (row-major index of
 * the logical tensor) under (seed, offset) -- the checkpointed SR state of
 * Appendix A.1.  Key = (seed lo, seed hi); counter = (i/8 lo, i/8 hi,
 * offset lo, offset hi); element i takes word (i mod 8)/2, low half if i is
 * even, high half if odd. */
uint32_t orc_sr_uniform16(uint64_t seed, uint64_t offset, uint64_t i)
{
    uint64_t g = i / 8;
    uint32_t ctr[4] = {(uint32_t)g, (uint32_t)(g >> 32), (uint32_t)offset, (uint32_t)(offset >> 32)};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t out[4];
    orc_philox4x32_10(ctr, key, out);
    uint32_t w = out[(i % 8) / 2];
    return (i % 2 == 0) ? (w & 0xFFFFu) : (w >> 16);
}

/* ------------------------------------------------------------------------ */
/* Fixed-sign H32 (Sec. 2.5, Eq. 10; Appendix A.1): R = H D / sqrt(32) with   */
/* the Sylvester Hadamard H32 and a sign diagonal D that repeats a 16-entry  */
/* vector over the two 16-value halves.  Applied as the signs, then the      */
/* butterfly stages of stride 1, 2, 4, 8 inside each half and finally the    */
/* cross-half stage of stride 16, each (a, b) -> (a + b, a - b) in binary32, */
/* then a binary32 multiply by fl32(1/sqrt(32)).                              */
/* ------------------------------------------------------------------------ */

float orc_inv_sqrt32_f32(void) { return (float)(1.0 / sqrt(32.0)); }

void orc_hadamard32_f32(float y[32], const int8_t signs[16])
{
    for (int i = 0; i < 32; ++i) y[i] = y[i] * (float)signs[i % 16];
    for (int h = 1; h < 32; h *= 2)
        for (int j = 0; j < 32; ++j)
            if ((j & h) == 0) {
                float a = y[j], b = y[j + h];
                y[j] = a + b;
                y[j + h] = a - b;
            }
    float s = orc_inv_sqrt32_f32();
    for (int i = 0; i < 32; ++i) y[i] = y[i] * s;
}

/* The same transform on every aligned 32-value block of every row of an
 * R x C binary32 matrix (in place). */
void orc_hadamard32_rows(float* x, int64_t R, int64_t C, const int8_t signs[16])
{
    for (int64_t r = 0; r < R; ++r)
        for (int64_t b = 0; b < C / 32; ++b) orc_hadamard32_f32(x + r * C + b * 32, signs);
}

/* Fixed-sign H16 ("Format-Aware Fusion for Fast FP4 Pretraining", Sec. 2.5
 * and Appendix A.1; the NVFP4 Wgrad transform and, with every sign +1,
 * the plain H16 of the operand-wise hybrid, Sec. 3.3): R = H16 D / 4 on
 * 16 binary32 values in place -- the 16 signs applied once, the butterflies
 * of stride 1, 2, 4 and 8 (a + b, a - b), then the multiply by 1/sqrt(16) =
 * 0.25 (exact). */
void orc_hadamard16_f32(float y[16], const int8_t signs[16])
{
    for (int i = 0; i < 16; ++i) y[i] = y[i] * (float)signs[i];
    for (int h = 1; h < 16; h *= 2)
        for (int j = 0; j < 16; ++j)
            if ((j & h) == 0) {
                float a = y[j], b = y[j + h];
                y[j] = a + b;
                y[j + h] = a - b;
            }
    for (int i = 0; i < 16; ++i) y[i] = y[i] * 0.25f;
}

/* The same transform on every aligned 16-value block of every row. */
void orc_hadamard16_rows(float* x, int64_t R, int64_t C, const int8_t signs[16])
{
    for (int64_t r = 0; r < R; ++r)
        for (int64_t b = 0; b < C / 16; ++b) orc_hadamard16_f32(x + r * C + b * 16, signs);
}

/* Explicit Sylvester matrix H_32 (entries +-1): H_1 = [1],
 * H_2n = [[H_n, H_n], [H_n, -H_n]].  Written row-major into h[32*32]. */
void orc_sylvester_h32(int8_t* h)
{
    h[0] = 1;
    for (int n = 1; n < 32; n *= 2)
        for (int i = 0; i < n; ++i)
            for (int j = 0; j < n; ++j) {
                int8_t v = h[i * 32 + j];
                h[i * 32 + (j + n)] = v;
                h[(i + n) * 32 + j] = v;
                h[(i + n) * 32 + (j + n)] = (int8_t)-v;
            }
}

/* ------------------------------------------------------------------------ */
/* Matrix quantizers.  Each quantizes the rows of a logical R x C matrix      */
/* with scale blocks along the row (the consumer's K axis): a row-facing     */
/* view Q_r(T) is this applied to T, a column-facing view Q_c(T) is this      */
/* applied to T^T (Sec. 2.3, the three contractions Eqs. 4-6).                */
/* Outputs: codes[R*C] (one 4-bit code per byte), scales[R*C/bs] bytes.      */
/* ------------------------------------------------------------------------ */

/* MXFP4, 32-value blocks with upward E8M0 scales (Sec. 2.2.1).  x holds
 * binary32 values (bf16 inputs widened exactly, or H32 outputs).  With
 * sr != 0 the values are rounded stochastically (Sec. 2.5) using the
 * row-major logical index of the element in the whole tensor,
 * index0 + r * ld + c: x may be a block of rows and columns of a larger
 * tensor whose element (0, 0) has logical index index0 and whose rows are
 * ld long (index0 = 0, ld = C for a whole tensor). */
void orc_mx_quantize_rows(const float* x, int64_t R, int64_t C, int sr, uint64_t seed,
                          uint64_t offset, uint64_t index0, int64_t ld, uint8_t* codes, uint8_t* scales)
{
    for (int64_t r = 0; r < R; ++r)
        for (int64_t b = 0; b < C / 32; ++b) {
            const float* blk = x + r * C + b * 32;
            double amax = 0.0;
            for (int j = 0; j < 32; ++j)
                if (fabs((double)blk[j]) > amax) amax = fabs((double)blk[j]);
            int e = orc_e8m0_exponent_up(amax);
            scales[r * (C / 32) + b] = (uint8_t)(e + 127);
            for (int j = 0; j < 32; ++j) {
                float v = (float)((double)blk[j] * ldexp(1.0, -e)); /* fl32 */
                int64_t i = r * C + b * 32 + j;
                uint64_t li = index0 + (uint64_t)(r * ld + b * 32 + j);
                codes[i] = sr ? orc_e2m1_sr((double)v, orc_sr_uniform16(seed, offset, li))
                              : orc_e2m1_rn((double)v);
            }
        }
}

/* MXFP4 2D32 weights (Sec. 2.4, Eqs. 7-8): one exponent per 32x32 tile chosen
 * by the adaptive rule, values rounded to nearest.  tile_exp[(R/32)*(C/32)]
 * receives the E8M0 bytes of the tiles; codes[R*C] the codes in logical
 * (row-major) order.  The row-facing view is (codes, tile scale replicated
 * along each row block); the column-facing view is the transpose. */
void orc_mx_quantize_weight2d(const float* x, int64_t R, int64_t C, uint8_t* codes,
                              uint8_t* tile_scale)
{
    for (int64_t tr = 0; tr < R / 32; ++tr)
        for (int64_t tc = 0; tc < C / 32; ++tc) {
            double amax = 0.0;
            for (int i = 0; i < 32; ++i)
                for (int j = 0; j < 32; ++j) {
                    double a = fabs((double)x[(tr * 32 + i) * C + tc * 32 + j]);
                    if (a > amax) amax = a;
                }
            int e = orc_mx_weight_tile_exponent(amax);
            tile_scale[tr * (C / 32) + tc] = (uint8_t)(e + 127);
            for (int i = 0; i < 32; ++i)
                for (int j = 0; j < 32; ++j) {
                    int64_t k = (tr * 32 + i) * C + tc * 32 + j;
                    float v = (float)((double)x[k] * ldexp(1.0, -e));
                    codes[k] = orc_e2m1_rn((double)v);
                }
        }
}

/* NVFP4, 16-value blocks with E4M3 scales under a binary32 outer factor
 * (Sec. 2.2.2).  senc_row[r] is the S_enc that applies to row r: one value
 * for the whole tensor (global NVFP4) or the factor of the row's 128-row
 * strip (CTA-local NVFP4).  sr, index0 and ld as for MXFP4. */
void orc_nv_quantize_rows(const float* x, int64_t R, int64_t C, const float* senc_row, int sr,
                          uint64_t seed, uint64_t offset, uint64_t index0, int64_t ld, uint8_t* codes,
                          uint8_t* scales)
{
    for (int64_t r = 0; r < R; ++r)
        for (int64_t b = 0; b < C / 16; ++b) {
            const float* blk = x + r * C + b * 16;
            float amax = 0.0f;
            for (int j = 0; j < 16; ++j)
                if (fabsf(blk[j]) > amax) amax = fabsf(blk[j]);
            float m;
            scales[r * (C / 16) + b] = orc_nv_block_scale(amax, senc_row[r], &m);
            for (int j = 0; j < 16; ++j) {
                float v = blk[j] * m; /* fl32 */
                int64_t i = r * C + b * 16 + j;
                uint64_t li = index0 + (uint64_t)(r * ld + b * 16 + j);
                codes[i] = sr ? orc_e2m1_sr((double)v, orc_sr_uniform16(seed, offset, li))
                              : orc_e2m1_rn((double)v);
            }
        }
}

/* NVFP4 2D16 weights (Sec. 2.4): one E4M3 scale per 16x16 tile under one
 * outer factor senc shared by both orientations. */
void orc_nv_quantize_weight2d(const float* x, int64_t R, int64_t C, float senc, uint8_t* codes,
                              uint8_t* tile_scale)
{
    for (int64_t tr = 0; tr < R / 16; ++tr)
        for (int64_t tc = 0; tc < C / 16; ++tc) {
            float amax = 0.0f;
            for (int i = 0; i < 16; ++i)
                for (int j = 0; j < 16; ++j) {
                    float a = fabsf(x[(tr * 16 + i) * C + tc * 16 + j]);
                    if (a > amax) amax = a;
                }
            float m;
            tile_scale[tr * (C / 16) + tc] = orc_nv_block_scale(amax, senc, &m);
            for (int i = 0; i < 16; ++i)
                for (int j = 0; j < 16; ++j) {
                    int64_t k = (tr * 16 + i) * C + tc * 16 + j;
                    float v = x[k] * m;
                    codes[k] = orc_e2m1_rn((double)v);
                }
        }
}

/* Largest magnitude over a binary32 array (exact). */
float orc_amax_f32(const float* x, int64_t n)
{
    float a = 0.0f;
    for (int64_t i = 0; i < n; ++i)
        if (fabsf(x[i]) > a) a = fabsf(x[i]);
    return a;
}

/* Widen bf16 bit patterns to binary32 (exact). */
void orc_bf16_to_f32(const uint16_t* h, int64_t n, float* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = bf16_value(h[i]);
}

/* ------------------------------------------------------------------------ */
/* Decode and contraction (Sec. 2.3, Eqs. 4-6; Sec. 2.2 Eq. 1):               */
/* x_hat = Q * delta_b / S.  Operands are K-major: A[M][K], B[N][K];         */
/* C[m][n] = sum_k A_hat[m][k] * B_hat[n][k], binary64.                       */
/* fmt: 0 = MXFP4 (E8M0 per 32), 1 = NVFP4 (E4M3 per 16).                    */
/* senc_row: per-row S_enc (NVFP4) or NULL.                                  */
/* ------------------------------------------------------------------------ */

static double block_scale_value(int fmt, uint8_t s)
{
    return fmt == 0 ? ldexp(1.0, (int)s - 127) : orc_e4m3_value(s);
}

void orc_dequantize(const uint8_t* codes, const uint8_t* scales, int fmt, int64_t R, int64_t C,
                    const float* senc_row, double* out)
{
    int bs = fmt == 0 ? 32 : 16;
    for (int64_t r = 0; r < R; ++r)
        for (int64_t c = 0; c < C; ++c) {
            double v = orc_e2m1_value(codes[r * C + c]) * block_scale_value(fmt, scales[r * (C / bs) + c / bs]);
            if (senc_row) v = v / (double)senc_row[r];
            out[r * C + c] = v;
        }
}

/* Full contraction C = A_hat * B_hat^T over dequantized operands. */
void orc_gemm_nt(const double* A, const double* B, int64_t M, int64_t N, int64_t K, double* C)
{
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double s = 0.0;
            for (int64_t k = 0; k < K; ++k) s += A[m * K + k] * B[n * K + k];
            C[m * N + n] = s;
        }
}

/* Sampled contraction straight from codes and scales: for each (m, n) pair,
 * out = sum_k A_hat[m][k] * B_hat[n][k] and absout = sum_k |A_hat B_hat|. */
void orc_gemm_sampled(const uint8_t* a_codes, const uint8_t* a_scales, const float* a_senc,
                      const uint8_t* b_codes, const uint8_t* b_scales, const float* b_senc, int fmt,
                      int64_t K, const int64_t* ms, const int64_t* ns, int64_t count, double* out,
                      double* absout)
{
    int bs = fmt == 0 ? 32 : 16;
    for (int64_t t = 0; t < count; ++t) {
        int64_t m = ms[t], n = ns[t];
        double s = 0.0, sa = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double a = orc_e2m1_value(a_codes[m * K + k]) * block_scale_value(fmt, a_scales[m * (K / bs) + k / bs]);
            double b = orc_e2m1_value(b_codes[n * K + k]) * block_scale_value(fmt, b_scales[n * (K / bs) + k / bs]);
            if (a_senc) a = a / (double)a_senc[m];
            if (b_senc) b = b / (double)b_senc[n];
            s += a * b;
            sa += fabs(a * b);
        }
        out[t] = s;
        absout[t] = sa;
    }
}

/* ------------------------------------------------------------------------ */
/* Fused producers' model arithmetic (Sec. 3.2): the unfused BF16 model's    */
/* rounding points, since fusion changes data movement, not the model.       */
/* ------------------------------------------------------------------------ */

/* SiLU gate forward: h = bf16(fl32(silu(a1)) * a3) with silu evaluated in
 * binary64 and rounded to binary32; the product is a binary32 multiply. */
void orc_swiglu_h(const uint16_t* a1, const uint16_t* a3, int64_t n, uint16_t* h)
{
    for (int64_t i = 0; i < n; ++i) {
        double x = (double)bf16_value(a1[i]);
        float s = (float)(x / (1.0 + exp(-x)));
        float p = s * bf16_value(a3[i]);
        h[i] = orc_bf16_round((double)p);
    }
}

/* SiLU gate backward given dh (bf16), a1, a3:
 *   da1 = bf16(dh * a3 * sigma(a1) * (1 + a1 * (1 - sigma(a1)))),
 *   da3 = bf16(dh * silu(a1)), evaluated in binary64. */
void orc_swiglu_bwd(const uint16_t* dh, const uint16_t* a1, const uint16_t* a3, int64_t n,
                    uint16_t* da1, uint16_t* da3)
{
    for (int64_t i = 0; i < n; ++i) {
        double g = (double)bf16_value(dh[i]);
        double x = (double)bf16_value(a1[i]);
        double u = (double)bf16_value(a3[i]);
        double sg = 1.0 / (1.0 + exp(-x));
        da1[i] = orc_bf16_round(g * u * sg * (1.0 + x * (1.0 - sg)));
        da3[i] = orc_bf16_round(g * x * sg);
    }
}

/* Residual + RMSNorm forward for rows of width C:
 *   r' = bf16(r + b); rstd = fl32(1 / sqrt(mean(r'^2) + eps)) (binary64 mean).
 * If use_rstd != 0, rstd is taken from rstd_in instead (lets a test feed the
 * kernel's own row statistic), then y = bf16(fl32(fl32(r' * rstd) * g)). */
void orc_residual_rmsnorm(const uint16_t* r, const uint16_t* b, const uint16_t* g, int64_t R,
                          int64_t C, double eps, int use_rstd, const float* rstd_in,
                          uint16_t* r_out, float* rstd_out, uint16_t* y)
{
    for (int64_t i = 0; i < R; ++i) {
        double ss = 0.0;
        for (int64_t j = 0; j < C; ++j) {
            uint16_t rp = orc_bf16_round((double)bf16_value(r[i * C + j]) + (double)bf16_value(b[i * C + j]));
            r_out[i * C + j] = rp;
            double v = (double)bf16_value(rp);
            ss += v * v;
        }
        float rs = (float)(1.0 / sqrt(ss / (double)C + eps));
        rstd_out[i] = rs;
        float use = use_rstd ? rstd_in[i] : rs;
        for (int64_t j = 0; j < C; ++j) {
            float t = bf16_value(r_out[i * C + j]) * use;
            float u = t * bf16_value(g[j]);
            y[i * C + j] = orc_bf16_round((double)u);
        }
    }
}

/* RMSNorm backward (plain BF16/FP32 model gradient) for one row set:
 *   xh = r' * rstd,  gy = dy * g,
 *   dr' = rstd * (gy - xh * mean(gy * xh)),
 *   dr  = bf16(dr' + dres) where dres is the gradient arriving on the
 *   residual stream.  Evaluated in binary64. */
void orc_rmsnorm_bwd(const uint16_t* dy, const uint16_t* rp, const float* rstd, const uint16_t* g,
                     const uint16_t* dres, int64_t R, int64_t C, uint16_t* dr)
{
    for (int64_t i = 0; i < R; ++i) {
        double s = 0.0;
        for (int64_t j = 0; j < C; ++j) {
            double xh = (double)bf16_value(rp[i * C + j]) * (double)rstd[i];
            double gy = (double)bf16_value(dy[i * C + j]) * (double)bf16_value(g[j]);
            s += gy * xh;
        }
        double mean = s / (double)C;
        for (int64_t j = 0; j < C; ++j) {
            double xh = (double)bf16_value(rp[i * C + j]) * (double)rstd[i];
            double gy = (double)bf16_value(dy[i * C + j]) * (double)bf16_value(g[j]);
            double d = (double)rstd[i] * (gy - xh * mean);
            dr[i * C + j] = orc_bf16_round(d + (double)bf16_value(dres[i * C + j]));
        }
    }
}

/* ------------------------------------------------------------------------ */
/* QKV producer with RoPE ("Format-Aware Fusion for Fast FP4 Pretraining",   */
/* Sec. 3.2: the Q/K projection applies RoPE and the attention layout; the   */
/* backward combines the inverse layout and RoPE with the QKV gradient        */
/* production).  Readings: Llama-3 heads of D values, the QKV columns laid    */
/* out [Q heads | K heads | V heads]; rotate-half pairs (i, i + D/2) turned   */
/* by p * theta^(-2i/D) at position p = token mod S; the outputs head-major   */
/* [heads][T][D].                                                             */
/* ------------------------------------------------------------------------ */

/* cos/sin of p * theta^(-2i/D) for p < S, i < D/2 in binary64, rounded to
 * binary32 ([S][D/2] each). */
void orc_rope_tables(int64_t S, int D, double theta, float* cos_t, float* sin_t)
{
    const int h = D / 2;
    for (int64_t p = 0; p < S; ++p)
        for (int i = 0; i < h; ++i) {
            double a = (double)p * pow(theta, -2.0 * (double)i / (double)D);
            cos_t[p * h + i] = (float)cos(a);
            sin_t[p * h + i] = (float)sin(a);
        }
}

/* One head of D bf16 values turned by the angles of one position (c, s of
 * D/2 each); binary32 products and sums, then bf16.  inverse != 0 applies
 * the transposed rotation (the gradient's). */
static void rope_head(const uint16_t* x, const float* c, const float* s, int D, int inverse, uint16_t* y)
{
    const int h = D / 2;
    for (int i = 0; i < h; ++i) {
        float a = bf16_value(x[i]), b = bf16_value(x[i + h]);
        float ac = a * c[i], bs = b * s[i], bc = b * c[i], as = a * s[i];
        float lo = inverse ? ac + bs : ac - bs;
        float hi = inverse ? bc - as : bc + as;
        y[i] = orc_bf16_round((double)lo);
        y[i + h] = orc_bf16_round((double)hi);
    }
}

/* Forward: qkv [T][(hq + 2 hkv) D] bf16 -> q [hq][T][D], k [hkv][T][D]
 * (turned), v [hkv][T][D] (copied). */
void orc_qkv_rope_fwd(const uint16_t* qkv, int64_t T, int64_t S, int hq, int hkv, int D, const float* cos_t,
                      const float* sin_t, uint16_t* q, uint16_t* k, uint16_t* v)
{
    const int64_t N = (int64_t)(hq + 2 * hkv) * D;
    for (int64_t t = 0; t < T; ++t) {
        const int64_t p = t % S;
        const float* c = cos_t + p * (D / 2);
        const float* s = sin_t + p * (D / 2);
        for (int hd = 0; hd < hq + 2 * hkv; ++hd) {
            const uint16_t* src = qkv + t * N + (int64_t)hd * D;
            if (hd < hq)
                rope_head(src, c, s, D, 0, q + ((int64_t)hd * T + t) * D);
            else if (hd < hq + hkv)
                rope_head(src, c, s, D, 0, k + ((int64_t)(hd - hq) * T + t) * D);
            else
                for (int i = 0; i < D; ++i) v[((int64_t)(hd - hq - hkv) * T + t) * D + i] = src[i];
        }
    }
}

/* Backward: dq [hq][T][D], dk, dv [hkv][T][D] -> dqkv [T][(hq + 2 hkv) D]
 * (dq, dk turned back, dv copied). */
void orc_qkv_rope_bwd(const uint16_t* dq, const uint16_t* dk, const uint16_t* dv, int64_t T, int64_t S, int hq,
                      int hkv, int D, const float* cos_t, const float* sin_t, uint16_t* dqkv)
{
    const int64_t N = (int64_t)(hq + 2 * hkv) * D;
    for (int64_t t = 0; t < T; ++t) {
        const int64_t p = t % S;
        const float* c = cos_t + p * (D / 2);
        const float* s = sin_t + p * (D / 2);
        for (int hd = 0; hd < hq + 2 * hkv; ++hd) {
            uint16_t* dst = dqkv + t * N + (int64_t)hd * D;
            if (hd < hq)
                rope_head(dq + ((int64_t)hd * T + t) * D, c, s, D, 1, dst);
            else if (hd < hq + hkv)
                rope_head(dk + ((int64_t)(hd - hq) * T + t) * D, c, s, D, 1, dst);
            else
                for (int i = 0; i < D; ++i) dst[i] = dv[((int64_t)(hd - hq - hkv) * T + t) * D + i];
        }
    }
}
