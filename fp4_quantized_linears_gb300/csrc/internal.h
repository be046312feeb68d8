// internal.h -- host-side interface between the C ABI (api.cu) and the
// kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/fp4lin.h"

namespace fp4 {

struct QuantParams {
    const uint16_t* x;  // bf16 [R][ld]
    int64_t R, C, ld;
    int row_route, col_route;  // FP4_ROUTE_* of each view (they differ in the operand-wise hybrid)
    unsigned views, flags;
    uint64_t seed, offset;
    uint32_t sr_keys[20];  // Philox round keys of `seed` (sr_round_keys)
    uint32_t sign_mask;  // bit j set: sign j of the H32 / H16 diagonal is -1
    uint8_t* row_codes;
    uint8_t* row_scales;
    float* row_outer;
    uint8_t* col_codes;
    uint8_t* col_scales;
    float* col_outer;
    uint32_t* amax_ws;  // NVFP4: amax bit slots [tensor, R/128 row strips, C/128 column strips,
                        // (H16 NVFP4 column view) transformed tensor]
    // Optional element-wise pre-op applied while the tile is loaded (the
    // residual-RMSNorm producer, Sec. 3.2):
    //   PRE_RMSNORM_FWD  x = r',  value = bf16(fl32(fl32(r' * rstd[r]) * g[c]))
    //   PRE_RMSNORM_BWD  x = dy,  value = bf16(fl32(fl32(rstd[r] * fl32(fl32(dy * g[c])
    //                                 - fl32(fl32(r' * rstd[r]) * mean_g[r]))) + dres))
    int pre;
    const float* rstd;
    const uint16_t* g;
    const float* mean_g;
    const uint16_t* rp;    // r' (bwd)
    const uint16_t* dres;  // incoming residual gradient (bwd), may be NULL
    uint16_t* tap;         // bf16 [R][C] copy of the values quantized (NULL: not written)
    int amax_ready;        // NVFP4: amax_ws already holds x's maxima (no pre-pass)
    //   PRE_ROPE_BWD     x = (dq, dk, dv) head-major [heads][R][128]; value = the
    //                    QKV-layout gradient [R][C], dq and dk turned back
    //                    (bf16(fl32(fl32(a c) + fl32(b s))), bf16(fl32(fl32(b c) - fl32(a s))))
    const uint16_t* rope_src[3];
    const float* rope_cos;  // [seq_len][64]
    const float* rope_sin;
    int64_t seq_len;
    int heads_q, heads_kv;
};

enum { PRE_NONE = 0, PRE_RMSNORM_FWD = 1, PRE_RMSNORM_BWD = 2, PRE_ROPE_BWD = 3 };

int launch_rmsnorm_fwd_stats(const uint16_t* r, const uint16_t* b, int64_t R, int64_t C, int64_t ld, float eps,
                             uint16_t* r_out, float* rstd, cudaStream_t stream);
// the same, and for an NVFP4 encode the maxima of y = bf16(r' * rstd * g)
// folded into the quantizer's amax slots (zeroed by the caller)
int launch_rmsnorm_fwd_stats_amax(const uint16_t* r, const uint16_t* b, const uint16_t* g, int64_t R, int64_t C,
                                  int64_t ld, float eps, uint16_t* r_out, float* rstd, uint32_t* amax_ws,
                                  cudaStream_t stream);
int launch_rmsnorm_bwd_stats(const uint16_t* dy, const uint16_t* rp, const float* rstd, const uint16_t* g, int64_t R,
                             int64_t C, float* mean_g, cudaStream_t stream);
// mean_g[row] = (sum over j in order of part[row][j]) / C
int launch_rms_parts_reduce(const float* part, int64_t R, int64_t nparts, int64_t C, float* mean_g,
                            cudaStream_t stream);

int launch_quantize(const QuantParams& p, cudaStream_t stream);
// amax slots (4 bytes each) a quantizer call needs in its workspace
size_t quant_workspace_slots(int64_t R, int64_t C, int row_route, int col_route, unsigned views, unsigned flags);
int quant_status(cudaStream_t stream, int* code, bool reset);

// C[M][N] = alpha(m,n) * A_hat[M][K] . B_hat[N][K]^T + beta * C
struct GemmParams {
    const uint8_t* a_codes;
    const uint8_t* a_scales;
    const float* a_outer;  // NVFP4: S_enc values (count a_outer_count) or NULL
    int a_outer_count;
    const uint8_t* b_codes;
    const uint8_t* b_scales;
    const float* b_outer;
    int b_outer_count;
    int64_t M, N, K;
    int nv;         // 0 = MXFP4 (E8M0 / 32), 1 = NVFP4 (E4M3 / 16)
    void* c;
    int out_dtype;  // FP4_OUT_F32 / FP4_OUT_BF16
    float beta;
    // fused producer epilogues (0 = plain store, 1 = SwiGLU forward, 2 = SwiGLU backward)
    int epi;
    int64_t b_rows;       // rows of the B code tensor (set by the launcher)
    int64_t f;            // SwiGLU inner width
    uint16_t* a1;         // bf16 [M][f]
    uint16_t* a3;
    uint16_t* tap0;       // fwd h / bwd dh, bf16 [M][f], optional
    uint16_t* tap1;       // bwd [da1 | da3], bf16 [M][2f], optional
    int quantize;         // MX views emitted by the epilogue
    uint8_t* q_row_codes;
    uint8_t* q_row_scales;
    uint8_t* q_col_codes;
    uint8_t* q_col_scales;
    uint64_t seed, offset;
    // epi 3: the QKV projection with RoPE -> head-major bf16 [heads][M][128]
    uint16_t* q_out;
    uint16_t* k_out;
    uint16_t* v_out;
    const float* rope_cos;  // [seq_len][64] binary32
    const float* rope_sin;
    int64_t seq_len;
    int heads_q, heads_kv;
    // plain bf16 store feeding a residual-RMSNorm backward: the row terms
    // part[m][n / 64] = sum over the 64-column block of fl32(c * g) * fl32(r' * rstd)
    const uint16_t* rms_rp;  // r' bf16 [M][N]
    const uint16_t* rms_g;   // g bf16 [N]
    const float* rms_rstd;   // [M]
    float* rms_part;         // [M][N / 64], or NULL
    // SwiGLU epilogues writing the bf16 tap for an NVFP4 encode: the tap's
    // maxima folded into the quantizer's amax slots (tensor, row strips,
    // column strips of the [M][f] or [M][2f] tensor), or NULL
    uint32_t* amax_ws;
};

int launch_gemm(const GemmParams& p, cudaStream_t stream);
int gemm_status(cudaStream_t stream, int* code, bool reset);
void gemm_set_wait_limit(uint64_t cycles);     // 0: the default bound
void gemm_test_skip_first_release(int enable);  // test hook (fp4_test_skip_accumulator_release)

}  // namespace fp4
