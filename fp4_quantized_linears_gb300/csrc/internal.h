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
    int route;
    unsigned views, flags;
    uint64_t seed, offset;
    uint32_t sign_mask;  // bit j set: sign j of the H32 diagonal is -1
    uint8_t* row_codes;
    uint8_t* row_scales;
    float* row_outer;
    uint8_t* col_codes;
    uint8_t* col_scales;
    float* col_outer;
    uint32_t* amax_ws;  // NVFP4: [1 + R/128 + C/128] amax bit slots
};

int launch_quantize(const QuantParams& p, cudaStream_t stream);
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
};

int launch_gemm(const GemmParams& p, cudaStream_t stream);
int gemm_status(cudaStream_t stream, int* code, bool reset);

}  // namespace fp4
