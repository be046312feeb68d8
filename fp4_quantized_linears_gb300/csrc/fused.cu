// fused.cu -- row statistics of the residual-RMSNorm producer (sm_103a).
//
// "Format-Aware Fusion for Fast FP4 Pretraining", Sec. 3.2: the
// residual-RMSNorm boundary retains the exact residual and its row
// statistics while producing the next quantized representations.  The row
// pass here produces the retained state; the quantizer kernel then reads it
// back (an L2-resident re-read for Llama-sized rows) through its RMSNorm
// pre-op and emits both FP4 views in the same pass.
//
//   forward   r' = bf16(r + b),  rstd = fl32(1 / sqrt(mean(r'^2) + eps))
//   backward  mean_g = mean_c(fl32(dy * g) * fl32(r' * rstd))  (per row, fp32)
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"

namespace fp4 {

namespace {

constexpr int ROW_THREADS = 256;

FP4_DEV float block_sum(float v, float* red) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    if (l == 0) red[w] = v;
    __syncthreads();
    if (w == 0) {
        v = l < (ROW_THREADS / 32) ? red[l] : 0.0f;
#pragma unroll
        for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
        if (l == 0) red[0] = v;
    }
    __syncthreads();
    return red[0];
}

// One CTA per row; 8 bf16 per 16-byte vector.
__global__ void __launch_bounds__(ROW_THREADS) rmsnorm_fwd_stats_kernel(const uint16_t* __restrict__ r,
                                                                       const uint16_t* __restrict__ b,
                                                                       int64_t C, int64_t ld, float eps,
                                                                       uint16_t* __restrict__ r_out,
                                                                       float* __restrict__ rstd) {
    __shared__ float red[ROW_THREADS / 32];
    const int64_t row = blockIdx.x;
    const uint16_t* rr = r + row * ld;
    const uint16_t* bb = b ? b + row * ld : nullptr;
    uint16_t* ro = r_out + row * C;
    float ss = 0.0f;
    for (int64_t c = (int64_t)threadIdx.x * 8; c < C; c += ROW_THREADS * 8) {
        uint4 x = *reinterpret_cast<const uint4*>(rr + c);
        uint4 y = bb ? *reinterpret_cast<const uint4*>(bb + c) : make_uint4(0, 0, 0, 0);
        uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w}, os[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            float a0 = __fadd_rn(bf16_lo(xs[k]), bf16_lo(ys[k]));
            float a1 = __fadd_rn(bf16_hi(xs[k]), bf16_hi(ys[k]));
            uint16_t h0 = f32_to_bf16_rn(a0), h1 = f32_to_bf16_rn(a1);
            float v0 = bf16_to_f32(h0), v1 = bf16_to_f32(h1);
            ss = fmaf(v0, v0, ss);
            ss = fmaf(v1, v1, ss);
            os[k] = (uint32_t)h0 | ((uint32_t)h1 << 16);
        }
        *reinterpret_cast<uint4*>(ro + c) = make_uint4(os[0], os[1], os[2], os[3]);
    }
    float tot = block_sum(ss, red);
    if (threadIdx.x == 0) rstd[row] = 1.0f / sqrtf(tot / (float)C + eps);
}

// The forward row pass for an NVFP4 encode: as above, and then the maxima of
// y = bf16(fl32(fl32(r' * rstd) * g)) that the encoder's outer factors need,
// folded into its amax slots [tensor, R/128 row strips, C/128 column
// strips]: CTAs of a grid sized to the resident slots take rows
// blockIdx.x, blockIdx.x + gridDim.x, ...; a row's maximum goes to its
// row-strip slot, the column-strip maxima collect in shared memory and reach
// global memory once per CTA, as does the tensor maximum.
__global__ void __launch_bounds__(ROW_THREADS) rmsnorm_fwd_stats_amax_kernel(
    const uint16_t* __restrict__ r, const uint16_t* __restrict__ b, const uint16_t* __restrict__ g, int64_t R,
    int64_t C, int64_t ld, float eps, uint16_t* __restrict__ r_out, float* __restrict__ rstd,
    uint32_t* __restrict__ ws) {
    __shared__ float red[ROW_THREADS / 32];
    __shared__ uint32_t redm[ROW_THREADS / 32];
    extern __shared__ uint32_t colmax[];  // C / 128 strips
    const int64_t n_strips = C / 128;
    for (int64_t i = threadIdx.x; i < n_strips; i += ROW_THREADS) colmax[i] = 0;
    uint32_t tmax = 0;  // this CTA's tensor maximum (thread 0)
    __syncthreads();
    for (int64_t row = blockIdx.x; row < R; row += gridDim.x) {
        const uint16_t* rr = r + row * ld;
        const uint16_t* bb = b ? b + row * ld : nullptr;
        uint16_t* ro = r_out + row * C;
        float ss = 0.0f;
        for (int64_t c = (int64_t)threadIdx.x * 8; c < C; c += ROW_THREADS * 8) {
            uint4 x = *reinterpret_cast<const uint4*>(rr + c);
            uint4 y = bb ? *reinterpret_cast<const uint4*>(bb + c) : make_uint4(0, 0, 0, 0);
            uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w}, os[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                float a0 = __fadd_rn(bf16_lo(xs[k]), bf16_lo(ys[k]));
                float a1 = __fadd_rn(bf16_hi(xs[k]), bf16_hi(ys[k]));
                uint16_t h0 = f32_to_bf16_rn(a0), h1 = f32_to_bf16_rn(a1);
                float v0 = bf16_to_f32(h0), v1 = bf16_to_f32(h1);
                ss = fmaf(v0, v0, ss);
                ss = fmaf(v1, v1, ss);
                os[k] = (uint32_t)h0 | ((uint32_t)h1 << 16);
            }
            *reinterpret_cast<uint4*>(ro + c) = make_uint4(os[0], os[1], os[2], os[3]);
        }
        const float tot = block_sum(ss, red);
        const float rs = 1.0f / sqrtf(tot / (float)C + eps);
        if (threadIdx.x == 0) rstd[row] = rs;
        // y over the row just written (this thread's own chunks)
        uint32_t rmax = 0;
        for (int64_t c = (int64_t)threadIdx.x * 8; c < C; c += ROW_THREADS * 8) {
            const uint4 x = *reinterpret_cast<const uint4*>(ro + c);
            const uint4 gv = *reinterpret_cast<const uint4*>(g + c);
            const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, gs[4] = {gv.x, gv.y, gv.z, gv.w};
            uint32_t m2 = 0;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float y0 = __fmul_rn(__fmul_rn(bf16_lo(xs[k]), rs), bf16_lo(gs[k]));
                const float y1 = __fmul_rn(__fmul_rn(bf16_hi(xs[k]), rs), bf16_hi(gs[k]));
                const uint32_t yw = (uint32_t)f32_to_bf16_rn(y0) | ((uint32_t)f32_to_bf16_rn(y1) << 16);
                m2 = __vmaxu2(m2, yw & 0x7FFF7FFFu);
            }
            const uint32_t m = max(m2 << 16, m2 & 0xFFFF0000u);
            atomicMax(&colmax[c >> 7], m);
            rmax = max(rmax, m);
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) rmax = max(rmax, __shfl_xor_sync(0xFFFFFFFFu, rmax, o));
        if ((threadIdx.x & 31) == 0) redm[threadIdx.x >> 5] = rmax;
        __syncthreads();
        if (threadIdx.x == 0) {
            for (int i = 1; i < ROW_THREADS / 32; ++i) rmax = max(rmax, redm[i]);
            atomicMax(&ws[1 + (row >> 7)], rmax);
            tmax = max(tmax, rmax);
        }
        __syncthreads();  // red / redm are reused by the next row
    }
    for (int64_t i = threadIdx.x; i < n_strips; i += ROW_THREADS)
        if (colmax[i]) atomicMax(&ws[1 + (R >> 7) + i], colmax[i]);
    if (threadIdx.x == 0 && tmax) atomicMax(&ws[0], tmax);
}

// mean_g[row] = (1/C) sum_c fl32(dy * g) * fl32(r' * rstd)
__global__ void __launch_bounds__(ROW_THREADS) rmsnorm_bwd_stats_kernel(const uint16_t* __restrict__ dy,
                                                                       const uint16_t* __restrict__ rp,
                                                                       const float* __restrict__ rstd,
                                                                       const uint16_t* __restrict__ g, int64_t C,
                                                                       float* __restrict__ mean_g) {
    __shared__ float red[ROW_THREADS / 32];
    const int64_t row = blockIdx.x;
    const float rs = rstd[row];
    float s = 0.0f;
    for (int64_t c = (int64_t)threadIdx.x * 8; c < C; c += ROW_THREADS * 8) {
        uint4 d = *reinterpret_cast<const uint4*>(dy + row * C + c);
        uint4 x = *reinterpret_cast<const uint4*>(rp + row * C + c);
        uint4 gg = *reinterpret_cast<const uint4*>(g + c);
        uint32_t ds[4] = {d.x, d.y, d.z, d.w}, xs[4] = {x.x, x.y, x.z, x.w}, gs[4] = {gg.x, gg.y, gg.z, gg.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            s = fmaf(__fmul_rn(bf16_lo(ds[k]), bf16_lo(gs[k])), __fmul_rn(bf16_lo(xs[k]), rs), s);
            s = fmaf(__fmul_rn(bf16_hi(ds[k]), bf16_hi(gs[k])), __fmul_rn(bf16_hi(xs[k]), rs), s);
        }
    }
    float tot = block_sum(s, red);
    if (threadIdx.x == 0) mean_g[row] = tot / (float)C;
}

// One thread per row: the row terms that a data-gradient epilogue wrote per
// 64-column block, summed in block order, divided by the row length.
__global__ void __launch_bounds__(256) rms_parts_reduce_kernel(const float* __restrict__ part, int64_t R,
                                                               int64_t nparts, int64_t C, float* __restrict__ mean_g) {
    const int64_t row = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (row >= R) return;
    const float* pr = part + row * nparts;
    float s = 0.0f;
    for (int64_t j = 0; j < nparts; ++j) s = __fadd_rn(s, pr[j]);
    mean_g[row] = s / (float)C;
}

}  // namespace

int launch_rms_parts_reduce(const float* part, int64_t R, int64_t nparts, int64_t C, float* mean_g,
                            cudaStream_t stream) {
    rms_parts_reduce_kernel<<<(unsigned)((R + 255) / 256), 256, 0, stream>>>(part, R, nparts, C, mean_g);
    return cudaGetLastError() == cudaSuccess ? FP4_OK : FP4_ERR_CUDA;
}

int launch_rmsnorm_fwd_stats(const uint16_t* r, const uint16_t* b, int64_t R, int64_t C, int64_t ld, float eps,
                             uint16_t* r_out, float* rstd, cudaStream_t stream) {
    rmsnorm_fwd_stats_kernel<<<(unsigned)R, ROW_THREADS, 0, stream>>>(r, b, C, ld, eps, r_out, rstd);
    return cudaGetLastError() == cudaSuccess ? FP4_OK : FP4_ERR_CUDA;
}

int launch_rmsnorm_fwd_stats_amax(const uint16_t* r, const uint16_t* b, const uint16_t* g, int64_t R, int64_t C,
                                  int64_t ld, float eps, uint16_t* r_out, float* rstd, uint32_t* amax_ws,
                                  cudaStream_t stream) {
    int dev = 0, sms = 1;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess)
        return FP4_ERR_CUDA;
    const int64_t slots = (int64_t)sms * 8;  // 256 threads: eight CTAs per SM
    const size_t smem = (size_t)(C / 128) * 4;
    if (smem > 48 * 1024) return FP4_ERR_UNSUPPORTED_SHAPE;
    rmsnorm_fwd_stats_amax_kernel<<<(unsigned)(R < slots ? R : slots), ROW_THREADS, smem, stream>>>(
        r, b, g, R, C, ld, eps, r_out, rstd, amax_ws);
    return cudaGetLastError() == cudaSuccess ? FP4_OK : FP4_ERR_CUDA;
}

int launch_rmsnorm_bwd_stats(const uint16_t* dy, const uint16_t* rp, const float* rstd, const uint16_t* g, int64_t R,
                             int64_t C, float* mean_g, cudaStream_t stream) {
    rmsnorm_bwd_stats_kernel<<<(unsigned)R, ROW_THREADS, 0, stream>>>(dy, rp, rstd, g, C, mean_g);
    return cudaGetLastError() == cudaSuccess ? FP4_OK : FP4_ERR_CUDA;
}

}  // namespace fp4
