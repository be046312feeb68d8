// gemm.cu -- block-scaled FP4 GEMM on the 5th-generation tensor cores
// (tcgen05) of sm_103a.
//
// Computes C[m][n] = alpha(m, n) * sum_k A_hat[m][k] B_hat[n][k] + beta * C[m][n]
// for the three contractions of "Format-Aware Fusion for Fast FP4
// Pretraining", Sec. 2.3 (Eqs. 4-6).  Every producer emits K-major operands,
// so Fprop, Dgrad and Wgrad are the same "TN" kernel over different views.
// alpha is 1 for MXFP4 and 1 / (S_enc,A[m/128] * S_enc,B[n/128]) for NVFP4,
// the CTA-local epilogue of Sec. 2.2.2 (the factors stay fixed over the whole
// K reduction and are applied together after it).
//
// Structure (one CTA per 128 x BN output tile, 192 threads):
//   warp 0      TMA producer: 2D tensor loads of the A and B code tiles
//               (128-byte swizzle) and 1D bulk copies of their scale atoms
//               into a STAGES-deep shared-memory ring guarded by mbarriers;
//   warp 1      allocates tensor memory; one thread copies each stage's scale
//               atoms into TMEM (tcgen05.cp 32x128b.warpx4) and issues the
//               block-scaled MMAs (kind::mxf4 with E8M0 scales, 2 per 64 K, or
//               kind::mxf4nvf4 with E4M3 scales, 4 per 64 K) into a 128 x BN
//               FP32 accumulator in TMEM; tcgen05.commit releases each stage;
//   warps 2-5   epilogue: tcgen05.ld of the accumulator (each warp its own
//               32-lane quarter), alpha / beta, 16-byte global stores.
// Every mbarrier wait is bounded: a wait that runs out sets the sticky status
// word to FP4_ERR_TIMEOUT, the roles drain what they issued and the CTA
// returns, releasing its tensor memory.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace fp4 {

__device__ unsigned int g_status_gemm;

namespace {

constexpr int BM = 128;
constexpr int BK = 256;          // FP4 elements per stage (128 bytes per row)
constexpr int BK_BYTES = BK / 2;
constexpr int STAGES = 4;
constexpr int THREADS = 192;
constexpr int TMEM_COLS = 512;
constexpr int SF_COL0 = 256;     // first TMEM column of the scale-factor region
constexpr long long WAIT_CYCLES = 4000000000LL;  // ~2 s at 2 GHz

// ------------------------------------------------------------ PTX wrappers -
FP4_DEV uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

FP4_DEV void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
FP4_DEV void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
FP4_DEV bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait; false (and the status word set) when the budget runs out.
FP4_DEV bool mbar_wait(uint64_t* bar, uint32_t parity) {
    long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > WAIT_CYCLES) {
            set_status(&g_status_gemm, FP4_ERR_TIMEOUT);
            return false;
        }
    }
    return true;
}

FP4_DEV void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(dst)),
        "l"((uint64_t)map), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}
FP4_DEV void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

FP4_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
FP4_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

FP4_DEV void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// shared-memory matrix descriptor (tcgen05): start, LBO, SBO (bytes >> 4),
// version 1 at bit 46, layout type at bits 61..63.
FP4_DEV uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t layout) {
    return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | ((uint64_t)layout << 61);
}
constexpr uint32_t LAYOUT_SW128 = 2;
constexpr uint32_t LAYOUT_NONE = 0;

// Instruction descriptor of the block-scaled kinds: E2M1 A and B (format 1),
// both K-major, N >> 3 at bit 17, scale type at bit 23 (1 = UE8M0,
// 0 = UE4M3), M >> 4 at bit 24, scale-factor byte ids at bits 29 (A) / 4 (B).
FP4_DEV uint32_t make_idesc(int n, bool ue8m0, uint32_t sfa_id, uint32_t sfb_id) {
    return (sfb_id << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((ue8m0 ? 1u : 0u) << 23) |
           ((uint32_t)(BM >> 4) << 24) | (sfa_id << 29);
}

FP4_DEV void mma_mxf4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t sfa, uint32_t sfb,
                      uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.u32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
        : "memory");
}
FP4_DEV void mma_nvf4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t sfa, uint32_t sfb,
                      uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.u32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
        : "memory");
}
FP4_DEV void tc_cp_sf(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

FP4_DEV void tmem_ld32(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ----------------------------------------------------------------- kernel -
struct KParams {
    const uint8_t* a_scales;
    const uint8_t* b_scales;
    const float* a_outer;
    const float* b_outer;
    int a_outer_count, b_outer_count;
    int64_t M, N, K;
    void* c;
    int out_dtype;
    float beta;
};

template <bool NV, int BN>
struct Cfg {
    static constexpr int SF_CHUNKS = NV ? 4 : 2;           // 512-byte atoms per 128 rows per stage
    static constexpr int A_BYTES = BM * BK_BYTES;          // 16 KB
    static constexpr int B_BYTES = BN * BK_BYTES;          // 16 / 32 KB
    static constexpr int SFA_BYTES = SF_CHUNKS * 512;
    static constexpr int SFB_BYTES = (BN / 128) * SF_CHUNKS * 512;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
    static constexpr int SF_COLS_A = SF_CHUNKS * 4;          // TMEM columns per stage
    static constexpr int SF_COLS_B = SF_CHUNKS * (BN / 32);
    static constexpr int SF_COLS = SF_COLS_A + SF_COLS_B;
    static constexpr int SMEM = STAGES * STAGE_BYTES + 1024 /*align*/ + 256 /*barriers*/;
    static_assert(SF_COL0 + STAGES * SF_COLS <= TMEM_COLS, "TMEM budget");
    static_assert(STAGE_BYTES % 1024 == 0, "stage alignment");
};

template <bool NV, int BN>
__global__ void __launch_bounds__(THREADS, 1)
    fp4_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, KParams p) {
    using C = Cfg<NV, BN>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * C::STAGE_BYTES);
    uint64_t* empty = full + STAGES;
    uint64_t* acc_full = empty + STAGES;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t m0 = (int64_t)blockIdx.y * BM, n0 = (int64_t)blockIdx.x * BN;
    const int num_kb = (int)(p.K / BK);

    auto stage_a = [&](int s) { return smem + s * C::STAGE_BYTES; };
    auto stage_b = [&](int s) { return smem + s * C::STAGE_BYTES + C::A_BYTES; };
    auto stage_sfa = [&](int s) { return smem + s * C::STAGE_BYTES + C::A_BYTES + C::B_BYTES; };
    auto stage_sfb = [&](int s) { return smem + s * C::STAGE_BYTES + C::A_BYTES + C::B_BYTES + C::SFA_BYTES; };

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(acc_full, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------ TMA producer ----
        const int64_t k_atoms_a = NV ? p.K / 64 : p.K / 128;  // atoms per 128-row block
        int last_issued = -1;
        for (int kb = 0; kb < num_kb; ++kb) {
            int s = kb % STAGES;
            if (kb >= STAGES) {
                if (*abort_flag || !mbar_wait(&empty[s], ((kb / STAGES) - 1) & 1)) {
                    *abort_flag = 1;
                    break;
                }
            }
            mbar_expect_tx(&full[s], C::STAGE_BYTES);
            tma_load_2d(stage_a(s), &tmA, kb * BK_BYTES, (int)m0, &full[s]);
            tma_load_2d(stage_b(s), &tmB, kb * BK_BYTES, (int)n0, &full[s]);
            const uint8_t* sfa = p.a_scales + ((m0 >> 7) * k_atoms_a + (int64_t)kb * C::SF_CHUNKS) * 512;
            bulk_load(stage_sfa(s), sfa, C::SFA_BYTES, &full[s]);
#pragma unroll
            for (int h = 0; h < BN / 128; ++h) {
                const uint8_t* sfb = p.b_scales + (((n0 >> 7) + h) * k_atoms_a + (int64_t)kb * C::SF_CHUNKS) * 512;
                bulk_load(stage_sfb(s) + h * C::SF_CHUNKS * 512, sfb, C::SF_CHUNKS * 512, &full[s]);
            }
            last_issued = kb;
        }
        if (*abort_flag) {
            // drain: wait (bounded) for the loads still in flight
            for (int kb = last_issued - STAGES + 1; kb <= last_issued; ++kb)
                if (kb >= 0) mbar_wait(&full[kb % STAGES], (kb / STAGES) & 1);
        }
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------ MMA issuer ------
        const uint32_t sf_base = tmem + SF_COL0;
        bool ok = true;
        for (int kb = 0; kb < num_kb; ++kb) {
            int s = kb % STAGES;
            if (*abort_flag || !mbar_wait(&full[s], (kb / STAGES) & 1)) {
                *abort_flag = 1;
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t sfa_col = sf_base + s * C::SF_COLS;
            const uint32_t sfb_col = sfa_col + C::SF_COLS_A;
            // scale atoms -> TMEM (replicated into the four lane quarters)
#pragma unroll
            for (int c = 0; c < C::SF_CHUNKS; ++c) {
                tc_cp_sf(sfa_col + 4 * c, smem_desc(smem_u32(stage_sfa(s) + c * 512), 0, 128, LAYOUT_NONE));
#pragma unroll
                for (int h = 0; h < BN / 128; ++h)
                    tc_cp_sf(sfb_col + c * (BN / 32) + 4 * h,
                             smem_desc(smem_u32(stage_sfb(s) + (h * C::SF_CHUNKS + c) * 512), 0, 128, LAYOUT_NONE));
            }
            const uint32_t a_base = smem_u32(stage_a(s)), b_base = smem_u32(stage_b(s));
#pragma unroll
            for (int kk = 0; kk < BK / 64; ++kk) {
                uint64_t ad = smem_desc(a_base + kk * 32, 16, 1024, LAYOUT_SW128);
                uint64_t bd = smem_desc(b_base + kk * 32, 16, 1024, LAYOUT_SW128);
                uint32_t acc = (kb > 0 || kk > 0) ? 1u : 0u;
                if (NV) {
                    uint32_t id = make_idesc(BN, false, 0, 0);
                    mma_nvf4(tmem, ad, bd, id, sfa_col + 4 * kk, sfb_col + kk * (BN / 32), acc);
                } else {
                    int c = kk >> 1;
                    uint32_t sid = (uint32_t)(kk & 1) * 2;
                    uint32_t id = make_idesc(BN, true, sid, sid);
                    mma_mxf4(tmem, ad, bd, id, sfa_col + 4 * c, sfb_col + c * (BN / 32), acc);
                }
            }
            tc_commit(&empty[s]);
        }
        tc_commit(acc_full);  // also the drain point of everything issued
        if (!ok) mbar_wait(acc_full, 0);
    } else if (warp >= 2) {
        // ------------------------------------------------ epilogue --------
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const bool ok = mbar_wait(acc_full, 0) && !*abort_flag;
        if (!ok) *abort_flag = 1;
        tc_fence_after();
        if (ok) {
            const int64_t m = m0 + q * 32 + lane;
            float sa = 1.0f;
            if (NV) sa = __fdiv_rn(1.0f, p.a_outer[p.a_outer_count == 1 ? 0 : (m0 >> 7)]);
#pragma unroll 1
            for (int cc = 0; cc < BN / 32; ++cc) {
                uint32_t r[32];
                tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + cc * 32, r);
                const int64_t n = n0 + cc * 32;
                float alpha = 1.0f;
                if (NV) alpha = __fmul_rn(sa, __fdiv_rn(1.0f, p.b_outer[p.b_outer_count == 1 ? 0 : (n >> 7)]));
                if (p.out_dtype == FP4_OUT_F32) {
                    float* dst = reinterpret_cast<float*>(p.c) + m * p.N + n;
#pragma unroll
                    for (int i = 0; i < 32; i += 4) {
                        float4 v = make_float4(__uint_as_float(r[i]) * alpha, __uint_as_float(r[i + 1]) * alpha,
                                               __uint_as_float(r[i + 2]) * alpha, __uint_as_float(r[i + 3]) * alpha);
                        if (p.beta != 0.0f) {
                            float4 o = *reinterpret_cast<const float4*>(dst + i);
                            v.x += p.beta * o.x; v.y += p.beta * o.y; v.z += p.beta * o.z; v.w += p.beta * o.w;
                        }
                        *reinterpret_cast<float4*>(dst + i) = v;
                    }
                } else {
                    uint16_t* dst = reinterpret_cast<uint16_t*>(p.c) + m * p.N + n;
#pragma unroll
                    for (int i = 0; i < 32; i += 8) {
                        uint32_t w[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            float x0 = __uint_as_float(r[i + 2 * j]) * alpha;
                            float x1 = __uint_as_float(r[i + 2 * j + 1]) * alpha;
                            if (p.beta != 0.0f) {
                                x0 += p.beta * bf16_to_f32(dst[i + 2 * j]);
                                x1 += p.beta * bf16_to_f32(dst[i + 2 * j + 1]);
                            }
                            w[j] = (uint32_t)f32_to_bf16_rn(x0) | ((uint32_t)f32_to_bf16_rn(x1) << 16);
                        }
                        *reinterpret_cast<uint4*>(dst + i) = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
    }
}

// ------------------------------------------------------------ host side ---
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool get_encode() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode != nullptr;
}

// K-major FP4 codes [rows][K/2] bytes as a 2D uint8 tensor, box 128 B x box_rows.
bool make_map(CUtensorMap* map, const void* codes, int64_t rows, int64_t K, int box_rows) {
    cuuint64_t dims[2] = {(cuuint64_t)(K / 2), (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(K / 2)};
    cuuint32_t box[2] = {(cuuint32_t)BK_BYTES, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(codes), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <bool NV, int BN>
int launch_t(const GemmParams& g, cudaStream_t stream) {
    using C = Cfg<NV, BN>;
    CUtensorMap ta, tb;
    if (!make_map(&ta, g.a_codes, g.M, g.K, BM) || !make_map(&tb, g.b_codes, g.N, g.K, BN)) return FP4_ERR_CUDA;
    KParams p;
    p.a_scales = g.a_scales;
    p.b_scales = g.b_scales;
    p.a_outer = g.a_outer;
    p.b_outer = g.b_outer;
    p.a_outer_count = g.a_outer_count;
    p.b_outer_count = g.b_outer_count;
    p.M = g.M;
    p.N = g.N;
    p.K = g.K;
    p.c = g.c;
    p.out_dtype = g.out_dtype;
    p.beta = g.beta;
    int dev = 0;
    cudaGetDevice(&dev);
    static bool attr_done[64] = {};
    if (dev < 64 && !attr_done[dev]) {
        if (cudaFuncSetAttribute(fp4_gemm_kernel<NV, BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) !=
            cudaSuccess)
            return FP4_ERR_CUDA;
        attr_done[dev] = true;
    }
    dim3 grid((unsigned)(g.N / BN), (unsigned)(g.M / BM));
    fp4_gemm_kernel<NV, BN><<<grid, THREADS, C::SMEM, stream>>>(ta, tb, p);
    return cudaGetLastError() == cudaSuccess ? FP4_OK : FP4_ERR_CUDA;
}

}  // namespace

int launch_gemm(const GemmParams& g, cudaStream_t stream) {
    if (!get_encode()) return FP4_ERR_CUDA;
    const bool wide = (g.N % 256) == 0;
    if (g.nv) return wide ? launch_t<true, 256>(g, stream) : launch_t<true, 128>(g, stream);
    return wide ? launch_t<false, 256>(g, stream) : launch_t<false, 128>(g, stream);
}

int gemm_status(cudaStream_t stream, int* code, bool reset) {
    unsigned int v = 0;
    if (reset) {
        return cudaMemcpyToSymbolAsync(g_status_gemm, &v, sizeof v, 0, cudaMemcpyHostToDevice, stream) == cudaSuccess
                   ? FP4_OK
                   : FP4_ERR_CUDA;
    }
    if (cudaMemcpyFromSymbolAsync(&v, g_status_gemm, sizeof v, 0, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
        return FP4_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return FP4_ERR_CUDA;
    *code = (int)v;
    return FP4_OK;
}

}  // namespace fp4
