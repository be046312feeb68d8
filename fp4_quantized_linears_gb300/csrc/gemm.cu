// gemm.cu -- block-scaled FP4 GEMM on the 5th-generation tensor cores
// (tcgen05) of sm_103a, with the fused producer epilogues.
//
// Computes C[m][n] = alpha(m, n) * sum_k A_hat[m][k] B_hat[n][k] + beta * C[m][n]
// for the three contractions of "Format-Aware Fusion for Fast FP4
// Pretraining", Sec. 2.3 (Eqs. 4-6).  Every producer emits K-major operands,
// so Fprop, Dgrad and Wgrad are the same "TN" kernel over different views.
// alpha is 1 for MXFP4 and 1 / (S_enc,A[m/128] * S_enc,B[n/128]) for NVFP4,
// the CTA-local epilogue of Sec. 2.2.2 (the factors stay fixed over the whole
// K reduction and are applied together after it).
//
// The same mainloop serves the gated-FFN boundary of Sec. 3.2:
//   EPI_SWIGLU_FWD  B tile = 128 rows of W1 + the matching 128 rows of W3, so
//                   one accumulator holds a1 and a3 of the same outputs; the
//                   epilogue writes the retained BF16 a1, a3 and emits
//                   h = SiLU(a1) * a3 directly as the FP4 row- and
//                   column-facing inputs of the W2 contractions;
//   EPI_SWIGLU_BWD  the W2 Dgrad accumulator dh is combined with the SiLU
//                   derivative (reading the retained a1, a3) and emitted as the
//                   FP4 views of [da1 | da3] for the W1/W3 Dgrad (row view,
//                   stochastic rounding) and Wgrad (column view).
//
// Structure: a persistent kernel, one CTA per SM (384 threads); with an even
// number of 128-row M blocks, CTA pairs (cta_group::2) share one M = 256 MMA
// whose B tile is split between the two CTAs by N halves:
//   warp 0      TMA producer: A tile (128 rows), this CTA's share of the B
//               tile, scale atoms, into a STAGES-deep ring of
//               mbarrier-guarded stages (pair: every load of both CTAs
//               completes on the pair leader's barrier);
//   warp 1      owns the TMEM allocation; one thread issues the block-scaled
//               MMAs (kind::mxf4 E8M0 / kind::mxf4nvf4 E4M3) into a
//               128 x BN FP32 accumulator per CTA; its commits release the
//               stage in both CTAs of a pair;
//   warps 10-11 one thread each copies half of each landed stage's scale
//               atoms into TMEM (tcgen05.cp 32x128b.warpx4) ahead of the MMA
//               thread, which waits for both copies' commits instead of the
//               landing;
//   warps 2-9   epilogue: drain the accumulator from TMEM into registers
//               (each warp one lane quarter x one column half), release it so
//               the next tile's MMAs start, then finish the tile while the
//               tensor core runs the next one: plain outputs go through a
//               swizzled 32-row shared buffer per warp and a TMA
//               tensor store (or TMA reduce-add for beta = 1), so every
//               global write is a bulk transfer of whole 32-byte sectors.
// Every operand load brings data into the issuing CTA's own shared memory;
// no load is multicast across the cluster.
// Every mbarrier wait is bounded: a wait that runs out sets the sticky status
// word to FP4_ERR_TIMEOUT, the roles drain what they issued and the CTA
// returns, releasing its tensor memory.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace fp4 {

__device__ unsigned int g_status_gemm;

namespace {

constexpr int BM = 128;
constexpr int BK = 256;  // FP4 elements per stage: 128-byte rows, 128-byte swizzle
constexpr int BK_BYTES = BK / 2;
constexpr int SMEM_LIMIT = 232448;  // opt-in shared memory per CTA
constexpr int MAX_STAGES = 8;
constexpr int EPI_WARPS = 8;  // epilogue warps (16 for the SwiGLU backward; warps 2 .. 2 + count - 1)
constexpr int SF_WARPS = 2;   // after the epilogue warps: each copies every SF_WARPS-th scale chunk of a stage
constexpr int TMEM_COLS = 512;
constexpr int SF_COL0 = 256;  // first TMEM column of the scale-factor region
constexpr long long WAIT_CYCLES = 4000000000LL;  // default wait bound, ~2 s at 2 GHz
constexpr int64_t L2_RESIDENT_BYTES = 40ll << 20;  // raster: budget for the operand kept in L2

// ------------------------------------------------------------ PTX wrappers -
FP4_DEV uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

FP4_DEV uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
FP4_DEV void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

FP4_DEV void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
FP4_DEV void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
FP4_DEV void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
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
// Bounded wait; false (and the status word set) when `limit` cycles pass.
FP4_DEV bool mbar_wait(uint64_t* bar, uint32_t parity, long long limit) {
    if (mbar_try_wait(bar, parity)) return true;
    long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > limit) {
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

// ---- CTA pair (cta_group::2) ----
// shared::cluster address of the same shared variable in CTA `rank` of the cluster
FP4_DEV uint32_t mapa_rank(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
// Tensor load into this CTA's shared memory whose completion is counted on
// an mbarrier of either CTA of the pair (here: the pair leader's).
FP4_DEV void tma_load_2d_pair(void* dst, const CUtensorMap* map, int x, int y, uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
        "%3}], [%4];" ::"r"(smem_u32(dst)),
        "l"((uint64_t)map), "r"(x), "r"(y), "r"(bar_cluster)
        : "memory");
}
// Arrive on a barrier of another CTA of the cluster.  CTA-scope release: the
// arrive publishes no data, only that this thread's prior tcgen05 work
// (ordered by tcgen05.fence::before_thread_sync) is done; a cluster-scope
// release made the arrive wait for the thread's earlier memory traffic.
FP4_DEV void mbar_arrive_cluster(uint32_t bar_cluster) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}

// TMA tensor store / reduce-add of a shared-memory box (bulk-group completion).
FP4_DEV void tma_store_2d(const CUtensorMap* map, const void* src, int x, int y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"((uint64_t)map),
                 "r"(smem_u32(src)), "r"(x), "r"(y)
                 : "memory");
}
FP4_DEV void tma_reduce_add_2d(const CUtensorMap* map, const void* src, int x, int y) {
    asm volatile("cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     (uint64_t)map),
                 "r"(smem_u32(src)), "r"(x), "r"(y)
                 : "memory");
}
FP4_DEV void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// 16-byte asynchronous global -> shared copy (L2 only) and its completion
FP4_DEV void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
FP4_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
FP4_DEV void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
// at most N committed bulk groups may still be reading their shared source
template <int N>
FP4_DEV void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
FP4_DEV void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
FP4_DEV void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

FP4_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
FP4_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

template <int G = 1>
FP4_DEV void tc_commit(uint64_t* bar) {
    if (G == 2)
        asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                     : "memory");
    else
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                     : "memory");
}
// tcgen05.commit of the pair leader: the arrive reaches the barrier at the
// same offset in both CTAs of the pair (`mask` = 3)
FP4_DEV void tc_commit_pair(uint64_t* bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"(mask)
        : "memory");
}

// shared-memory matrix descriptor (tcgen05): start, LBO, SBO (bytes >> 4),
// version 1 at bit 46, layout type at bits 61..63.
FP4_DEV uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t layout) {
    return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | ((uint64_t)layout << 61);
}
constexpr uint32_t LAYOUT_SW128 = 2;
constexpr uint32_t LAYOUT_SW64 = 4;
// operand tiles: K-major rows of BK_BYTES, swizzled across 8-row groups
constexpr uint32_t AB_LAYOUT = BK_BYTES == 128 ? LAYOUT_SW128 : LAYOUT_SW64;
constexpr uint32_t AB_SBO = 8 * BK_BYTES;
constexpr uint32_t LAYOUT_NONE = 0;

// Instruction descriptor of the block-scaled kinds: E2M1 A and B (format 1),
// both K-major, N >> 3 at bit 17, scale type at bit 23 (1 = UE8M0,
// 0 = UE4M3), M >> 4 at bit 24, scale-factor byte ids at bits 29 (A) / 4 (B).
FP4_DEV uint32_t make_idesc(int n, bool ue8m0, uint32_t sfa_id, uint32_t sfb_id, int m = BM) {
    return (sfb_id << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((ue8m0 ? 1u : 0u) << 23) |
           ((uint32_t)(m >> 4) << 24) | (sfa_id << 29);
}

// G = 2: one MMA over the CTA pair (M = 256: A rows from each CTA's shared
// memory, B split by N halves across the two, D into each CTA's TMEM).
template <int G = 1>
FP4_DEV void mma_mxf4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t sfa, uint32_t sfb,
                      uint32_t accumulate) {
    if (G == 2)
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.u32 p, %6, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
                d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.u32 p, %6, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
                d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
            : "memory");
}
template <int G = 1>
FP4_DEV void mma_nvf4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t sfa, uint32_t sfb,
                      uint32_t accumulate) {
    if (G == 2)
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.u32 p, %6, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], "
            "p;\n\t}" ::"r"(d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.u32 p, %6, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], "
            "p;\n\t}" ::"r"(d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
            : "memory");
}
// one 512-byte scale atom into TMEM, replicated into the four lane quarters
// (G = 2: in each CTA of the pair, from its own shared memory)
template <int G = 1>
FP4_DEV void tc_cp_sf(uint32_t taddr, uint64_t sdesc) {
    if (G == 2)
        asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
    else
        asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
// 32 lanes x 64 / 128 columns of 32-bit accumulator in one load; the wait
// is part of the same asm statement, so no use of the registers can be
// scheduled before it, and one wait covers the whole drain.
FP4_DEV void tmem_ld64(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 {"
        "%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, "
        "%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, "
        "%48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63"
        "}, [%64];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
          "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
          "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
          "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
          "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
        : "r"(taddr)
        : "memory");
}
FP4_DEV void tmem_ld32(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {"
        "%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31"
        "}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}
// Two 32-column loads (at ta and tb) under one wait.
FP4_DEV void tmem_ld32x2(uint32_t ta, uint32_t tb, uint32_t* a, uint32_t* b) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {"
        "%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31"
        "}, [%64];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {"
        "%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, "
        "%48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63"
        "}, [%65];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]), "=r"(a[7]),
          "=r"(a[8]), "=r"(a[9]), "=r"(a[10]), "=r"(a[11]), "=r"(a[12]), "=r"(a[13]), "=r"(a[14]), "=r"(a[15]),
          "=r"(a[16]), "=r"(a[17]), "=r"(a[18]), "=r"(a[19]), "=r"(a[20]), "=r"(a[21]), "=r"(a[22]), "=r"(a[23]),
          "=r"(a[24]), "=r"(a[25]), "=r"(a[26]), "=r"(a[27]), "=r"(a[28]), "=r"(a[29]), "=r"(a[30]), "=r"(a[31]),
          "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3]), "=r"(b[4]), "=r"(b[5]), "=r"(b[6]), "=r"(b[7]),
          "=r"(b[8]), "=r"(b[9]), "=r"(b[10]), "=r"(b[11]), "=r"(b[12]), "=r"(b[13]), "=r"(b[14]), "=r"(b[15]),
          "=r"(b[16]), "=r"(b[17]), "=r"(b[18]), "=r"(b[19]), "=r"(b[20]), "=r"(b[21]), "=r"(b[22]), "=r"(b[23]),
          "=r"(b[24]), "=r"(b[25]), "=r"(b[26]), "=r"(b[27]), "=r"(b[28]), "=r"(b[29]), "=r"(b[30]), "=r"(b[31])
        : "r"(ta), "r"(tb)
        : "memory");
}
FP4_DEV void tmem_ld128(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x128.b32 {"
        "%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, "
        "%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, "
        "%48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, "
        "%64, %65, %66, %67, %68, %69, %70, %71, %72, %73, %74, %75, %76, %77, %78, %79, "
        "%80, %81, %82, %83, %84, %85, %86, %87, %88, %89, %90, %91, %92, %93, %94, %95, "
        "%96, %97, %98, %99, %100, %101, %102, %103, %104, %105, %106, %107, %108, %109, %110, %111, "
        "%112, %113, %114, %115, %116, %117, %118, %119, %120, %121, %122, %123, %124, %125, %126, %127"
        "}, [%128];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
          "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
          "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
          "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
          "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]),
          "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]),
          "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]),
          "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]),
          "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]),
          "=r"(r[96]), "=r"(r[97]), "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]),
          "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]), "=r"(r[110]), "=r"(r[111]),
          "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]), "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]),
          "=r"(r[120]), "=r"(r[121]), "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127])
        : "r"(taddr)
        : "memory");
}


// ------------------------------------------------------ epilogue helpers --
// Bring `bytes` (a multiple of 16, 16-byte aligned) of global memory into L2.
FP4_DEV void bulk_prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

FP4_DEV int atom_off(int r, int j) { return (j >> 2) * 512 + (r & 31) * 16 + (r >> 5) * 4 + (j & 3); }


// Largest |bf16| of n words, as fp32 bits, reduced over the warp.
template <int N>
FP4_DEV uint32_t warp_amax_words(const uint32_t* w) {
    uint32_t m2 = 0;
#pragma unroll
    for (int i = 0; i < N; i += 2) m2 = __vimax3_u16x2(m2, w[i] & 0x7FFF7FFFu, w[i + 1] & 0x7FFF7FFFu);
    uint32_t m = max(m2 << 16, m2 & 0xFFFF0000u);
#pragma unroll
    for (int o = 16; o; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    return m;
}

// fp32 bit pattern of the larger magnitude in a word of two bf16 maxima
FP4_DEV uint32_t lanes_max_f32bits(uint32_t m2) { return max(m2 << 16, m2 & 0xFFFF0000u); }

// MX block of the 32 bf16 values of 16 words (logical indices 8*g0 ..), with
// stochastic rounding: scale byte and 16 bytes of codes.  The block maximum
// is taken on the bf16 magnitudes (their unsigned order is the numeric one;
// a NaN still ends at or above the infinity pattern).
FP4_DEV uint32_t mx_words_sr(const uint32_t* w, uint64_t g0, const uint32_t* rk, uint64_t offset, uint4& packed) {
    uint32_t m2 = 0;
#pragma unroll
    for (int i = 0; i < 16; i += 2) m2 = __vimax3_u16x2(m2, w[i] & 0x7FFF7FFFu, w[i + 1] & 0x7FFF7FFFu);
    const uint32_t am = lanes_max_f32bits(m2);
    if (am >= 0x7F800000u) set_status(&g_status_gemm, FP4_ERR_NONFINITE);
    const int e = e8m0_exponent_up(am);
    const float mult = exp2_neg(e);
    uint32_t out[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) out[q] = e2m1x8_sr_bf16<false>(w + 4 * q, mult, sr_bits8(g0 + q, rk, offset));
    packed = make_uint4(out[0], out[1], out[2], out[3]);
    return (uint32_t)(e + 127);
}

// MX block of the 32 bf16 values of 16 words, round to nearest: scale byte
// and 16 bytes of codes.
FP4_DEV uint32_t mx_words_rn(const uint32_t* w, uint4& packed) {
    uint32_t m2 = 0;
#pragma unroll
    for (int i = 0; i < 16; i += 2) m2 = __vimax3_u16x2(m2, w[i] & 0x7FFF7FFFu, w[i + 1] & 0x7FFF7FFFu);
    const uint32_t am = lanes_max_f32bits(m2);
    if (am >= 0x7F800000u) set_status(&g_status_gemm, FP4_ERR_NONFINITE);
    const int e = e8m0_exponent_up(am);
    const float mult = exp2_neg(e);
    uint32_t out[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        float s8[8];
#pragma unroll
        for (int b = 0; b < 4; ++b)
            f32x2_mul(s8[2 * b], s8[2 * b + 1], bf16_lo(w[4 * q + b]), bf16_hi(w[4 * q + b]), mult, mult);
        out[q] = e2m1x8_rn(s8[0], s8[1], s8[2], s8[3], s8[4], s8[5], s8[6], s8[7]);
    }
    packed = make_uint4(out[0], out[1], out[2], out[3]);
    return (uint32_t)(e + 127);
}


// Two binary32 values rounded to nearest-even bf16 and packed (lo in the low
// half), one conversion instruction; the same rounding as f32_to_bf16_rn.
FP4_DEV uint32_t bf16x2_rn(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

FP4_DEV void store_bf16x32(uint16_t* dst, const float* v) {
#pragma unroll
    for (int i = 0; i < 32; i += 8) {
        uint32_t w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            w[j] = (uint32_t)f32_to_bf16_rn(v[i + 2 * j]) | ((uint32_t)f32_to_bf16_rn(v[i + 2 * j + 1]) << 16);
        *reinterpret_cast<uint4*>(dst + i) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// ----------------------------------------------------------------- kernel -
// EPI_STORE_RMS: the plain store (bf16) that also writes the adjacent
// RMSNorm backward's row terms (a separate instantiation, so that the plain
// store's register allocation is untouched)
enum { EPI_STORE = 0, EPI_SWIGLU_FWD = 1, EPI_SWIGLU_BWD = 2, EPI_QKV_ROPE = 3, EPI_STORE_RMS = 4 };
__host__ __device__ constexpr bool is_store(int epi) { return epi == EPI_STORE || epi == EPI_STORE_RMS; }
// The SwiGLU epilogues (the gate or its derivative, the row views, the
// transposed column views per tile) are latency-bound: they run on 16 warps,
// each thread holding one row x 32 columns; the others on 8 (one row x 64 or
// 128 columns).
__host__ __device__ constexpr int epi_warps(int epi) {
    return epi == EPI_SWIGLU_BWD || epi == EPI_SWIGLU_FWD ? 16 : EPI_WARPS;
}
__host__ __device__ constexpr int kthreads(int epi) { return 32 * (2 + epi_warps(epi) + SF_WARPS); }

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
    // fused SwiGLU
    int64_t f;             // inner width (W1/W3 rows); B rows of W3 start at f
    uint16_t* a1;          // bf16 [M][f]: written (fwd) / read (bwd)
    uint16_t* a3;
    uint16_t* tap0;        // fwd: h;  bwd: dh            (bf16 [M][f], optional)
    uint16_t* tap1;        // bwd: [da1 | da3]            (bf16 [M][2f], optional)
    int quantize;          // emit the MX views below
    uint8_t* q_row_codes;  // fwd: Q_r(h) [M][f];   bwd: Q_r(da13) [M][2f]
    uint8_t* q_row_scales;
    uint8_t* q_col_codes;  // fwd: Q_c(h) [f][M];   bwd: Q_c(da13) [2f][M]
    uint8_t* q_col_scales;
    uint64_t seed, offset;
    uint32_t sr_keys[SR_ROUND_KEYS];  // Philox round keys of `seed`
    // QKV producer with RoPE: head-major bf16 outputs [heads][M][128]
    uint16_t* q_out;
    uint16_t* k_out;
    uint16_t* v_out;
    const float* rope_cos;  // [seq_len][64]
    const float* rope_sin;
    int64_t seq_len;
    int heads_q, heads_kv;
    // plain bf16 store: the adjacent RMSNorm backward's row terms
    const uint16_t* rms_rp;
    const uint16_t* rms_g;
    const float* rms_rstd;
    float* rms_part;
    long long wait_cycles;   // bound of every mbarrier wait
    int skip_first_release;  // test hook: the epilogue's first accumulator release is skipped
    // raster: bands of `band` units along M (n_inner = 0: M fastest inside a
    // band, the band's A tiles reused from L2 while B streams) or along N
    // (n_inner = 1: N fastest, the band's B tiles reused while A streams)
    int n_inner;
    int64_t band;
    uint32_t* amax_ws;  // SwiGLU taps for an NVFP4 encode: maxima slots, or NULL
};

constexpr int cmin(int a, int b) { return a < b ? a : b; }

// The ring is as deep as shared memory and the TMEM scale-factor region
// allow (up to MAX_STAGES): the operand loads of the next stages are what
// hides the L2/HBM latency.  (Halving BK to deepen the ring measured slower:
// 64-byte rows cost more than the extra depth gains.)
// P2: the CTA-pair kernel, where each CTA's stage holds its own 128 rows of
// A, its N-half of the B tile and the scale atoms of the whole B tile.
template <bool NV, int BN, int EPI, bool P2 = false>
struct Cfg {
    static constexpr int SF_CHUNKS = NV ? BK / 64 : BK / 128;  // 512-byte atoms per 128 rows per stage
    static constexpr int A_BYTES = BM * BK_BYTES;
    static constexpr int B_BYTES = (P2 ? BN / 2 : BN) * BK_BYTES;
    static constexpr int SFA_BYTES = SF_CHUNKS * 512;
    static constexpr int SFB_BYTES = (BN / 128) * SF_CHUNKS * 512;
    static constexpr int TX_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;  // bytes landing per stage
    static constexpr int STAGE_BYTES = (TX_BYTES + 1023) / 1024 * 1024;           // ring slot, 1 KiB aligned
    static constexpr int SF_COLS_A = SF_CHUNKS * 4;
    static constexpr int SF_COLS_B = SF_CHUNKS * (BN / 32);
    static constexpr int SF_COLS = SF_COLS_A + SF_COLS_B;
    static constexpr int RESERVED = 256;  // barriers (the dynamic shared base is 1 KiB aligned; checked)
    static constexpr int fit(int staging) {
        return cmin(MAX_STAGES, cmin((SMEM_LIMIT - RESERVED - staging) / STAGE_BYTES, (TMEM_COLS - SF_COL0) / SF_COLS));
    }
    // STORE: each epilogue warp stages its rows in one buffer of 32 rows x
    // 32 bytes (one sector per row) and writes it with a TMA store.  Of the
    // box widths (16 to 128 bytes per row, one or two buffers) this is the
    // fastest: the operand loads share the SM's TMA unit with these stores,
    // and short stores hold it up least, while 16-byte rows write half
    // sectors; pacing the stores over the tile gains nothing.
    static constexpr int OUT_ROW = 32;  // bytes per box row
    static constexpr int OUT_BOX = 32 * OUT_ROW;
    static constexpr int OUT_BUFS = is_store(EPI) ? 1 : 0;
    // SwiGLU backward on CTA pairs: each epilogue thread's retained a1 / a3
    // row segments (2 x 64 bytes) of the next tile land in a slot of its own
    static constexpr bool BWD_PREFETCH = EPI == EPI_SWIGLU_BWD && P2;
    static constexpr int PREFETCH_BYTES = BWD_PREFETCH ? epi_warps(EPI) * 32 * 128 : 0;
    // SwiGLU forward: one 2 KB box (32 rows x 64 bytes) per epilogue warp,
    // and the row and column scale atoms of two tiles
    static constexpr int FWD_BOX = 32 * 64;
    // SwiGLU backward: one 2 KB box per epilogue warp for its column views,
    // the four scale atoms (row da1, row da3, column da1, column da3) of two
    // tiles, and the a1 / a3 prefetch slots
    static constexpr int STAGING =
        is_store(EPI)          ? EPI_WARPS * OUT_BUFS * OUT_BOX
        : EPI == EPI_QKV_ROPE  ? EPI_WARPS * 1024
        : EPI == EPI_SWIGLU_FWD ? epi_warps(EPI) * FWD_BOX + 4 * 512
                               : epi_warps(EPI) * FWD_BOX + 2 * 4 * 512 + PREFETCH_BYTES;
    static constexpr int STAGES = fit(STAGING);
    static constexpr int SMEM = STAGES * STAGE_BYTES + STAGING + RESERVED;
    static_assert(STAGES >= 3, "pipeline depth");
    static_assert(SF_COL0 + STAGES * SF_COLS <= TMEM_COLS, "TMEM budget");
    static_assert(SMEM <= SMEM_LIMIT, "shared memory budget");
    static_assert(3 * MAX_STAGES * 8 + 64 <= 256, "barrier area");
};

template <bool NV, int BN, int EPI, int CM, bool P2 = false>
__global__ void __launch_bounds__(kthreads(EPI), 1)
    fp4_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmSA,
                    const __grid_constant__ CUtensorMap tmSB, const __grid_constant__ CUtensorMap tmX,
                    const __grid_constant__ CUtensorMap tmY, const __grid_constant__ KParams p) {
    using C = Cfg<NV, BN, EPI, P2>;
    static_assert(P2 ? CM == 2 : CM == 1, "clusters are CTA pairs");
    static_assert(!P2 || BN == 256 || EPI == EPI_STORE || EPI == EPI_SWIGLU_BWD, "pair tile widths");
    constexpr int G = P2 ? 2 : 1;       // tcgen05 CTA group
    constexpr int MMA_M = P2 ? 2 * BM : BM;
    constexpr int STAGES = C::STAGES;
    constexpr int EW = epi_warps(EPI);  // epilogue warps
    constexpr int SF_WARP = 2 + EW;     // the first of the warps that move scale factors into TMEM
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // The ring's 128-byte-swizzled stages need 1 KiB alignment, and the
    // budget leaves no slack to realign: a kernel whose dynamic shared base
    // is not aligned reports an error before touching anything (uniform
    // across the grid, so no CTA is left waiting at a cluster barrier).
    if ((reinterpret_cast<uintptr_t>(smem_raw) & 1023) != 0) {
        if (threadIdx.x == 0) set_status(&g_status_gemm, FP4_ERR_CUDA);
        return;
    }
    uint8_t* smem = smem_raw;
    uint8_t* staging = smem + STAGES * C::STAGE_BYTES;
    uint64_t* full = reinterpret_cast<uint64_t*>(staging + C::STAGING);
    uint64_t* empty = full + STAGES;
    uint64_t* sf_full = empty + STAGES;   // the stage's scale factors are in TMEM
    uint64_t* acc_full = sf_full + STAGES;
    uint64_t* acc_empty = acc_full + 1;
    uint64_t* drain_bar = acc_empty + 1;  // MMA completion point at the end
    uint64_t* epi_bar = drain_bar + 1;    // bounded barrier among the epilogue warps
    uint64_t* sf_drain = epi_bar + 1;     // completion point of the last scale-factor copies
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sf_drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = CM > 1 ? cluster_rank() : 0;
    const long long lim = p.wait_cycles;
    const int num_kb = (int)(p.K / BK);
    const int64_t m_units = p.M / (BM * CM);
    const int64_t n_blocks = EPI == EPI_SWIGLU_FWD ? p.f / 128 : p.N / BN;
    const int64_t n_units = m_units * n_blocks;
    const int64_t cluster_id = blockIdx.x / CM, n_clusters = gridDim.x / CM;

    auto unit_coords = [&](int64_t u, int64_t& m0, int64_t& n0) {
        int64_t mu, nb;
        if (p.n_inner) {
            const int64_t per_group = p.band * m_units;
            const int64_t g = u / per_group, within = u % per_group;
            const int64_t n_first = g * p.band;
            const int64_t gs = min(p.band, n_blocks - n_first);
            nb = n_first + within % gs;
            mu = within / gs;
        } else {
            const int64_t per_group = p.band * n_blocks;
            const int64_t g = u / per_group, within = u % per_group;
            const int64_t m_first = g * p.band;
            const int64_t gs = min(p.band, m_units - m_first);
            mu = m_first + within % gs;
            nb = within / gs;
        }
        m0 = (mu * CM + rank) * BM;
        n0 = nb * (EPI == EPI_SWIGLU_FWD ? 128 : BN);
    };
    // global row of B where 128-row half h of the tile starts
    auto b_row = [&](int64_t n0, int h) -> int64_t {
        return EPI == EPI_SWIGLU_FWD ? h * p.f + n0 : n0 + 128 * h;
    };

    auto stage_a = [&](int s) { return smem + s * C::STAGE_BYTES; };
    auto stage_b = [&](int s) { return smem + s * C::STAGE_BYTES + C::A_BYTES; };
    auto stage_sfa = [&](int s) { return smem + s * C::STAGE_BYTES + C::A_BYTES + C::B_BYTES; };
    auto stage_sfb = [&](int s) { return smem + s * C::STAGE_BYTES + C::A_BYTES + C::B_BYTES + C::SFA_BYTES; };

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);  // pair: the leader's commit reaches each CTA once
            mbar_init(&sf_full[s], SF_WARPS);
        }
        mbar_init(sf_drain, SF_WARPS);
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, P2 ? 2 * EW : EW);  // pair: both CTAs' epilogues, on the leader
        mbar_init(drain_bar, 1);
        mbar_init(epi_bar, EW);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        if (P2) {
            // both CTAs of the pair allocate the same columns together
            asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                             smem_u32(tmem_slot)),
                         "r"(TMEM_COLS)
                         : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
        } else {
            asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                             smem_u32(tmem_slot)),
                         "r"(TMEM_COLS)
                         : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        }
    }
    if (warp == 0 && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmA) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmB) : "memory");
        if (P2) {
            asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmSA) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmSB) : "memory");
        }
    }
    tc_fence_before();
    __syncthreads();
    if (CM > 1) cluster_sync();  // the peer's barriers are initialised before any remote arrive
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------ TMA producer ----
        const int64_t k_atoms = NV ? p.K / 64 : p.K / 128;  // scale atoms per 128-row block
        int stage = 0;
        uint32_t phase = 0;
        int64_t issued = 0;
        bool ok = true;
        for (int64_t u = cluster_id; u < n_units && ok; u += n_clusters) {
            int64_t m0, n0;
            unit_coords(u, m0, n0);
            for (int kb = 0; kb < num_kb; ++kb) {
                if (*abort_flag || !mbar_wait(&empty[stage], phase ^ 1, lim)) {
                    *abort_flag = 1;
                    ok = false;
                    break;
                }
                if (P2) {
                    // this CTA's A rows, its N-half of B, its A scales and the
                    // whole B tile's scales; completion counted on the leader
                    const uint32_t fb = mapa_rank(smem_u32(&full[stage]), 0);
                    if (rank == 0) mbar_expect_tx(&full[stage], 2 * C::TX_BYTES);
                    tma_load_2d_pair(stage_a(stage), &tmA, kb * BK_BYTES, (int)m0, fb);
                    // B rows of this CTA's N-half: 128 rows of W1 / W3 (SwiGLU
                    // forward), else rows [n0 + rank * BN/2, + BN/2)
                    const int64_t brow = EPI == EPI_SWIGLU_FWD ? b_row(n0, (int)rank) : n0 + (int64_t)rank * (BN / 2);
                    tma_load_2d_pair(stage_b(stage), &tmB, kb * BK_BYTES, (int)brow, fb);
                    tma_load_2d_pair(stage_sfa(stage), &tmSA, 0, (int)((m0 >> 7) * k_atoms + kb * C::SF_CHUNKS), fb);
#pragma unroll
                    for (int h = 0; h < BN / 128; ++h)
                        tma_load_2d_pair(stage_sfb(stage) + h * C::SF_CHUNKS * 512, &tmSB, 0,
                                         (int)((b_row(n0, h) >> 7) * k_atoms + kb * C::SF_CHUNKS), fb);
                    ++issued;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                    continue;
                }
                mbar_expect_tx(&full[stage], C::TX_BYTES);
                tma_load_2d(stage_a(stage), &tmA, kb * BK_BYTES, (int)m0, &full[stage]);
                for (int h = 0; h < BN / 128; ++h)
                    tma_load_2d(stage_b(stage) + h * 128 * BK_BYTES, &tmB, kb * BK_BYTES, (int)b_row(n0, h),
                                &full[stage]);
                const uint8_t* sfa = p.a_scales + ((m0 >> 7) * k_atoms + (int64_t)kb * C::SF_CHUNKS) * 512;
                bulk_load(stage_sfa(stage), sfa, C::SFA_BYTES, &full[stage]);
#pragma unroll
                for (int h = 0; h < BN / 128; ++h) {
                    const uint8_t* sfb =
                        p.b_scales + ((b_row(n0, h) >> 7) * k_atoms + (int64_t)kb * C::SF_CHUNKS) * 512;
                    bulk_load(stage_sfb(stage) + h * C::SF_CHUNKS * 512, sfb, C::SF_CHUNKS * 512, &full[stage]);
                }
                ++issued;
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1;
                }
            }
        }
        if ((!ok || *abort_flag) && (!P2 || rank == 0)) {
            // drain: wait (bounded) for the loads of the stages still in flight
            // when this or another role gave up (pair: the leader's barriers
            // count the loads of both CTAs)
            int s = stage;
            uint32_t ph = phase;
            for (int i = 0; i < STAGES && i < issued; ++i) {
                if (--s < 0) {
                    s = STAGES - 1;
                    ph ^= 1;
                }
                mbar_wait(&full[s], ph, lim);
            }
        }
    } else if (warp == 1 && lane == 0 && (!P2 || rank == 0)) {
        // ------------------------------------------------ MMA issuer ------
        // (pair: the leader issues for both CTAs)
        const uint32_t sf_base = tmem + SF_COL0;
        int stage = 0;
        uint32_t phase = 0, acc_phase = 0;
        bool ok = true;
        for (int64_t u = cluster_id; u < n_units && ok; u += n_clusters) {
            if (*abort_flag || !mbar_wait(acc_empty, acc_phase ^ 1, lim)) {
                *abort_flag = 1;
                ok = false;
                break;
            }
            tc_fence_after();
            for (int kb = 0; kb < num_kb; ++kb) {
                // the stage has landed and its scale factors are in TMEM
                if (*abort_flag || !mbar_wait(&sf_full[stage], phase, lim)) {
                    *abort_flag = 1;
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sfa_col = sf_base + stage * C::SF_COLS;
                const uint32_t sfb_col = sfa_col + C::SF_COLS_A;
                const uint32_t a_base = smem_u32(stage_a(stage)), b_base = smem_u32(stage_b(stage));
                constexpr int MMAS_PER_CHUNK = (BK / 64) / C::SF_CHUNKS;
#pragma unroll
                for (int c = 0; c < C::SF_CHUNKS; ++c) {
#pragma unroll
                    for (int q = 0; q < MMAS_PER_CHUNK; ++q) {
                        const int kk = c * MMAS_PER_CHUNK + q;
                        // each MMA's 64 FP4 values start 32 bytes further into the rows
                        const uint64_t ad = smem_desc(a_base + kk * 32, 16, AB_SBO, AB_LAYOUT);
                        const uint64_t bd = smem_desc(b_base + kk * 32, 16, AB_SBO, AB_LAYOUT);
                        const uint32_t acc = (kb > 0 || kk > 0) ? 1u : 0u;
                        if (NV) {
                            mma_nvf4<G>(tmem, ad, bd, make_idesc(BN, false, 0, 0, MMA_M), sfa_col + 4 * kk,
                                        sfb_col + kk * (BN / 32), acc);
                        } else {
                            const uint32_t sid = (uint32_t)(kk & 1) * 2;
                            mma_mxf4<G>(tmem, ad, bd, make_idesc(BN, true, sid, sid, MMA_M), sfa_col + 4 * c,
                                        sfb_col + c * (BN / 32), acc);
                        }
                    }
                }
                if (P2)
                    tc_commit_pair(&empty[stage], (uint16_t)3);
                else
                    tc_commit(&empty[stage]);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            if (!ok) break;
            if (P2)
                tc_commit_pair(acc_full, (uint16_t)3);
            else
                tc_commit(acc_full);
            acc_phase ^= 1;
        }
        // drain point of everything issued (its own barrier, so that no
        // epilogue wait on acc_full can see an extra phase)
        tc_commit<G>(drain_bar);
        mbar_wait(drain_bar, 0, lim);
    } else if (warp >= SF_WARP && lane == 0 && (!P2 || rank == 0)) {
        // ------------------------------------------------ scale factors ---
        // Each landed stage's scale atoms go to that stage's TMEM columns
        // (replicated into the four lane quarters), issued from this thread
        // so that the copies run beside the MMAs of earlier stages rather
        // than in the MMA thread's in-order stream; the commit on sf_full
        // tells the MMA thread they are complete.  Region `stage` is free
        // again once the stage lands anew: the producer refills it only after
        // the MMAs that read the previous copies have completed.
        // (pair: the leader copies for both CTAs, each from its own stage)
        // Two such threads, in two warps, share each stage's chunks: one
        // thread's copies (12 per stage for NVFP4) took about as long as the
        // stage's MMAs.  Both commit to sf_full (arrival count SF_WARPS).
        const int sfi = warp - SF_WARP;
        const uint32_t sf_base = tmem + SF_COL0;
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int64_t u = cluster_id; u < n_units && ok; u += n_clusters) {
            for (int kb = 0; kb < num_kb; ++kb) {
                if (*abort_flag || !mbar_wait(&full[stage], phase, lim)) {
                    *abort_flag = 1;
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sfa_col = sf_base + stage * C::SF_COLS;
                const uint32_t sfb_col = sfa_col + C::SF_COLS_A;
#pragma unroll
                for (int c = sfi; c < C::SF_CHUNKS; c += SF_WARPS) {
                    tc_cp_sf<G>(sfa_col + 4 * c,
                                smem_desc(smem_u32(stage_sfa(stage) + c * 512), 0, 128, LAYOUT_NONE));
#pragma unroll
                    for (int h = 0; h < BN / 128; ++h)
                        tc_cp_sf<G>(sfb_col + c * (BN / 32) + 4 * h,
                                    smem_desc(smem_u32(stage_sfb(stage) + (h * C::SF_CHUNKS + c) * 512), 0, 128,
                                              LAYOUT_NONE));
                }
                tc_commit<G>(&sf_full[stage]);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1;
                }
            }
        }
        // every copy issued has completed before TMEM can be released
        tc_commit<G>(sf_drain);
        mbar_wait(sf_drain, 0, lim);
    } else if (warp >= 2 && warp < 2 + EW) {
        // ------------------------------------------------ epilogue --------
        const int q = warp & 3;               // TMEM lane quarter this warp may access
        const int half = (warp - 2) >> 2;     // column half (SwiGLU backward: column quarter)
        const int lr = q * 32 + lane;         // row within the tile
        const int et = (warp - 2) * 32 + lane;  // epilogue thread index 0 .. 32 * EW - 1
        uint32_t acc_phase = 0, epi_phase = 0;
        bool epi_ok = true;
        bool skip_release = p.skip_first_release != 0;  // test hook, first tile only
        uint32_t tensor_amax = 0;  // SwiGLU taps: this warp's running maximum (fp32 bits)
        // the accumulator is free once every epilogue warp has read it; in
        // pair mode the MMA thread waits on the leader's barrier for the
        // warps of both CTAs
        auto release_acc = [&]() {
            if (skip_release) {
                skip_release = false;
                return;
            }
            if (lane == 0) {
                if (P2 && rank != 0)
                    mbar_arrive_cluster(mapa_rank(smem_u32(acc_empty), 0));
                else
                    mbar_arrive(acc_empty);
            }
        };
        // bounded barrier among the epilogue warps: one arrive per warp after
        // the warp's own lanes have synchronised
        auto epi_sync = [&]() {
            __syncwarp();
            if (lane == 0) mbar_arrive(epi_bar);
            if (!mbar_wait(epi_bar, epi_phase, lim)) {
                *abort_flag = 1;
                epi_ok = false;
            }
            epi_phase ^= 1;
        };
        // SwiGLU backward (pairs): this thread's a1 / a3 row segments of a
        // tile are copied into shared memory one tile ahead, so that their
        // latency hides behind the previous tile's work.  Chunk-major layout:
        // 16-byte chunk i (a1: 0-3, a3: 4-7) of epilogue thread et sits at
        // (i * 32 * EW + et) * 16, so a warp's accesses to one chunk are 512
        // contiguous bytes (no bank conflicts).
        const uint32_t slot = smem_u32(staging + EW * C::FWD_BOX + 2 * 4 * 512) + (uint32_t)et * 16;
        constexpr uint32_t CHUNK_STRIDE = 32 * EW * 16;
        auto prefetch_a13 = [&](int64_t u2) {
            if constexpr (C::BWD_PREFETCH) {
                if (u2 < n_units) {
                    int64_t m2, n2;
                    unit_coords(u2, m2, n2);
                    const int64_t off = (m2 + lr) * p.f + n2 + 32 * half;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        cp_async16(slot + i * CHUNK_STRIDE, p.a1 + off + 8 * i);
                        cp_async16(slot + (4 + i) * CHUNK_STRIDE, p.a3 + off + 8 * i);
                    }
                }
                cp_async_commit();
            }
        };
        prefetch_a13(cluster_id);
        for (int64_t u = cluster_id; u < n_units && epi_ok; u += n_clusters) {
            int64_t m0, n0;
            unit_coords(u, m0, n0);
            if constexpr (EPI == EPI_SWIGLU_BWD && !C::BWD_PREFETCH) {
                // this thread's retained a1 / a3 (one 64-byte row segment
                // each) do not depend on the accumulator: start moving them
                // into L2 while the tile's MMAs run
                const int64_t off = (m0 + lr) * p.f + n0 + 32 * half;
                bulk_prefetch_l2(p.a1 + off, 64);
                bulk_prefetch_l2(p.a3 + off, 64);
            }
            if (!mbar_wait(acc_full, acc_phase, lim)) {
                *abort_flag = 1;
                break;
            }
            tc_fence_after();
            const int64_t m = m0 + lr;
            const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
            if constexpr (is_store(EPI)) {
                constexpr int NC = BN / 64;  // 32-column chunks per thread
                uint32_t r[NC * 32];
                if constexpr (NC == 4)
                    tmem_ld128(lane_base + half * (BN / 2), r);
                else
                    tmem_ld64(lane_base + half * (BN / 2), r);
                tc_fence_before();
                release_acc();
                float sa = 1.0f;
                if (NV) sa = __fdiv_rn(1.0f, p.a_outer[p.a_outer_count == 1 ? 0 : (m0 >> 7)]);
                // EPI_STORE_RMS (bf16 only): the consumer is a residual-RMSNorm
                // backward, whose row mean needs sum_n fl32(dy * g) *
                // fl32(r' * rstd) over the bf16 values this store writes.  Each
                // thread adds its row's terms box by box, in column order, and
                // writes one binary32 partial per 64-column block (no atomics:
                // the blocks are summed in a fixed order later).
                float rms_acc = 0.0f, rms_rs = 0.0f;
                if constexpr (EPI == EPI_STORE_RMS) rms_rs = p.rms_rstd[m];
                const bool tma_out = p.beta == 0.0f || p.beta == 1.0f;
                if (tma_out) {
                    // rows [32q, 32q+32) of the tile through this warp's
                    // swizzled 32 x OUT_ROW-byte buffers and TMA stores
                    constexpr int ROW = C::OUT_ROW, WORDS = ROW / 4;  // 32-bit words per box row
                    uint8_t* wbuf = staging + (warp - 2) * C::OUT_BUFS * C::OUT_BOX;
                    const bool f32 = p.out_dtype == FP4_OUT_F32;
                    constexpr int NB = (BN / 2) / WORDS;  // boxes per thread (fp32; bf16 needs half)
                    const int nbox = f32 ? NB : NB / 2;
#pragma unroll
                    for (int bi = 0; bi < NB; ++bi) {
                        if (bi >= nbox) break;
                        uint8_t* buf = wbuf;
                        // the store previously issued from this buffer must have read it
                        if (lane == 0) bulk_wait_read<0>();
                        __syncwarp();
                        const int cols = f32 ? WORDS : 2 * WORDS;
                        const int64_t n = n0 + half * (BN / 2) + cols * bi;
                        float alpha = 1.0f;
                        if (NV) alpha = __fmul_rn(sa, __fdiv_rn(1.0f, p.b_outer[p.b_outer_count == 1 ? 0 : (n >> 7)]));
                        uint32_t w[WORDS];
                        if (f32) {
#pragma unroll
                            for (int i = 0; i < WORDS; ++i)
                                w[i] = __float_as_uint(__uint_as_float(r[WORDS * bi + i]) * alpha);
                        } else {
#pragma unroll
                            for (int i = 0; i < WORDS; ++i)
                                w[i] = (uint32_t)f32_to_bf16_rn(__uint_as_float(r[2 * WORDS * bi + 2 * i]) * alpha) |
                                       ((uint32_t)f32_to_bf16_rn(__uint_as_float(r[2 * WORDS * bi + 2 * i + 1]) * alpha)
                                        << 16);
                            if constexpr (EPI == EPI_STORE_RMS) {
                                const uint16_t* xr = p.rms_rp + m * p.N + n;
                                const uint16_t* gr = p.rms_g + n;
#pragma unroll
                                for (int c8 = 0; c8 < WORDS / 4; ++c8) {  // 8 columns per 16-byte load
                                    const uint4 xv = *reinterpret_cast<const uint4*>(xr + 8 * c8);
                                    const uint4 gv = *reinterpret_cast<const uint4*>(gr + 8 * c8);
                                    const uint32_t xs[4] = {xv.x, xv.y, xv.z, xv.w}, gs[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
                                    for (int k = 0; k < 4; ++k) {
                                        const uint32_t dw = w[4 * c8 + k];
                                        rms_acc = fmaf(__fmul_rn(bf16_lo(dw), bf16_lo(gs[k])),
                                                       __fmul_rn(bf16_lo(xs[k]), rms_rs), rms_acc);
                                        rms_acc = fmaf(__fmul_rn(bf16_hi(dw), bf16_hi(gs[k])),
                                                       __fmul_rn(bf16_hi(xs[k]), rms_rs), rms_acc);
                                    }
                                }
                                if (((bi + 1) * 2 * WORDS) % 64 == 0) {  // a 64-column block is complete
                                    p.rms_part[m * (p.N >> 6) + ((n + 2 * WORDS - 64) >> 6)] = rms_acc;
                                    rms_acc = 0.0f;
                                }
                            }
                        }
                        // this lane's row: 16-byte chunk k lands at k ^ ((row >> 2) & 1)
                        // (32B swizzle: no bank conflicts across the 8 lanes of a phase)
                        static_assert(ROW == 32, "box row width");
#pragma unroll
                        for (int k = 0; k < ROW / 16; ++k) {
                            const int sw = (lane >> 2) & 1;
                            *reinterpret_cast<uint4*>(buf + lane * ROW + ((k ^ sw) << 4)) =
                                make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
                        }
                        fence_proxy_async();
                        __syncwarp();
                        if (lane == 0) {
                            if (p.beta == 0.0f)
                                tma_store_2d(&tmC, buf, (int)n, (int)(m0 + q * 32));
                            else
                                tma_reduce_add_2d(&tmC, buf, (int)n, (int)(m0 + q * 32));
                            bulk_commit();
                        }
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < NC; ++c) {
                        const int64_t n = n0 + half * (BN / 2) + 32 * c;
                        float alpha = 1.0f;
                        if (NV) alpha = __fmul_rn(sa, __fdiv_rn(1.0f, p.b_outer[p.b_outer_count == 1 ? 0 : (n >> 7)]));
                        const uint32_t* rc = r + 32 * c;
                        if (p.out_dtype == FP4_OUT_F32) {
                            float* dst = reinterpret_cast<float*>(p.c) + m * p.N + n;
#pragma unroll
                            for (int i = 0; i < 32; i += 4) {
                                float4 v = make_float4(__uint_as_float(rc[i]) * alpha,
                                                       __uint_as_float(rc[i + 1]) * alpha,
                                                       __uint_as_float(rc[i + 2]) * alpha,
                                                       __uint_as_float(rc[i + 3]) * alpha);
                                const float4 o = *reinterpret_cast<const float4*>(dst + i);
                                v.x += p.beta * o.x;
                                v.y += p.beta * o.y;
                                v.z += p.beta * o.z;
                                v.w += p.beta * o.w;
                                *reinterpret_cast<float4*>(dst + i) = v;
                            }
                        } else {
                            uint16_t* dst = reinterpret_cast<uint16_t*>(p.c) + m * p.N + n;
                            float v[32];
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                v[i] = __uint_as_float(rc[i]) * alpha + p.beta * bf16_to_f32(dst[i]);
                            store_bf16x32(dst, v);
                        }
                    }
                }
            } else if constexpr (EPI == EPI_QKV_ROPE) {
                // this thread's 128 columns are exactly one head of token m:
                // bf16(acc), RoPE on Q and K heads (rotate-half pairs (i, i+64),
                // binary32 products and sums, then bf16), head-major TMA stores
                // (direct 16-byte stores from the lanes were 4-7 % slower)
                uint32_t pk[64];  // bf16x2 of the head's 128 values
                {
                    uint32_t r[128];
                    tmem_ld128(lane_base + 128 * half, r);
                    tc_fence_before();
                    release_acc();
                    float alpha = 1.0f;
                    if (NV)
                        alpha = __fmul_rn(__fdiv_rn(1.0f, p.a_outer[p.a_outer_count == 1 ? 0 : (m0 >> 7)]),
                                          __fdiv_rn(1.0f, p.b_outer[p.b_outer_count == 1 ? 0 : ((n0 >> 7) + half)]));
#pragma unroll
                    for (int i = 0; i < 64; ++i)
                        pk[i] = bf16x2_rn(__uint_as_float(r[2 * i]) * alpha, __uint_as_float(r[2 * i + 1]) * alpha);
                }
                const int head = (int)((n0 >> 7) + half);
                const int hqk = p.heads_q + p.heads_kv;
                if (head < hqk) {
                    // RoPE in place: pair (i, i + 64) of the head is words (j, 32 + j)
                    const int64_t pos = m % p.seq_len;
                    const float4* cp = reinterpret_cast<const float4*>(p.rope_cos + pos * 64);
                    const float4* sp = reinterpret_cast<const float4*>(p.rope_sin + pos * 64);
#pragma unroll
                    for (int g = 0; g < 8; ++g) {  // pairs i = 8g .. 8g+7
                        const float4 c0 = cp[2 * g], c1 = cp[2 * g + 1], s0 = sp[2 * g], s1 = sp[2 * g + 1];
                        const float cv[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
                        const float sv[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const uint32_t wa = pk[4 * g + j], wb = pk[32 + 4 * g + j];
                            float l[2], h[2];
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                const float a = e ? bf16_hi(wa) : bf16_lo(wa);
                                const float b = e ? bf16_hi(wb) : bf16_lo(wb);
                                const float c = cv[2 * j + e], sn = sv[2 * j + e];
                                l[e] = __fsub_rn(__fmul_rn(a, c), __fmul_rn(b, sn));
                                h[e] = __fadd_rn(__fmul_rn(b, c), __fmul_rn(a, sn));
                            }
                            pk[4 * g + j] = bf16x2_rn(l[0], l[1]);
                            pk[32 + 4 * g + j] = bf16x2_rn(h[0], h[1]);
                        }
                    }
                }
                // head-major rows: this warp's 32 tokens of one head are 32
                // consecutive rows of the [heads * M][128] view, stored as eight
                // 32-row x 32-byte boxes through the warp's 1 KB buffer
                const CUtensorMap* map = head < p.heads_q ? &tmC : head < hqk ? &tmX : &tmY;
                const int hl = head < p.heads_q ? head : head < hqk ? head - p.heads_q : head - hqk;
                const int row0 = (int)((int64_t)hl * p.M + m0 + q * 32);
                uint8_t* buf = staging + (warp - 2) * 1024;
#pragma unroll
                for (int b = 0; b < 8; ++b) {
                    if (lane == 0) bulk_wait_read<0>();
                    __syncwarp();
#pragma unroll
                    for (int k = 0; k < 2; ++k)
                        *reinterpret_cast<uint4*>(buf + lane * 32 + ((k ^ ((lane >> 2) & 1)) << 4)) =
                            make_uint4(pk[8 * b + 4 * k], pk[8 * b + 4 * k + 1], pk[8 * b + 4 * k + 2], pk[8 * b + 4 * k + 3]);
                    fence_proxy_async();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(map, buf, 16 * b, row0);
                        bulk_commit();
                    }
                }
            } else if constexpr (EPI == EPI_SWIGLU_FWD) {
                // This thread: row lr, output columns [oc, oc + 32) of the
                // 128-wide tile (a1 in accumulator columns oc .., a3 in
                // 128 + oc ..); this warp: the 32 x 32 block of rows
                // [32q, 32q + 32).  The block's retained a1 and a3 leave
                // through the warp's own 2 KB box (64-byte rows, 64B swizzle)
                // by TMA tensor stores; the box then holds the block's h, read
                // down its columns for the column view (the block is exactly
                // one 32-row block of 32 stored rows of Q_c(h)).
                const int oc = 32 * half;
                const int64_t n = n0 + oc;
                uint32_t p1[16], p3[16];  // bf16x2 of the retained a1, a3
                {
                    uint32_t r1[32], r3[32];
                    tmem_ld32x2(lane_base + oc, lane_base + 128 + oc, r1, r3);
                    tc_fence_before();
                    release_acc();
                    float alpha = 1.0f;
                    if (NV)
                        alpha = __fmul_rn(__fdiv_rn(1.0f, p.a_outer[p.a_outer_count == 1 ? 0 : (m0 >> 7)]),
                                          __fdiv_rn(1.0f, p.b_outer[0]));
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        p1[i] = bf16x2_rn(__uint_as_float(r1[2 * i]) * alpha, __uint_as_float(r1[2 * i + 1]) * alpha);
                        p3[i] = bf16x2_rn(__uint_as_float(r3[2 * i]) * alpha, __uint_as_float(r3[2 * i + 1]) * alpha);
                    }
                }
                uint8_t* box = staging + (warp - 2) * C::FWD_BOX;
                uint8_t* atoms = staging + EW * C::FWD_BOX + (acc_phase & 1) * 1024;  // row, then column atom
                // this lane's row: 16-byte chunk k at k ^ ((row >> 1) & 3) (64B swizzle)
                auto put_row = [&](const uint32_t* w) {
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        *reinterpret_cast<uint4*>(box + lane * 64 + ((k ^ ((lane >> 1) & 3)) << 4)) =
                            make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
                };
                auto box_free = [&]() {  // the previous bulk store from the box has read it
                    if (lane == 0) bulk_wait_read<0>();
                    __syncwarp();
                };
                auto store_box = [&](const CUtensorMap* map) {
                    fence_proxy_async();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(map, box, (int)n, (int)(m0 + q * 32));
                        bulk_commit();
                    }
                };
                box_free();
                put_row(p1);
                store_box(&tmX);
                uint32_t hp[16];  // bf16x2 of h = bf16(fl32(SiLU(a1)) * a3)
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float hv[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const float x1 = e ? bf16_hi(p1[i]) : bf16_lo(p1[i]);
                        const float x3 = e ? bf16_hi(p3[i]) : bf16_lo(p3[i]);
                        const float sl = x1 * __fdividef(1.0f, 1.0f + __expf(-x1));
                        hv[e] = __fmul_rn(sl, x3);
                    }
                    hp[i] = bf16x2_rn(hv[0], hv[1]);
                }
                box_free();
                put_row(p3);
                store_box(&tmY);
                if (p.tap0) {  // the h tap through the box as well (tmC maps it)
                    box_free();
                    put_row(hp);
                    store_box(&tmC);
                }
                if (p.amax_ws) {
                    // the tap's maxima for the NVFP4 encode that follows: the
                    // tile's 128-row strip, its 128-column strip, the tensor
                    const uint32_t mw = warp_amax_words<16>(hp);
                    if (lane == 0) {
                        atomicMax(&p.amax_ws[1 + (m0 >> 7)], mw);
                        atomicMax(&p.amax_ws[1 + (p.M >> 7) + (n0 >> 7)], mw);
                        tensor_amax = max(tensor_amax, mw);
                    }
                }
                if (p.quantize) {
                    uint4 pk;
                    const uint32_t sc = mx_words_rn(hp, pk);
                    *reinterpret_cast<uint4*>(p.q_row_codes + m * (p.f >> 1) + (n >> 1)) = pk;
                    atoms[atom_off(lr, half)] = (uint8_t)sc;
                    // the block's h into the box, then each lane takes one
                    // column (one stored row of Q_c(h)) down the 32 rows
                    box_free();
                    put_row(hp);
                    __syncwarp();
                    uint32_t w[16];
                    {
                        const int k = lane >> 3, b = (lane & 7) * 2;
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const int r0 = 2 * i, r1 = 2 * i + 1;
                            const uint32_t lo = *reinterpret_cast<const uint16_t*>(box + r0 * 64 + ((k ^ ((r0 >> 1) & 3)) << 4) + b);
                            const uint32_t hi = *reinterpret_cast<const uint16_t*>(box + r1 * 64 + ((k ^ ((r1 >> 1) & 3)) << 4) + b);
                            w[i] = lo | (hi << 16);
                        }
                    }
                    uint4 pkc;
                    const uint32_t scc = mx_words_rn(w, pkc);
                    const int c = oc + lane;
                    *reinterpret_cast<uint4*>(p.q_col_codes + (n0 + c) * (p.M >> 1) + ((m0 + 32 * q) >> 1)) = pkc;
                    atoms[512 + atom_off(c, q)] = (uint8_t)scc;
                    // the tile's scale atoms (double-buffered by tile, so one
                    // barrier per tile suffices)
                    epi_sync();
                    if (!epi_ok) break;
                    if (et < 32) {
                        const int64_t a = (m0 >> 7) * (p.f >> 7) + (n0 >> 7);
                        *reinterpret_cast<uint4*>(p.q_row_scales + a * 512 + et * 16) =
                            *reinterpret_cast<const uint4*>(atoms + et * 16);
                    } else if (et < 64) {
                        const int64_t a = (n0 >> 7) * (p.M >> 7) + (m0 >> 7);
                        *reinterpret_cast<uint4*>(p.q_col_scales + a * 512 + (et - 32) * 16) =
                            *reinterpret_cast<const uint4*>(atoms + 512 + (et - 32) * 16);
                    }
                }
            } else {
                // EPI_SWIGLU_BWD: dh for output columns [oc, oc + 32) of this
                // thread's row
                const int oc = 32 * half;
                const int64_t n = n0 + oc;
                uint32_t dp[16];  // bf16x2 of dh
                {
                    uint32_t r[32];
                    tmem_ld32(lane_base + oc, r);
                    tc_fence_before();
                    release_acc();
                    float alpha = 1.0f;
                    if (NV)
                        alpha = __fmul_rn(__fdiv_rn(1.0f, p.a_outer[p.a_outer_count == 1 ? 0 : (m0 >> 7)]),
                                          __fdiv_rn(1.0f, p.b_outer[p.b_outer_count == 1 ? 0 : (n0 >> 7)]));
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        dp[i] = bf16x2_rn(__uint_as_float(r[2 * i]) * alpha, __uint_as_float(r[2 * i + 1]) * alpha);
                }
                uint8_t* box = staging + (warp - 2) * C::FWD_BOX;
                // row da1, row da3, column da1, column da3; double-buffered by tile
                uint8_t* atoms = staging + EW * C::FWD_BOX + (acc_phase & 1) * 2048;
                const int64_t f2 = 2 * p.f;
                // The taps leave through this warp's 2 KB box (its 32 x 32
                // block: 32 rows x 64 bytes, 64B swizzle) by TMA tensor stores
                // (tmY maps dh, tmX [da1 | da3]); direct 16-byte stores from
                // the lanes were ~10 % slower on the NVFP4 route.
                auto tap_store = [&](const uint32_t* w, const CUtensorMap* map, int x) {
                    if (lane == 0) bulk_wait_read<0>();  // the box's previous store has read it
                    __syncwarp();
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        *reinterpret_cast<uint4*>(box + lane * 64 + ((k ^ ((lane >> 1) & 3)) << 4)) =
                            make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
                    fence_proxy_async();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(map, box, x, (int)(m0 + q * 32));
                        bulk_commit();
                    }
                };
                if (p.tap0) tap_store(dp, &tmY, (int)n);
                // da1 = bf16(dh * a3 * SiLU'(a1)), da3 = bf16(dh * SiLU(a1)), as bf16x2 words
                uint32_t q1[16], q3[16];
                {
                    uint4 v1[4], v3[4];
                    if constexpr (C::BWD_PREFETCH) {
                        cp_async_wait_all();  // this thread's own copies of this tile's segments
                        const uint8_t* s13 = staging + EW * C::FWD_BOX + 2 * 4 * 512 + et * 16;
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            v1[i] = *reinterpret_cast<const uint4*>(s13 + i * CHUNK_STRIDE);
                            v3[i] = *reinterpret_cast<const uint4*>(s13 + (4 + i) * CHUNK_STRIDE);
                        }
                    } else {
                        const uint4* pa1 = reinterpret_cast<const uint4*>(p.a1 + m * p.f + n);
                        const uint4* pa3 = reinterpret_cast<const uint4*>(p.a3 + m * p.f + n);
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            v1[i] = pa1[i];
                            v3[i] = pa3[i];
                        }
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint32_t w1[4] = {v1[i].x, v1[i].y, v1[i].z, v1[i].w};
                        const uint32_t w3[4] = {v3[i].x, v3[i].y, v3[i].z, v3[i].w};
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const uint32_t wg = dp[4 * i + j];
                            float o1[2], o3[2];
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                const float x = e ? bf16_hi(w1[j]) : bf16_lo(w1[j]);
                                const float y = e ? bf16_hi(w3[j]) : bf16_lo(w3[j]);
                                const float g = e ? bf16_hi(wg) : bf16_lo(wg);
                                const float sg = __fdividef(1.0f, 1.0f + __expf(-x));
                                const float dsilu = sg * (1.0f + x * (1.0f - sg));
                                o1[e] = g * y * dsilu;
                                o3[e] = g * (x * sg);
                            }
                            q1[4 * i + j] = bf16x2_rn(o1[0], o1[1]);
                            q3[4 * i + j] = bf16x2_rn(o3[0], o3[1]);
                        }
                    }
                }
                // the slot's values are consumed: the next tile's segments may land
                prefetch_a13(u + n_clusters);
                if (p.tap1) {
                    tap_store(q1, &tmX, (int)n);
                    tap_store(q3, &tmX, (int)(p.f + n));
                }
                if (p.amax_ws) {
                    // maxima of the [da1 | da3] tap: the tile's row strip
                    // spans both, the column strips are da1's and da3's
                    const uint32_t m1 = warp_amax_words<16>(q1), m3 = warp_amax_words<16>(q3);
                    if (lane == 0) {
                        atomicMax(&p.amax_ws[1 + (m0 >> 7)], max(m1, m3));
                        atomicMax(&p.amax_ws[1 + (p.M >> 7) + (n0 >> 7)], m1);
                        atomicMax(&p.amax_ws[1 + (p.M >> 7) + ((p.f + n0) >> 7)], m3);
                        tensor_amax = max(tensor_amax, max(m1, m3));
                    }
                }
                if (p.quantize) {
                    // row views of [da1 | da3] (stochastic rounding), one block each
                    uint4 pk;
                    uint32_t sc = mx_words_sr(q1, (uint64_t)(m * f2 + n) >> 3, p.sr_keys, p.offset, pk);
                    *reinterpret_cast<uint4*>(p.q_row_codes + m * p.f + (n >> 1)) = pk;
                    atoms[atom_off(lr, half)] = (uint8_t)sc;
                    sc = mx_words_sr(q3, (uint64_t)(m * f2 + p.f + n) >> 3, p.sr_keys, p.offset, pk);
                    *reinterpret_cast<uint4*>(p.q_row_codes + m * p.f + ((p.f + n) >> 1)) = pk;
                    atoms[512 + atom_off(lr, half)] = (uint8_t)sc;
                    // column views: this warp's 32 x 32 block of da1, then of
                    // da3, through its box (64B swizzle); each lane encodes
                    // one column (one stored row of Q_c(da13)) down the block
#pragma unroll 1
                    for (int which = 0; which < 2; ++which) {
                        const uint32_t* src = which ? q3 : q1;
                        if (lane == 0) bulk_wait_read<0>();  // a tap store may still read the box
                        __syncwarp();  // the previous reads of the box are done
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            *reinterpret_cast<uint4*>(box + lane * 64 + ((k ^ ((lane >> 1) & 3)) << 4)) =
                                make_uint4(src[4 * k], src[4 * k + 1], src[4 * k + 2], src[4 * k + 3]);
                        __syncwarp();
                        uint32_t w[16];
                        const int ck = lane >> 3, cb = (lane & 7) * 2;
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const int r0 = 2 * i, r1 = 2 * i + 1;
                            const uint32_t lo =
                                *reinterpret_cast<const uint16_t*>(box + r0 * 64 + ((ck ^ ((r0 >> 1) & 3)) << 4) + cb);
                            const uint32_t hi =
                                *reinterpret_cast<const uint16_t*>(box + r1 * 64 + ((ck ^ ((r1 >> 1) & 3)) << 4) + cb);
                            w[i] = lo | (hi << 16);
                        }
                        uint4 pkc;
                        const uint32_t scc = mx_words_rn(w, pkc);
                        const int64_t srow = (which ? p.f : 0) + n + lane;
                        *reinterpret_cast<uint4*>(p.q_col_codes + srow * (p.M >> 1) + ((m0 + 32 * q) >> 1)) = pkc;
                        atoms[1024 + which * 512 + atom_off(oc + lane, q)] = (uint8_t)scc;
                    }
                    // the tile's four scale atoms (double-buffered by tile, so
                    // one barrier per tile suffices)
                    epi_sync();
                    if (!epi_ok) break;
                    if (et < 128) {
                        const int which = et >> 5, part = et & 31;
                        int64_t a;
                        if (which < 2)  // row views of da1 / da3 in [M][2f]
                            a = (m0 >> 7) * (f2 >> 7) + ((which ? p.f : 0) + n0) / 128;
                        else  // column views in [2f][M]
                            a = (((which == 3 ? p.f : 0) + n0) >> 7) * (p.M >> 7) + (m0 >> 7);
                        uint8_t* dst = (which < 2 ? p.q_row_scales : p.q_col_scales) + a * 512 + part * 16;
                        *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(atoms + which * 512 + part * 16);
                    }
                }
            }
            acc_phase ^= 1;
        }
        if ((EPI == EPI_SWIGLU_FWD || EPI == EPI_SWIGLU_BWD) && p.amax_ws && lane == 0 && tensor_amax)
            atomicMax(&p.amax_ws[0], tensor_amax);
    }
    if ((is_store(EPI) || EPI == EPI_SWIGLU_FWD || EPI == EPI_SWIGLU_BWD || EPI == EPI_QKV_ROPE) && warp >= 2 &&
        lane == 0)
        bulk_wait_all();  // TMA stores done with shared memory
    if (Cfg<NV, BN, EPI, P2>::BWD_PREFETCH && warp >= 2 && warp < 2 + EW) cp_async_wait_all();
    tc_fence_before();
    __syncthreads();
    if (CM > 1) cluster_sync();  // the peer no longer arrives on this CTA's barriers
    if (warp == 1) {
        tc_fence_after();
        if (P2)
            asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS)
                         : "memory");
        else
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS)
                         : "memory");
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

// K-major FP4 codes [rows][K/2] bytes as a 2D uint8 tensor, box 128 B x
// `box_rows` rows (128, or 64 for the B half of a 128-wide pair tile).
bool make_map(CUtensorMap* map, const void* codes, int64_t rows, int64_t K, int box_rows = 128) {
    cuuint64_t dims[2] = {(cuuint64_t)(K / 2), (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(K / 2)};
    cuuint32_t box[2] = {(cuuint32_t)BK_BYTES, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(codes), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, BK_BYTES == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Scale atoms [atoms][512 bytes] as a 2D uint32 tensor, box = `chunk`
// consecutive atoms (the pair kernel loads its scales through TMA so that
// their completion can be counted on the pair leader's barrier).
bool make_sf_map(CUtensorMap* map, const void* scales, int64_t atoms, int chunk) {
    cuuint64_t dims[2] = {128u, (cuuint64_t)atoms};
    cuuint64_t strides[1] = {512u};
    cuuint32_t box[2] = {128u, (cuuint32_t)chunk};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(scales), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Row-major output [M][N] (fp32 or bf16), box `row_bytes` (128, 64 or 32) x
// 32 rows with the swizzle of that width.
bool make_out_map(CUtensorMap* map, void* c, int64_t M, int64_t N, int out_dtype, int row_bytes) {
    const bool f32 = out_dtype == FP4_OUT_F32;
    const int es = f32 ? 4 : 2;
    cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)M};
    cuuint64_t strides[1] = {(cuuint64_t)(N * es)};
    cuuint32_t box[2] = {(cuuint32_t)(row_bytes / es), 32u};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, c, dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          row_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                          : row_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                            : CU_TENSOR_MAP_SWIZZLE_32B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int sm_count() {
    static int cached[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 64) dev = 63;
    if (!cached[dev]) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cached[dev] = n > 0 ? n : 1;
    }
    return cached[dev];
}

template <bool NV, int BN, int EPI, int CM, bool P2 = false>
int launch_t(const GemmParams& g, const KParams& kp, int64_t n_units, cudaStream_t stream) {
    using C = Cfg<NV, BN, EPI, P2>;
    CUtensorMap ta, tb, tc, tsa, tsb, tx, ty;
    if (!make_map(&ta, g.a_codes, g.M, g.K) || !make_map(&tb, g.b_codes, g.b_rows, g.K, P2 ? BN / 2 : 128))
        return FP4_ERR_CUDA;
    memset(&tc, 0, sizeof tc);
    memset(&tsa, 0, sizeof tsa);
    memset(&tsb, 0, sizeof tsb);
    memset(&tx, 0, sizeof tx);
    memset(&ty, 0, sizeof ty);
    // QKV + RoPE: q, k, v as [heads * M][128] views with 32-byte row boxes
    if (EPI == EPI_QKV_ROPE && (!make_out_map(&tc, g.q_out, (int64_t)g.heads_q * g.M, 128, FP4_OUT_BF16, 32) ||
                                !make_out_map(&tx, g.k_out, (int64_t)g.heads_kv * g.M, 128, FP4_OUT_BF16, 32) ||
                                !make_out_map(&ty, g.v_out, (int64_t)g.heads_kv * g.M, 128, FP4_OUT_BF16, 32)))
        return FP4_ERR_CUDA;
    // the SwiGLU taps' maps: the forward's h in the output map's slot, the
    // backward's [da1 | da3] and dh in the a1 / a3 slots it does not use
    if (EPI == EPI_SWIGLU_FWD && g.tap0 && !make_out_map(&tc, g.tap0, g.M, g.f, FP4_OUT_BF16, 64)) return FP4_ERR_CUDA;
    if (EPI == EPI_SWIGLU_BWD && g.tap1 && !make_out_map(&tx, g.tap1, g.M, 2 * g.f, FP4_OUT_BF16, 64)) return FP4_ERR_CUDA;
    if (EPI == EPI_SWIGLU_BWD && g.tap0 && !make_out_map(&ty, g.tap0, g.M, g.f, FP4_OUT_BF16, 64)) return FP4_ERR_CUDA;
    if (EPI == EPI_SWIGLU_FWD && (!make_out_map(&tx, g.a1, g.M, g.f, FP4_OUT_BF16, 64) ||
                                  !make_out_map(&ty, g.a3, g.M, g.f, FP4_OUT_BF16, 64)))
        return FP4_ERR_CUDA;
    if (P2) {
        const int64_t k_atoms = NV ? g.K / 64 : g.K / 128;
        if (!make_sf_map(&tsa, g.a_scales, (g.M / 128) * k_atoms, C::SF_CHUNKS) ||
            !make_sf_map(&tsb, g.b_scales, (g.b_rows / 128) * k_atoms, C::SF_CHUNKS))
            return FP4_ERR_CUDA;
    }
    if (is_store(EPI) && (g.beta == 0.0f || g.beta == 1.0f) && !make_out_map(&tc, g.c, g.M, g.N, g.out_dtype, C::OUT_ROW))
        return FP4_ERR_CUDA;
    auto kern = fp4_gemm_kernel<NV, BN, EPI, CM, P2>;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FP4_ERR_CUDA;
    static std::mutex mu;
    static bool attr_done[64] = {};
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!attr_done[dev]) {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
                return FP4_ERR_CUDA;
            attr_done[dev] = true;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.blockDim = dim3(kthreads(EPI));
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = stream;
    int max_clusters = sm_count() / CM;
    if (CM > 1) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = CM;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cfg.gridDim = dim3((unsigned)(max_clusters * CM));
        int active = 0;
        if (cudaOccupancyMaxActiveClusters(&active, (void*)kern, &cfg) == cudaSuccess && active > 0)
            max_clusters = active;
    }
    const int64_t clusters = n_units < max_clusters ? n_units : max_clusters;
    cfg.gridDim = dim3((unsigned)(clusters * CM));
    // Raster: the operand with fewer code bytes stays in L2 (a band of its
    // tiles as wide as the budget allows, all of it when it fits) while the
    // other streams through once per band.
    KParams k = kp;
    {
        const int64_t m_units = g.M / (BM * CM);
        const int64_t n_blocks = EPI == EPI_SWIGLU_FWD ? g.f / 128 : g.N / BN;
        const int64_t a_unit = (int64_t)BM * CM * (g.K / 2), b_unit = (int64_t)(EPI == EPI_SWIGLU_FWD ? 256 : BN) * (g.K / 2);
        const bool n_inner = b_unit * n_blocks < a_unit * m_units;
        const int64_t unit_bytes = n_inner ? b_unit : a_unit, units = n_inner ? n_blocks : m_units;
        int64_t band = L2_RESIDENT_BYTES / (unit_bytes > 0 ? unit_bytes : 1);
        k.n_inner = n_inner ? 1 : 0;
        k.band = band < 1 ? 1 : (band > units ? units : band);
    }
    if (cudaLaunchKernelEx(&cfg, kern, ta, tb, tc, tsa, tsb, tx, ty, k) != cudaSuccess) return FP4_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? FP4_OK : FP4_ERR_CUDA;
}

KParams kparams_of(const GemmParams& g) {
    KParams p{};
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
    p.f = g.f;
    p.a1 = g.a1;
    p.a3 = g.a3;
    p.tap0 = g.tap0;
    p.tap1 = g.tap1;
    p.quantize = g.quantize;
    p.q_row_codes = g.q_row_codes;
    p.q_row_scales = g.q_row_scales;
    p.q_col_codes = g.q_col_codes;
    p.q_col_scales = g.q_col_scales;
    p.seed = g.seed;
    p.offset = g.offset;
    sr_round_keys(g.seed, p.sr_keys);
    p.q_out = g.q_out;
    p.k_out = g.k_out;
    p.v_out = g.v_out;
    p.rope_cos = g.rope_cos;
    p.rope_sin = g.rope_sin;
    p.seq_len = g.seq_len;
    p.heads_q = g.heads_q;
    p.heads_kv = g.heads_kv;
    p.rms_rp = g.rms_rp;
    p.rms_g = g.rms_g;
    p.rms_rstd = g.rms_rstd;
    p.rms_part = g.rms_part;
    p.amax_ws = g.amax_ws;
    return p;
}

}  // namespace

std::atomic<long long> g_wait_cycles{WAIT_CYCLES};
std::atomic<int> g_skip_first_release{0};

int launch_gemm(const GemmParams& g0, cudaStream_t stream) {
    if (!get_encode()) return FP4_ERR_CUDA;
    GemmParams g = g0;
    const bool pair = (g.M / BM) % 2 == 0;
    KParams kp = kparams_of(g);
    kp.wait_cycles = g_wait_cycles.load();
    kp.skip_first_release = g_skip_first_release.load();
    if (g.epi == 1) {  // SwiGLU forward: B = [W1; W3] with 2f rows, output width f
        g.b_rows = 2 * g.f;
        const int64_t units_1 = (g.M / BM) * (g.f / 128);
        if (g.nv) return pair ? launch_t<true, 256, EPI_SWIGLU_FWD, 2, true>(g, kp, units_1 / 2, stream)
                              : launch_t<true, 256, EPI_SWIGLU_FWD, 1>(g, kp, units_1, stream);
        return pair ? launch_t<false, 256, EPI_SWIGLU_FWD, 2, true>(g, kp, units_1 / 2, stream)
                    : launch_t<false, 256, EPI_SWIGLU_FWD, 1>(g, kp, units_1, stream);
    }
    g.b_rows = g.N;
    if (g.epi == 3) {  // QKV projection with RoPE into head-major outputs
        const int64_t units_1 = (g.M / BM) * (g.N / 256);
        if (g.nv) return pair ? launch_t<true, 256, EPI_QKV_ROPE, 2, true>(g, kp, units_1 / 2, stream)
                              : launch_t<true, 256, EPI_QKV_ROPE, 1>(g, kp, units_1, stream);
        return pair ? launch_t<false, 256, EPI_QKV_ROPE, 2, true>(g, kp, units_1 / 2, stream)
                    : launch_t<false, 256, EPI_QKV_ROPE, 1>(g, kp, units_1, stream);
    }
    if (g.epi == 2) {  // SwiGLU backward: W2 Dgrad, output [M][f]
        const int64_t units_1 = (g.M / BM) * (g.N / 128);
        if (g.nv) return pair ? launch_t<true, 128, EPI_SWIGLU_BWD, 2, true>(g, kp, units_1 / 2, stream)
                              : launch_t<true, 128, EPI_SWIGLU_BWD, 1>(g, kp, units_1, stream);
        return pair ? launch_t<false, 128, EPI_SWIGLU_BWD, 2, true>(g, kp, units_1 / 2, stream)
                    : launch_t<false, 128, EPI_SWIGLU_BWD, 1>(g, kp, units_1, stream);
    }
    const bool wide = (g.N % 256) == 0;
    const int64_t units_1 = (g.M / BM) * (g.N / (wide ? 256 : 128));
    if (g.rms_part) {  // bf16 store + RMSNorm row terms: the pair kernel, else 128-wide single CTAs
        const int64_t units_128 = (g.M / BM) * (g.N / 128);
        if (g.nv) return wide && pair ? launch_t<true, 256, EPI_STORE_RMS, 2, true>(g, kp, units_1 / 2, stream)
                                      : launch_t<true, 128, EPI_STORE_RMS, 1>(g, kp, units_128, stream);
        return wide && pair ? launch_t<false, 256, EPI_STORE_RMS, 2, true>(g, kp, units_1 / 2, stream)
                            : launch_t<false, 128, EPI_STORE_RMS, 1>(g, kp, units_128, stream);
    }
    if (g.nv) {
        // an even number of M blocks runs on CTA pairs (M = 256 MMAs), 256 or
        // 128 columns wide; an odd number on single CTAs
        if (wide) return pair ? launch_t<true, 256, EPI_STORE, 2, true>(g, kp, units_1 / 2, stream)
                              : launch_t<true, 256, EPI_STORE, 1>(g, kp, units_1, stream);
        return pair ? launch_t<true, 128, EPI_STORE, 2, true>(g, kp, units_1 / 2, stream)
                    : launch_t<true, 128, EPI_STORE, 1>(g, kp, units_1, stream);
    }
    if (wide) return pair ? launch_t<false, 256, EPI_STORE, 2, true>(g, kp, units_1 / 2, stream)
                          : launch_t<false, 256, EPI_STORE, 1>(g, kp, units_1, stream);
    return pair ? launch_t<false, 128, EPI_STORE, 2, true>(g, kp, units_1 / 2, stream)
                : launch_t<false, 128, EPI_STORE, 1>(g, kp, units_1, stream);
}

void gemm_set_wait_limit(uint64_t cycles) {
    g_wait_cycles.store(cycles == 0 || cycles > (uint64_t)WAIT_CYCLES * 1000 ? WAIT_CYCLES : (long long)cycles);
}
void gemm_test_skip_first_release(int enable) { g_skip_first_release.store(enable ? 1 : 0); }

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
