// api.cu -- the extern "C" boundary of libfp4lin (declared in include/fp4lin.h).
//
// Host-side argument validation and dispatch only: every step of the path
// runs in the kernels of quantize.cu / gemm.cu / fused.cu.  Nothing here
// allocates or synchronises, except fp4_status() which reads the device
// status words.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

using namespace fp4;

namespace {

bool route_ok(int route) {
    return route == FP4_ROUTE_MXFP4 || route == FP4_ROUTE_NVFP4_GLOBAL || route == FP4_ROUTE_NVFP4_LOCAL;
}

int block_size(int route) { return route == FP4_ROUTE_MXFP4 ? 32 : 16; }

int32_t outer_count_of(int route, int64_t rows, unsigned flags) {
    if (route == FP4_ROUTE_MXFP4) return 0;
    if (route == FP4_ROUTE_NVFP4_GLOBAL || (flags & FP4_FLAG_WEIGHT_2D)) return 1;
    return (int32_t)(rows / 128);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" {

int fp4_version(void) { return FP4LIN_VERSION; }

const char* fp4_status_string(int code) {
    switch (code) {
        case FP4_OK: return "ok";
        case FP4_ERR_INVALID_ARG: return "invalid argument";
        case FP4_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
        case FP4_ERR_ROUTE_MISMATCH: return "route mismatch";
        case FP4_ERR_WORKSPACE: return "workspace too small";
        case FP4_ERR_CUDA: return "CUDA error";
        case FP4_ERR_TIMEOUT: return "device wait timed out";
        case FP4_ERR_NONFINITE: return "non-finite input";
        default: return "unknown status";
    }
}

int fp4_tensor_bytes(int route, int64_t rows, int64_t cols, unsigned flags, size_t* codes_bytes, size_t* scale_bytes,
                     int32_t* outer_count) {
    if (!route_ok(route) || rows < 0 || cols < 0) return FP4_ERR_INVALID_ARG;
    if (rows % 128 || cols % 128) return FP4_ERR_UNSUPPORTED_SHAPE;
    if (codes_bytes) *codes_bytes = (size_t)(rows * cols / 2);
    if (scale_bytes) *scale_bytes = (size_t)(rows * cols / block_size(route));
    if (outer_count) *outer_count = outer_count_of(route, rows, flags);
    return FP4_OK;
}

int fp4_quantize_workspace_bytes(int route, int64_t rows, int64_t cols, unsigned views, unsigned flags,
                                 size_t* bytes) {
    return fp4_quantize_hybrid_workspace_bytes(route, route, rows, cols, views, flags, bytes);
}

int fp4_quantize_hybrid_workspace_bytes(int row_route, int col_route, int64_t rows, int64_t cols, unsigned views,
                                        unsigned flags, size_t* bytes) {
    if (!route_ok(row_route) || !route_ok(col_route) || !bytes || rows < 0 || cols < 0) return FP4_ERR_INVALID_ARG;
    if ((views & ~3u) || (flags & ~15u)) return FP4_ERR_INVALID_ARG;
    if (rows % 128 || cols % 128) return FP4_ERR_UNSUPPORTED_SHAPE;
    *bytes = quant_workspace_slots(rows, cols, row_route, col_route, views ? views : 3u, flags) * 4;
    return FP4_OK;
}

// Validate a quantizer call and fill its parameters; nothing is enqueued.
// x may be NULL when the caller produces it in an earlier kernel (pre-ops).
static int prepare_quant(const void* x, bool x_from_pre, int64_t rows, int64_t cols, int64_t ld, int row_route,
                         int col_route, unsigned views, unsigned flags, uint64_t sr_seed, uint64_t sr_offset,
                         const int8_t* hadamard_signs, fp4_tensor* row_out, fp4_tensor* col_out, void* workspace,
                         size_t workspace_bytes, QuantParams* p) {
    if (!route_ok(row_route) || !route_ok(col_route)) return FP4_ERR_INVALID_ARG;
    if ((views & ~3u) || views == 0 || (flags & ~15u)) return FP4_ERR_INVALID_ARG;
    if (rows < 0 || cols < 0 || ld < cols) return FP4_ERR_INVALID_ARG;
    if (rows % 128 || cols % 128) return FP4_ERR_UNSUPPORTED_SHAPE;
    const unsigned had_any = FP4_FLAG_HADAMARD_COL | FP4_FLAG_HADAMARD16_COL;
    if ((flags & FP4_FLAG_WEIGHT_2D) && (flags & (FP4_FLAG_SR_ROW | had_any))) return FP4_ERR_ROUTE_MISMATCH;
    if ((flags & FP4_FLAG_HADAMARD_COL) && (flags & FP4_FLAG_HADAMARD16_COL)) return FP4_ERR_INVALID_ARG;
    if ((flags & FP4_FLAG_HADAMARD_COL) && col_route != FP4_ROUTE_MXFP4) return FP4_ERR_ROUTE_MISMATCH;
    const bool do_row = views & FP4_VIEW_ROW, do_col = views & FP4_VIEW_COL;
    if ((do_row && !row_out) || (do_col && !col_out)) return FP4_ERR_INVALID_ARG;
    for (int v = 0; v < 2; ++v) {
        fp4_tensor* t = v == 0 ? (do_row ? row_out : nullptr) : (do_col ? col_out : nullptr);
        if (!t) continue;
        if (!t->codes || !t->scales || !aligned16(t->codes) || !aligned16(t->scales)) return FP4_ERR_INVALID_ARG;
        if ((v == 0 ? row_route : col_route) != FP4_ROUTE_MXFP4 && !t->outer) return FP4_ERR_INVALID_ARG;
    }
    uint32_t sign_mask = 0;
    if (flags & had_any) {
        if (!hadamard_signs) return FP4_ERR_INVALID_ARG;
        for (int j = 0; j < 16; ++j) {
            if (hadamard_signs[j] != 1 && hadamard_signs[j] != -1) return FP4_ERR_INVALID_ARG;
            if (hadamard_signs[j] < 0) sign_mask |= 1u << j;
        }
    }
    const size_t need = quant_workspace_slots(rows, cols, row_route, col_route, views, flags) * 4;
    if (need > 0 && (!workspace || workspace_bytes < need)) return FP4_ERR_WORKSPACE;
    if (rows > 0 && cols > 0 && !x_from_pre && (!x || !aligned16(x) || ld % 8)) return FP4_ERR_INVALID_ARG;

    if (do_row) {
        row_out->rows = rows;
        row_out->cols = cols;
        row_out->route = row_route;
        row_out->outer_count = outer_count_of(row_route, rows, flags);
    }
    if (do_col) {
        col_out->rows = cols;
        col_out->cols = rows;
        col_out->route = col_route;
        col_out->outer_count = outer_count_of(col_route, cols, flags);
    }
    *p = QuantParams{};
    p->x = static_cast<const uint16_t*>(x);
    p->R = rows;
    p->C = cols;
    p->ld = ld;
    p->row_route = row_route;
    p->col_route = col_route;
    p->views = views;
    p->flags = flags;
    p->seed = sr_seed;
    p->offset = sr_offset;
    sr_round_keys(sr_seed, p->sr_keys);
    p->sign_mask = sign_mask;
    if (do_row) {
        p->row_codes = static_cast<uint8_t*>(row_out->codes);
        p->row_scales = static_cast<uint8_t*>(row_out->scales);
        p->row_outer = row_out->outer;
    }
    if (do_col) {
        p->col_codes = static_cast<uint8_t*>(col_out->codes);
        p->col_scales = static_cast<uint8_t*>(col_out->scales);
        p->col_outer = col_out->outer;
    }
    p->amax_ws = static_cast<uint32_t*>(workspace);
    return FP4_OK;
}

int fp4_quantize(const void* x, int64_t rows, int64_t cols, int64_t ld, int route, unsigned views, unsigned flags,
                 uint64_t sr_seed, uint64_t sr_offset, const int8_t* hadamard_signs, fp4_tensor* row_out,
                 fp4_tensor* col_out, void* workspace, size_t workspace_bytes, fp4_stream_t stream) {
    QuantParams p;
    int rc = prepare_quant(x, false, rows, cols, ld, route, route, views, flags, sr_seed, sr_offset, hadamard_signs,
                           row_out, col_out, workspace, workspace_bytes, &p);
    if (rc != FP4_OK || rows == 0 || cols == 0) return rc;
    return launch_quantize(p, reinterpret_cast<cudaStream_t>(stream));
}

int fp4_quantize_hybrid(const void* x, int64_t rows, int64_t cols, int64_t ld, int row_route, int col_route,
                        unsigned views, unsigned flags, uint64_t sr_seed, uint64_t sr_offset,
                        const int8_t* hadamard_signs, fp4_tensor* row_out, fp4_tensor* col_out, void* workspace,
                        size_t workspace_bytes, fp4_stream_t stream) {
    QuantParams p;
    int rc = prepare_quant(x, false, rows, cols, ld, row_route, col_route, views, flags, sr_seed, sr_offset,
                           hadamard_signs, row_out, col_out, workspace, workspace_bytes, &p);
    if (rc != FP4_OK || rows == 0 || cols == 0) return rc;
    return launch_quantize(p, reinterpret_cast<cudaStream_t>(stream));
}

int fp4_residual_rmsnorm_fwd(int route, unsigned views, const void* r, const void* b, const void* g, int64_t rows,
                             int64_t cols, int64_t ld, float eps, void* r_out, float* rstd, fp4_tensor* y_row,
                             fp4_tensor* y_col, void* y_tap, void* workspace, size_t workspace_bytes,
                             fp4_stream_t stream) {
    QuantParams p;
    int rc = prepare_quant(r_out, true, rows, cols, cols, route, route, views, 0, 0, 0, nullptr, y_row, y_col,
                           workspace, workspace_bytes, &p);
    if (rc != FP4_OK || rows == 0 || cols == 0) return rc;
    if (ld < cols || ld % 8) return FP4_ERR_INVALID_ARG;
    if (!r || !g || !r_out || !rstd || !aligned16(r) || !aligned16(g) || !aligned16(r_out) || (b && !aligned16(b)) ||
        (y_tap && !aligned16(y_tap)))
        return FP4_ERR_INVALID_ARG;
    if (!(eps >= 0.0f)) return FP4_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const size_t slots = quant_workspace_slots(rows, cols, route, route, views, 0);
    if (slots) {
        // NVFP4: the row pass also folds the maxima of y, so the encoder
        // needs no pass of its own over the rows before it
        if (cudaMemsetAsync(p.amax_ws, 0, slots * 4, s) != cudaSuccess) return FP4_ERR_CUDA;
        rc = launch_rmsnorm_fwd_stats_amax(static_cast<const uint16_t*>(r), static_cast<const uint16_t*>(b),
                                           static_cast<const uint16_t*>(g), rows, cols, ld, eps,
                                           static_cast<uint16_t*>(r_out), rstd, p.amax_ws, s);
        p.amax_ready = 1;
    } else {
        rc = launch_rmsnorm_fwd_stats(static_cast<const uint16_t*>(r), static_cast<const uint16_t*>(b), rows, cols,
                                      ld, eps, static_cast<uint16_t*>(r_out), rstd, s);
    }
    if (rc != FP4_OK) return rc;
    p.pre = PRE_RMSNORM_FWD;
    p.rstd = rstd;
    p.g = static_cast<const uint16_t*>(g);
    p.tap = static_cast<uint16_t*>(y_tap);
    return launch_quantize(p, s);
}

int fp4_rmsnorm_bwd_workspace_bytes(int route, int64_t rows, int64_t cols, size_t* bytes) {
    if (!bytes) return FP4_ERR_INVALID_ARG;
    size_t q = 0;
    int rc = fp4_quantize_workspace_bytes(route, rows, cols, 3, 0, &q);
    if (rc != FP4_OK) return rc;
    size_t stats = ((size_t)rows * 4 + 255) / 256 * 256;
    *bytes = stats + q;
    return FP4_OK;
}

// The residual-RMSNorm backward: the row means from a pass over dy (part
// NULL) or from the per-block row terms a data-gradient epilogue wrote.
static int rmsnorm_bwd(int route, unsigned views, int sr, const void* dy, const float* part, const void* r_prime,
                       const float* rstd, const void* g, const void* dres, int64_t rows, int64_t cols,
                       uint64_t sr_seed, uint64_t sr_offset, void* dr, fp4_tensor* dr_row, fp4_tensor* dr_col,
                       void* workspace, size_t workspace_bytes, fp4_stream_t stream) {
    if (!route_ok(route) || rows < 0 || cols < 0) return FP4_ERR_INVALID_ARG;
    if (rows % 128 || cols % 128) return FP4_ERR_UNSUPPORTED_SHAPE;
    size_t need = 0;
    fp4_rmsnorm_bwd_workspace_bytes(route, rows, cols, &need);
    const size_t stats = ((size_t)rows * 4 + 255) / 256 * 256;
    if (rows > 0 && cols > 0 && (!workspace || workspace_bytes < need)) return FP4_ERR_WORKSPACE;
    void* qws = workspace ? static_cast<uint8_t*>(workspace) + stats : nullptr;
    QuantParams p;
    int rc = prepare_quant(dy, false, rows, cols, cols, route, route, views, sr ? FP4_FLAG_SR_ROW : 0, sr_seed,
                           sr_offset, nullptr, dr_row, dr_col, qws, workspace ? workspace_bytes - stats : 0, &p);
    if (rc != FP4_OK || rows == 0 || cols == 0) return rc;
    if (!r_prime || !rstd || !g || !dr || !aligned16(r_prime) || !aligned16(g) || !aligned16(dr) ||
        (dres && !aligned16(dres)))
        return FP4_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    float* mean_g = static_cast<float*>(workspace);
    rc = part ? launch_rms_parts_reduce(part, rows, cols / 64, cols, mean_g, s)
              : launch_rmsnorm_bwd_stats(static_cast<const uint16_t*>(dy), static_cast<const uint16_t*>(r_prime),
                                         rstd, static_cast<const uint16_t*>(g), rows, cols, mean_g, s);
    if (rc != FP4_OK) return rc;
    p.pre = PRE_RMSNORM_BWD;
    p.rstd = rstd;
    p.g = static_cast<const uint16_t*>(g);
    p.mean_g = mean_g;
    p.rp = static_cast<const uint16_t*>(r_prime);
    p.dres = static_cast<const uint16_t*>(dres);
    p.tap = static_cast<uint16_t*>(dr);
    return launch_quantize(p, s);
}

int fp4_residual_rmsnorm_bwd(int route, unsigned views, int sr, const void* dy, const void* r_prime,
                             const float* rstd, const void* g, const void* dres, int64_t rows, int64_t cols,
                             uint64_t sr_seed, uint64_t sr_offset, void* dr, fp4_tensor* dr_row, fp4_tensor* dr_col,
                             void* workspace, size_t workspace_bytes, fp4_stream_t stream) {
    return rmsnorm_bwd(route, views, sr, dy, nullptr, r_prime, rstd, g, dres, rows, cols, sr_seed, sr_offset, dr,
                       dr_row, dr_col, workspace, workspace_bytes, stream);
}

int fp4_residual_rmsnorm_bwd_parts(int route, unsigned views, int sr, const void* dy, const float* part,
                                   const void* r_prime, const float* rstd, const void* g, const void* dres,
                                   int64_t rows, int64_t cols, uint64_t sr_seed, uint64_t sr_offset, void* dr,
                                   fp4_tensor* dr_row, fp4_tensor* dr_col, void* workspace, size_t workspace_bytes,
                                   fp4_stream_t stream) {
    if (!part && rows > 0 && cols > 0) return FP4_ERR_INVALID_ARG;
    return rmsnorm_bwd(route, views, sr, dy, part, r_prime, rstd, g, dres, rows, cols, sr_seed, sr_offset, dr,
                       dr_row, dr_col, workspace, workspace_bytes, stream);
}

// The adjacent RMSNorm backward's row terms, computed in a plain bf16 store
// epilogue (see fp4_linear_dgrad_rmsnorm).
struct RmsTerms {
    const void* r_prime;
    const float* rstd;
    const void* g;
    float* part;
};

static int linear(const fp4_tensor* a, const fp4_tensor* b, void* c, int out_dtype, float beta, fp4_stream_t stream,
                  const RmsTerms* rms = nullptr) {
    if (!a || !b || !c) return FP4_ERR_INVALID_ARG;
    if (out_dtype != FP4_OUT_F32 && out_dtype != FP4_OUT_BF16) return FP4_ERR_INVALID_ARG;
    if (!route_ok(a->route) || !route_ok(b->route)) return FP4_ERR_INVALID_ARG;
    if (a->route != b->route) return FP4_ERR_ROUTE_MISMATCH;
    if (a->cols != b->cols) return FP4_ERR_UNSUPPORTED_SHAPE;
    const int64_t M = a->rows, N = b->rows, K = a->cols;
    if (M < 0 || N < 0 || K < 0) return FP4_ERR_INVALID_ARG;
    if (M % 128 || N % 128 || K % 256) return FP4_ERR_UNSUPPORTED_SHAPE;
    const bool nv = a->route != FP4_ROUTE_MXFP4;
    for (const fp4_tensor* t : {a, b}) {
        if (!t->codes || !t->scales || !aligned16(t->codes) || !aligned16(t->scales)) return FP4_ERR_INVALID_ARG;
        if (nv && (!t->outer || (t->outer_count != 1 && t->outer_count != t->rows / 128))) return FP4_ERR_INVALID_ARG;
    }
    if (!aligned16(c)) return FP4_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return FP4_OK;
    if (K == 0) return FP4_ERR_UNSUPPORTED_SHAPE;
    GemmParams g{};
    g.a_codes = static_cast<const uint8_t*>(a->codes);
    g.a_scales = static_cast<const uint8_t*>(a->scales);
    g.a_outer = nv ? a->outer : nullptr;
    g.a_outer_count = a->outer_count;
    g.b_codes = static_cast<const uint8_t*>(b->codes);
    g.b_scales = static_cast<const uint8_t*>(b->scales);
    g.b_outer = nv ? b->outer : nullptr;
    g.b_outer_count = b->outer_count;
    g.M = M;
    g.N = N;
    g.K = K;
    g.nv = nv ? 1 : 0;
    g.c = c;
    g.out_dtype = out_dtype;
    g.beta = beta;
    if (rms) {
        g.rms_rp = static_cast<const uint16_t*>(rms->r_prime);
        g.rms_g = static_cast<const uint16_t*>(rms->g);
        g.rms_rstd = rms->rstd;
        g.rms_part = rms->part;
    }
    return launch_gemm(g, reinterpret_cast<cudaStream_t>(stream));
}

static bool view_ok(const fp4_tensor* t) {
    return t && t->codes && t->scales && aligned16(t->codes) && aligned16(t->scales);
}

static void set_view(fp4_tensor* t, int64_t rows, int64_t cols, int route) {
    t->rows = rows;
    t->cols = cols;
    t->route = route;
    t->outer_count = 0;
}

static void fill_operands(GemmParams& g, const fp4_tensor* a, const fp4_tensor* b) {
    const bool nv = a->route != FP4_ROUTE_MXFP4;
    g.a_codes = static_cast<const uint8_t*>(a->codes);
    g.a_scales = static_cast<const uint8_t*>(a->scales);
    g.a_outer = nv ? a->outer : nullptr;
    g.a_outer_count = a->outer_count;
    g.b_codes = static_cast<const uint8_t*>(b->codes);
    g.b_scales = static_cast<const uint8_t*>(b->scales);
    g.b_outer = nv ? b->outer : nullptr;
    g.b_outer_count = b->outer_count;
    g.nv = nv ? 1 : 0;
}

static int check_operand(const fp4_tensor* t) {
    if (!t || !route_ok(t->route)) return FP4_ERR_INVALID_ARG;
    if (!view_ok(t)) return FP4_ERR_INVALID_ARG;
    if (t->route != FP4_ROUTE_MXFP4 && (!t->outer || (t->outer_count != 1 && t->outer_count != t->rows / 128)))
        return FP4_ERR_INVALID_ARG;
    return FP4_OK;
}

int fp4_qkv_rope_fwd(const fp4_tensor* x_row, const fp4_tensor* wqkv_row, const float* rope_cos,
                     const float* rope_sin, int64_t seq_len, int heads_q, int heads_kv, void* q, void* k, void* v,
                     fp4_stream_t stream) {
    int rc;
    if ((rc = check_operand(x_row)) != FP4_OK || (rc = check_operand(wqkv_row)) != FP4_OK) return rc;
    if (x_row->route != wqkv_row->route) return FP4_ERR_ROUTE_MISMATCH;
    if (heads_q <= 0 || heads_kv <= 0 || seq_len <= 0) return FP4_ERR_INVALID_ARG;
    const int64_t T = x_row->rows, d = x_row->cols, N = (int64_t)(heads_q + 2 * heads_kv) * 128;
    if (wqkv_row->rows != N || wqkv_row->cols != d) return FP4_ERR_UNSUPPORTED_SHAPE;
    if (T <= 0 || T % 128 || N % 256 || d % 256) return FP4_ERR_UNSUPPORTED_SHAPE;
    if (!q || !k || !v || !rope_cos || !rope_sin || !aligned16(q) || !aligned16(k) || !aligned16(v) ||
        !aligned16(rope_cos) || !aligned16(rope_sin))
        return FP4_ERR_INVALID_ARG;
    GemmParams g{};
    fill_operands(g, x_row, wqkv_row);
    g.M = T;
    g.N = N;
    g.K = d;
    g.epi = 3;
    g.q_out = static_cast<uint16_t*>(q);
    g.k_out = static_cast<uint16_t*>(k);
    g.v_out = static_cast<uint16_t*>(v);
    g.rope_cos = rope_cos;
    g.rope_sin = rope_sin;
    g.seq_len = seq_len;
    g.heads_q = heads_q;
    g.heads_kv = heads_kv;
    return launch_gemm(g, reinterpret_cast<cudaStream_t>(stream));
}

int fp4_qkv_rope_bwd(int route, unsigned views, int sr, const void* dq, const void* dk, const void* dv,
                     const float* rope_cos, const float* rope_sin, int64_t rows, int64_t seq_len, int heads_q,
                     int heads_kv, uint64_t sr_seed, uint64_t sr_offset, void* dqkv_tap, fp4_tensor* dqkv_row,
                     fp4_tensor* dqkv_col, void* workspace, size_t workspace_bytes, fp4_stream_t stream) {
    if (heads_q <= 0 || heads_kv <= 0 || seq_len <= 0) return FP4_ERR_INVALID_ARG;
    const int64_t cols = (int64_t)(heads_q + 2 * heads_kv) * 128;
    QuantParams p;
    int rc = prepare_quant(nullptr, true, rows, cols, cols, route, route, views, sr ? FP4_FLAG_SR_ROW : 0, sr_seed,
                           sr_offset, nullptr, dqkv_row, dqkv_col, workspace, workspace_bytes, &p);
    if (rc != FP4_OK || rows == 0) return rc;
    if (!dq || !dk || !dv || !rope_cos || !rope_sin || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) ||
        !aligned16(rope_cos) || !aligned16(rope_sin) || (dqkv_tap && !aligned16(dqkv_tap)))
        return FP4_ERR_INVALID_ARG;
    p.pre = PRE_ROPE_BWD;
    p.rope_src[0] = static_cast<const uint16_t*>(dq);
    p.rope_src[1] = static_cast<const uint16_t*>(dk);
    p.rope_src[2] = static_cast<const uint16_t*>(dv);
    p.rope_cos = rope_cos;
    p.rope_sin = rope_sin;
    p.seq_len = seq_len;
    p.heads_q = heads_q;
    p.heads_kv = heads_kv;
    p.tap = static_cast<uint16_t*>(dqkv_tap);
    return launch_quantize(p, reinterpret_cast<cudaStream_t>(stream));
}

// Workspace of the NVFP4 gated-FFN producers: the amax slots of the tensor
// that is encoded (h [T][f] forward, [da1 | da3] [T][2f] backward), padded to
// 256 bytes, then its bf16 copy unless the caller passes a tap for it.
static size_t swiglu_slots_bytes(int64_t T, int64_t cols) {
    return ((size_t)(1 + T / 128 + cols / 128) * 4 + 255) / 256 * 256;
}

int fp4_swiglu_workspace_bytes(int route, int64_t T, int64_t f, int backward, int with_tap, size_t* bytes) {
    if (!route_ok(route) || !bytes || T < 0 || f < 0) return FP4_ERR_INVALID_ARG;
    if (T % 128 || f % 128) return FP4_ERR_UNSUPPORTED_SHAPE;
    const int64_t cols = backward ? 2 * f : f;
    *bytes = route == FP4_ROUTE_MXFP4 ? 0 : swiglu_slots_bytes(T, cols) + (with_tap ? 0 : (size_t)(T * cols * 2));
    return FP4_OK;
}

// The NVFP4 encode of a gated-FFN tap: the epilogue has already written the
// tap and folded its maxima into the slots (zeroed before the contraction).
static int encode_tap(const uint16_t* tap, int64_t T, int64_t cols, int route, unsigned flags, uint64_t seed,
                      uint64_t offset, fp4_tensor* row, fp4_tensor* col, void* slots, size_t slots_bytes,
                      cudaStream_t s) {
    QuantParams q;
    int rc = prepare_quant(tap, false, T, cols, cols, route, route, 3, flags, seed, offset, nullptr, row, col, slots,
                           slots_bytes, &q);
    if (rc != FP4_OK) return rc;
    q.amax_ready = 1;
    return launch_quantize(q, s);
}

int fp4_swiglu_fwd(const fp4_tensor* x_row, const fp4_tensor* w13_row, int64_t f, void* a1, void* a3,
                   fp4_tensor* h_row, fp4_tensor* h_col, void* h_tap, void* workspace, size_t workspace_bytes,
                   fp4_stream_t stream) {
    int rc;
    if ((rc = check_operand(x_row)) != FP4_OK || (rc = check_operand(w13_row)) != FP4_OK) return rc;
    if (x_row->route != w13_row->route) return FP4_ERR_ROUTE_MISMATCH;
    const int64_t T = x_row->rows, d = x_row->cols;
    if (f <= 0 || w13_row->rows != 2 * f || w13_row->cols != d) return FP4_ERR_UNSUPPORTED_SHAPE;
    if (T % 128 || f % 128 || d % 256 || T <= 0) return FP4_ERR_UNSUPPORTED_SHAPE;
    if (!a1 || !a3 || !aligned16(a1) || !aligned16(a3) || (h_tap && !aligned16(h_tap))) return FP4_ERR_INVALID_ARG;
    const bool mx = x_row->route == FP4_ROUTE_MXFP4;
    if (w13_row->route != FP4_ROUTE_MXFP4 && w13_row->outer_count != 1) return FP4_ERR_INVALID_ARG;
    if ((h_row == nullptr) != (h_col == nullptr)) return FP4_ERR_INVALID_ARG;
    if (h_row && (!view_ok(h_row) || !view_ok(h_col))) return FP4_ERR_INVALID_ARG;
    if (!h_row && !h_tap) return FP4_ERR_INVALID_ARG;
    const bool nv_views = !mx && h_row;
    size_t need = 0;
    if (nv_views) {
        if ((rc = fp4_swiglu_workspace_bytes(x_row->route, T, f, 0, h_tap != nullptr, &need)) != FP4_OK) return rc;
        if (!workspace || workspace_bytes < need || !aligned16(workspace)) return FP4_ERR_WORKSPACE;
        if (!h_row->outer || !h_col->outer) return FP4_ERR_INVALID_ARG;
    }
    GemmParams g{};
    fill_operands(g, x_row, w13_row);
    g.M = T;
    g.N = f;
    g.K = d;
    g.epi = 1;
    g.f = f;
    g.a1 = static_cast<uint16_t*>(a1);
    g.a3 = static_cast<uint16_t*>(a3);
    g.tap0 = static_cast<uint16_t*>(h_tap);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (mx && h_row) {
        g.quantize = 1;
        g.q_row_codes = static_cast<uint8_t*>(h_row->codes);
        g.q_row_scales = static_cast<uint8_t*>(h_row->scales);
        g.q_col_codes = static_cast<uint8_t*>(h_col->codes);
        g.q_col_scales = static_cast<uint8_t*>(h_col->scales);
        set_view(h_row, T, f, FP4_ROUTE_MXFP4);
        set_view(h_col, f, T, FP4_ROUTE_MXFP4);
        return launch_gemm(g, s);
    }
    if (!nv_views) return launch_gemm(g, s);
    // NVFP4: every strip factor depends on values from the whole strip (all f
    // columns for the row view, all T tokens for the column view), so h goes
    // through one bf16 copy: the epilogue writes it and folds its maxima, the
    // encoder reads it once
    const size_t sb = swiglu_slots_bytes(T, f);
    uint32_t* slots = static_cast<uint32_t*>(workspace);
    g.tap0 = h_tap ? static_cast<uint16_t*>(h_tap) : reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(workspace) + sb);
    g.amax_ws = slots;
    if (cudaMemsetAsync(slots, 0, sb, s) != cudaSuccess) return FP4_ERR_CUDA;
    if ((rc = launch_gemm(g, s)) != FP4_OK) return rc;
    return encode_tap(g.tap0, T, f, x_row->route, 0, 0, 0, h_row, h_col, slots, sb, s);
}

int fp4_swiglu_bwd(const fp4_tensor* dy2_row, const fp4_tensor* w2_col, int64_t f, const void* a1, const void* a3,
                   uint64_t sr_seed, uint64_t sr_offset, fp4_tensor* da13_row, fp4_tensor* da13_col, void* dh_tap,
                   void* da13_tap, void* workspace, size_t workspace_bytes, fp4_stream_t stream) {
    int rc;
    if ((rc = check_operand(dy2_row)) != FP4_OK || (rc = check_operand(w2_col)) != FP4_OK) return rc;
    if (dy2_row->route != w2_col->route) return FP4_ERR_ROUTE_MISMATCH;
    const int64_t T = dy2_row->rows, d = dy2_row->cols;
    if (f <= 0 || w2_col->rows != f || w2_col->cols != d) return FP4_ERR_UNSUPPORTED_SHAPE;
    if (T % 128 || f % 128 || d % 256 || T <= 0) return FP4_ERR_UNSUPPORTED_SHAPE;
    if (!a1 || !a3 || !aligned16(a1) || !aligned16(a3) || (dh_tap && !aligned16(dh_tap)) ||
        (da13_tap && !aligned16(da13_tap)))
        return FP4_ERR_INVALID_ARG;
    const bool mx = dy2_row->route == FP4_ROUTE_MXFP4;
    if ((da13_row == nullptr) != (da13_col == nullptr)) return FP4_ERR_INVALID_ARG;
    if (da13_row && (!view_ok(da13_row) || !view_ok(da13_col))) return FP4_ERR_INVALID_ARG;
    if (!da13_row && !da13_tap) return FP4_ERR_INVALID_ARG;
    const bool nv_views = !mx && da13_row;
    size_t need = 0;
    if (nv_views) {
        if ((rc = fp4_swiglu_workspace_bytes(dy2_row->route, T, f, 1, da13_tap != nullptr, &need)) != FP4_OK)
            return rc;
        if (!workspace || workspace_bytes < need || !aligned16(workspace)) return FP4_ERR_WORKSPACE;
        if (!da13_row->outer || !da13_col->outer) return FP4_ERR_INVALID_ARG;
    }
    GemmParams g{};
    fill_operands(g, dy2_row, w2_col);
    g.M = T;
    g.N = f;
    g.K = d;
    g.epi = 2;
    g.f = f;
    g.a1 = const_cast<uint16_t*>(static_cast<const uint16_t*>(a1));
    g.a3 = const_cast<uint16_t*>(static_cast<const uint16_t*>(a3));
    g.tap0 = static_cast<uint16_t*>(dh_tap);
    g.tap1 = static_cast<uint16_t*>(da13_tap);
    g.seed = sr_seed;
    g.offset = sr_offset;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (mx && da13_row) {
        g.quantize = 1;
        g.q_row_codes = static_cast<uint8_t*>(da13_row->codes);
        g.q_row_scales = static_cast<uint8_t*>(da13_row->scales);
        g.q_col_codes = static_cast<uint8_t*>(da13_col->codes);
        g.q_col_scales = static_cast<uint8_t*>(da13_col->scales);
        set_view(da13_row, T, 2 * f, FP4_ROUTE_MXFP4);
        set_view(da13_col, 2 * f, T, FP4_ROUTE_MXFP4);
        return launch_gemm(g, s);
    }
    if (!nv_views) return launch_gemm(g, s);
    // NVFP4: [da1 | da3] through one bf16 copy, its maxima from the epilogue
    const size_t sb = swiglu_slots_bytes(T, 2 * f);
    uint32_t* slots = static_cast<uint32_t*>(workspace);
    g.tap1 = da13_tap ? static_cast<uint16_t*>(da13_tap)
                      : reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(workspace) + sb);
    g.amax_ws = slots;
    if (cudaMemsetAsync(slots, 0, sb, s) != cudaSuccess) return FP4_ERR_CUDA;
    if ((rc = launch_gemm(g, s)) != FP4_OK) return rc;
    return encode_tap(g.tap1, T, 2 * f, dy2_row->route, FP4_FLAG_SR_ROW, sr_seed, sr_offset, da13_row, da13_col,
                      slots, sb, s);
}

int fp4_linear_fprop(const fp4_tensor* x_row, const fp4_tensor* w_row, void* y, int out_dtype, float beta,
                     fp4_stream_t stream) {
    return linear(x_row, w_row, y, out_dtype, beta, stream);
}

int fp4_linear_dgrad(const fp4_tensor* dy_row, const fp4_tensor* w_col, void* dx, int out_dtype, float beta,
                     fp4_stream_t stream) {
    return linear(dy_row, w_col, dx, out_dtype, beta, stream);
}

int fp4_linear_dgrad_rmsnorm(const fp4_tensor* dy_row, const fp4_tensor* w_col, void* dx, const void* r_prime,
                             const float* rstd, const void* g, float* part, fp4_stream_t stream) {
    if (!r_prime || !rstd || !g || !part || !aligned16(r_prime) || !aligned16(g) ||
        (reinterpret_cast<uintptr_t>(rstd) & 3u) || (reinterpret_cast<uintptr_t>(part) & 3u))
        return FP4_ERR_INVALID_ARG;
    const RmsTerms rms{r_prime, rstd, g, part};
    return linear(dy_row, w_col, dx, FP4_OUT_BF16, 0.0f, stream, &rms);
}

int fp4_linear_wgrad(const fp4_tensor* dy_col, const fp4_tensor* x_col, float* dw, float beta, fp4_stream_t stream) {
    return linear(dy_col, x_col, dw, FP4_OUT_F32, beta, stream);
}

// ---------------------------------------------------------------------------
// Allocation-free quantizer entry point.
//
// Some callers cannot call cudaMalloc at the moment they quantize: a runtime
// that owns all device memory through its own pool and forbids raw
// allocations, a serving process that reserves every byte at start-up, or code
// on a latency-critical path where cudaMalloc's implicit device
// synchronisation is not acceptable.  fp4_quantize_noalloc serves them by
// taking the NVFP4 amax scratch from a fixed array in static device memory
// instead of a caller-provided workspace.
//
// The array is FP4_NOALLOC_SCRATCH_BYTES (16 KiB) per GPU that loads this
// library, held until the process exits, shared by every call on that GPU.
// Each call clears the slots it uses before its amax pass, but the array keeps
// the last call's contents, so calls whose kernels overlap on the GPU (other
// streams, or concurrent host threads) race on it and must be serialised by
// the caller.
#define FP4_NOALLOC_SCRATCH_BYTES 16384
static __device__ __align__(256) uint32_t g_noalloc_scratch[FP4_NOALLOC_SCRATCH_BYTES / 4];

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// with cudaGetSymbolAddress once per device (with that device current) and
// cached.
static void* noalloc_scratch(void) {
    static std::mutex mu;
    static void* addr[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess) return nullptr;
        addr[dev] = ptr;
    }
    return addr[dev];
}

int fp4_quantize_noalloc(const void* x, int64_t rows, int64_t cols, int64_t ld, int route, unsigned views,
                         unsigned flags, uint64_t sr_seed, uint64_t sr_offset, const int8_t* hadamard_signs,
                         fp4_tensor* row_out, fp4_tensor* col_out, fp4_stream_t stream) {
    size_t need = 0;
    int rc = fp4_quantize_workspace_bytes(route, rows, cols, views, flags, &need);
    if (rc != FP4_OK) return rc;
    // Every argument check of fp4_quantize comes first (on copies of the
    // views, with a stand-in workspace of the needed size that is never
    // touched), so an invalid call fails the same way as there; only then is
    // the shape held against the scratch array's size.
    {
        fp4_tensor r_chk = row_out ? *row_out : fp4_tensor{};
        fp4_tensor c_chk = col_out ? *col_out : fp4_tensor{};
        QuantParams chk;
        static uint32_t stand_in;
        rc = prepare_quant(x, false, rows, cols, ld, route, route, views, flags, sr_seed, sr_offset, hadamard_signs,
                           row_out ? &r_chk : nullptr, col_out ? &c_chk : nullptr, need ? &stand_in : nullptr, need,
                           &chk);
        if (rc != FP4_OK) return rc;
    }
    if (need > FP4_NOALLOC_SCRATCH_BYTES) return FP4_ERR_WORKSPACE;
    void* ws = nullptr;
    if (need > 0 && rows > 0 && cols > 0) {
        ws = noalloc_scratch();
        if (!ws) return FP4_ERR_CUDA;
    }
    return fp4_quantize(x, rows, cols, ld, route, views, flags, sr_seed, sr_offset, hadamard_signs, row_out, col_out,
                        ws, need, stream);
}

int fp4_status(fp4_stream_t stream, int* code) {
    if (!code) return FP4_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int a = 0, b = 0, r;
    if ((r = quant_status(s, &a, false)) != FP4_OK) return r;
    if ((r = gemm_status(s, &b, false)) != FP4_OK) return r;
    *code = a ? a : b;
    return FP4_OK;
}

int fp4_set_wait_limit(uint64_t cycles) {
    gemm_set_wait_limit(cycles);
    return FP4_OK;
}

int fp4_test_skip_accumulator_release(int enable) {
    gemm_test_skip_first_release(enable);
    return FP4_OK;
}

int fp4_status_reset(fp4_stream_t stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int r;
    if ((r = quant_status(s, nullptr, true)) != FP4_OK) return r;
    return gemm_status(s, nullptr, true);
}

}  // extern "C"
