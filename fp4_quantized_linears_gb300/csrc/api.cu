// api.cu -- the extern "C" boundary of libfp4lin (declared in include/fp4lin.h).
//
// Host-side argument validation and dispatch only: every step of the path
// runs in the kernels of quantize.cu / gemm.cu / fused.cu.  Nothing here
// allocates or synchronises, except fp4_status() which reads the device
// status words.
#include <cuda_runtime.h>
#include <stdint.h>

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
    (void)views;
    (void)flags;
    if (!route_ok(route) || !bytes || rows < 0 || cols < 0) return FP4_ERR_INVALID_ARG;
    if (rows % 128 || cols % 128) return FP4_ERR_UNSUPPORTED_SHAPE;
    *bytes = route == FP4_ROUTE_MXFP4 ? 0 : (size_t)(1 + rows / 128 + cols / 128) * 4;
    return FP4_OK;
}

int fp4_quantize(const void* x, int64_t rows, int64_t cols, int64_t ld, int route, unsigned views, unsigned flags,
                 uint64_t sr_seed, uint64_t sr_offset, const int8_t* hadamard_signs, fp4_tensor* row_out,
                 fp4_tensor* col_out, void* workspace, size_t workspace_bytes, fp4_stream_t stream) {
    if (!route_ok(route)) return FP4_ERR_INVALID_ARG;
    if ((views & ~3u) || views == 0 || (flags & ~7u)) return FP4_ERR_INVALID_ARG;
    if (rows < 0 || cols < 0 || ld < cols) return FP4_ERR_INVALID_ARG;
    if (rows % 128 || cols % 128) return FP4_ERR_UNSUPPORTED_SHAPE;
    if ((flags & FP4_FLAG_WEIGHT_2D) && (flags & (FP4_FLAG_SR_ROW | FP4_FLAG_HADAMARD_COL)))
        return FP4_ERR_ROUTE_MISMATCH;
    if ((flags & FP4_FLAG_HADAMARD_COL) && route != FP4_ROUTE_MXFP4) return FP4_ERR_ROUTE_MISMATCH;
    const bool do_row = views & FP4_VIEW_ROW, do_col = views & FP4_VIEW_COL;
    if ((do_row && !row_out) || (do_col && !col_out)) return FP4_ERR_INVALID_ARG;
    const int32_t oc_row = outer_count_of(route, rows, flags), oc_col = outer_count_of(route, cols, flags);
    for (int v = 0; v < 2; ++v) {
        fp4_tensor* t = v == 0 ? (do_row ? row_out : nullptr) : (do_col ? col_out : nullptr);
        if (!t) continue;
        if (!t->codes || !t->scales || !aligned16(t->codes) || !aligned16(t->scales)) return FP4_ERR_INVALID_ARG;
        if (route != FP4_ROUTE_MXFP4 && !t->outer) return FP4_ERR_INVALID_ARG;
    }
    uint32_t sign_mask = 0;
    if (flags & FP4_FLAG_HADAMARD_COL) {
        if (!hadamard_signs) return FP4_ERR_INVALID_ARG;
        for (int j = 0; j < 16; ++j) {
            if (hadamard_signs[j] != 1 && hadamard_signs[j] != -1) return FP4_ERR_INVALID_ARG;
            if (hadamard_signs[j] < 0) sign_mask |= 1u << j;
        }
    }
    size_t need = 0;
    fp4_quantize_workspace_bytes(route, rows, cols, views, flags, &need);
    if (need > 0 && (!workspace || workspace_bytes < need)) return FP4_ERR_WORKSPACE;
    if (rows > 0 && cols > 0 && (!x || !aligned16(x) || ld % 8)) return FP4_ERR_INVALID_ARG;

    if (do_row) {
        row_out->rows = rows;
        row_out->cols = cols;
        row_out->route = route;
        row_out->outer_count = oc_row;
    }
    if (do_col) {
        col_out->rows = cols;
        col_out->cols = rows;
        col_out->route = route;
        col_out->outer_count = oc_col;
    }
    if (rows == 0 || cols == 0) return FP4_OK;

    QuantParams p{};
    p.x = static_cast<const uint16_t*>(x);
    p.R = rows;
    p.C = cols;
    p.ld = ld;
    p.route = route;
    p.views = views;
    p.flags = flags;
    p.seed = sr_seed;
    p.offset = sr_offset;
    p.sign_mask = sign_mask;
    if (do_row) {
        p.row_codes = static_cast<uint8_t*>(row_out->codes);
        p.row_scales = static_cast<uint8_t*>(row_out->scales);
        p.row_outer = row_out->outer;
    }
    if (do_col) {
        p.col_codes = static_cast<uint8_t*>(col_out->codes);
        p.col_scales = static_cast<uint8_t*>(col_out->scales);
        p.col_outer = col_out->outer;
    }
    p.amax_ws = static_cast<uint32_t*>(workspace);
    return launch_quantize(p, reinterpret_cast<cudaStream_t>(stream));
}

static int linear(const fp4_tensor* a, const fp4_tensor* b, void* c, int out_dtype, float beta, fp4_stream_t stream) {
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
    return launch_gemm(g, reinterpret_cast<cudaStream_t>(stream));
}

int fp4_linear_fprop(const fp4_tensor* x_row, const fp4_tensor* w_row, void* y, int out_dtype, float beta,
                     fp4_stream_t stream) {
    return linear(x_row, w_row, y, out_dtype, beta, stream);
}

int fp4_linear_dgrad(const fp4_tensor* dy_row, const fp4_tensor* w_col, void* dx, int out_dtype, float beta,
                     fp4_stream_t stream) {
    return linear(dy_row, w_col, dx, out_dtype, beta, stream);
}

int fp4_linear_wgrad(const fp4_tensor* dy_col, const fp4_tensor* x_col, float* dw, float beta, fp4_stream_t stream) {
    return linear(dy_col, x_col, dw, FP4_OUT_F32, beta, stream);
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

int fp4_status_reset(fp4_stream_t stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int r;
    if ((r = quant_status(s, nullptr, true)) != FP4_OK) return r;
    return gemm_status(s, nullptr, true);
}

}  // extern "C"
