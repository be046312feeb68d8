/*
 * fp4lin.h -- C ABI of the format-aware FP4 linear-layer boundary
 * ("Format-Aware Fusion for Fast FP4 Pretraining"), hand-written CUDA for
 * sm_103a (GB300).
 *
 * Two halves, as in the paper's boundary contract (Sec. 3.1):
 *   producers  fp4_quantize(_hybrid), fp4_swiglu_fwd/bwd, fp4_residual_rmsnorm_fwd/bwd(_parts),
 *              fp4_qkv_rope_fwd/bwd turn BF16 tensors into E2M1 codes plus
 *              scales (or the BF16 attention inputs) in the physical
 *              layout the next contraction consumes;
 *   consumers  fp4_linear_fprop/dgrad/wgrad (and fp4_linear_dgrad_rmsnorm,
 *              a Dgrad that also emits the next RMSNorm backward's row
 *              terms), block-scaled tcgen05 GEMMs.
 *
 * General conventions
 *  - Every pointer named "device" is caller-owned CUDA device memory.  The
 *    library never allocates, frees or synchronises; each call enqueues its
 *    kernels on `stream` and returns.  Host pointers are read during the call
 *    only.
 *  - Every call returns an fp4 status code (FP4_OK == 0).  Argument errors are
 *    detected on the host before anything is enqueued.  Device-side conditions
 *    (non-finite input, a bounded wait that ran out) set a sticky device status
 *    word that fp4_status() reads.
 *  - BF16 tensors are row-major with a leading dimension `ld` in elements
 *    (ld >= cols, ld % 8 == 0, base 16-byte aligned).
 *
 * Quantized tensor layout (fp4_tensor)
 *  A quantized view is stored K-major: `rows` stored rows of `cols` values,
 *  where cols is the reduction axis K of the consuming contraction.
 *   - The row-facing view Q_r(T) of a logical R x C tensor T has rows = R,
 *     cols = C.  The column-facing view Q_c(T) has rows = C, cols = R (it holds
 *     T transposed).  (Sec. 2.3, Eqs. 4-6.)
 *   - codes: rows * cols / 2 bytes; stored row r occupies bytes
 *     [r * cols/2, (r+1) * cols/2); value k of the row sits in byte k/2, in the
 *     low nibble when k is even and the high nibble when k is odd.  A nibble is
 *     an E2M1 code: bit 3 sign, bits 2..1 exponent, bit 0 fraction.
 *   - scales: one byte per block of bs values along a stored row (bs = 32,
 *     E8M0, for MXFP4; bs = 16, E4M3, for NVFP4).  The bytes are grouped in
 *     512-byte atoms of 128 stored rows x 4 consecutive blocks:
 *       atom  = (r / 128) * (cols / (4 * bs)) + (j / 4)     j = k / bs
 *       byte  = atom * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + (j % 4)
 *     which is the layout the tcgen05 block-scaled MMA reads after a
 *     32x128b.warpx4 copy into tensor memory.  scale bytes = rows * cols / bs.
 *   - outer: NVFP4 encode factors S_enc (binary32).  outer_count = 1 for global
 *     NVFP4 and for every 2D16 weight; rows / 128 (one per 128-row strip of the
 *     stored view) for CTA-local activations and gradients; 0 and NULL for
 *     MXFP4.  Decoded value = code * block scale / S_enc.
 *  Shape rules: rows % 128 == 0 and cols % 128 == 0.
 */
#ifndef FP4LIN_H
#define FP4LIN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FP4LIN_VERSION 110 /* 1.1.0 */

/* Exported symbols keep default visibility (the library builds with hidden
 * visibility for everything else). */
#if defined(__GNUC__)
#define FP4_API __attribute__((visibility("default")))
#else
#define FP4_API
#endif

/* A cudaStream_t.  NULL selects the legacy default stream. */
typedef struct CUstream_st* fp4_stream_t;

/* Status codes. */
enum fp4_status_code {
    FP4_OK = 0,
    FP4_ERR_INVALID_ARG = 1,       /* null pointer, bad enum, bad leading dimension */
    FP4_ERR_UNSUPPORTED_SHAPE = 2, /* a dimension breaks the shape rules */
    FP4_ERR_ROUTE_MISMATCH = 3,    /* operands of different routes / a flag the route forbids */
    FP4_ERR_WORKSPACE = 4,         /* workspace missing or smaller than required */
    FP4_ERR_CUDA = 5,              /* a CUDA runtime call failed */
    FP4_ERR_TIMEOUT = 6,           /* (device) a bounded pipeline wait ran out */
    FP4_ERR_NONFINITE = 7          /* (device) a quantizer saw Inf or NaN */
};

/* Routes: the three scale contracts of Sec. 2.2. */
enum fp4_route {
    FP4_ROUTE_MXFP4 = 0,        /* 32-value blocks, upward-rounded E8M0 scales (Sec. 2.2.1) */
    FP4_ROUTE_NVFP4_GLOBAL = 1, /* 16-value E4M3 blocks under one tensor-amax factor (Sec. 2.2.2) */
    FP4_ROUTE_NVFP4_LOCAL = 2   /* 16-value E4M3 blocks under per-128-strip factors (Sec. 2.2.2, Eq. 3) */
};

/* Views requested from a producer (bit mask). */
enum fp4_view { FP4_VIEW_ROW = 1, FP4_VIEW_COL = 2 };

/* Producer flags (bit mask). */
enum fp4_flag {
    FP4_FLAG_WEIGHT_2D = 1,     /* 2D32 (MX, adaptive finer scale when a/s < 0.87) or 2D16 (NV) weight
                                   encoding shared by both views (Sec. 2.4, Eqs. 7-8) */
    FP4_FLAG_SR_ROW = 2,        /* stochastic rounding of the row view (Sec. 2.5, Eq. 9) */
    FP4_FLAG_HADAMARD_COL = 4,  /* fixed-sign H32 on the column view before quantization
                                   (Sec. 2.5, Eq. 10; MXFP4 only) */
    FP4_FLAG_HADAMARD16_COL = 8 /* fixed-sign H16 on the column view before quantization
                                   (Sec. 2.5: the NVFP4 Wgrad transform; with every sign
                                   +1 the plain H16 of the operand-wise hybrid, Sec. 3.3);
                                   any route */
};

/* GEMM output element types. */
enum fp4_out_dtype { FP4_OUT_F32 = 0, FP4_OUT_BF16 = 1 };

/* One quantized view.  All pointers are caller-owned device memory sized by
 * fp4_tensor_bytes(); the producer fills every field. */
typedef struct fp4_tensor {
    void* codes;         /* device, rows * cols / 2 bytes */
    void* scales;        /* device, rows * cols / bs bytes, atom layout above */
    float* outer;        /* device, outer_count binary32 S_enc values, or NULL */
    int64_t rows;        /* stored rows (M or N of the consumer) */
    int64_t cols;        /* stored columns (K of the consumer) */
    int32_t route;       /* enum fp4_route */
    int32_t outer_count; /* 0, 1 or rows / 128 */
} fp4_tensor;

/* Library version (FP4LIN_VERSION). */
FP4_API int fp4_version(void);

/* Human-readable name of a status code (static string). */
FP4_API const char* fp4_status_string(int code);

/* Sizes of one quantized view with `rows` stored rows of `cols` values:
 * codes and scale bytes, and the number of S_enc values (0 for MXFP4; 1 for
 * global NVFP4 or with FP4_FLAG_WEIGHT_2D; rows / 128 for CTA-local).
 * Host only; nothing is enqueued. */
FP4_API int fp4_tensor_bytes(int route, int64_t rows, int64_t cols, unsigned flags, size_t* codes_bytes,
                     size_t* scale_bytes, int32_t* outer_count);

/* Workspace bytes fp4_quantize needs for this route, shape, views and flags
 * (0 for MXFP4; (1 + rows/128 + cols/128) * 4 for NVFP4, the amax slots of the
 * outer-factor pre-pass, plus 4 when the column view is H16-transformed).
 * Host only. */
FP4_API int fp4_quantize_workspace_bytes(int route, int64_t rows, int64_t cols, unsigned views, unsigned flags,
                                 size_t* bytes);

/* Quantize a BF16 tensor x (device, rows x cols, leading dimension ld) into
 * the requested views (Sec. 2.2-2.5, Sec. 3.1).
 *  route          enum fp4_route
 *  views          FP4_VIEW_ROW and/or FP4_VIEW_COL
 *  flags          FP4_FLAG_WEIGHT_2D: one shared 2D encoding (views decode
 *                 identically, Eq. 8; no SR, no H32);
 *                 FP4_FLAG_SR_ROW: Philox4x32-10 stochastic rounding of the row
 *                 view only; element i = r * cols + c of the logical tensor uses
 *                 16 bits of Philox(key = sr_seed, counter = (i/8, sr_offset)),
 *                 word (i%8)/2, low half for even i;
 *                 FP4_FLAG_HADAMARD_COL: H32 = Sylvester H32 x diag(signs
 *                 repeated over both halves) / sqrt(32) on every aligned
 *                 32-value block of the column view (MXFP4 only);
 *                 FP4_FLAG_HADAMARD16_COL: H16 = Sylvester H16 x diag(signs)
 *                 / 4 on every aligned 16-value block of the column view (any
 *                 route; an NVFP4 view then takes its outer factors from the
 *                 transformed values).  The two are exclusive, and neither
 *                 combines with WEIGHT_2D.
 *  hadamard_signs host array of 16 int8 values, each +1 or -1 (read only when
 *                 a Hadamard flag is set; all +1 gives plain H16).
 *  row_out/col_out caller-filled codes/scales/outer pointers for each requested
 *                 view (may be NULL for a view not requested); the call sets
 *                 rows, cols, route and outer_count.
 *  workspace      device scratch of fp4_quantize_workspace_bytes() bytes
 *                 (NULL allowed when that is 0); its contents are overwritten.
 * Errors: FP4_ERR_INVALID_ARG, FP4_ERR_UNSUPPORTED_SHAPE (rows or cols not a
 * multiple of 128), FP4_ERR_ROUTE_MISMATCH (SR with WEIGHT_2D, H32 on NVFP4 or
 * with WEIGHT_2D), FP4_ERR_WORKSPACE, FP4_ERR_CUDA (launch failure). */
FP4_API int fp4_quantize(const void* x, int64_t rows, int64_t cols, int64_t ld, int route, unsigned views,
                 unsigned flags, uint64_t sr_seed, uint64_t sr_offset, const int8_t* hadamard_signs,
                 fp4_tensor* row_out, fp4_tensor* col_out, void* workspace, size_t workspace_bytes,
                 fp4_stream_t stream);

/* The operand-wise hybrid producer ("Format-Aware Fusion for Fast FP4
 * Pretraining", Sec. 3.3): one read of x emits the row view under row_route
 * and the column view under col_route.  For the hybrid linear, the gradient
 * dY takes (NVFP4_LOCAL row view with FP4_FLAG_SR_ROW -> Dgrad, MXFP4 column
 * view with FP4_FLAG_HADAMARD16_COL (plain, all signs +1) or
 * FP4_FLAG_HADAMARD_COL -> Wgrad) and the weight W takes (MXFP4 2D32 row view
 * -> Fprop, NVFP4_LOCAL 2D16 column view under the tensor factor -> Dgrad),
 * with FP4_FLAG_WEIGHT_2D giving each view its own format's 2D encoding.
 * Every argument is as for fp4_quantize, with each view's rules taken from
 * its own route (H32 needs an MXFP4 column view; an NVFP4 view needs an
 * `outer` array).  fp4_quantize(route) is this call with both routes equal.
 * workspace: fp4_quantize_hybrid_workspace_bytes() bytes. */
FP4_API int fp4_quantize_hybrid(const void* x, int64_t rows, int64_t cols, int64_t ld, int row_route, int col_route,
                                unsigned views, unsigned flags, uint64_t sr_seed, uint64_t sr_offset,
                                const int8_t* hadamard_signs, fp4_tensor* row_out, fp4_tensor* col_out,
                                void* workspace, size_t workspace_bytes, fp4_stream_t stream);

/* Workspace bytes of fp4_quantize_hybrid: 4 bytes per amax slot when any
 * requested view is NVFP4 (1 + rows/128 + cols/128 slots, one more when the
 * NVFP4 column view is H16-transformed), else 0.  Host only. */
FP4_API int fp4_quantize_hybrid_workspace_bytes(int row_route, int col_route, int64_t rows, int64_t cols,
                                                unsigned views, unsigned flags, size_t* bytes);

/* fp4_quantize without a workspace argument, for callers that cannot
 * allocate device memory when they quantize (a runtime whose pool owns all
 * device memory, a server that reserves everything at start-up, a path that
 * cannot afford cudaMalloc's implicit synchronisation).  The paper has no
 * counterpart to this call; it is a deployment convenience.
 *  - Same arguments, results and errors as fp4_quantize, except that the NVFP4
 *    amax scratch comes from a 16 KiB array in static device memory that
 *    every GPU loading this library holds until exit.  A shape needing more
 *    (1 + rows/128 + cols/128 > 4096 slots) returns FP4_ERR_WORKSPACE.
 *  - The call allocates nothing and frees nothing.
 *  - All calls on a GPU share the array and each clears it before use: calls
 *    whose kernels overlap on the GPU race, so the caller must order them
 *    (one stream, or explicit synchronisation).
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current); make that first call
 *    before any stream capture begins. */
FP4_API int fp4_quantize_noalloc(const void* x, int64_t rows, int64_t cols, int64_t ld, int route, unsigned views,
                                 unsigned flags, uint64_t sr_seed, uint64_t sr_offset, const int8_t* hadamard_signs,
                                 fp4_tensor* row_out, fp4_tensor* col_out, fp4_stream_t stream);

/* The three contractions of Sec. 2.3 (Eqs. 4-6).  Each computes
 *   C[m][n] = alpha(m, n) * sum_k A_hat[m][k] * B_hat[n][k] + beta * C[m][n]
 * over K-major operands with FP32 tensor-core accumulation, where A_hat/B_hat
 * are code * block scale and alpha = 1 (MXFP4) or 1 / (S_enc,A * S_enc,B)
 * with the factor of each operand's row strip (NVFP4; the CTA-local epilogue
 * of Sec. 2.2.2).  Output C is row-major [M][N] (ldc = N) in out_dtype; beta
 * = 0 does not read C.  A.cols == B.cols, M % 128 == 0, N % 128 == 0,
 * K % 256 == 0; both operands of one route.
 *   fprop:  Y  [T x out] = Q_r(X)  [T x in]  . Q_r(W)  [out x in]^T
 *   dgrad:  dX [T x in]  = Q_r(dY) [T x out] . Q_c(W)  [in x out]^T
 *   wgrad:  dW [out x in]= Q_c(dY) [out x T] . Q_c(X)  [in x T]^T   (FP32 only) */
FP4_API int fp4_linear_fprop(const fp4_tensor* x_row, const fp4_tensor* w_row, void* y, int out_dtype, float beta,
                     fp4_stream_t stream);
FP4_API int fp4_linear_dgrad(const fp4_tensor* dy_row, const fp4_tensor* w_col, void* dx, int out_dtype, float beta,
                     fp4_stream_t stream);
FP4_API int fp4_linear_wgrad(const fp4_tensor* dy_col, const fp4_tensor* x_col, float* dw, float beta,
                     fp4_stream_t stream);

/* QKV producer with RoPE ("Format-Aware Fusion for Fast FP4 Pretraining",
 * Sec. 3.2: the Q/K projection applies RoPE and the layout attention
 * consumes).  One contraction qkv = bf16(X Wqkv^T) (x_row: Q_r(X) [T][d];
 * wqkv_row: Q_r(Wqkv) [(heads_q + 2 heads_kv) * 128][d], same route) whose
 * epilogue writes head-major bf16
 *   q [heads_q][T][128], k [heads_kv][T][128]  turned by RoPE,
 *   v [heads_kv][T][128]                       copied,
 * with the QKV columns laid out [Q heads | K heads | V heads] and heads of
 * 128 values.  RoPE (the rotate-half pairs (i, i + 64) of each head, token t
 * at position p = t mod seq_len): with c = rope_cos[p][i], s = rope_sin[p][i]
 * (device binary32 tables [seq_len][64], e.g. cos/sin of p theta^(-i/64)),
 *   y_i = bf16(fl32(fl32(x_i c) - fl32(x_{i+64} s))),
 *   y_{i+64} = bf16(fl32(fl32(x_{i+64} c) + fl32(x_i s))).
 * T a multiple of 128, (heads_q + 2 heads_kv) * 128 a multiple of 256, d a
 * multiple of 256; q, k, v, tables 16-byte aligned.  Errors as
 * fp4_linear_fprop, FP4_ERR_UNSUPPORTED_SHAPE for other shapes. */
FP4_API int fp4_qkv_rope_fwd(const fp4_tensor* x_row, const fp4_tensor* wqkv_row, const float* rope_cos,
                             const float* rope_sin, int64_t seq_len, int heads_q, int heads_kv, void* q, void* k,
                             void* v, fp4_stream_t stream);

/* The matching backward producer (Sec. 3.2: inverse layout and RoPE combined
 * with the QKV gradient production).  From the head-major gradients dq, dk,
 * dv (device bf16, layouts as the forward's outputs) it forms the QKV-layout
 * gradient dqkv [rows][(heads_q + 2 heads_kv) * 128] -- dq and dk turned back
 * by the transposed rotation
 *   g_i = bf16(fl32(fl32(a_i c) + fl32(a_{i+64} s))),
 *   g_{i+64} = bf16(fl32(fl32(a_{i+64} c) - fl32(a_i s))),
 * dv copied -- and quantizes it in the same pass under `route` into the
 * views requested (row view with FP4_FLAG_SR_ROW semantics under sr_seed /
 * sr_offset when `sr` is non-zero: the QKV Dgrad operand; column view: the
 * QKV Wgrad operand).  dqkv_tap (optional, device bf16 [rows][...]) receives
 * the gradient that was quantized.  workspace: fp4_quantize_workspace_bytes()
 * bytes for (route, rows, (heads_q + 2 heads_kv) * 128).  Errors as
 * fp4_quantize. */
FP4_API int fp4_qkv_rope_bwd(int route, unsigned views, int sr, const void* dq, const void* dk, const void* dv,
                             const float* rope_cos, const float* rope_sin, int64_t rows, int64_t seq_len, int heads_q,
                             int heads_kv, uint64_t sr_seed, uint64_t sr_offset, void* dqkv_tap,
                             fp4_tensor* dqkv_row, fp4_tensor* dqkv_col, void* workspace, size_t workspace_bytes,
                             fp4_stream_t stream);

/* Fused gated-FFN forward producer (Sec. 3.2).  One contraction over the
 * paired projections,
 *   a1 = X W1^T, a3 = X W3^T     (x_row: Q_r(X) [T][d]; w13_row: Q_r of the
 *                                 stacked [W1; W3] [2f][d], rows [0,f) = W1),
 * whose epilogue writes the retained BF16 values a1, a3 (device bf16
 * [T][f], the exact values autograd needs) and h = bf16(fl32(silu(a1)) * a3),
 * emitted as Q_r(h) [T][f] (the W2 Fprop input) and Q_c(h) [f][T] (the W2
 * Wgrad input) into h_row / h_col (both or neither):
 *   MXFP4  directly from the epilogue; workspace unused (may be NULL);
 *   NVFP4  every outer factor of h needs its whole strip's maximum (all f
 *          columns for the row view, all T tokens for the column view), so
 *          h passes through one bf16 copy: the epilogue writes it and folds
 *          its strip and tensor maxima into slots in `workspace`, then the
 *          encoder reads it once (no separate maximum pass).  The copy is
 *          h_tap when given, else it lives in the workspace;
 *          fp4_swiglu_workspace_bytes gives the size (caller-owned device
 *          memory, 16-byte aligned; FP4_ERR_WORKSPACE if smaller).
 * With h_row = h_col = NULL only h_tap (device bf16 [T][f]) is written.
 * T % 128 == 0, f % 128 == 0, d % 256 == 0.  Errors: FP4_ERR_INVALID_ARG,
 * FP4_ERR_UNSUPPORTED_SHAPE, FP4_ERR_ROUTE_MISMATCH, FP4_ERR_WORKSPACE,
 * FP4_ERR_CUDA. */
FP4_API int fp4_swiglu_fwd(const fp4_tensor* x_row, const fp4_tensor* w13_row, int64_t f, void* a1, void* a3,
                           fp4_tensor* h_row, fp4_tensor* h_col, void* h_tap, void* workspace,
                           size_t workspace_bytes, fp4_stream_t stream);

/* Fused gated-FFN backward producer (Sec. 3.2).  The W2 data-gradient
 * contraction dh = dY2 W2 (dy2_row: Q_r(dY2) [T][d]; w2_col: Q_c(W2) [f][d])
 * with, in its epilogue, dh = bf16(acc) and the SiLU derivative from the
 * retained a1, a3 (device bf16 [T][f]):
 *   da1 = bf16(dh * a3 * s * (1 + a1 * (1 - s))),  da3 = bf16(dh * a1 * s),
 *   s = 1 / (1 + exp(-a1)),
 * laid out as one logical tensor da13 = [da1 | da3] of [T][2f], emitted as
 * Q_r(da13) [T][2f] with stochastic rounding (Philox under sr_seed /
 * sr_offset, element index t * 2f + c; the W1/W3 Dgrad operand, K = 2f) and
 * Q_c(da13) [2f][T] (the W1/W3 Wgrad operand) into da13_row / da13_col:
 *   MXFP4  directly from the epilogue;
 *   NVFP4  through one bf16 copy of da13 (da13_tap, else in the workspace)
 *          whose maxima the epilogue folds, as for the forward
 *          (fp4_swiglu_workspace_bytes with backward = 1).
 * dh_tap (bf16 [T][f]) and da13_tap (bf16 [T][2f]) are optional debug
 * copies; with da13_row = da13_col = NULL only the taps are written. */
FP4_API int fp4_swiglu_bwd(const fp4_tensor* dy2_row, const fp4_tensor* w2_col, int64_t f, const void* a1,
                           const void* a3, uint64_t sr_seed, uint64_t sr_offset, fp4_tensor* da13_row,
                           fp4_tensor* da13_col, void* dh_tap, void* da13_tap, void* workspace,
                           size_t workspace_bytes, fp4_stream_t stream);

/* Workspace bytes of the NVFP4 gated-FFN producers (0 for MXFP4): the
 * maximum slots of the encoded tensor (h [T][f], or da13 [T][2f] when
 * backward != 0), padded to 256 bytes, plus its bf16 copy unless with_tap
 * (the caller passes h_tap / da13_tap).  Host only. */
FP4_API int fp4_swiglu_workspace_bytes(int route, int64_t T, int64_t f, int backward, int with_tap, size_t* bytes);

/* Residual + RMSNorm producer, forward (Sec. 3.2: the residual-RMSNorm
 * boundary retains the exact residual and its row statistics while producing
 * the next quantized representations).  For each row of r, b (device bf16,
 * rows x cols, leading dimension ld; b may be NULL for b = 0) and gain g
 * (device bf16 [cols]):
 *   r_out = r' = bf16(r + b)                  device bf16 [rows][cols], retained
 *   rstd  = fl32(1 / sqrt(mean(r'^2) + eps))   device binary32 [rows], retained
 *   y     = bf16(fl32(fl32(r' * rstd) * g))   quantized into y_row / y_col
 * exactly as fp4_quantize would quantize y under (route, views, flags 0);
 * y_tap (device bf16 [rows][cols], optional) receives y itself.
 * workspace: fp4_quantize_workspace_bytes(route, rows, cols, ...) bytes.
 * Errors as fp4_quantize. */
FP4_API int fp4_residual_rmsnorm_fwd(int route, unsigned views, const void* r, const void* b, const void* g,
                                     int64_t rows, int64_t cols, int64_t ld, float eps, void* r_out, float* rstd,
                                     fp4_tensor* y_row, fp4_tensor* y_col, void* y_tap, void* workspace,
                                     size_t workspace_bytes, fp4_stream_t stream);

/* Residual + RMSNorm producer, backward.  dy (device bf16 [rows][cols]) is the
 * gradient of y, r_prime / rstd the state retained by the forward, g the gain
 * and dres (device bf16 [rows][cols], may be NULL) the gradient arriving on the
 * residual stream.  Computes, per row, mean_g = mean(fl32(dy * g) * fl32(r' * rstd))
 * and
 *   dr = bf16(fl32(fl32(rstd * fl32(fl32(dy * g) - fl32(fl32(r' * rstd) * mean_g))) + dres))
 * written to dr (device bf16 [rows][cols], the residual gradient), and
 * quantizes dr into dr_row (with FP4_FLAG_SR_ROW semantics under sr_seed /
 * sr_offset when `sr` is non-zero) and dr_col: the gradient producer of the
 * preceding linear.
 * workspace: fp4_rmsnorm_bwd_workspace_bytes() bytes. */
FP4_API int fp4_residual_rmsnorm_bwd(int route, unsigned views, int sr, const void* dy, const void* r_prime,
                                     const float* rstd, const void* g, const void* dres, int64_t rows, int64_t cols,
                                     uint64_t sr_seed, uint64_t sr_offset, void* dr, fp4_tensor* dr_row,
                                     fp4_tensor* dr_col, void* workspace, size_t workspace_bytes,
                                     fp4_stream_t stream);

/* Data-gradient contraction whose consumer is a residual-RMSNorm backward
 * (Sec. 3.2: the backward combines QKV gradient production with the adjacent
 * RMSNorm reduction when their data dependencies align).  Computes
 * dx = dY . W exactly as fp4_linear_dgrad(dy_row, w_col, dx, FP4_OUT_BF16, 0)
 * and, in the same epilogue, for every row m and 64-column block j of dx,
 *   part[m][j] = sum over the block's columns n, in increasing order, of
 *                fl32(dx[m][n] * g[n]) * fl32(r'[m][n] * rstd[m])
 * (binary32, fused multiply-add accumulation), the terms of the RMSNorm
 * backward's row mean over the bf16 values written to dx.
 * r_prime: device bf16 [rows][cols] (the forward's retained r'), rstd: device
 * binary32 [rows], g: device bf16 [cols], part: device binary32
 * [rows][cols / 64] written by the call (rows = dy_row->rows, cols =
 * w_col->rows); r_prime and g 16-byte aligned.  Errors as fp4_linear_dgrad,
 * FP4_ERR_INVALID_ARG for a missing or misaligned pointer. */
FP4_API int fp4_linear_dgrad_rmsnorm(const fp4_tensor* dy_row, const fp4_tensor* w_col, void* dx, const void* r_prime,
                                     const float* rstd, const void* g, float* part, fp4_stream_t stream);

/* fp4_residual_rmsnorm_bwd with the row means taken from the partial sums
 * that fp4_linear_dgrad_rmsnorm wrote for this dy:
 *   mean_g[m] = (sum over j = 0 .. cols/64 - 1, in order, of part[m][j]) / cols
 * instead of a second pass over dy; everything else as
 * fp4_residual_rmsnorm_bwd (same workspace).  part: device binary32
 * [rows][cols / 64]. */
FP4_API int fp4_residual_rmsnorm_bwd_parts(int route, unsigned views, int sr, const void* dy, const float* part,
                                           const void* r_prime, const float* rstd, const void* g, const void* dres,
                                           int64_t rows, int64_t cols, uint64_t sr_seed, uint64_t sr_offset,
                                           void* dr, fp4_tensor* dr_row, fp4_tensor* dr_col, void* workspace,
                                           size_t workspace_bytes, fp4_stream_t stream);

/* Workspace of fp4_residual_rmsnorm_bwd: rows * 4 bytes of row statistics
 * plus the quantizer's workspace, rounded up to 256 bytes.  Host only. */
FP4_API int fp4_rmsnorm_bwd_workspace_bytes(int route, int64_t rows, int64_t cols, size_t* bytes);

/* Read the sticky device status word (first device-side error since the last
 * reset, FP4_OK if none) into *code.  Synchronises `stream`. */
FP4_API int fp4_status(fp4_stream_t stream, int* code);

/* Clear the sticky device status word (enqueued on `stream`). */
FP4_API int fp4_status_reset(fp4_stream_t stream);

/* Bound of every mbarrier wait in the GEMM kernels, in SM clock cycles, for
 * the launches that follow this call (process-wide).  A wait that runs out
 * sets FP4_ERR_TIMEOUT in the status word; the kernel then waits (again
 * bounded) for the copies it issued, releases its tensor memory and returns,
 * so the context stays usable.  cycles = 0 restores the default (4e9, about
 * 2 s at 2 GHz).  Host only; returns FP4_OK. */
FP4_API int fp4_set_wait_limit(uint64_t cycles);

/* Test hook for the timeout path above: with enable != 0, the GEMM launches
 * that follow skip their epilogue's first accumulator release, so the MMA
 * thread's next wait for the accumulator cannot be satisfied and runs out
 * after the wait limit (a barrier that no copy targets; nothing faults).
 * enable = 0 restores normal operation.  Not for production use; results of
 * launches made while it is set are invalid.  Host only; returns FP4_OK. */
FP4_API int fp4_test_skip_accumulator_release(int enable);

#ifdef __cplusplus
}
#endif

#endif /* FP4LIN_H */
