/*
 * mxg.h -- C ABI of the GB300 (sm_103a) grouped block-scaled quantize +
 * grouped GEMM library (libmxg.so).
 *
 * The operations follow three public pages:
 *   [TE-gemm]  TransformerEngine transformer_engine/jax/cpp_extensions/gemm.py
 *              (commit 070b5b7): swizzled_scale, grouped_gemm,
 *              _jax_scaled_matmul, _get_nvfp4_tensor_scale_inv.
 *   [PR2763]   TransformerEngine PR #2763 "[JAX] MXFP8 Grouped Quant+GEMM".
 *   [PR3661]   TransformerEngine PR #3661 "Add row-scaled NVFP4 support to
 *              grouped-tensor GEMM".
 *
 * Conventions for every entry point
 *   - All buffers are caller-owned DEVICE memory unless stated otherwise.
 *     The library never allocates, frees or synchronises on these calls, so
 *     each of them may be captured in a CUDA graph.
 *   - Work is enqueued on `stream` (NULL = the legacy default stream).
 *   - Host-detectable errors (null pointers, sizes, alignment, unsupported
 *     combinations, a device that is not sm_103) are returned synchronously
 *     and nothing is launched.  MXG_ERR_LAUNCH reports a failed launch.
 *   - Data-dependent errors cannot be known on the host without a sync; the
 *     kernels record them in a caller-owned sticky device word `dev_status`
 *     (int32, atomicOr of the MXG_DEV_* bits) and clamp so that no access
 *     leaves the buffers.  Read it after the stream or graph has completed.
 *     `dev_status` may be NULL (then nothing is recorded).
 *   - Rows are dense (a [rows, cols] matrix has leading dimension cols),
 *     except the GEMM operands' data, whose leading dimension the operand
 *     descriptor gives.
 *   - bf16 is IEEE bfloat16 stored as uint16; E4M3 is the "fn" variant.
 *   - The grouped matrices are 128-row aligned: every group size, K, N and
 *     rows_capacity is a multiple of 128 (the alignment [PR2763] states for
 *     the grouped quantize and GEMM setup kernels).
 */
#ifndef MXG_H_
#define MXG_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* CUDA stream handle (same type as cudaStream_t / CUstream). */
struct CUstream_st;
typedef struct CUstream_st* mxg_stream_t;

typedef enum {
  MXG_OK = 0,
  MXG_ERR_INVALID_ARG = 1,         /* null pointer, bad size or enum value      */
  MXG_ERR_ALIGNMENT = 2,           /* size not a multiple of 128, pointer not   */
                                   /* 16-byte aligned                           */
  MXG_ERR_UNSUPPORTED_ARCH = 3,    /* current device is not sm_103 (GB300)      */
  MXG_ERR_LAUNCH = 4,              /* the CUDA launch failed                    */
  MXG_ERR_WORKSPACE_TOO_SMALL = 5, /* workspace smaller than the size query     */
  MXG_ERR_UNSUPPORTED = 6          /* valid but not implemented combination     */
} mxg_status_t;

/* Sticky device status bits (atomicOr into dev_status). */
#define MXG_DEV_NEG_SIZE 1          /* a group size was negative: used as 0       */
#define MXG_DEV_MISALIGNED 2        /* a group size was not a multiple of 128:    */
                                    /* rounded down                               */
#define MXG_DEV_SUM_OVER_CAPACITY 4 /* the sizes summed past rows_capacity: the   */
                                    /* rows beyond it were dropped                */
#define MXG_DEV_BOUNDS 8            /* an index check failed (debug builds)       */
#define MXG_DEV_TIMEOUT 16          /* a pipeline wait ran out; the kernel gave   */
                                    /* up on its tile and returned                */

typedef enum {
  MXG_MXFP8_E4M3 = 1,     /* E4M3 data, one E8M0 scale per 1x32 block          */
  MXG_NVFP4_ROWSCALED = 2 /* E2M1 data, one E4M3 scale per 1x16 block, plus an  */
                          /* FP32 outer scale per row                           */
} mxg_format_t;

typedef enum { MXG_ROWWISE = 1, MXG_COLWISE = 2, MXG_BOTH = 3 } mxg_qlayout_t;

typedef enum {
  MXG_FPROP_TN = 0, /* ragged output rows:  C[M_cap, N] = X[M_cap, K] . W[g]^T  */
  MXG_WGRAD_NT = 1, /* ragged contraction:  dW[G, N, K] = dY_g^T . X_g          */
  MXG_DGRAD_NN = 2  /* ragged output rows:  dX[M_cap, K] = dY[M_cap, N] . W[g]  */
} mxg_gemm_mode_t;

typedef enum { MXG_OUT_F32 = 0, MXG_OUT_BF16 = 1 } mxg_out_t;

/* One quantized GEMM operand: rowwise-quantized rows of the contraction dim
 * ([PR2763] GEMM-setup review thread: per-group operand pointers come from
 * the offsets and the leading dimensions).
 *   data  : E4M3 bytes [rows, cols] (MXFP8) or packed E2M1 [rows, cols/2]
 *           (NVFP4, element 2i in the low nibble of byte i), consecutive rows
 *           ld elements apart.
 *   scale : block scales in the swizzled layout of [TE-gemm] swizzled_scale
 *           for the [rows, cols/32] (MXFP8) or [rows, cols/16] (NVFP4) scale
 *           matrix: 128x4 tiles of 512 contiguous bytes, byte
 *           ((r/128 * C/4 + c/4) * 32 + r%32) * 16 + (r%128)/32 * 4 + c%4.
 *           Always dense (the swizzle fixes its layout).
 *   outer : NVFP4 only: FP32 outer scale per row [rows]; NULL for MXFP8.
 *   rows, cols : the operand's rows and contraction length in elements, as
 *           the GEMM mode implies them (listed at mxg_grouped_gemm); 0 means
 *           "as implied" (no check), any other value must match.
 *   ld    : elements from one row of data to the next; 0 means cols (dense).
 *           Otherwise ld >= cols and ld bytes (ld for MXFP8, ld/2 for NVFP4,
 *           ld even) a multiple of 16, so that an operand can be a view of
 *           rows inside a wider buffer.
 * data and scale must be 16-byte aligned. */
typedef struct {
  const void* data;
  const uint8_t* scale;
  const float* outer;
  int64_t rows;
  int64_t cols;
  int64_t ld;
} mxg_operand_t;

/* ------------------------------------------------------------------------- */
/* Group sizes -> int64 sizes + element offsets ([PR2763] description: int32 */
/* sizes widened to int64 with a multiplier; offsets-kernel review thread:   */
/* exclusive prefix sum of size * last_dim, G+1 values; workspace review     */
/* thread: layout [G int64 sizes | G+1 int64 offsets]).                      */
/* ------------------------------------------------------------------------- */

/* Bytes of the offsets workspace: (2G + 1) * 8.  Returns 0 if G < 1. */
size_t mxg_offsets_workspace_bytes(int G);

/* sizes          : device int32[G] (sizes_is_int64 = 0) or int64[G] (= 1).
 * multiplier     : rows per size unit (1 when sizes are row counts).
 * last_dim       : elements per row, used for the element offsets.
 * rows_capacity  : rows of the buffers the groups live in.
 * ws             : device int64[2G+1]; written as
 *                  ws[g] = s_g (sanitised rows of group g),
 *                  ws[G] = 0, ws[G+1+g] = ws[G+g] + s_g * last_dim.
 * Sanitisation (recorded in dev_status): a negative size counts as 0
 * (NEG_SIZE); a size not a multiple of 128 is rounded down (MISALIGNED);
 * rows past rows_capacity are dropped (SUM_OVER_CAPACITY).
 * A size times the multiplier is formed exactly (no 64-bit overflow): a
 * product past rows_capacity is clamped to it.
 * Errors: MXG_ERR_INVALID_ARG for null sizes/ws, G < 1 or G > 65536,
 * multiplier < 1 or > 2^31, last_dim < 1, rows_capacity < 0 or > 2^62, or
 * rows_capacity * last_dim beyond int64. */
mxg_status_t mxg_group_offsets(const void* sizes, int sizes_is_int64, int G, int64_t multiplier,
                               int64_t last_dim, int64_t rows_capacity, int64_t* ws,
                               int32_t* dev_status, mxg_stream_t stream);

/* ------------------------------------------------------------------------- */
/* Grouped quantize with the swizzled scale layout written directly         */
/* ([PR2763] description: swizzle fused into the grouped quantize;          */
/* [PR3661] description: row-scaled NVFP4 cast writes swizzled scales).     */
/* ------------------------------------------------------------------------- */
/* x             : bf16 [rows_capacity, cols], 16-byte aligned.
 * group_ws      : offsets workspace from mxg_group_offsets (its first G
 *                 entries are the rows of each group); the live rows are
 *                 their sum, clamped to rows_capacity.  NULL: all
 *                 rows_capacity rows are live (weights, [TE-gemm]
 *                 grouped_gemm quantizes the kernel with no group sizes).
 * Rows at or beyond the live count are neither read nor written.
 *
 * MXG_MXFP8_E4M3, rowwise (layout ROWWISE or BOTH):
 *   q_row  : E4M3 [rows_capacity, cols]
 *   sf_row : E8M0 swizzled [rows_capacity, cols/32]; group g's scales start
 *            at byte row_off_g * cols / 32 ([PR2763]: scale offset = data
 *            offset / 32).
 *   Per 1x32 block: amax -> e = ceil(log2(amax / 448)) clamped to
 *   [-127, 127] (all-zero block: e = -127), byte e + 127, data
 *   E4M3_RNE(x * 2^-e).
 * MXG_MXFP8_E4M3, colwise (layout COLWISE or BOTH), written transposed:
 *   q_col  : E4M3 [cols, rows_capacity], q_col[k, m] = Q(x[m, k]) over
 *            32x1 blocks along rows
 *   sf_col : E8M0 swizzled [cols, rows_capacity/32] ([TE-gemm]
 *            swizzled_scale, colwise: the scale matrix is transposed first).
 * MXG_NVFP4_ROWSCALED, rowwise (layout ROWWISE or BOTH):
 *   q_row     : packed E2M1 [rows_capacity, cols/2]
 *   sf_row    : E4M3 swizzled [rows_capacity, cols/16]
 *   outer_row : FP32 [rows_capacity], s_r = amax_r / 2688
 *               ([TE-gemm] _get_nvfp4_tensor_scale_inv: amax / (6 * 448)).
 *   Per 1x16 block, fp32 round-to-nearest steps: S = 2688 / amax_r,
 *   sb = E4M3_RNE_satfinite((amax_b / 6) * S), code =
 *   E2M1_RNE_satfinite(x * (S / sb)) (signed zeros when sb or amax_r is 0).
 * MXG_NVFP4_ROWSCALED, colwise (layout COLWISE or BOTH), written transposed
 * for wgrad ([PR3661]: columnwise amax per column, split per expert):
 *   q_col     : packed E2M1 [cols, rows_capacity/2]; byte q_col[k, m/2] holds
 *               rows m (low nibble) and m+1 of column k
 *   sf_col    : E4M3 swizzled [cols, rows_capacity/16] (16-row blocks)
 *   outer_col : FP32 [G, cols] (G = 1 when group_ws is NULL):
 *               A[g, k] / 2688 with A the amax of column k over group g's
 *               rows; the same block rule as rowwise runs down the column.
 *               Groups with no rows get 0.  Requires G <= 1024.
 * Unused output pointers may be NULL.
 * Errors: INVALID_ARG (null required pointer, bad enum, NVFP4 colwise with
 * G > 1024), ALIGNMENT (rows_capacity or cols not a multiple of 128, pointer
 * not 16-byte aligned), UNSUPPORTED_ARCH, LAUNCH. */
mxg_status_t mxg_group_quantize(mxg_format_t fmt, mxg_qlayout_t layout, const void* x,
                                int64_t rows_capacity, int64_t cols, const int64_t* group_ws,
                                int G, void* q_row, uint8_t* sf_row, void* q_col, uint8_t* sf_col,
                                float* outer_row, float* outer_col, int32_t* dev_status,
                                mxg_stream_t stream);

/* ------------------------------------------------------------------------- */
/* Grouped block-scaled GEMM ([TE-gemm] grouped_gemm; [PR2763] V2 grouped    */
/* GEMM consuming pre-swizzled scales; [PR3661] row-scaled NVFP4: neutral    */
/* outer scales, FP32 accumulation, outer scales applied afterwards).       */
/* ------------------------------------------------------------------------- */
/* MXG_FPROP_TN (ragged rows):
 *   A = activations, rowwise: data [M_cap, K]; B = weights, rowwise:
 *   data [G*N, K] (expert g owns rows g*N .. g*N+N-1).
 *   C[off_g + i, n] = alpha_g * sum_k A[off_g+i, k] * B[g*N+n, k]
 *                     + beta_g * C[off_g + i, n];   C is [M_cap, N].
 *   Rows of C at or beyond the live count are not written.
 *   NVFP4: A.outer [M_cap] and B.outer [G*N] are required, and the result is
 *   multiplied by A.outer[row] * B.outer[g*N + n].
 * MXG_WGRAD_NT (ragged contraction; MXFP8, or row-scaled NVFP4 whose
 * operands are the colwise copies with A.outer = dY's outer_col [G, N] and
 * B.outer = X's outer_col [G, K], applied as
 * dW[g, n, k] *= A.outer[g, n] * B.outer[g, k]):
 *   A = colwise copy of dY: data [N, M_cap], scale [N, M_cap/32];
 *   B = colwise copy of X:  data [K, M_cap], scale [K, M_cap/32].
 *   dW[g, n, k] = alpha_g * sum_{m in group g} A[n, m] * B[k, m]
 *                 + beta_g * dW[g, n, k];   C = dW is [G, N, K].
 *   An empty group writes beta_g * dW[g] (zeros when beta is NULL or
 *   beta_g is 0).  With M_cap = 0 every group is empty and A and B are not
 *   read (their pointers must still be non-NULL).
 * MXG_DGRAD_NN (ragged rows, weights not transposed, MXFP8; [TE-gemm]
 * _quantize_gemm_operands: an RHS whose contraction dim is not last is
 * quantized colwise):
 *   A = rowwise dY: data [M_cap, N], scale [M_cap, N/32];
 *   B = colwise copy of W viewed as [G*N, K]: data [K, G*N], scale
 *       [K, G*N/32] (mxg_group_quantize(MXFP8, COLWISE, W, G*N, K, NULL, ...)).
 *   dX[off_g + i, k] = alpha_g * sum_n A[off_g+i, n] * B[k, g*N + n]
 *                      + beta_g * dX[off_g + i, k];   C = dX is [M_cap, K].
 * M_cap = 0: fprop and dgrad have no output rows and launch nothing.
 * group_ws : offsets workspace of mxg_group_offsets (first G entries used).
 * alpha, beta : device float[G] or NULL (alpha = 1, beta = 0).
 * bias  : device float [G, N] (fprop) or [G, K] (dgrad), or NULL: per-group
 *         bias ([TE-gemm] grouped_gemm: bias of shape (G, N)); the output is
 *         alpha_g * acc + bias[g, col] + beta_g * C.  Rejected for wgrad.
 * workspace : not needed by this implementation (size query returns 0);
 *             may be NULL.
 * Accumulation is FP32 in tensor memory; the FP32 output is the parity
 * output, bf16 is rounded to nearest even from it.
 * Operand shapes (rows x cols of mxg_operand_t, checked when nonzero):
 *   FPROP_TN: A M_cap x K, B G*N x K;  WGRAD_NT: A N x M_cap, B K x M_cap;
 *   DGRAD_NN: A M_cap x N, B K x G*N.
 * Errors: INVALID_ARG (nulls, G < 1 or G > 1024, NVFP4 dgrad, beta with
 * NVFP4 -- rejected as on [PR3661] --, an operand's rows or cols not the
 * mode's, ld < cols), ALIGNMENT (M_cap, N, K not multiples of 128;
 * data/scale/C not 16-byte aligned; ld bytes not a multiple of 16),
 * UNSUPPORTED_ARCH, LAUNCH. */
mxg_status_t mxg_grouped_gemm(mxg_format_t fmt, mxg_gemm_mode_t mode, const mxg_operand_t* A,
                              const mxg_operand_t* B, const int64_t* group_ws, int G,
                              int64_t M_cap, int64_t N, int64_t K, const float* alpha,
                              const float* beta, const float* bias, void* C, mxg_out_t out_type,
                              void* workspace, size_t workspace_bytes, int32_t* dev_status,
                              mxg_stream_t stream);

/* Test entry point (no counterpart on the pages): mxg_grouped_gemm with the
 * kernel choices that the parity tests need to reach every variant, and a
 * hook for the failure path of the bounded pipeline waits.  Same arguments
 * and checks as mxg_grouped_gemm, plus:
 *   tile_n          : 0 -- the default kernel choice (the CTA-pair kernel
 *                     with 256 x 256 units when B has at least 256 rows);
 *                     256 or 128 -- the single-CTA kernel with 128 x 256 or
 *                     128 x 128 tiles (256 only where the output width is a
 *                     multiple of 256, else 128).
 *   stage_bytes     : 0 -- default; 128 -- 128 bytes of K per pipeline stage
 *                     where the default takes 256 (MXFP8 fprop, K % 256 == 0).
 *   inject_flags    : bit 0 -- CTA 0 withholds the arrival that tells its
 *                     epilogue that its first accumulator is ready, so the
 *                     epilogue's wait runs out; 0 -- a normal run.
 *   wait_timeout_ns : bound on every pipeline wait, in ns (0 = 1 s default).
 * With bit 0 set the launch ends with MXG_DEV_TIMEOUT in dev_status, the
 * affected CTA drains its copies and MMAs, frees its tensor memory and
 * returns; the output is undefined and the device stays usable.
 * Errors: as mxg_grouped_gemm, plus INVALID_ARG for another tile_n or
 * stage_bytes value or unknown inject bits. */
mxg_status_t mxg_grouped_gemm_debug(mxg_format_t fmt, mxg_gemm_mode_t mode, const mxg_operand_t* A,
                                    const mxg_operand_t* B, const int64_t* group_ws, int G,
                                    int64_t M_cap, int64_t N, int64_t K, const float* alpha,
                                    const float* beta, const float* bias, void* C,
                                    mxg_out_t out_type, int32_t* dev_status, int tile_n,
                                    int stage_bytes, int inject_flags, int64_t wait_timeout_ns,
                                    mxg_stream_t stream);

/* Workspace bytes mxg_grouped_gemm needs (0 for every combination here). */
size_t mxg_grouped_gemm_workspace_bytes(mxg_format_t fmt, mxg_gemm_mode_t mode, int G,
                                        int64_t M_cap, int64_t N);

/* ------------------------------------------------------------------------- */
/* Group sizes that are not multiples of 128 (MXFP8).  [PR2763] review       */
/* thread on the V2 alignment rule: the 128-row requirement comes from how   */
/* the grouped quantize and the GEMM setup compute per-group scale offsets,  */
/* not from the GEMM; [TE-gemm] grouped_gemm: padding belongs to the group   */
/* and is zero-filled so that it does not change the result; [TE-gemm]      */
/* apply_padding_to_scale_inv pads scale matrices of non-128 dims.  Here     */
/* each group's scales, and its slab of a colwise copy, are padded to a      */
/* multiple of 128 rows with zeros; rowwise data stays dense.                */
/* ------------------------------------------------------------------------- */

/* Rows of the padded layouts: rows_capacity + 128 * G (an upper bound on
 * the sum over groups of each group's rows rounded up to 128).  Returns 0
 * if rows_capacity < 0 or G < 1. */
int64_t mxg_unaligned_rows_capacity(int64_t rows_capacity, int G);

/* As mxg_group_offsets, but sizes are kept as given: no rounding and no
 * MISALIGNED bit (negative sizes and rows past rows_capacity are sanitised
 * as there).  Same workspace layout. */
mxg_status_t mxg_group_offsets_unaligned(const void* sizes, int sizes_is_int64, int G,
                                         int64_t multiplier, int64_t last_dim,
                                         int64_t rows_capacity, int64_t* ws, int32_t* dev_status,
                                         mxg_stream_t stream);

/* MXFP8 grouped quantize for groups of any size.  group_ws (required) is a
 * workspace of mxg_group_offsets_unaligned; group g owns data rows
 * [row_off_g, row_off_g + M_g) and padded rows [prow_off_g, prow_off_g +
 * P_g) with P_g = M_g rounded up to 128 and prow_off the prefix sum of P.
 * With R_pad = mxg_unaligned_rows_capacity(rows_capacity, G):
 *   q_row  : E4M3 [rows_capacity, cols], dense (row r of group g at row_off_g + r);
 *   sf_row : E8M0 swizzled [R_pad, cols/32]; group g's scale rows start at
 *            prow_off_g; its padding rows get byte 0;
 *   q_col  : E4M3 [cols, R_pad], transposed; group g's slab is columns
 *            [prow_off_g, prow_off_g + P_g), its padding columns 0x00;
 *   sf_col : E8M0 swizzled [cols, R_pad/32]; 32-row blocks start at each
 *            group's first row (a block never spans two groups).
 * Each group is quantized as if it were its own tensor, zero-padded to P_g
 * rows, with the block rules of mxg_group_quantize.  Rows and columns past
 * the padded groups are not written.  Unused output pointers may be NULL.
 * Errors: INVALID_ARG (null x or group_ws, G < 1 or G > 1024, bad layout,
 * null required output, rows_capacity + 128 * G above 2^31 - 128),
 * ALIGNMENT (rows_capacity or cols not multiples of 128, pointers not
 * 16-byte aligned), UNSUPPORTED_ARCH, LAUNCH. */
mxg_status_t mxg_group_quantize_unaligned(mxg_qlayout_t layout, const void* x,
                                          int64_t rows_capacity, int64_t cols,
                                          const int64_t* group_ws, int G, uint8_t* q_row,
                                          uint8_t* sf_row, uint8_t* q_col, uint8_t* sf_col,
                                          int32_t* dev_status, mxg_stream_t stream);

/* MXFP8 grouped GEMM for groups of any size (operands from
 * mxg_group_quantize_unaligned, weights from mxg_group_quantize).  Same
 * formulas, arguments and epilogue as mxg_grouped_gemm, with group_ws from
 * mxg_group_offsets_unaligned and these operand shapes (R_pad as above):
 *   FPROP_TN : A data [M_cap, K] dense, A scale [R_pad, K/32] padded;
 *   WGRAD_NT : A = dY colwise [N, R_pad] + [N, R_pad/32], B = X colwise
 *              [K, R_pad] + [K, R_pad/32]; each group contracts over its
 *              padded slab (the zero padding adds nothing);
 *   DGRAD_NN : A data [M_cap, N] dense, A scale [R_pad, N/32] padded
 *              (WGRAD_NT operands are R_pad columns long).
 * Output rows are the dense data rows; rows past a group are not written.
 * Errors: as mxg_grouped_gemm, plus INVALID_ARG when B has fewer than 256
 * rows (G * N for fprop, K otherwise) or M_cap + 128 * G exceeds 2^31 - 128. */
mxg_status_t mxg_grouped_gemm_unaligned(mxg_gemm_mode_t mode, const mxg_operand_t* A,
                                        const mxg_operand_t* B, const int64_t* group_ws, int G,
                                        int64_t M_cap, int64_t N, int64_t K, const float* alpha,
                                        const float* beta, const float* bias, void* C,
                                        mxg_out_t out_type, int32_t* dev_status,
                                        mxg_stream_t stream);

/* ------------------------------------------------------------------------- */
/* Dequantize ([PR2763] dequantizer: inverse swizzle of the scales, then    */
/* data * scale).  Test helper; not on the timed path.                      */
/* ------------------------------------------------------------------------- */
/* ROWWISE: q [rows, cols] (NVFP4: [rows, cols/2]), sf swizzled [rows,
 *          cols/32 or cols/16], outer [rows] (NVFP4) -> out [rows, cols].
 * COLWISE: (MXFP8 only) q is the transposed copy [cols, rows], sf swizzled
 *          [cols, rows/32] -> out [rows, cols] (transposed back).
 * out is FP32 or bf16 (round to nearest even).
 * Errors: INVALID_ARG, ALIGNMENT (rows or cols not multiples of 128),
 * UNSUPPORTED (NVFP4 colwise), UNSUPPORTED_ARCH, LAUNCH. */
mxg_status_t mxg_dequantize(mxg_format_t fmt, mxg_qlayout_t layout, const void* q,
                            const uint8_t* sf, const float* outer, int64_t rows, int64_t cols,
                            void* out, mxg_out_t out_type, mxg_stream_t stream);

/* Human-readable name of a status code (static string). */
const char* mxg_status_string(mxg_status_t status);

/* Library version: major * 10000 + minor * 100 + patch. */
int mxg_version(void);

/* Number of kernel launches this library has issued in this process
 * (all entry points, all devices).  For launch accounting in benchmarks. */
uint64_t mxg_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* MXG_H_ */
