/*
 * nvfp4.h -- C ABI of libnvfp4: NVFP4 quantize / dequantize on one GB300 GPU.
 *
 * What the library computes (web pages; titles and sections):
 *   [TE-3206] TransformerEngine PR #3206 "NVFP4: enable row-scaled transpose
 *             quantization for backward": a row-scaled NVFP4 quantize that emits
 *             both the rowwise (fprop) and the columnwise / transposed (wgrad)
 *             output in one pass, after a per-row and per-column amax pre-pass
 *             (sequence diagram; description).
 *   [TE-3454] TransformerEngine PR #3454 "row-scaled nvfp4 path: fuse row/col
 *             amax into a single TMA-tiled kernel": one kernel for the row and
 *             column amax, byte-identical to two separate reductions; a noop flag
 *             that must leave the amax buffers untouched (description; flowchart;
 *             review comment on compute_fused_amax).
 *   [AO-9]    torchao PR #9 "Add NVFP4 four-over-six grouped GEMM for MoE
 *             training": per-block four-over-six choice with bound 448 or 256;
 *             grouped quantize whose per-group amax is expanded to a per-row
 *             vector over contiguous token groups given by group-end offsets
 *             (description).
 *   [AO-8]    torchao PR #8 "Add backward overrides and 1x16 weights to NVFP4
 *             four-over-six": dequantize = code * ((scale * amax) * factor_inv)
 *             with a correctly rounded FP32 reciprocal; 1x16 or 16x16 weight
 *             blocks; BF16 or FP32 output (description).
 *
 * Encode recipe (the pages fix the formats and the dequantize formula but print
 * no encode formula; this is the plain reading the library implements, FP32 with
 * round-to-nearest-even, one operation at a time):
 *   F  = bound * 6                          (6 = largest E2M1 magnitude)
 *   S  = F / a (a = amax of the line or tensor; S = 1 if a == 0; FLT_MAX if F/a
 *        overflows)
 *   per 16-element block (or 16x16 tile) with max |x| = b, for T = 6 (and T = 4
 *   when four-over-six is on):
 *     s8 = E4M3_satfinite((b / T) * S)      block scale byte
 *     e  = S / decode(s8)  (0 if decode(s8) == 0)
 *     c  = E2M1_satfinite(x * e)            4-bit code, sign kept
 *   four-over-six keeps T = 4 only if its squared error, summed in element order
 *   after dequantizing with the formula above, is strictly smaller.
 *
 * Layouts (all row-major, compact):
 *   x            [rows][cols] BF16 or FP32, row stride = cols elements.
 *   rowwise      codes  [rows][ceil(cols/2)]  two codes per byte, low nibble = even column
 *                scales [rows][ceil(cols/16)] one E4M3 byte per 1x16 block
 *                amax   [rows] (row-scaled) or [1] (per-tensor)
 *   columnwise   the rowwise layout of x^T: codes [cols][ceil(rows/2)],
 *                scales [cols][ceil(rows/16)], amax [cols] or [1].
 *
 * Conventions for every entry point:
 *   - All data pointers are DEVICE pointers on the current CUDA device; the
 *     caller allocates and owns every buffer.  The library allocates nothing
 *     (its own device memory, the status word and the static GEMM workspace, is
 *     reserved when its device code loads),
 *     never synchronizes and never reads device memory on the host, so a call
 *     can be captured in a CUDA graph (after the first call on a device, which
 *     loads the kernels; nothing is claimed here for nvfp4_gemm_static_ws).
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default
 *     stream) on the current device.
 *   - noop: optional device float; if non-NULL and *noop == 1.0f at run time,
 *     the call writes nothing at all (no amax, codes or scales).
 *   - Return value: NVFP4_OK once the work is enqueued.  NVFP4_ERR_INVALID for
 *     bad arguments (NULL required pointer, negative size, bound not 448/256,
 *     16x16 blocks with row-scaled mode, unknown dtype); nothing is enqueued
 *     then.  NVFP4_ERR_CUDA if a launch failed.  The reason is available from
 *     nvfp4_last_error() (per host thread).
 *   - Problems found on the device (invalid group ends, a wait that gave up)
 *     set bits in the library's device status word, read with
 *     nvfp4_device_status().
 *   - rows == 0 or cols == 0 is valid: amax buffers of the non-empty extent are
 *     written with 0 and no code or scale byte exists.
 */
#ifndef NVFP4_H
#define NVFP4_H

#include <stdint.h>

#if defined(__GNUC__)
#define NVFP4_API __attribute__((visibility("default")))
#else
#define NVFP4_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *nvfp4_stream_t;

typedef enum {
    NVFP4_OK = 0,
    NVFP4_ERR_INVALID = 1,
    NVFP4_ERR_UNSUPPORTED = 2,
    NVFP4_ERR_CUDA = 3,
    NVFP4_ERR_TIMEOUT = 4
} nvfp4_status;

typedef enum { NVFP4_IN_BF16 = 0, NVFP4_IN_FP32 = 1 } nvfp4_in_dtype;
typedef enum { NVFP4_OUT_BF16 = 0, NVFP4_OUT_FP32 = 1 } nvfp4_out_dtype;

/* PER_TENSOR: one amax for the whole tensor (both directions use it).
 * ROW_SCALED: rowwise output uses the per-row amax, columnwise output uses the
 * per-column amax [TE-3206]. */
typedef enum { NVFP4_PER_TENSOR = 0, NVFP4_ROW_SCALED = 1 } nvfp4_amax_mode;

/* Device status bits (nvfp4_device_status). */
#define NVFP4_DEVICE_TIMEOUT 1    /* a kernel gave up a bounded wait */
#define NVFP4_DEVICE_BAD_GROUPS 2 /* group ends not non-decreasing / last != rows */

typedef struct {
    int32_t mode;          /* nvfp4_amax_mode */
    float bound;           /* E4M3 bound of the global scale: 448 or 256 [AO-9] */
    int32_t four_over_six; /* 0: T = 6 only; 1: per-block choice of T = 4 or 6 by MSE */
    int32_t block_2d;      /* 0: 1x16 blocks; 1: 16x16 blocks (PER_TENSOR only) [AO-8] */
} nvfp4_config;

/* One output direction. */
typedef struct {
    uint8_t *codes;        /* [lines][ceil(n/2)] */
    uint8_t *scales;       /* [lines][ceil(n/16)] */
    float *amax;           /* [lines] or [1]: receives the amax the codes were made with */
    const float *amax_in;  /* NULL: compute amax from x; else [lines] or [1] to use (may equal amax) */
} nvfp4_out;

/*
 * nvfp4_amax -- exact amax of x, rows and columns in one pass over x [TE-3454].
 *   row_amax [rows], col_amax [cols], tensor_amax [1]: each may be NULL (at least
 *   one must be given).  Values are max |x| (an empty line gives 0); the result
 *   does not depend on the order of reduction.
 */
NVFP4_API nvfp4_status nvfp4_amax(const void *x, int32_t in_dtype, int64_t rows, int64_t cols,
                        float *row_amax, float *col_amax, float *tensor_amax,
                        const float *noop, nvfp4_stream_t stream);

/*
 * nvfp4_quantize_rowwise / _columnwise / _both -- NVFP4 quantize of x [TE-3206].
 *   cfg: see nvfp4_config.  row / col: the output direction(s); amax length is
 *   rows / cols for ROW_SCALED and 1 for PER_TENSOR.  The _both variant reads x
 *   for the amax pass and once more for the encode pass (a global amax must be
 *   known before the first code), in one stream-ordered sequence of kernels; with
 *   four-over-six and 1x16 blocks the encode runs as one pass per direction (x is
 *   read once more; faster than one pass holding both directions' block routines).
 */
NVFP4_API nvfp4_status nvfp4_quantize_rowwise(const void *x, int32_t in_dtype, int64_t rows, int64_t cols,
                                    const nvfp4_config *cfg, const nvfp4_out *row,
                                    const float *noop, nvfp4_stream_t stream);
NVFP4_API nvfp4_status nvfp4_quantize_columnwise(const void *x, int32_t in_dtype, int64_t rows,
                                       int64_t cols, const nvfp4_config *cfg,
                                       const nvfp4_out *col, const float *noop,
                                       nvfp4_stream_t stream);
NVFP4_API nvfp4_status nvfp4_quantize_both(const void *x, int32_t in_dtype, int64_t rows, int64_t cols,
                                 const nvfp4_config *cfg, const nvfp4_out *row,
                                 const nvfp4_out *col, const float *noop, nvfp4_stream_t stream);

/*
 * nvfp4_dequantize -- value = code * ((decode(scale) * amax) * fl(1/(bound*6)))
 * [AO-8], written as FP32 or rounded to nearest-even BF16.
 *   codes [rows][ceil(cols/2)], scales [rows][ceil(cols/16)], amax [rows]
 *   (ROW_SCALED) or [1] (PER_TENSOR); out [rows][cols].  For a columnwise output
 *   pass rows = original cols, cols = original rows.
 */
NVFP4_API nvfp4_status nvfp4_dequantize(const uint8_t *codes, const uint8_t *scales, const float *amax,
                              int32_t mode, int64_t rows, int64_t cols, float bound, void *out,
                              int32_t out_dtype, nvfp4_stream_t stream);

/*
 * nvfp4_grouped_amax -- per-group amax over contiguous row groups [AO-9].
 *   group_ends: device int64 [num_groups], cumulative row ends, non-decreasing,
 *   last == rows (an empty group is allowed and gets amax 0).
 *   group_amax [num_groups] (required); row_amax_expanded [rows] (optional)
 *   receives each row's group amax (it also holds the row maxima between the
 *   call's kernels).  Invalid ends set NVFP4_DEVICE_BAD_GROUPS and nothing is
 *   written.  num_groups <= 4096.
 */
NVFP4_API nvfp4_status nvfp4_grouped_amax(const void *x, int32_t in_dtype, int64_t rows, int64_t cols,
                                const int64_t *group_ends, int32_t num_groups, float *group_amax,
                                float *row_amax_expanded, const float *noop,
                                nvfp4_stream_t stream);

/*
 * nvfp4_grouped_quantize_rowwise -- rowwise quantize of grouped tokens [AO-9].
 *   cfg->mode PER_TENSOR: each group uses its own amax (the group amax expanded
 *   to every row), bit-identical to quantizing each group separately;
 *   cfg->mode ROW_SCALED: per-row amax (groups do not change the result).
 *   row->amax [rows] receives the per-row amax used; row->amax_in must be NULL.
 *   group_amax [num_groups] (optional with ROW_SCALED, required otherwise).
 */
NVFP4_API nvfp4_status nvfp4_grouped_quantize_rowwise(const void *x, int32_t in_dtype, int64_t rows,
                                            int64_t cols, const int64_t *group_ends,
                                            int32_t num_groups, const nvfp4_config *cfg,
                                            const nvfp4_out *row, float *group_amax,
                                            const float *noop, nvfp4_stream_t stream);

/*
 * nvfp4_grouped_quantize_rowwise_padded -- rowwise quantize of grouped tokens
 * straight from the ragged (unpadded) tensor into the padded layout that "Add NVFP4
 * four-over-six grouped GEMM for MoE training" (torchao PR #9, description) pads
 * each group to; the result is bit-identical to zero-padding x into that layout and
 * calling nvfp4_grouped_quantize_rowwise (NVFP4_PER_TENSOR: each group's amax),
 * without reading or materialising the padding rows.
 *   x: device [tokens][cols] (BF16 or FP32), the groups' rows back to back.
 *   ragged_ends: device int64 [num_groups], cumulative token ends (last == tokens).
 *   padded_ends: device int64 [num_groups], cumulative padded ends (last ==
 *   padded_rows); every padded group is at least as long as its ragged group and
 *   starts on a multiple of 128 rows.
 *   row->codes [padded_rows][ceil(cols/2)], row->scales [padded_rows][ceil(cols/16)],
 *   row->amax [padded_rows] receives each padded row's group amax; row->amax_in must be
 *   NULL.  Padding rows get zero codes and zero scales.
 *   group_amax [num_groups] (required).
 *   cfg->mode must be NVFP4_PER_TENSOR (NVFP4_ERR_UNSUPPORTED otherwise), cfg->block_2d 0.
 *   Invalid ends or layouts set NVFP4_DEVICE_BAD_GROUPS and nothing is written.
 */
NVFP4_API nvfp4_status nvfp4_grouped_quantize_rowwise_padded(
    const void *x, int32_t in_dtype, int64_t tokens, int64_t cols, const int64_t *ragged_ends,
    const int64_t *padded_ends, int32_t num_groups, int64_t padded_rows, const nvfp4_config *cfg,
    const nvfp4_out *row, float *group_amax, const float *noop, nvfp4_stream_t stream);

/*
 * nvfp4_grouped_quantize_columnwise -- columnwise (transposed, wgrad) quantize of
 * grouped tokens with each group's own amax: the columnwise operand of the
 * per-expert weight-gradient GEMMs of "Add NVFP4 four-over-six grouped GEMM for MoE
 * training" (torchao PR #9, description), in the row-scaled columnwise form of
 * "NVFP4: enable row-scaled transpose quantization for backward" (TransformerEngine
 * PR #3206, description).  Equal to quantizing each group's rows on their own
 * columnwise and placing the results side by side along the token axis.
 *   x: device [rows][cols]; group_ends: device int64 [num_groups], cumulative, every
 *   end a multiple of 128 (groups of whole 128-row tiles, as padded MoE tokens are),
 *   last == rows.
 *   col->codes [cols][rows/2], col->scales [cols][rows/16] (the columnwise layout of x).
 *   cfg->mode NVFP4_ROW_SCALED: col->amax [num_groups][cols], column c's amax over
 *   group g's rows; NVFP4_PER_TENSOR: col->amax [num_groups], each group's amax.
 *   col->amax_in: optional amax of that shape (else computed).  cfg->block_2d must
 *   be 0.  The rows of x must be 16-byte aligned (NVFP4_ERR_UNSUPPORTED otherwise).
 *   Invalid or unaligned ends set NVFP4_DEVICE_BAD_GROUPS and nothing is written.
 */
NVFP4_API nvfp4_status nvfp4_grouped_quantize_columnwise(const void *x, int32_t in_dtype,
                                               int64_t rows, int64_t cols,
                                               const int64_t *group_ends, int32_t num_groups,
                                               const nvfp4_config *cfg, const nvfp4_out *col,
                                               const float *noop, nvfp4_stream_t stream);

/*
 * nvfp4_rht16 -- random Hadamard transform (RHT) of x along its rows, per column and
 * per block of 16 consecutive rows (one columnwise 1x16 block).  [TE-3206]'s
 * description names an RHT of the transposed path without defining it; the reading
 * implemented is y = (1/4) H16 diag(s) x, H16 the Sylvester Hadamard matrix (entry
 * (i, j) = (-1)^popcount(i & j)), s_j = -1 where bit j of sign_mask is set, else +1.
 * It is orthonormal, so a wgrad product of two operands transformed with the same
 * signs equals the product of the originals.  FP32 steps: the signs, the four
 * natural-order butterfly stages of the fast Walsh-Hadamard transform (h = 1, 2, 4, 8:
 * rows i and i + h, i & h == 0, become u + v and u - v), then the product with 0.25.
 *   x [rows][cols] BF16 or FP32; y [rows][cols] FP32, caller-owned.  y may equal x
 *   when x is FP32 (in place); any other overlap of the two byte ranges is rejected
 *   (NVFP4_ERR_INVALID, nothing enqueued).  rows must be a multiple of 16
 *   (NVFP4_ERR_UNSUPPORTED otherwise); sign_mask < 2^16 (NVFP4_ERR_INVALID otherwise).
 */
NVFP4_API nvfp4_status nvfp4_rht16(const void *x, int32_t in_dtype, int64_t rows, int64_t cols,
                                   uint32_t sign_mask, float *y, nvfp4_stream_t stream);

/*
 * nvfp4_quantize_columnwise_rht -- the columnwise quantization (as
 * nvfp4_quantize_columnwise, every cfg) of nvfp4_rht16(x, sign_mask): the wgrad
 * operand with its 16-row blocks rotated before the amax and the encode.
 *   1x16 blocks (cfg->block_2d == 0): the transform is fused; the amax pass and the
 *   encode pass each read x and transform the blocks they read, and nothing else is
 *   written (workspace unused, may be NULL).  col->amax_in, if given, is taken as
 *   the amax of the transformed operand.
 *   16x16 blocks: workspace, an FP32 device buffer of rows * cols elements
 *   (ws_bytes at least 4 * rows * cols), receives the transformed operand, which is
 *   then quantized from there; a workspace that overlaps x or an output buffer is
 *   rejected (NVFP4_ERR_INVALID, nothing enqueued).
 *   noop as for every call: the transform is skipped as well.  rows a multiple of 16
 *   (NVFP4_ERR_UNSUPPORTED otherwise).
 */
NVFP4_API nvfp4_status nvfp4_quantize_columnwise_rht(const void *x, int32_t in_dtype, int64_t rows,
                                                     int64_t cols, uint32_t sign_mask,
                                                     const nvfp4_config *cfg,
                                                     const nvfp4_out *col, float *workspace,
                                                     uint64_t ws_bytes, const float *noop,
                                                     nvfp4_stream_t stream);

/*
 * nvfp4_grouped_quantize_columnwise_rht -- nvfp4_grouped_quantize_columnwise of the
 * transform nvfp4_rht16(x, sign_mask): each group's rows rotated block by block and
 * quantized columnwise with that group's amax of the transform (the wgrad operands
 * of the per-expert GEMMs with their 16-token blocks rotated).  Every rule of
 * nvfp4_grouped_quantize_columnwise applies (group ends multiples of 128, 1x16
 * blocks, 16-byte aligned rows of x); sign_mask < 2^16.  col->amax_in, if given, is
 * taken as the groups' amax of the transform.
 */
NVFP4_API nvfp4_status nvfp4_grouped_quantize_columnwise_rht(const void *x, int32_t in_dtype,
                                                   int64_t rows, int64_t cols,
                                                   const int64_t *group_ends,
                                                   int32_t num_groups, uint32_t sign_mask,
                                                   const nvfp4_config *cfg,
                                                   const nvfp4_out *col, const float *noop,
                                                   nvfp4_stream_t stream);

/*
 * nvfp4_quantize_both_rht -- both directions in one call (one encode pass; two, one per
 * direction, with four-over-six), the transform on the
 * transposed side only ([TE-3206]: the fprop operand as it is, the wgrad operand
 * rotated): row = nvfp4_quantize_rowwise(x, cfg), col =
 * nvfp4_quantize_columnwise_rht(x, sign_mask, cfg), byte for byte.
 *   cfg: 1x16 blocks only (block_2d == 1: NVFP4_ERR_UNSUPPORTED); both modes;
 *   four-over-six allowed.  With NVFP4_PER_TENSOR each direction has its own tensor
 *   amax (of x, of the transform).  row->amax_in / col->amax_in, if given, are taken
 *   as the amax of x / of the transform.
 *   rows a multiple of 16; x rows 16-byte aligned (cols * element size a multiple of
 *   16, x 16-byte aligned), else NVFP4_ERR_UNSUPPORTED.  Nothing is enqueued when a
 *   check fails.  noop as for every call.
 */
NVFP4_API nvfp4_status nvfp4_quantize_both_rht(const void *x, int32_t in_dtype, int64_t rows,
                                               int64_t cols, uint32_t sign_mask,
                                               const nvfp4_config *cfg, const nvfp4_out *row,
                                               const nvfp4_out *col, const float *noop,
                                               nvfp4_stream_t stream);

/*
 * One operand of nvfp4_gemm: an NVFP4 tensor in K-major layout -- a rowwise output
 * (lines = rows of x) or a columnwise output (lines = columns of x, the operand
 * that enters the GEMM transposed).
 */
typedef struct {
    const uint8_t *codes;   /* [lines][k/2], 16-byte aligned */
    const uint8_t *scales;  /* [lines][k/16]; a 16x16-block operand carries its tile's
                               scale on each of the tile's lines, as the quantize
                               entry points write it */
    const float *amax;      /* [lines] (NVFP4_ROW_SCALED) or [1] (NVFP4_PER_TENSOR) */
    int32_t mode;           /* nvfp4_amax_mode of amax */
    float bound;            /* 448 or 256: the bound the operand was quantized with */
} nvfp4_operand;

/*
 * nvfp4_gemm -- the GEMM that consumes two NVFP4 operands, with the bilateral amax
 * post-scale of "NVFP4: enable row-scaled transpose quantization for backward"
 * (TransformerEngine PR #3206, sequence diagram: the fprop output is scaled by the
 * activation's per-row amax and the weight's amax, the wgrad output by the outer
 * product of both operands' per-line amax).  Defined as the product of the two
 * dequantized operands:
 *   d[i][j] = sum_c value_a(i, c) * value_b(j, c),
 *   value   = code * decode(scale) * amax / (bound * 6)
 * for a: m lines, b: n lines, both with k values per line.  Computed on the
 * tensor cores with one E4M3 scale per 16 values and FP32 accumulation, then
 * d = fl(fl(acc * alpha_i) * beta_j) with alpha_i = amax_a[i] * fl(1/(bound_a*6)),
 * beta_j = amax_b[j] * fl(1/(bound_b*6)), written row-major [m][n] as BF16 (round
 * to nearest even) or FP32 (out_dtype).  Not bit-identical to an FP64 product:
 * the FP32 accumulation order is the tensor core's.
 *   k: a multiple of 32 (NVFP4_ERR_UNSUPPORTED otherwise); k == 0 writes zeros;
 *   m == 0 or n == 0 writes nothing.
 *   workspace: device, 256-byte aligned, at least nvfp4_gemm_workspace_size(m, n,
 *   k) bytes, owned by the caller and used by the call (the scales rewritten in
 *   the tensor core's chunk layout); two calls in flight at once need two
 *   workspaces.
 *   A wait that gives up sets NVFP4_DEVICE_TIMEOUT and d is left unwritten.
 */
NVFP4_API nvfp4_status nvfp4_gemm_workspace_size(int64_t m, int64_t n, int64_t k, uint64_t *bytes);
NVFP4_API nvfp4_status nvfp4_gemm(const nvfp4_operand *a, const nvfp4_operand *b, int64_t m,
                        int64_t n, int64_t k, void *d, int32_t out_dtype, void *workspace,
                        uint64_t workspace_bytes, nvfp4_stream_t stream);

/*
 * nvfp4_grouped_gemm -- the per-expert GEMM of "Add NVFP4 four-over-six grouped GEMM
 * for MoE training" (torchao PR #9, description: token groups A (rows, k) times
 * expert weights B (groups, n, k) with group-end offsets), with the same bilateral
 * post-scale as nvfp4_gemm: for group g with rows [s_g, e_g) of a,
 *   d[i][j] = sum_c value_a(i, c) * value_b(g * n + j, c),  s_g <= i < e_g,
 * i.e. nvfp4_gemm of a's rows of the group with b's rows [g*n, (g+1)*n).
 *   a: rows lines (the padded MoE tokens, as the grouped quantize entry points write
 *      them), amax [rows] (NVFP4_ROW_SCALED: per row, e.g. the group amax expanded
 *      to its rows) or [1];
 *   b: num_groups * n lines, amax [num_groups * n] (NVFP4_ROW_SCALED) or
 *      [num_groups] (NVFP4_PER_TENSOR: one amax per expert);
 *   group_ends: device int64 [num_groups], cumulative, non-decreasing, every end a
 *      multiple of 128, last == rows (empty groups allowed); num_groups <= 4096;
 *   n: a multiple of 256 (NVFP4_ERR_UNSUPPORTED otherwise); d [rows][n].
 *   Invalid or unaligned ends set NVFP4_DEVICE_BAD_GROUPS and write nothing.
 *   workspace: at least nvfp4_grouped_gemm_workspace_size(rows, n, k, num_groups)
 *   bytes, as for nvfp4_gemm.
 */
NVFP4_API nvfp4_status nvfp4_grouped_gemm_workspace_size(int64_t rows, int64_t n, int64_t k,
                                               int32_t num_groups, uint64_t *bytes);
NVFP4_API nvfp4_status nvfp4_grouped_gemm(const nvfp4_operand *a, const nvfp4_operand *b,
                                const int64_t *group_ends, int32_t num_groups, int64_t rows,
                                int64_t n, int64_t k, void *d, int32_t out_dtype,
                                void *workspace, uint64_t workspace_bytes,
                                nvfp4_stream_t stream);

/*
 * nvfp4_grouped_gemm_wgrad -- the per-expert weight-gradient GEMM of the same MoE
 * layout: group g's token range [s_g, e_g) is the reduction dimension,
 *   d[g][i][j] = sum_{s_g <= c < e_g} value_a(i, c) * value_b(j, c),
 * with the bilateral post-scale of nvfp4_gemm using group g's amax.  The operands
 * are columnwise outputs of nvfp4_grouped_quantize_columnwise (lines = features, the
 * tokens along K): a = dY^T (m lines), b = X^T (n lines), each [lines][tokens/2];
 * a->amax [num_groups * m] (NVFP4_ROW_SCALED: group g's per-line amax at g*m) or
 * [num_groups] (NVFP4_PER_TENSOR: one per group); b->amax likewise with n.
 *   group_ends: device int64 [num_groups], cumulative token ends, every end a
 *   multiple of 256 (so that no 256-token K tile spans two groups), last == tokens;
 *   an empty group gets a zero block.  d: [num_groups][m][n].
 *   Invalid or unaligned ends set NVFP4_DEVICE_BAD_GROUPS and write nothing.
 *   workspace: nvfp4_gemm_workspace_size(m, n, tokens) bytes.
 */
NVFP4_API nvfp4_status nvfp4_grouped_gemm_wgrad(const nvfp4_operand *a, const nvfp4_operand *b,
                                      const int64_t *group_ends, int32_t num_groups, int64_t m,
                                      int64_t n, int64_t tokens, void *d, int32_t out_dtype,
                                      void *workspace, uint64_t workspace_bytes,
                                      nvfp4_stream_t stream);

/*
 * nvfp4_gemm_static_ws -- nvfp4_gemm with its workspace in the library's own static
 * device memory instead of a caller buffer: NVFP4_GEMM_STATIC_WS_BYTES per device,
 * reserved when the library's device code is loaded, so the call allocates nothing.
 * The pages have no counterpart for it (an interface for callers that cannot pass a
 * workspace); it computes exactly what nvfp4_gemm computes, byte for byte.
 *   A shape whose nvfp4_gemm_workspace_size exceeds NVFP4_GEMM_STATIC_WS_BYTES returns
 *   NVFP4_ERR_UNSUPPORTED and enqueues nothing.
 *   Every call on a device uses the same workspace: calls must not overlap in time
 *   (issue them on one stream or order them otherwise).
 */
#define NVFP4_GEMM_STATIC_WS_BYTES (64ull << 20)
NVFP4_API nvfp4_status nvfp4_gemm_static_ws(const nvfp4_operand *a, const nvfp4_operand *b,
                                  int64_t m, int64_t n, int64_t k, void *d,
                                  int32_t out_dtype, nvfp4_stream_t stream);

/* Message for the last non-OK status returned on this host thread ("" if none). */
NVFP4_API const char *nvfp4_last_error(void);

/*
 * nvfp4_device_status -- read (and if reset != 0, clear) the device status word
 * of the current device.  Synchronizes the device; not for use inside graph
 * capture.  *status receives NVFP4_DEVICE_* bits (0 = nothing happened).
 * Returns NVFP4_ERR_TIMEOUT when the word holds NVFP4_DEVICE_TIMEOUT (a kernel
 * gave up a bounded wait, so some outputs of the calls since the last reset
 * are incomplete); *status is filled (and reset, if asked) in that case too.
 */
NVFP4_API nvfp4_status nvfp4_device_status(int32_t *status, int32_t reset);

/*
 * nvfp4_selftest_scale_division -- diagnostic: the encode factor fl(S / sd) as the
 * encode kernels compute it (a reciprocal and two FMA steps in place of the IEEE
 * division; the IEEE division for S outside [2^-90, 2^90]), for each of n FP32
 * values S and each E4M3 byte s8 = 0 .. 126 (sd its value; 0 when sd == 0):
 * e_out[i * 127 + s8], device buffers.  Lets a test compare every block scale's
 * quotient with the correctly rounded one.
 */
NVFP4_API nvfp4_status nvfp4_selftest_scale_division(const float *S, int64_t n, float *e_out,
                                                     nvfp4_stream_t stream);

/*
 * nvfp4_selftest_wait_timeout -- diagnostic of the failure path every pipeline
 * kernel shares (their mbarrier waits are bounded, 2 s): one warp waits on a
 * shared-memory mbarrier that nothing ever arrives on, bounded by limit_ns
 * nanoseconds (0 .. 1e9; NVFP4_ERR_INVALID otherwise).  The wait gives up, the
 * kernel sets NVFP4_DEVICE_TIMEOUT in the status word and returns without
 * writing *out (device uint32; it would be set to 1 only had the wait
 * completed).  No copy or tensor-memory allocation is in flight, so the context
 * stays usable.  A test calls it, then nvfp4_device_status, which returns
 * NVFP4_ERR_TIMEOUT.
 */
NVFP4_API nvfp4_status nvfp4_selftest_wait_timeout(int64_t limit_ns, uint32_t *out,
                                                   nvfp4_stream_t stream);

/*
 * nvfp4_selftest_convert -- diagnostic: run the device conversions used by the
 * kernels over n FP32 inputs: e2m1_out[i] = E2M1 code of in[i] (one code per
 * byte) and e4m3_out[i] = E4M3 byte of in[i] (either output may be NULL).  Lets
 * a test compare the hardware conversions with the oracle on every bit pattern.
 */
NVFP4_API nvfp4_status nvfp4_selftest_convert(const float *in, int64_t n, uint8_t *e2m1_out,
                                    uint8_t *e4m3_out, nvfp4_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_H */
