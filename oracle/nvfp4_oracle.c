/*
 * nvfp4_oracle.c -- plain, slow CPU oracle for NVFP4 quantize / dequantize.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package's smoke check and
 * the CPU-baseline leg of the benchmark may load this library.  It shares no code,
 * header, table or constant with the CUDA path and must never be used as a
 * fallback for it.
 *
 * Sources (web pages; titles and sections):
 *   [TE-3206] TransformerEngine PR #3206 "NVFP4: enable row-scaled transpose
 *             quantization for backward" -- Greptile summary, sequence diagram,
 *             description (row-scaled rowwise + columnwise outputs, per-row amax
 *             for rows, per-column amax for the transposed output).
 *   [TE-3454] TransformerEngine PR #3454 "row-scaled nvfp4 path: fuse row/col
 *             amax into a single TMA-tiled kernel" -- description (amax is an
 *             exact max, fused == two-kernel byte for byte), flowchart and review
 *             comment (noop flag must leave amax untouched).
 *   [AO-9]    torchao PR #9 "Add NVFP4 four-over-six grouped GEMM for MoE
 *             training" -- description (four-over-six, bound 256, group amax
 *             expanded per row == per-split quantize, zero-padded rows).
 *   [AO-8]    torchao PR #8 "Add backward overrides and 1x16 weights to NVFP4
 *             four-over-six" -- description (dequantize = (scale * amax) *
 *             factor_inv with a correctly rounded FP32 reciprocal; 1x16 vs 16x16
 *             weight blocks; bound 256/448; bf16/fp32 output).
 *
 * Precision: every floating-point step is ONE IEEE-754 binary32 operation with
 * round-to-nearest-even, in the order written.  The pages fix FP32 for the global
 * scales and for the dequantize factor, E4M3 for the block scales and E2M1 for
 * the codes, so the oracle works in FP32 rather than FP64.  It must be compiled
 * with -ffp-contract=off (no fused multiply-add) and without -ffast-math; the
 * build script in this directory does that and the tests check it.
 *
 * Readings where the pages are silent (the pages give no explicit formula
 * for the encode path; only the dequantize formula is stated):
 *   R1  global scale  S = F / a with F = bound * 6 (6 = E2M1 max), a = amax of
 *       the line (row, column or tensor); a == 0 gives S = 1; an infinite
 *       quotient is replaced by FLT_MAX.
 *   R2  block scale   s32 = (b / T) * S, b = block amax, T = 6 (or 4 for the
 *       four-over-six candidate); s8 = E4M3(s32) with RNE and saturation to 448.
 *   R3  encode factor e = S / decode(s8) (IEEE division), 0 when decode(s8) is 0.
 *   R4  codes         c = E2M1(x * e), RNE, saturating at 6, sign kept (so a
 *       negative value that rounds to zero gives code 0x8).
 *   R5  four-over-six error: each candidate is dequantized with the dequantize
 *       formula, err = sum over the block, in element order, of (x - deq)^2
 *       computed as separate FP32 multiply and add; T = 4 wins only if its error
 *       is strictly smaller.
 *   R6  16x16 blocks (per-tensor only): one scale per 16x16 tile, block amax over
 *       the tile, error sum in row-major order inside the tile; the rowwise and
 *       columnwise outputs then hold the same codes, transposed.
 *   R7  tails: a partial last block uses only the elements present; an odd final
 *       element packs with a zero high nibble.
 *   R8  layouts: codes two per byte, low nibble = even element; scales one byte
 *       per block, row-major [lines][ceil(n/16)], no GEMM swizzle.
 *   R9  noop: a non-NULL flag equal to 1.0f means nothing at all is written.
 *   R13 GEMM consumer (sequence diagram of [TE-3206]: output times the outer
 *       product of the operands' per-line amax): the matrix product of the two
 *       dequantized operands, each element code * decode(scale) * amax /
 *       (bound * 6) as a real number; computed here in FP64, not FP32, because it
 *       is the exact target that the GPU's FP32 accumulation is bounded against.
 *   R14 random Hadamard transform (RHT) of the columnwise operand: [TE-3206]'s
 *       description names it only among what that PR leaves out (no RHT or
 *       four-over-six fusion on the transposed path); its definition comes from
 *       outside the pages. Along each column, every run of 16 consecutive rows (one
 *       columnwise 1x16 block) x is replaced by y = (1/4) H16 diag(s) x, where H16 is
 *       the Sylvester Hadamard matrix (H1 = [1], H2n = [[Hn, Hn], [Hn, -Hn]]; entry
 *       (i, j) is (-1)^popcount(i & j)), s_j = -1 where bit j of a caller-given
 *       16-bit sign mask is set and +1 elsewhere, and 1/4 = 1/sqrt(16) makes the
 *       map orthonormal. FP32 steps: the signs (exact); then the four butterfly
 *       stages of the fast Walsh-Hadamard transform in natural order (h = 1, 2, 4,
 *       8: the pair at rows (i, i + h), i & h == 0, becomes (u + v, u - v)); then
 *       the product with 0.25. The columnwise output is the quantization of y.
 *
 * Parity pins: every function here is checked in tests/ against something other
 * than itself (brute force, library conversions, closed forms, invariants from
 * the pages).  No function is "parity unpinned".
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_API __attribute__((visibility("default")))

/* ------------------------------------------------------------------------- */
/* Number formats                                                             */
/* ------------------------------------------------------------------------- */

/* BF16 is the top half of an FP32 bit pattern, so widening is exact. */
ORACLE_API float oracle_bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* FP32 -> BF16, round to nearest, ties to even (used for BF16 dequantize
 * output, [AO-8] "bf16/fp32 out").  NaN stays NaN. */
ORACLE_API uint16_t oracle_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t upper = u >> 16;
    uint32_t lower = u & 0xffffu;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;
    return (uint16_t)upper;
}

/* E2M1 magnitudes in code order: 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit. */
static const float kE2M1Magnitude[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};

ORACLE_API float oracle_e2m1_decode(uint8_t code)
{
    float m = kE2M1Magnitude[code & 7u];
    return (code & 8u) ? -m : m;
}

/* FP32 -> E2M1: nearest magnitude, a tie goes to the even code (even mantissa
 * bit), values at or beyond 6 saturate to 6, the sign bit is copied (R4). */
ORACLE_API uint8_t oracle_e2m1_encode(float y)
{
    uint8_t sign = signbit(y) ? 8u : 0u;
    float m = fabsf(y);
    if (!(m < 6.0f)) return (uint8_t)(sign | 7u);
    int best = 0;
    double best_dist = (double)m; /* distance to magnitude 0 */
    for (int k = 1; k < 8; ++k) {
        double dist = fabs((double)m - (double)kE2M1Magnitude[k]);
        if (dist < best_dist || (dist == best_dist && (k & 1) == 0)) {
            best = k;
            best_dist = dist;
        }
    }
    return (uint8_t)(sign | (uint8_t)best);
}

/* E4M3 ("fn" variant): bias 7, subnormals m * 2^-9, largest finite 448 (0x7E),
 * 0x7F / 0xFF are NaN, no infinities. */
ORACLE_API float oracle_e4m3_decode(uint8_t s)
{
    int e = (s >> 3) & 15;
    int m = s & 7;
    if (e == 15 && m == 7) return NAN;
    float mag = (e == 0) ? ldexpf((float)m, -9) : ldexpf(1.0f + (float)m / 8.0f, e - 7);
    return (s & 0x80u) ? -mag : mag;
}

/* FP32 -> E4M3: nearest finite value, tie to the even code, saturating at 448
 * (R2).  Linear search over the 127 non-negative finite codes. */
ORACLE_API uint8_t oracle_e4m3_encode(float s)
{
    uint8_t sign = signbit(s) ? 0x80u : 0u;
    float m = fabsf(s);
    if (!(m < 448.0f)) return (uint8_t)(sign | 0x7Eu);
    int best = 0;
    double best_dist = (double)m;
    for (int k = 1; k <= 0x7E; ++k) {
        double dist = fabs((double)m - (double)oracle_e4m3_decode((uint8_t)k));
        if (dist < best_dist || (dist == best_dist && (k & 1) == 0)) {
            best = k;
            best_dist = dist;
        }
    }
    return (uint8_t)(sign | (uint8_t)best);
}

/* Array helpers so the tests can sweep the conversions. */
ORACLE_API void oracle_e2m1_encode_array(const float *y, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e2m1_encode(y[i]);
}

ORACLE_API void oracle_e4m3_encode_array(const float *s, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_encode(s[i]);
}

ORACLE_API void oracle_bf16_to_f32_array(const uint16_t *h, int64_t n, float *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_to_f32(h[i]);
}

/* Probe used by the tests: returns a*b + c written the same way as the
 * four-over-six error update.  With -ffp-contract=off this is two roundings. */
ORACLE_API float oracle_fp_contract_probe(float a, float b, float c)
{
    return c + a * b;
}

/* ------------------------------------------------------------------------- */
/* Global scale and the block recipe                                          */
/* ------------------------------------------------------------------------- */

/* R1: per-line (or per-tensor) FP32 global encode scale. */
ORACLE_API float oracle_global_scale(float amax, float bound)
{
    float F = bound * 6.0f; /* exact: 2688 or 1536 */
    if (amax == 0.0f) return 1.0f;
    float S = F / amax;
    if (isinf(S)) S = FLT_MAX;
    return S;
}

/* Dequantize factor of one block: (decode(s8) * amax) * fl(1/F)  [AO-8]. */
static float dequant_factor(uint8_t s8, float amax, float bound)
{
    float F_inv = 1.0f / (bound * 6.0f);
    float sd = oracle_e4m3_decode(s8);
    float t = sd * amax;
    return t * F_inv;
}

/* One candidate of R2-R4 for a block of n values whose amax is b. */
static void encode_candidate(const float *v, int n, float b, float T, float S,
                             uint8_t *codes, uint8_t *s8_out)
{
    float q = b / T;
    float s32 = q * S;
    uint8_t s8 = oracle_e4m3_encode(s32);
    float sd = oracle_e4m3_decode(s8);
    float e = (sd == 0.0f) ? 0.0f : S / sd;
    for (int i = 0; i < n; ++i) {
        float y = v[i] * e;
        codes[i] = oracle_e2m1_encode(y);
    }
    *s8_out = s8;
}

/* R5: squared error of one candidate, in element order, multiply then add. */
static float candidate_error(const float *v, int n, const uint8_t *codes, uint8_t s8,
                             float amax, float bound)
{
    float D = dequant_factor(s8, amax, bound);
    float err = 0.0f;
    for (int i = 0; i < n; ++i) {
        float deq = oracle_e2m1_decode(codes[i]) * D;
        float d = v[i] - deq;
        float d2 = d * d;
        err = err + d2;
    }
    return err;
}

/* Quantize one block (1x16 line segment, or a 16x16 tile in row-major order).
 * n <= 256.  amax is the line/tensor amax a that produced S (used by R5).
 * four_over_six: 0 = T 6 only, 1 = pick the lower-error of T 6 / T 4,
 * 2 = T 4 only (a test hook so the choice can be checked from outside). */
static void quantize_block(const float *v, int n, float S, float amax, float bound,
                           int four_over_six, uint8_t *codes, uint8_t *s8_out)
{
    float b = 0.0f;
    for (int i = 0; i < n; ++i) {
        float t = fabsf(v[i]);
        if (t > b) b = t;
    }
    if (four_over_six == 2) { /* test hook: the T = 4 candidate alone */
        encode_candidate(v, n, b, 4.0f, S, codes, s8_out);
        return;
    }
    uint8_t c6[256], s6;
    encode_candidate(v, n, b, 6.0f, S, c6, &s6);
    if (!four_over_six) {
        memcpy(codes, c6, (size_t)n);
        *s8_out = s6;
        return;
    }
    uint8_t c4[256], s4;
    encode_candidate(v, n, b, 4.0f, S, c4, &s4);
    float err6 = candidate_error(v, n, c6, s6, amax, bound);
    float err4 = candidate_error(v, n, c4, s4, amax, bound);
    if (err4 < err6) {
        memcpy(codes, c4, (size_t)n);
        *s8_out = s4;
    } else {
        memcpy(codes, c6, (size_t)n);
        *s8_out = s6;
    }
}

static void put_code(uint8_t *packed, int64_t idx, uint8_t code)
{
    if (idx & 1) packed[idx >> 1] = (uint8_t)(packed[idx >> 1] | (uint8_t)(code << 4));
    else packed[idx >> 1] = (uint8_t)(packed[idx >> 1] | code);
}

/* Quantize one line of n values read with the given stride (1x16 blocks).
 * codes: ceil(n/2) bytes, scales: ceil(n/16) bytes. */
ORACLE_API void oracle_quantize_line(const float *x, int64_t n, int64_t stride, float amax,
                                     float bound, int four_over_six, uint8_t *codes,
                                     uint8_t *scales)
{
    float S = oracle_global_scale(amax, bound);
    memset(codes, 0, (size_t)((n + 1) / 2));
    for (int64_t blk = 0; blk * 16 < n; ++blk) {
        int len = (int)((n - blk * 16) < 16 ? (n - blk * 16) : 16);
        float v[16];
        uint8_t c[16];
        for (int i = 0; i < len; ++i) v[i] = x[(blk * 16 + i) * stride];
        quantize_block(v, len, S, amax, bound, four_over_six, c, &scales[blk]);
        for (int i = 0; i < len; ++i) put_code(codes, blk * 16 + i, c[i]);
    }
}

/* ------------------------------------------------------------------------- */
/* amax  [TE-3206] pre-pass amax_rowwise / amax_columnwise; [TE-3454] fused  */
/* ------------------------------------------------------------------------- */

/* Each output may be NULL.  Exact maxima of |x|; an empty line gives 0. */
ORACLE_API void oracle_amax(const float *x, int64_t rows, int64_t cols, float *row_amax,
                            float *col_amax, float *tensor_amax)
{
    if (col_amax)
        for (int64_t c = 0; c < cols; ++c) col_amax[c] = 0.0f;
    float t = 0.0f;
    for (int64_t r = 0; r < rows; ++r) {
        float m = 0.0f;
        for (int64_t c = 0; c < cols; ++c) {
            float a = fabsf(x[r * cols + c]);
            if (a > m) m = a;
            if (col_amax && a > col_amax[c]) col_amax[c] = a;
        }
        if (row_amax) row_amax[r] = m;
        if (m > t) t = m;
    }
    if (tensor_amax) *tensor_amax = t;
}

/* ------------------------------------------------------------------------- */
/* Quantize (dense)                                                           */
/* ------------------------------------------------------------------------- */

enum { ORACLE_PER_TENSOR = 0, ORACLE_ROW_SCALED = 1 };

static int noop_set(const float *noop) { return noop != NULL && *noop == 1.0f; }

/* 16x16 tiles, per-tensor amax a (R6), one direction.  transpose = 0 writes
 * the rowwise layout of x, transpose = 1 the columnwise layout (x^T); the tile
 * grid, tile maxima and error order are those of x in both cases, so the two
 * layouts hold the same codes. */
static void quantize_2d(const float *x, int64_t rows, int64_t cols, float a, float bound,
                        int four_over_six, int transpose, uint8_t *codes, uint8_t *scales)
{
    float S = oracle_global_scale(a, bound);
    int64_t lines = transpose ? cols : rows, n = transpose ? rows : cols;
    int64_t cb = (n + 1) / 2, sb = (n + 15) / 16;
    memset(codes, 0, (size_t)(lines * cb));
    for (int64_t ti = 0; ti * 16 < rows; ++ti) {
        for (int64_t tj = 0; tj * 16 < cols; ++tj) {
            int h = (int)((rows - ti * 16) < 16 ? (rows - ti * 16) : 16);
            int w = (int)((cols - tj * 16) < 16 ? (cols - tj * 16) : 16);
            float v[256];
            uint8_t c[256], s8;
            for (int i = 0; i < h; ++i)
                for (int j = 0; j < w; ++j) v[i * w + j] = x[(ti * 16 + i) * cols + tj * 16 + j];
            quantize_block(v, h * w, S, a, bound, four_over_six, c, &s8);
            for (int i = 0; i < h; ++i) {
                for (int j = 0; j < w; ++j) {
                    int64_t r = ti * 16 + i, col = tj * 16 + j;
                    int64_t line = transpose ? col : r, pos = transpose ? r : col;
                    put_code(codes + line * cb, pos, c[i * w + j]);
                    scales[line * sb + pos / 16] = s8;
                }
            }
        }
    }
}

/*
 * Dense quantize of x [rows][cols] (FP32 values; BF16 callers widen first).
 *   mode: 0 per-tensor, 1 row-scaled (rowwise uses row amax, columnwise uses
 *         column amax [TE-3206]); block_2d only with per-tensor.
 *   row_*: rowwise outputs (codes [rows][ceil(cols/2)], scales [rows][ceil(cols/16)],
 *          amax [rows] or [1]); all NULL to skip the direction.
 *   col_*: columnwise outputs, i.e. the rowwise quantize of x^T with column amax
 *          (codes [cols][ceil(rows/2)], scales [cols][ceil(rows/16)], amax [cols] or [1]).
 *   row_amax_in / col_amax_in: NULL to compute amax, else used (and copied out).
 * Returns 0, or -1 for an invalid combination.
 */
ORACLE_API int oracle_quantize(const float *x, int64_t rows, int64_t cols, int mode, float bound,
                               int four_over_six, int block_2d, const float *row_amax_in,
                               const float *col_amax_in, uint8_t *row_codes, uint8_t *row_scales,
                               float *row_amax, uint8_t *col_codes, uint8_t *col_scales,
                               float *col_amax, const float *noop)
{
    if (bound != 448.0f && bound != 256.0f) return -1;
    if (block_2d && mode != ORACLE_PER_TENSOR) return -1;
    if (noop_set(noop)) return 0;
    int do_row = row_codes != NULL, do_col = col_codes != NULL;

    /* Line amax values: a direction given amax_in uses it, otherwise the amax
     * is computed from x (row amax for rows, column amax for columns, or the
     * tensor amax in per-tensor mode). */
    int64_t nra = (mode == ORACLE_ROW_SCALED) ? rows : 1;
    int64_t nca = (mode == ORACLE_ROW_SCALED) ? cols : 1;
    float *ra = (float *)calloc((size_t)(nra > 0 ? nra : 1), sizeof(float));
    float *ca = (float *)calloc((size_t)(nca > 0 ? nca : 1), sizeof(float));
    if (mode == ORACLE_ROW_SCALED) {
        if (row_amax_in) memcpy(ra, row_amax_in, (size_t)rows * sizeof(float));
        else if (do_row) oracle_amax(x, rows, cols, ra, NULL, NULL);
        if (col_amax_in) memcpy(ca, col_amax_in, (size_t)cols * sizeof(float));
        else if (do_col) oracle_amax(x, rows, cols, NULL, ca, NULL);
    } else {
        float t = 0.0f;
        if ((do_row && !row_amax_in) || (do_col && !col_amax_in))
            oracle_amax(x, rows, cols, NULL, NULL, &t);
        ra[0] = row_amax_in ? row_amax_in[0] : t;
        ca[0] = col_amax_in ? col_amax_in[0] : t;
    }

    if (block_2d) {
        if (do_row) quantize_2d(x, rows, cols, ra[0], bound, four_over_six, 0, row_codes, row_scales);
        if (do_col) quantize_2d(x, rows, cols, ca[0], bound, four_over_six, 1, col_codes, col_scales);
    } else {
        if (do_row)
            for (int64_t r = 0; r < rows; ++r) {
                float a = ra[mode == ORACLE_ROW_SCALED ? r : 0];
                oracle_quantize_line(x + r * cols, cols, 1, a, bound, four_over_six,
                                     row_codes + r * ((cols + 1) / 2),
                                     row_scales + r * ((cols + 15) / 16));
            }
        if (do_col)
            for (int64_t c = 0; c < cols; ++c) {
                float a = ca[mode == ORACLE_ROW_SCALED ? c : 0];
                oracle_quantize_line(x + c, rows, cols, a, bound, four_over_six,
                                     col_codes + c * ((rows + 1) / 2),
                                     col_scales + c * ((rows + 15) / 16));
            }
    }
    if (do_row && row_amax) memcpy(row_amax, ra, (size_t)nra * sizeof(float));
    if (do_col && col_amax) memcpy(col_amax, ca, (size_t)nca * sizeof(float));
    free(ra);
    free(ca);
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Dequantize  [AO-8]: value = code * ((scale * amax) * factor_inv)           */
/* ------------------------------------------------------------------------- */

/* codes [rows][ceil(cols/2)], scales [rows][ceil(cols/16)], amax [rows]
 * (row_scaled) or [1].  out_bf16 != 0 writes BF16 bit patterns to out (uint16),
 * else FP32 values. */
ORACLE_API void oracle_dequantize(const uint8_t *codes, const uint8_t *scales, const float *amax,
                                  int row_scaled, int64_t rows, int64_t cols, float bound,
                                  void *out, int out_bf16)
{
    int64_t cb = (cols + 1) / 2, sb = (cols + 15) / 16;
    for (int64_t r = 0; r < rows; ++r) {
        float a = amax[row_scaled ? r : 0];
        for (int64_t c = 0; c < cols; ++c) {
            uint8_t byte = codes[r * cb + c / 2];
            uint8_t code = (c & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15u);
            float D = dequant_factor(scales[r * sb + c / 16], a, bound);
            float value = oracle_e2m1_decode(code) * D;
            if (out_bf16) ((uint16_t *)out)[r * cols + c] = oracle_f32_to_bf16(value);
            else ((float *)out)[r * cols + c] = value;
        }
    }
}

/* ------------------------------------------------------------------------- */
/* Grouped  [AO-9]: group amax expanded to a per-row amax vector              */
/* ------------------------------------------------------------------------- */

/* group_ends: cumulative row ends, non-decreasing, last == rows.  Returns -1 if
 * they are not (and writes nothing). */
ORACLE_API int oracle_grouped_amax(const float *x, int64_t rows, int64_t cols,
                                   const int64_t *group_ends, int num_groups, float *group_amax,
                                   float *row_amax_expanded, const float *noop)
{
    if (num_groups < 1) return -1;
    int64_t prev = 0;
    for (int g = 0; g < num_groups; ++g) {
        if (group_ends[g] < prev || group_ends[g] > rows) return -1;
        prev = group_ends[g];
    }
    if (prev != rows) return -1;
    if (noop_set(noop)) return 0;
    int64_t start = 0;
    for (int g = 0; g < num_groups; ++g) {
        int64_t end = group_ends[g];
        float t = 0.0f;
        if (end > start) oracle_amax(x + start * cols, end - start, cols, NULL, NULL, &t);
        if (group_amax) group_amax[g] = t;
        if (row_amax_expanded)
            for (int64_t r = start; r < end; ++r) row_amax_expanded[r] = t;
        start = end;
    }
    return 0;
}

/* Grouped rowwise quantize.  mode 0: per-group amax expanded per row; mode 1:
 * plain per-row amax (groups do not change the result).  row_amax receives the
 * [rows] amax vector actually used. */
ORACLE_API int oracle_grouped_quantize_rowwise(const float *x, int64_t rows, int64_t cols,
                                               const int64_t *group_ends, int num_groups,
                                               int mode, float bound, int four_over_six,
                                               uint8_t *codes, uint8_t *scales, float *row_amax,
                                               float *group_amax, const float *noop)
{
    if (bound != 448.0f && bound != 256.0f) return -1;
    float *expanded = (float *)calloc((size_t)(rows > 0 ? rows : 1), sizeof(float));
    float *gam = (float *)calloc((size_t)(num_groups > 0 ? num_groups : 1), sizeof(float));
    int rc = oracle_grouped_amax(x, rows, cols, group_ends, num_groups, gam, expanded, NULL);
    if (rc != 0 || noop_set(noop)) {
        free(expanded);
        free(gam);
        return rc;
    }
    if (mode == ORACLE_ROW_SCALED) oracle_amax(x, rows, cols, expanded, NULL, NULL);
    rc = oracle_quantize(x, rows, cols, ORACLE_ROW_SCALED, bound, four_over_six, 0, expanded, NULL,
                         codes, scales, row_amax, NULL, NULL, NULL, NULL);
    if (group_amax) memcpy(group_amax, gam, (size_t)num_groups * sizeof(float));
    free(expanded);
    free(gam);
    return rc;
}

/* ------------------------------------------------------------------------- */
/* GEMM consumer [TE-3206]: D = dequant(A) x dequant(B)^T                     */
/* ------------------------------------------------------------------------- */

/* The value an NVFP4 element stands for, as a real number: code * decode(scale)
 * * amax / (bound * 6).  In FP64 the product is exact (at most 2 + 4 + 24
 * significant bits) and the division rounds once. */
static double element_value(const uint8_t *codes, const uint8_t *scales, const float *amax,
                            int row_scaled, float bound, int64_t k, int64_t r, int64_t c)
{
    uint8_t byte = codes[r * (k / 2) + c / 2];
    uint8_t code = (c & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15u);
    double sd = (double)oracle_e4m3_decode(scales[r * (k / 16) + c / 16]);
    double a = (double)amax[row_scaled ? r : 0];
    return (double)oracle_e2m1_decode(code) * sd * a / ((double)bound * 6.0);
}

/* The GEMM that consumes two NVFP4 operands (sequence diagram of [TE-3206]: the
 * fprop GEMM scales its output by the activation's per-row amax and the weight's
 * amax; the wgrad GEMM by the outer product of both operands' per-line amax).
 * Its plain definition: the matrix product of the two dequantized operands.
 *   A: codes [m][k/2], scales [m][k/16], amax [m] (a_row_scaled) or [1];
 *   B: codes [n][k/2], scales [n][k/16], amax [n] or [1]  (both K-major, the
 *      layout of a rowwise output, or of a columnwise output for the transposed
 *      operand); k even and a multiple of 16 here.
 *   d [m][n] = sum over c of value_A(i, c) * value_B(j, c), summed in FP64 in
 *   column order; d_abs (optional) [m][n] = sum of |value_A * value_B|, the
 *   magnitude the tests scale their rounding bound by. */
ORACLE_API void oracle_gemm(const uint8_t *a_codes, const uint8_t *a_scales, const float *a_amax,
                            int a_row_scaled, float a_bound, const uint8_t *b_codes,
                            const uint8_t *b_scales, const float *b_amax, int b_row_scaled,
                            float b_bound, int64_t m, int64_t n, int64_t k, double *d,
                            double *d_abs)
{
    double *va = (double *)malloc((size_t)(k > 0 ? k : 1) * sizeof(double));
    for (int64_t i = 0; i < m; ++i) {
        for (int64_t c = 0; c < k; ++c)
            va[c] = element_value(a_codes, a_scales, a_amax, a_row_scaled, a_bound, k, i, c);
        for (int64_t j = 0; j < n; ++j) {
            double s = 0.0, sa = 0.0;
            for (int64_t c = 0; c < k; ++c) {
                double t = va[c] *
                           element_value(b_codes, b_scales, b_amax, b_row_scaled, b_bound, k, j, c);
                s += t;
                sa += fabs(t);
            }
            d[i * n + j] = s;
            if (d_abs) d_abs[i * n + j] = sa;
        }
    }
    free(va);
}

/* ------------------------------------------------------------------------- */
/* R14 random Hadamard transform of the columnwise operand                    */
/* ------------------------------------------------------------------------- */

/* y [rows][cols] = the transform of x [rows][cols] along rows, per column, in
 * blocks of 16 rows (R14).  rows must be a multiple of 16; returns -1 otherwise
 * and writes nothing. */
ORACLE_API int oracle_rht16(const float *x, int64_t rows, int64_t cols, uint32_t sign_mask,
                            float *y)
{
    if (rows < 0 || cols < 0 || rows % 16 != 0) return -1;
    for (int64_t c = 0; c < cols; ++c) {
        for (int64_t r0 = 0; r0 < rows; r0 += 16) {
            float v[16];
            for (int j = 0; j < 16; ++j) {
                float t = x[(r0 + j) * cols + c];
                v[j] = ((sign_mask >> j) & 1u) ? -t : t;
            }
            for (int h = 1; h < 16; h *= 2) {
                for (int i = 0; i < 16; ++i) {
                    if (i & h) continue;
                    float u = v[i], w = v[i + h];
                    v[i] = u + w;
                    v[i + h] = u - w;
                }
            }
            for (int j = 0; j < 16; ++j) y[(r0 + j) * cols + c] = v[j] * 0.25f;
        }
    }
    return 0;
}
