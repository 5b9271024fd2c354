// device_common.cuh -- device helpers shared by the NVFP4 kernels (sm_103a).
//
// Number formats and the encode recipe follow the pages listed in
// include/nvfp4.h: E2M1 codes and E4M3 block scales ("NVFP4: enable row-scaled
// transpose quantization for backward", TransformerEngine PR #3206), the
// four-over-six choice with bound 448/256 ("Add NVFP4 four-over-six grouped GEMM
// for MoE training", torchao PR #9) and the dequantize formula ("Add backward
// overrides and 1x16 weights to NVFP4 four-over-six", torchao PR #8).
//
// Every floating-point step of the recipe is one correctly rounded FP32 operation,
// as in the oracle: explicitly rounded scalar operations (__fmul_rn / __fadd_rn /
// __fsub_rn), packed pairs whose products cannot be contracted (mul2_fma), and two
// divisions replaced by FMA sequences proven to return the correctly rounded
// quotient (div6_short, div_by_scale).  The conversions use the sm_100-family cvt
// instructions (RNE, satfinite).  The four-over-six choice is first tried on an
// estimate of the two errors with a proven bound (fos_bounded_pick); the exact
// sums decide whenever the bound does not.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace nvfp4 {

constexpr int kStatusTimeout = 1;    // NVFP4_DEVICE_TIMEOUT
constexpr int kStatusBadGroups = 2;  // NVFP4_DEVICE_BAD_GROUPS

// ---------------------------------------------------------------- flags / status

__device__ __forceinline__ bool noop_set(const float* noop) {
  return noop != nullptr && *noop == 1.0f;
}

__device__ __forceinline__ void raise_status(int* status, int bits) {
  if (status != nullptr) atomicOr(status, bits);
}

// Group ends are valid when non-decreasing, within [0, M], and the last equals M.
// Must be called by every thread of the block.
__device__ __forceinline__ bool groups_valid(const int64_t* ends, int G, int64_t M) {
  int bad = 0;
  for (int g = threadIdx.x; g < G; g += blockDim.x) {
    const int64_t e = ends[g];
    const int64_t p = g ? ends[g - 1] : 0;
    if (e < p || e > M || (g == G - 1 && e != M)) bad = 1;
  }
  return !__syncthreads_or(bad);
}

// Every group end a multiple of n (groups made of whole tiles).  Every thread of
// the block must call it.
__device__ __forceinline__ bool ends_aligned(const int64_t* ends, int G, int64_t n) {
  int bad = 0;
  for (int g = threadIdx.x; g < G; g += blockDim.x)
    if (ends[g] % n != 0) bad = 1;
  return !__syncthreads_or(bad);
}

// Ragged tokens quantized into a padded layout: group g has ragged rows
// [rag_ends[g-1], rag_ends[g]) of x and padded output rows [pad_ends[g-1],
// pad_ends[g]).  Valid when both are non-decreasing, end at their row counts, every
// padded group is at least as long as its ragged one and starts on a 128-row tile
// boundary.  Every thread of the block must call it.
__device__ __forceinline__ bool pad_layout_valid(const int64_t* rag_ends, const int64_t* pad_ends,
                                                 int G, int64_t in_rows, int64_t out_rows) {
  int bad = 0;
  for (int g = threadIdx.x; g < G; g += blockDim.x) {
    const int64_t re = rag_ends[g], rp = g ? rag_ends[g - 1] : 0;
    const int64_t pe = pad_ends[g], pp = g ? pad_ends[g - 1] : 0;
    if (re < rp || re > in_rows || (g == G - 1 && re != in_rows)) bad = 1;
    if (pe < pp || pe > out_rows || (g == G - 1 && pe != out_rows)) bad = 1;
    if (pe - pp < re - rp || (pp & 127) != 0) bad = 1;
  }
  return !__syncthreads_or(bad);
}

// ---------------------------------------------------------------- BF16 helpers

// The two BF16 halves of a packed pair, widened exactly to FP32.
__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// Lane-wise max of |a|, |b| over packed BF16 pairs.  The sign bits of the
// result are meaningless (xorsign); callers mask them off.
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// max of the two magnitudes held in a packed pair, as FP32 (exact).
__device__ __forceinline__ float bf16x2_hmax_f32(uint32_t v) {
  uint32_t m = v & 0x7fff7fffu;
  uint32_t lo = m << 16, hi = m & 0xffff0000u;
  return __uint_as_float(lo > hi ? lo : hi);
}

// ---------------------------------------------------------------- conversions

// Eight FP32 values -> eight E2M1 codes packed in 32 bits; value k lands in
// nibble k (low nibble of byte 0 = value 0).  RNE, saturating at +-6, sign kept.
// cvt...e2m1x2 puts its first source in the high nibble, so each pair is
// passed high-then-low.
__device__ __forceinline__ uint32_t e2m1x8(float v0, float v1, float v2, float v3, float v4,
                                           float v5, float v6, float v7) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "f"(v0), "f"(v1), "f"(v2), "f"(v3), "f"(v4), "f"(v5), "f"(v6), "f"(v7));
  return r;
}

// FP16 bit pattern -> FP32 (exact).
__device__ __forceinline__ float f16_bits_to_f32(uint32_t h) {
  float f;
  asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"((uint16_t)(h & 0xffffu)));
  return f;
}

// FP32 -> E4M3 byte (RNE, satfinite: anything beyond 448, inf included, gives 448).
__device__ __forceinline__ uint32_t e4m3_byte(float s) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(s));
  return r & 0xffu;
}

// E4M3 byte -> FP32 (exact; every E4M3 value is an FP16 value).
__device__ __forceinline__ float e4m3_value(uint32_t s8) {
  uint32_t h2;
  uint16_t in = (uint16_t)s8;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
  return f16_bits_to_f32(h2);
}

// Two E2M1 codes (one byte, low nibble first) -> their FP32 values (exact).
__device__ __forceinline__ void e2m1x2_values(uint32_t byte, float& lo, float& hi) {
  uint32_t h2;
  uint16_t in = (uint16_t)(byte & 0xffu);
  asm("{\n\t.reg .b8 t;\n\tcvt.u8.u16 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
      : "=r"(h2)
      : "h"(in));
  lo = f16_bits_to_f32(h2);
  hi = f16_bits_to_f32(h2 >> 16);
}

// ---------------------------------------------------------------- recipe steps

// Global encode scale S = F / a (1 if a == 0, FLT_MAX if the quotient overflows).
__device__ __forceinline__ float global_scale(float a, float F) {
  if (a == 0.0f) return 1.0f;
  float S = __fdiv_rn(F, a);
  return S > 3.402823466e38f ? 3.402823466e38f : S;
}

// Block scale byte and encode factor for block max b and target T (6 or 4).
struct BlockEnc {
  uint32_t s8;  // E4M3 byte
  float sd;     // its value
  float e;      // S / sd, or 0
};

// fl(b / 6) for a b with at most 8 significant bits (every BF16 value): the
// product with fl(1/6) = 0x3E2AAAAB, then one FMA correction step (Markstein's
// division with a correctly rounded reciprocal).  The residual b - 6 q0 is exact,
// and for each of the 32639 positive finite BF16 values (subnormal quotients
// included) the corrected quotient equals the IEEE quotient, checked in exact
// rational arithmetic.
__device__ __forceinline__ float div6_short(float b) {
  const float r = __uint_as_float(0x3E2AAAABu);
  const float q0 = __fmul_rn(b, r);
  const float rem = __fmaf_rn(-q0, 6.0f, b);
  return __fmaf_rn(rem, r, q0);
}

// fl(S / sd) for a positive E4M3 value sd (the decoded block scale): Markstein's
// division.  r = rcp.approx(sd) is the correctly rounded reciprocal of each of the
// 126 positive E4M3 values on sm_100-family GPUs (a device test checks all of
// them); q0 = fl(S r), the residual S - q0 sd is exact (one FMA), and
// q1 = fl(q0 + residual r) is the correctly rounded quotient for every FP32
// significand of S and every E4M3 significand of sd (checked exhaustively in exact
// integer arithmetic on the CPU).  The argument needs every intermediate in the
// normal range, so S outside [2^-90, 2^90] takes the IEEE division instead.
__device__ __forceinline__ float div_by_scale(float S, float sd) {
  if (!(S >= 0x1p-90f && S <= 0x1p90f)) return __fdiv_rn(S, sd);
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(sd));
  const float q0 = __fmul_rn(S, r);
  const float rem = __fmaf_rn(-q0, sd, S);
  return __fmaf_rn(rem, r, q0);
}

// SHORT: b is a BF16 value (the block max of BF16 inputs), so fl(b / 6) may use
// div6_short; otherwise it is an IEEE division.
template <int T, bool SHORT = false>
__device__ __forceinline__ BlockEnc block_encode(float b, float S) {
  const float q = (T == 4) ? __fmul_rn(b, 0.25f)  // b/4 == b*0.25 exactly
                  : SHORT  ? div6_short(b)
                           : __fdiv_rn(b, (float)T);
  const float s32 = __fmul_rn(q, S);
  BlockEnc r;
  r.s8 = e4m3_byte(s32);
  r.sd = e4m3_value(r.s8);
  r.e = (r.sd == 0.0f) ? 0.0f : div_by_scale(S, r.sd);
  return r;
}

// Dequantize factor (decode(s8) * a) * F_inv of a block.
__device__ __forceinline__ float dequant_factor(float sd, float a, float F_inv) {
  return __fmul_rn(__fmul_rn(sd, a), F_inv);
}

// Two IEEE round-to-nearest products with one packed FP32x2 multiply (sm_100+):
// (ra, rb) = (fl(a * e), fl(b * e)), each rounded exactly like __fmul_rn.
__device__ __forceinline__ void mul2_rn(float a, float b, float e, float& ra, float& rb) {
  asm("{\n\t.reg .b64 t, u, v;\n\t"
      "mov.b64 t, {%2, %3};\n\t"
      "mov.b64 u, {%4, %4};\n\t"
      "mul.rn.f32x2 v, t, u;\n\t"
      "mov.b64 {%0, %1}, v;\n\t}"
      : "=f"(ra), "=f"(rb)
      : "f"(a), "f"(b), "f"(e));
}

// (ra, rb) = (fl(a0 * b0), fl(a1 * b1)): one packed multiply of two pairs.  The
// compiler may contract a packed multiply into an addition that uses it (mul2_fma is
// the form that cannot be), so this is for products where one rounding fewer is
// harmless.
__device__ __forceinline__ void mul2_pair(float a0, float a1, float b0, float b1, float& ra,
                                          float& rb) {
  asm("{\n\t.reg .b64 a, b, d;\n\t"
      "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
      "mul.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "=f"(ra), "=f"(rb)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// The two four-over-six candidates of a block at once: the steps of block_encode<6>
// and block_encode<4> (and of dequant_factor for each), with the products paired in
// packed multiplies and the two scale bytes converted, and decoded, by one
// instruction each (cvt ...e4m3x2: the second source lands in the low byte, which
// decodes into the low half).  Every value is rounded as in the separate steps.
template <bool SHORT>
__device__ __forceinline__ void block_encode_pair(float b, float S, float a, float F_inv,
                                                  BlockEnc& e6, BlockEnc& e4, float& D6,
                                                  float& D4) {
  const float q6 = SHORT ? div6_short(b) : __fdiv_rn(b, 6.0f);
  const float q4 = __fmul_rn(b, 0.25f);  // b/4 == b*0.25 exactly
  float s6, s4;
  mul2_rn(q6, q4, S, s6, s4);
  uint16_t pr;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(pr) : "f"(s4), "f"(s6));
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(pr));
  e6.s8 = pr & 0xffu;
  e4.s8 = (uint32_t)pr >> 8;
  e6.sd = f16_bits_to_f32(h2);
  e4.sd = f16_bits_to_f32(h2 >> 16);
  e6.e = (e6.sd == 0.0f) ? 0.0f : div_by_scale(S, e6.sd);
  e4.e = (e4.sd == 0.0f) ? 0.0f : div_by_scale(S, e4.sd);
  float t6, t4;
  mul2_rn(e6.sd, e4.sd, a, t6, t4);
  mul2_rn(t6, t4, F_inv, D6, D4);
}

// Eight codes of x[0..7] scaled by e (products via packed multiplies).
__device__ __forceinline__ uint32_t codes8(const float* x, float e) {
  float y[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) mul2_rn(x[2 * i], x[2 * i + 1], e, y[2 * i], y[2 * i + 1]);
  return e2m1x8(y[0], y[1], y[2], y[3], y[4], y[5], y[6], y[7]);
}

// (d0, d1) = (fl(a0 b0), fl(a1 b1)): one fma.rn.f32x2 whose addend is -0.0, which
// leaves every product as the plain rounded product (a nonzero product plus -0 is
// itself, +0 + -0 is +0, -0 + -0 is -0).  negz must hold -0.0 at run time (a kernel
// argument): the compiler then cannot see the addend, so it cannot turn the
// instruction into a multiply and contract that multiply into the add or subtract
// that consumes it (it does so with packed multiplies, despite their .rn).
__device__ __forceinline__ void mul2_fma(float a0, float a1, float b0, float b1, float negz,
                                         float& d0, float& d1) {
  asm("{\n\t.reg .b64 a, b, c, d;\n\t"
      "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\tmov.b64 c, {%6, %6};\n\t"
      "fma.rn.f32x2 d, a, b, c;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(negz));
}

// (d0, d1) = (fl(a0 - b0), fl(a1 - b1)), one packed subtraction.
__device__ __forceinline__ void sub2_rn(float a0, float a1, float b0, float b1, float& d0,
                                        float& d1) {
  asm("{\n\t.reg .b64 a, b, d;\n\t"
      "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
      "sub.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

__device__ __forceinline__ uint32_t byte_perm(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// |value| of the four E2M1 codes in nibbles 0..3 of m (their sign bits clear), as
// FP32, by table lookup: the FP32 pattern of magnitude code k is hi[k] << 24 |
// lo[k] << 16 with hi = 00 3F 3F 3F 40 40 40 40 and lo = 00 00 80 C0 00 40 80 C0
// (0, 0.5, 1, 1.5, 2, 3, 4, 6).  Two byte permutes look up the hi and lo bytes of
// the four codes; one more per value places them, its two low bytes copying the
// (clear) sign bit of a hi byte.
__device__ __forceinline__ void e2m1_magnitudes4(uint32_t m, float (&v)[4]) {
  const uint32_t hi = byte_perm(0x3F3F3F00u, 0x40404040u, m);
  const uint32_t lo = byte_perm(0xC0800000u, 0xC0804000u, m);
  v[0] = __uint_as_float(byte_perm(lo, hi, 0x40CCu));
  v[1] = __uint_as_float(byte_perm(lo, hi, 0x51DDu));
  v[2] = __uint_as_float(byte_perm(lo, hi, 0x62EEu));
  v[3] = __uint_as_float(byte_perm(lo, hi, 0x73FFu));
}

// Four-over-six error of one candidate: err continued over 16 values in order,
// err = fl(err + fl(d_i * d_i)) with d_i = fl(x_i - fl(v_i * D)), v_i the value of
// code i (c0: values 0..7, c1: 8..15) and D the candidate's dequantize factor.
// Two ways of decoding, so that the two candidates load different pipes:
//   sse16_magnitudes: from |x| and the codes' magnitudes (table lookup).  The
//     sign of a nonzero code is the sign of its x, so |x_i| - |v_i D| is d_i up to
//     its sign, and d_i * d_i is the same.
//   sse16_signed: from x and the signed values (hardware E2M1 -> FP16 conversion).
// The dequantized values, the differences and the squares are formed two at a time
// (packed); the additions stay one at a time, in order.
__device__ __forceinline__ float sse16_magnitudes(float err, const float* x, uint32_t c0,
                                                  uint32_t c1, float D, float negz) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t w = q < 2 ? c0 : c1;
    float v[4], g[4], d[4], p[4];
    e2m1_magnitudes4(((q & 1) ? (w >> 16) : w) & 0x7777u, v);
    mul2_fma(v[0], v[1], D, D, negz, g[0], g[1]);
    mul2_fma(v[2], v[3], D, D, negz, g[2], g[3]);
    sub2_rn(fabsf(x[4 * q]), fabsf(x[4 * q + 1]), g[0], g[1], d[0], d[1]);
    sub2_rn(fabsf(x[4 * q + 2]), fabsf(x[4 * q + 3]), g[2], g[3], d[2], d[3]);
    mul2_fma(d[0], d[1], d[0], d[1], negz, p[0], p[1]);
    mul2_fma(d[2], d[3], d[2], d[3], negz, p[2], p[3]);
#pragma unroll
    for (int k = 0; k < 4; ++k) err = __fadd_rn(err, p[k]);
  }
  return err;
}

__device__ __forceinline__ float sse16_signed(float err, const float* x, uint32_t c0, uint32_t c1,
                                              float D, float negz) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t w = (q < 2 ? c0 : c1) >> (16 * (q & 1));
    float v[4], g[4], d[4], p[4];
    e2m1x2_values(w, v[0], v[1]);
    e2m1x2_values(w >> 8, v[2], v[3]);
    mul2_fma(v[0], v[1], D, D, negz, g[0], g[1]);
    mul2_fma(v[2], v[3], D, D, negz, g[2], g[3]);
    sub2_rn(x[4 * q], x[4 * q + 1], g[0], g[1], d[0], d[1]);
    sub2_rn(x[4 * q + 2], x[4 * q + 3], g[2], g[3], d[2], d[3]);
    mul2_fma(d[0], d[1], d[0], d[1], negz, p[0], p[1]);
    mul2_fma(d[2], d[3], d[2], d[3], negz, p[2], p[3]);
#pragma unroll
    for (int k = 0; k < 4; ++k) err = __fadd_rn(err, p[k]);
  }
  return err;
}

// (sa, sb) = (fl(r0 r0 + sa), fl(r1 r1 + sb)): one packed FMA.
__device__ __forceinline__ void sq2_acc(float r0, float r1, float& sa, float& sb) {
  asm("{\n\t.reg .b64 r, s;\n\t"
      "mov.b64 r, {%2, %3};\n\tmov.b64 s, {%0, %1};\n\t"
      "fma.rn.f32x2 s, r, r, s;\n\tmov.b64 {%0, %1}, s;\n\t}"
      : "+f"(sa), "+f"(sb)
      : "f"(r0), "f"(r1));
}

// Codes of x[0..7] scaled by e (as codes8), and the squared residuals of the scaled
// values added into (sa, sb), even i into sa and odd i into sb: r_i = fl(v_i - y_i)
// with y_i = fl(x_i e) and v_i the value of code i (its FP16 form from the hardware
// conversion, subtracted from y_i in one mixed-precision instruction), then
// fl(r_i r_i + s) as packed FMAs.  The sum only estimates the candidate's error;
// fos_bounded_pick bounds how far the estimate can be from the exact sum.
__device__ __forceinline__ uint32_t codes8_residual(const float* x, float e, float& sa,
                                                    float& sb) {
  float y[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) mul2_rn(x[2 * i], x[2 * i + 1], e, y[2 * i], y[2 * i + 1]);
  uint32_t w, h[4];
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %8, %7;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %10, %9;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %12, %11;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %4, b3;\n\t}"
      : "=r"(w), "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "f"(y[0]), "f"(y[1]), "f"(y[2]), "f"(y[3]), "f"(y[4]), "f"(y[5]), "f"(y[6]),
        "f"(y[7]));
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float r0, r1;  // v - y: FP16 value minus FP32 value, one rounding each
    asm("{\n\t.reg .f16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
        "sub.rn.f32.f16 %0, a, %3;\n\tsub.rn.f32.f16 %1, b, %4;\n\t}"
        : "=f"(r0), "=f"(r1)
        : "r"(h[k]), "f"(y[2 * k]), "f"(y[2 * k + 1]));
    sq2_acc(r0, r1, sa, sb);
  }
  return w;
}

// Four-over-six without the exact error sums, where a bound settles the choice.
// Per candidate T, with D its dequantize factor and A = sum (y_i - v_i)^2 from
// codes8_residual, E' = fl(fl(D D) A) estimates the exact error err (the
// definition's FP32 sum of fl(x_i - fl(v_i D))^2 in element order).  Both are
// within a few rounding errors of the real sum of t_i^2, t_i = x_i - v_i D:
//   * e D = 1 + phi with |phi| <= 5u (u = 2^-24: the roundings of S = F/a, e = S/sd,
//     fl(1/F), fl(sd a) and D), so D y_i = x_i (1 + theta_i), |theta_i| <= 6u;
//   * fl(b e) <= 6.5 bounds every |y_i| by 6.5 and every |y_i - v_i| by 1 (half the
//     E2M1 spacing, or the distance to 6 past it), so |t_i| <= D (1 + 40u) and
//     b <= 6.5001 D;
//   * forward error analysis of the 16 terms then gives |err - sum t_i^2| <= 528.1 u D^2
//     (the products, differences and squares, and the in-order sum of 16 non-negative
//     terms) and |E' - sum t_i^2| <= 1568.3 u D^2 (the x_i theta_i terms, the rounding
//     of each r_i, the two 8-term FMA chains and their sum, the final product), plus
//     underflow terms below 100 * 2^-150 (D^2 + 1) that D in [2^-62, 2^61] makes
//     negligible against 2^-12 D^2.
// So |err - E'| <= 2096.4 u D^2 < 2^-12 D^2 / 1.9, and err4 < err6 holds whenever
// E'4 - E'6 < -2^-12 (D4^2 + D6^2) (after the roundings of that comparison), and fails
// whenever the difference exceeds +2^-12 (D4^2 + D6^2).  Returns 1 (T = 4), 0 (T = 6)
// or -1: the estimates are too close, or the block is outside the ranges above (inf,
// NaN and saturated blocks included), and the exact sums decide.  The ranges take
// three comparisons: fl(b/4) >= fl(b/6) and every rounding step is monotonic, so the
// T = 4 scale is at least the T = 6 one, hence D4 >= D6 and fl(b e4) <= fl(b e6).
// The paired products round as the scalar ones (a contraction into the difference or
// the sum that follows would only drop a rounding, which the margin covers).
__device__ __forceinline__ int fos_bounded_pick(float b, float e6, float D6, float D4, float A6,
                                                float A4) {
  const float y6 = __fmul_rn(b, e6);
  if (!(y6 <= 6.5f && D6 >= 0x1p-62f && D4 <= 0x1p61f)) return -1;
  float q6, q4, E6, E4;
  mul2_pair(D6, D4, D6, D4, q6, q4);
  mul2_pair(q6, q4, A6, A4, E6, E4);
  const float diff = __fsub_rn(E4, E6);
  const float tol = __fmul_rn(0x1p-12f, __fadd_rn(q4, q6));
  return diff < -tol ? 1 : (diff > tol ? 0 : -1);
}

// The same transform of two blocks at once (two adjacent columns), every add,
// subtract and product formed as a packed pair: each half of add.rn.f32x2 /
// sub.rn.f32x2 / mul.rn.f32x2 is the IEEE operation of the scalar steps, so a and b
// come out bit for bit as rht16_block would make them.
__device__ __forceinline__ void rht16_block2(float (&a)[16], float (&b)[16], uint32_t mask) {
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const uint32_t sb = ((mask >> j) & 1u) << 31;
    a[j] = __uint_as_float(__float_as_uint(a[j]) ^ sb);
    b[j] = __uint_as_float(__float_as_uint(b[j]) ^ sb);
  }
#pragma unroll
  for (int h = 1; h < 16; h *= 2) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (i & h) continue;
      float s0, s1, d0, d1;
      asm("{\n\t.reg .b64 u, w, s, d;\n\t"
          "mov.b64 u, {%4, %5};\n\tmov.b64 w, {%6, %7};\n\t"
          "add.rn.f32x2 s, u, w;\n\tsub.rn.f32x2 d, u, w;\n\t"
          "mov.b64 {%0, %1}, s;\n\tmov.b64 {%2, %3}, d;\n\t}"
          : "=f"(s0), "=f"(s1), "=f"(d0), "=f"(d1)
          : "f"(a[i]), "f"(b[i]), "f"(a[i + h]), "f"(b[i + h]));
      a[i] = s0, b[i] = s1, a[i + h] = d0, b[i + h] = d1;
    }
  }
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    float p0, p1;
    asm("{\n\t.reg .b64 u, q, d;\n\t"
        "mov.b64 u, {%2, %3};\n\tmov.b64 q, {%4, %4};\n\t"
        "mul.rn.f32x2 d, u, q;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(p0), "=f"(p1)
        : "f"(a[j]), "f"(b[j]), "f"(0.25f));
    a[j] = p0, b[j] = p1;
  }
}

// Random Hadamard transform of one 16-value block, in place: v = (1/4) H16 diag(s) v
// with H16 the Sylvester Hadamard matrix and s_j = -1 where bit j of mask is set.
// FP32 steps in this order: the signs (exact), the four natural-order butterfly
// stages (h = 1, 2, 4, 8: entries i and i + h, i & h == 0, become u + v and u - v),
// then the product with 0.25.
__device__ __forceinline__ void rht16_block(float (&v)[16], uint32_t mask) {
#pragma unroll
  for (int j = 0; j < 16; ++j)
    v[j] = __uint_as_float(__float_as_uint(v[j]) ^ (((mask >> j) & 1u) << 31));
#pragma unroll
  for (int h = 1; h < 16; h *= 2) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (i & h) continue;
      const float u = v[i], w = v[i + h];
      v[i] = __fadd_rn(u, w);
      v[i + h] = __fsub_rn(u, w);
    }
  }
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = __fmul_rn(v[j], 0.25f);
}

// The exact four-over-six choice of one block: 1 when the T = 4 error (codes d0, d1,
// factor D4) is below the T = 6 error (codes c0, c1, factor D6).  Out of line: it
// runs only for the blocks that fos_bounded_pick leaves open, and its code is then
// not repeated in every unrolled block of the encode loops.
static __device__ __noinline__ int fos_exact_pick(float4 xa, float4 xb, float4 xc,
                                                  float4 xd, uint32_t c0, uint32_t c1,
                                                  uint32_t d0, uint32_t d1, float D6, float D4,
                                                  float negz) {
  const float x[16] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w,
                       xc.x, xc.y, xc.z, xc.w, xd.x, xd.y, xd.z, xd.w};
  const float err4 = sse16_signed(0.0f, x, d0, d1, D4, negz);
  const float err6 = sse16_magnitudes(0.0f, x, c0, c1, D6, negz);
  return err4 < err6;
}

// Both four-over-six candidates of a block, their codes, and the choice the bounded
// estimate makes: pick 1 (T = 4), 0 (T = 6) or -1 (open: the exact sums decide).
struct FosEstimate {
  uint32_t c0, c1, d0, d1;  // T = 6 and T = 4 code words
  uint32_t s6, s4;          // scale bytes
  float D6, D4;             // dequantize factors
  int pick;
};
template <bool SHORT>
__device__ __forceinline__ FosEstimate fos_estimate(const float* x, float b, float S, float a,
                                                    float F_inv) {
  FosEstimate f;
  BlockEnc e6, e4;
  block_encode_pair<SHORT>(b, S, a, F_inv, e6, e4, f.D6, f.D4);
  float s6a = 0.0f, s6b = 0.0f, s4a = 0.0f, s4b = 0.0f;
  f.c0 = codes8_residual(x, e6.e, s6a, s6b);
  f.c1 = codes8_residual(x + 8, e6.e, s6a, s6b);
  f.d0 = codes8_residual(x, e4.e, s4a, s4b);
  f.d1 = codes8_residual(x + 8, e4.e, s4a, s4b);
  f.s6 = e6.s8;
  f.s4 = e4.s8;
  // one scale byte: the same codes and errors, and a tie keeps T = 6
  f.pick = e4.s8 == e6.s8 ? 0
                          : fos_bounded_pick(b, e6.e, f.D6, f.D4, __fadd_rn(s6a, s6b),
                                             __fadd_rn(s4a, s4b));
  return f;
}

// Four-over-six with the open blocks left to the caller: writes the chosen codes and
// returns the scale byte; for an open block (open = true) those of T = 6, which the
// caller replaces with the exact choice (quantize16_exact) before storing them.
template <bool SHORT>
__device__ __forceinline__ uint32_t quantize16_est(const float* x, float b, float S, float a,
                                                   float F_inv, uint32_t& c0, uint32_t& c1,
                                                   bool& open) {
  const FosEstimate f = fos_estimate<SHORT>(x, b, S, a, F_inv);
  open = f.pick < 0;
  const bool four = f.pick > 0;
  c0 = four ? f.d0 : f.c0;
  c1 = four ? f.d1 : f.c1;
  return four ? f.s4 : f.s6;
}

// The exact four-over-six choice of one block (the in-order error sums of both
// candidates): writes the codes and returns the scale byte.
template <bool SHORT>
__device__ __forceinline__ uint32_t quantize16_exact(const float* x, float b, float S, float a,
                                                     float F_inv, float negz, uint32_t& c0,
                                                     uint32_t& c1) {
  BlockEnc e6, e4;
  float D6, D4;
  block_encode_pair<SHORT>(b, S, a, F_inv, e6, e4, D6, D4);
  c0 = codes8(x, e6.e);
  c1 = codes8(x + 8, e6.e);
  if (e4.s8 == e6.s8) return e6.s8;
  const uint32_t d0 = codes8(x, e4.e), d1 = codes8(x + 8, e4.e);
  const float err4 = sse16_signed(0.0f, x, d0, d1, D4, negz);
  const float err6 = sse16_magnitudes(0.0f, x, c0, c1, D6, negz);
  if (err4 < err6) {
    c0 = d0;
    c1 = d1;
    return e4.s8;
  }
  return e6.s8;
}

// Quantize 16 FP32 values of one block whose max |x| is b: writes the two code
// words (value k in nibble k) and returns the scale byte.  FOS: four-over-six
// (needs the line amax a and F_inv for the error of each candidate, and negz =
// -0.0 at run time, see mul2_fma).  The choice is that of the exact in-order error
// sums: the bounded estimate settles it where it provably agrees with them, the
// exact sums (out of line) elsewhere.
template <bool FOS, bool SHORT = false>
__device__ __forceinline__ uint32_t quantize16(const float* x, float b, float S, float a,
                                               float F_inv, float negz, uint32_t& c0,
                                               uint32_t& c1) {
  if constexpr (!FOS) {
    const BlockEnc e6 = block_encode<6, SHORT>(b, S);
    c0 = codes8(x, e6.e);
    c1 = codes8(x + 8, e6.e);
    return e6.s8;
  } else {
    const FosEstimate f = fos_estimate<SHORT>(x, b, S, a, F_inv);
    int pick = f.pick;
    if (pick < 0)  // the exact sums
      pick = fos_exact_pick(make_float4(x[0], x[1], x[2], x[3]),
                            make_float4(x[4], x[5], x[6], x[7]),
                            make_float4(x[8], x[9], x[10], x[11]),
                            make_float4(x[12], x[13], x[14], x[15]), f.c0, f.c1, f.d0, f.d1,
                            f.D6, f.D4, negz);
    c0 = pick ? f.d0 : f.c0;
    c1 = pick ? f.d1 : f.c1;
    return pick ? f.s4 : f.s6;
  }
}

// Codes of 16 values with a given encode factor (16x16 blocks: the tile's scale).
__device__ __forceinline__ void codes16(const float* x, float e, uint32_t& c0, uint32_t& c1) {
  c0 = codes8(x, e);
  c1 = codes8(x + 8, e);
}

// ---------------------------------------------------------------- mbarrier / TMA

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait on an mbarrier phase: gives up after limit_ns of %globaltimer
// (2 s unless a self-test passes a shorter limit) or 2^28 polls, whichever comes
// first, and returns false; the caller then records a timeout and leaves.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint64_t limit_ns = 2000000000ull) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0; it < (1u << 28); ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 255u && global_timer_ns() - t0 > limit_ns) break;
  }
  return false;
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2D tiled TMA load global -> shared, completing on `bar`; x = innermost (column)
// coordinate, y = row coordinate.  policy: an L2 cache policy from createpolicy.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int32_t x, int32_t y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// 2D tiled TMA store shared -> global (bulk-group completion).  Elements outside
// the tensor's extent are not written.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int32_t x,
                                             int32_t y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group.L2::cache_hint"
      " [%0, {%1, %2}], [%3], %4;" ::"l"(reinterpret_cast<uint64_t>(map)),
      "r"(x), "r"(y), "r"(smem_addr(src)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// wait until the committed bulk stores have finished reading shared memory
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// wait until at most N committed bulk-store groups are still reading shared memory
template <int N>
__device__ __forceinline__ void bulk_wait_read_allow() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// wait until the committed bulk stores are complete
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// make generic-proxy shared-memory writes visible to the async (TMA) proxy
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 16-byte global load with an L2 cache policy (read-only data).
__device__ __forceinline__ uint4 ldg_v4_policy(const void* p, uint64_t policy) {
  uint4 v;
  asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(policy));
  return v;
}

// One 32-byte store (a whole L2 sector); p must be 32-byte aligned.
__device__ __forceinline__ void stg_v8(void* p, const uint32_t* w) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]),
               "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

// Streaming stores for outputs that are not read again by this kernel.
__device__ __forceinline__ void stg_v4_cs(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ void sts_v4(void* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(smem_addr(p)), "r"(a), "r"(b),
               "r"(c), "r"(d)
               : "memory");
}
__device__ __forceinline__ void sts_v2(void* p, uint32_t a, uint32_t b) {
  asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(smem_addr(p)), "r"(a), "r"(b) : "memory");
}
// One full 32-byte sector per thread (256-bit store, sm_100+); p 32-byte aligned.
__device__ __forceinline__ void stg_v8_cs(void* p, const uint32_t* w) {
  asm volatile("st.global.cs.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]),
               "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

// Stores that should stay in L2 until their 32-byte sector is complete (scale
// bytes written in pieces by consecutive tiles).
__device__ __forceinline__ void stg_v2_keep(void* p, uint32_t a, uint32_t b, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v2.u32 [%0], {%1, %2}, %3;" ::"l"(p), "r"(a), "r"(b),
               "l"(pol)
               : "memory");
}
__device__ __forceinline__ void stg_u32_keep(void* p, uint32_t a, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.u32 [%0], %1, %2;" ::"l"(p), "r"(a), "l"(pol) : "memory");
}
__device__ __forceinline__ void stg_u16_keep(void* p, uint32_t a, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.u16 [%0], %1, %2;" ::"l"(p), "h"((uint16_t)a), "l"(pol)
               : "memory");
}
__device__ __forceinline__ void stg_v2_cs(void* p, uint32_t a, uint32_t b) {
  asm volatile("st.global.cs.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(a), "r"(b) : "memory");
}
__device__ __forceinline__ void stg_u32_cs(void* p, uint32_t a) {
  asm volatile("st.global.cs.u32 [%0], %1;" ::"l"(p), "r"(a) : "memory");
}
__device__ __forceinline__ void stg_u16_cs(void* p, uint32_t a) {
  asm volatile("st.global.cs.u16 [%0], %1;" ::"l"(p), "h"((uint16_t)a) : "memory");
}

// Write n bytes (n <= 16) of the little-endian words w[] to p, with the widest
// stores the alignment of p and n allow.
__device__ __forceinline__ void store_bytes(uint8_t* p, const uint32_t* w, int n) {
  if (n == 16 && (reinterpret_cast<uintptr_t>(p) & 15u) == 0) {
    stg_v4_cs(p, make_uint4(w[0], w[1], w[2], w[3]));
    return;
  }
  if (n == 8 && (reinterpret_cast<uintptr_t>(p) & 7u) == 0) {
    stg_v2_cs(p, w[0], w[1]);
    return;
  }
  if ((n & 3) == 0 && (reinterpret_cast<uintptr_t>(p) & 3u) == 0) {
    for (int i = 0; i < n / 4; ++i) stg_u32_cs(p + 4 * i, w[i]);
    return;
  }
  for (int i = 0; i < n; ++i) p[i] = (uint8_t)(w[i >> 2] >> (8 * (i & 3)));
}

}  // namespace nvfp4
