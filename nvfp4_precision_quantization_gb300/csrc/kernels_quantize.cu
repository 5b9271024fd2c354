// kernels_quantize.cu -- NVFP4 encode of x into rowwise and/or columnwise codes.
//
// "NVFP4: enable row-scaled transpose quantization for backward"
// (TransformerEngine PR #3206, description and sequence diagram): one pass emits
// the rowwise (fprop) and the columnwise / transposed (wgrad) output, with the
// per-row amax scaling rows and the per-column amax scaling columns.
// Four-over-six and the 1x16 / 16x16 block choice follow "Add NVFP4
// four-over-six grouped GEMM for MoE training" (torchao PR #9) and "Add
// backward overrides and 1x16 weights to NVFP4 four-over-six" (torchao PR #8).
//
// Design (sm_103a): a persistent grid of 2 CTAs per SM; each CTA walks its chunk
// of the strip-major tile order backwards (see tile_pipeline.cuh).  Warp 8 is the
// producer: lane 0 issues the two TMA boxes of a tile into a 3-stage ring, then
// the warp stages the tile's per-row and per-column amax and global scale
// S = F / amax in shared memory (one division per row / column instead of one per
// thread).  Warps 0-7 consume: with both directions, warps 0-3 encode rows (a
// thread = one row, 128 bytes of each box) and warps 4-7 encode columns (a thread
// = a column pair over 64 rows).  Each consumer warp releases a stage through an
// "empty" mbarrier, so warps never wait for each other.  Shared-memory reads are
// bank-conflict free under the swizzle.  Output paths (OutMode):
//   sector  code pitches multiples of 32 bytes: whole 32-byte sectors, one 256-bit
//           store per thread; with both directions (no four-over-six) the two
//           halves of a row's or a column's run sit in neighbouring lanes (PAIRED),
//           columnwise only the two 32-row halves of a column's run do (CPAIR).
//           A rowwise thread keeps its row's scale bytes for the 4 tiles of a
//           super-strip row and writes the 32-byte sector once; columnwise scale
//           bytes are collected per 4 tile rows or written per tile with an L2
//           evict_last hint so the sector completes in L2.
//   TMA     code pitches multiples of 16 bytes: per-warp shared-memory staging and
//           TMA tensor stores.
//   direct  any pitch: the widest stores the pitch and base allow on interior
//           tiles (both directions, no four-over-six: rowwise rows staged per warp
//           and written back row by row), bytes on edge tiles.
// Four-over-six with 1x16 blocks and both directions is launched as two
// single-direction passes (see launch_quantize).  RHT: the columnwise warps
// transform each 16-row block in registers before encoding it.
#include <algorithm>
#include <cstring>

#include "device_common.cuh"
#include "internal.h"
#include "tile_pipeline.cuh"

namespace nvfp4 {

namespace {


struct EncodeArgs {
  const void* x;
  int64_t M, K;
  TileGrid grid;
  uint8_t* row_codes;
  uint8_t* row_scales;
  const float* row_amax;
  uint8_t* col_codes;
  uint8_t* col_scales;
  const float* col_amax;
  int64_t row_cpitch, row_spitch, col_cpitch, col_spitch;
  int row_scaled;
  float F, F_inv;
  float* copy_dst;
  const float* copy_src;
  const float* noop;
  int* status;
  const int64_t* ends;
  int G;
  int full_m, full_n;  // tiles with tm < full_m and tn < full_n lie entirely inside x
  int vec_ok;          // output pitches / bases allow the 16-byte stores
  // widest store (16, 8, 4, 2 or 1 bytes) that the pitch and base of each output
  // allow: row codes, row scales, column codes, column scales
  int rc_g, rs_g, cc_g, cs_g;
  // ragged x into a padded output (grouped tokens): group g's output rows
  // [pad_ends[g-1], pad_ends[g]) take x rows from rag_ends[g-1] on, as many as the
  // group has; the rest of the group's rows are padding (zero codes and scales).
  const int64_t* pad_ends;
  const int64_t* rag_ends;
  int64_t in_rows;
  // grouped columns: col_amax is [G][K] (or [G] with col_grouped_pt), one row per group
  // of ends (multiples of kTileRows); the producer stages each tile's column scales
  int col_grouped, col_grouped_pt;
  uint32_t rht_mask;  // sign mask of the columnwise transform (RHT kernels only)
  int row_scale_groups;  // rowwise scales of a super-strip row go out as one 32-byte sector
  int col_scale_sectors;  // columnwise scales of four tile rows go out as one 32-byte sector
  float neg_zero;         // -0.0, the addend of the four-over-six products (see mul2_fma)
  int reverse_walk;       // walk each chunk the other way (a second pass over x)
  int load_normal;        // x's tiles at the normal L2 priority (else evict-first)
};

// Per-stage values staged by the producer: the tile's per-row and per-column
// global scales, and (four-over-six or 16x16 blocks only) the amax values and the
// 16x16 sub-tile scales.  FULL = false keeps only the scales (smaller footprint).
template <bool FULL>
struct StageMetaT {
  float rowS[kTileRows], colS[128];
  int nrows;  // rows of the tile that hold data (the rest are padding rows)
  float rowA_[FULL ? kTileRows : 1], colA_[FULL ? 128 : 1];
  uint32_t s2d_[FULL ? 64 : 1];
  float e2d_[FULL ? 64 : 1];
  __device__ __forceinline__ float rowA(int i) const {
    if constexpr (FULL) return rowA_[i];
    else return 0.0f;
  }
  __device__ __forceinline__ float colA(int i) const {
    if constexpr (FULL) return colA_[i];
    else return 0.0f;
  }
  __device__ __forceinline__ uint32_t s2d(int i) const {
    if constexpr (FULL) return s2d_[i];
    else return 0u;
  }
  __device__ __forceinline__ float e2d(int i) const {
    if constexpr (FULL) return e2d_[i];
    else return 0.0f;
  }
  __device__ __forceinline__ void set_rowA(int i, float v) {
    if constexpr (FULL) rowA_[i] = v;
  }
  __device__ __forceinline__ void set_colA(int i, float v) {
    if constexpr (FULL) colA_[i] = v;
  }
  __device__ __forceinline__ void set_2d(int i, uint32_t s8, float e) {
    if constexpr (FULL) {
      s2d_[i] = s8;
      e2d_[i] = e;
    }
  }
};

__device__ __forceinline__ uint4 lds128(const uint8_t* p) {
  return *reinterpret_cast<const uint4*>(p);
}

// max |.| over 8 packed BF16 pairs, as FP32
__device__ __forceinline__ float absmax8_bf16(const uint4& v0, const uint4& v1) {
  uint32_t m = absmax_bf16x2(absmax_bf16x2(absmax_bf16x2(v0.x, v0.y), absmax_bf16x2(v0.z, v0.w)),
                             absmax_bf16x2(absmax_bf16x2(v1.x, v1.y), absmax_bf16x2(v1.z, v1.w)));
  return bf16x2_hmax_f32(m);
}

__device__ __forceinline__ float absmax16_f32(const float* x) {
  float b = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) b = fmaxf(b, fabsf(x[i]));
  return b;
}

// Edge tiles: write the first n (<= 32) bytes of the little-endian words w0..w7,
// one byte at a time (bounds and alignment of the destination are arbitrary).
// The words are passed by value so that the fast path keeps them in registers.
__device__ __noinline__ void store_tail(uint8_t* p, int n, uint32_t w0, uint32_t w1, uint32_t w2,
                                        uint32_t w3, uint32_t w4, uint32_t w5, uint32_t w6,
                                        uint32_t w7) {
  for (int i = 0; i < n; ++i) {
    const int k = i >> 2;
    const uint32_t w = k == 0 ? w0 : k == 1 ? w1 : k == 2 ? w2 : k == 3 ? w3
                     : k == 4 ? w4 : k == 5 ? w5 : k == 6 ? w6 : w7;
    p[i] = (uint8_t)(w >> (8 * (i & 3)));
  }
}

template <int NW>
__device__ __forceinline__ void store_tail_words(uint8_t* p, const uint32_t (&w)[NW], int n) {
  store_tail(p, n, w[0], NW > 1 ? w[1 < NW ? 1 : 0] : 0u, NW > 2 ? w[2 < NW ? 2 : 0] : 0u,
             NW > 3 ? w[3 < NW ? 3 : 0] : 0u, NW > 4 ? w[4 < NW ? 4 : 0] : 0u,
             NW > 5 ? w[5 < NW ? 5 : 0] : 0u, NW > 6 ? w[6 < NW ? 6 : 0] : 0u,
             NW > 7 ? w[7 < NW ? 7 : 0] : 0u);
}

template <bool FOS, bool B2D, bool SHORT>
__device__ __forceinline__ uint32_t encode_block(const float* x, float b, float S, float a,
                                                 float F_inv, float negz, uint32_t s2d, float e2d,
                                                 uint32_t& c0, uint32_t& c1) {
  if constexpr (B2D) {
    codes16(x, e2d, c0, c1);
    return s2d;
  } else {
    return quantize16<FOS, SHORT>(x, b, S, a, F_inv, negz, c0, c1);
  }
}

// ---------------------------------------------------------------- rowwise

// Block j of a box row (row pointer rowp, swizzle sw) as 16 FP32 values; returns
// the block max (MAX) or 0.
template <typename T, bool MAX>
__device__ __forceinline__ float load_row_block(const uint8_t* rowp, int j, int sw,
                                                float (&x)[16]) {
  if constexpr (sizeof(T) == 2) {
    const uint4 v0 = lds128(rowp + (((2 * j) ^ sw) << 4));
    const uint4 v1 = lds128(rowp + (((2 * j + 1) ^ sw) << 4));
    const uint32_t u[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      x[2 * i] = bf16_lo(u[i]);
      x[2 * i + 1] = bf16_hi(u[i]);
    }
    return MAX ? absmax8_bf16(v0, v1) : 0.0f;
  } else {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint4 v = lds128(rowp + (((4 * j + k) ^ sw) << 4));
      x[4 * k] = __uint_as_float(v.x);
      x[4 * k + 1] = __uint_as_float(v.y);
      x[4 * k + 2] = __uint_as_float(v.z);
      x[4 * k + 3] = __uint_as_float(v.w);
    }
    return MAX ? absmax16_f32(x) : 0.0f;
  }
}

// The exact four-over-six choice of block j of a box row, its values read again from
// the stage: codes in x, y, scale byte in z.  For the blocks the bound left open;
// out of line, so that its code stays out of the encode loop.
template <typename T>
__device__ __noinline__ uint3 row_block_exact(const uint8_t* rowp, int j, int sw, float S,
                                              float A, float F_inv, float negz) {
  float x[16];
  const float b = load_row_block<T, true>(rowp, j, sw, x);
  uint3 r;
  r.z = quantize16_exact<sizeof(T) == 2>(x, b, S, A, F_inv, negz, r.x, r.y);
  return r;
}

// Codes and scales of row r of boxes [b0, b0 + NBOX): w[box][word], sc[box].
// Rows / columns outside x were zero-filled by the load, so they encode to 0;
// the caller decides what is stored.  rot = 4 (BF16) makes step j read block
// j ^ 2 of the box row (its results land in the slots of block j).  With
// four-over-six the bound settles each block; the blocks it leaves open are redone
// with the exact sums after the loop (one test per row instead of one per block).
template <typename T, int NBOX, bool FOS, bool B2D, typename M>
__device__ __forceinline__ void rowwise_compute(const uint8_t* stage, const M& m,
                                                const EncodeArgs& a, int r, int b0, float S_t,
                                                float A_t,
                                                uint32_t (&w)[NBOX][TileGeo<T>::BOXC / 8],
                                                uint32_t (&sc)[NBOX], int rot = 0) {
  using G = TileGeo<T>;
  constexpr int NB = G::BOXC / 16;  // blocks per box row
  constexpr bool DEFER = FOS && !B2D;
  const float S = a.row_scaled ? m.rowS[r] : S_t;
  const float A = a.row_scaled ? m.rowA(r) : A_t;
  const int sw = (r & 7) ^ rot;
  uint32_t open_mask = 0;
#pragma unroll
  for (int bi = 0; bi < NBOX; ++bi) {
    const int box = b0 + bi;
    const uint8_t* rowp = stage + box * kBoxBytes + r * 128;
    sc[bi] = 0;
#pragma unroll
    for (int j = 0; j < NB; ++j) {
      float x[16];
      const float b = load_row_block<T, !B2D>(rowp, j, sw, x);
      if constexpr (DEFER) {
        bool open;
        sc[bi] |= quantize16_est<sizeof(T) == 2>(x, b, S, A, a.F_inv, w[bi][2 * j],
                                                 w[bi][2 * j + 1], open)
                  << (8 * j);
        open_mask |= (uint32_t)open << (bi * NB + j);
      } else {
        uint32_t s2 = 0;
        float e2 = 0.0f;
        if constexpr (B2D) {
          const int sub = (r >> 4) * (G::TILEC / 16) + box * NB + j;
          s2 = m.s2d(sub);
          e2 = m.e2d(sub);
        }
        sc[bi] |= encode_block<FOS, B2D, sizeof(T) == 2>(x, b, S, A, a.F_inv, a.neg_zero, s2,
                                                         e2, w[bi][2 * j], w[bi][2 * j + 1])
                  << (8 * j);
      }
    }
  }
  if constexpr (DEFER) {
    if (open_mask != 0) {
#pragma unroll
      for (int bi = 0; bi < NBOX; ++bi) {
#pragma unroll
        for (int j = 0; j < NB; ++j) {
          if (open_mask & (1u << (bi * NB + j))) {
            const uint3 e = row_block_exact<T>(stage + (b0 + bi) * kBoxBytes + r * 128, j, sw,
                                               S, A, a.F_inv, a.neg_zero);
            w[bi][2 * j] = e.x;
            w[bi][2 * j + 1] = e.y;
            sc[bi] = (sc[bi] & ~(0xffu << (8 * j))) | (e.z << (8 * j));
          }
        }
      }
    }
  }
}

// NW code words (4 NW bytes) to p: 16-byte stores when g >= 16, 4-byte stores when
// g >= 4, else bytes (g: the widest store that the output's pitch and base allow, the
// same for every thread of a launch).
template <int NW>
__device__ __forceinline__ void store_words_g(uint8_t* p, const uint32_t* w, int g) {
  if (NW % 4 == 0 && g >= 16) {
#pragma unroll
    for (int q = 0; q < NW / 4; ++q)
      stg_v4_cs(p + 16 * q, make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]));
  } else if (g >= 4) {
#pragma unroll
    for (int q = 0; q < NW; ++q) stg_u32_cs(p + 4 * q, w[q]);
  } else {
#pragma unroll 4
    for (int i = 0; i < 4 * NW; ++i) p[i] = (uint8_t)(w[i >> 2] >> (8 * (i & 3)));
  }
}

// N (1, 2 or 4) scale bytes to p, one store when g >= N, else bytes; kept in L2 (scale
// sectors fill up over several tiles).
template <int N>
__device__ __forceinline__ void store_scales_g(uint8_t* p, uint32_t s, int g, uint64_t keep) {
  if (g >= N) {
    if constexpr (N == 4) stg_u32_keep(p, s, keep);
    else if constexpr (N == 2) stg_u16_keep(p, s, keep);
    else p[0] = (uint8_t)s;
  } else {
#pragma unroll
    for (int i = 0; i < N; ++i) p[i] = (uint8_t)(s >> (8 * i));
  }
}

// Direct stores of one row's codes and scales (no TMA for the outputs): whole
// stores of the widest size the output allows on tiles inside x, bytes on edge tiles.
template <typename T, int NBOX>
__device__ __forceinline__ void rowwise_store(const EncodeArgs& a, int r, int b0, int tm, int tn,
                                              const uint32_t (&w)[NBOX][TileGeo<T>::BOXC / 8],
                                              const uint32_t (&sc)[NBOX], bool interior) {
  using G = TileGeo<T>;
  constexpr int NB = G::BOXC / 16;
  const int64_t gr = (int64_t)tm * kTileRows + r;
  if (gr >= a.M) return;
#pragma unroll
  for (int bi = 0; bi < NBOX; ++bi) {
    const int64_t gc0 = (int64_t)tn * G::TILEC + (b0 + bi) * G::BOXC;
    if (gc0 >= a.K) return;
    uint8_t* cp = a.row_codes + gr * a.row_cpitch + gc0 / 2;
    uint8_t* sp = a.row_scales + gr * a.row_spitch + gc0 / 16;
    if (interior) {
      store_words_g<2 * NB>(cp, w[bi], a.rc_g);
      store_scales_g<NB>(sp, sc[bi], a.rs_g, policy_evict_last());
    } else {
      const int64_t rem = a.K - gc0;
      const int ncols = rem < G::BOXC ? (int)rem : G::BOXC;
      store_tail_words<2 * NB>(cp, w[bi], (ncols + 1) / 2);
      store_tail(sp, (ncols + 15) / 16, sc[bi], 0, 0, 0, 0, 0, 0, 0);
    }
  }
}

// Rowwise stores through per-warp shared-memory staging (direct output path, tiles
// inside x).  A thread holds one row's codes and scales of the tile; stored from
// registers, each warp request would touch 32 rows, one piece of a sector each.
// Instead the warp stages its rows one box at a time (both directions: 32 rows of
// one box per phase) or 16 rows at a time (rowwise only: one box per thread) and
// writes them back row by row: a request then covers a few whole rows with stores
// of the widest size that the output's pitch and base allow (codes: 4, 8 or 16
// bytes, rc_g >= 4; scales: 1 to 4 bytes, rs_g).
template <typename T, int NBOX>
struct RowStage {
  static constexpr int NB = TileGeo<T>::BOXC / 16;  // scale bytes of a row per box
  static constexpr int UB = TileGeo<T>::BOXC / 2;   // code bytes of a row per box
  static constexpr int NR = NBOX == 2 ? 32 : 16;    // rows per phase
  // staging pitch of a row: an odd number of 16-byte units (no bank conflicts on
  // the 16-byte writes of 8 consecutive lanes)
  static constexpr int RP = (UB / 16) % 2 == 0 ? UB + 16 : UB;
  static constexpr int kBytes = NR * RP + NR * NB;  // per warp
};

template <int W>
__device__ __forceinline__ void stg_piece(uint8_t* p, const uint8_t* src) {
  if constexpr (W == 16) {
    const uint4 v = *reinterpret_cast<const uint4*>(src);
    stg_v4_cs(p, v);
  } else if constexpr (W == 8) {
    const uint2 v = *reinterpret_cast<const uint2*>(src);
    stg_v2_cs(p, v.x, v.y);
  } else {
    stg_u32_cs(p, *reinterpret_cast<const uint32_t*>(src));
  }
}

template <int SW>
__device__ __forceinline__ void stg_scale_piece(uint8_t* p, const uint8_t* src, uint64_t keep) {
  if constexpr (SW == 4) {
    stg_u32_keep(p, *reinterpret_cast<const uint32_t*>(src), keep);
  } else if constexpr (SW == 2) {
    stg_u16_keep(p, *reinterpret_cast<const uint16_t*>(src), keep);
  } else {
    *p = *src;
  }
}

// NR staged rows of B bytes each (staging pitch P) to row0, row0 + pitch, ...:
// B / W pieces per row, taken by consecutive lanes, 32 / (B / W) rows per request.
template <int NR, int B, int P, int W, bool SCALES>
__device__ __forceinline__ void staged_rows_out(uint8_t* row0, int64_t pitch, const uint8_t* st,
                                                int lane, uint64_t keep) {
  constexpr int PPR = B / W, RPI = 32 / PPR < NR ? 32 / PPR : NR;
  if (lane >= RPI * PPR) return;
  const int j = lane / PPR, i = lane % PPR;
  uint8_t* dst = row0 + j * pitch + i * W;
  const uint8_t* src = st + j * P + i * W;
  const int64_t step = RPI * pitch;
#pragma unroll 1
  for (int it = 0; it < NR / RPI; ++it, dst += step, src += RPI * P) {
    if constexpr (SCALES) stg_scale_piece<W>(dst, src, keep);
    else stg_piece<W>(dst, src);
  }
}

// r: this thread's row of the tile (rows r - lane .. r - lane + 31 belong to the
// warp), b0: its first box.  Every lane of the warp must call this.
template <typename T, int NBOX>
__device__ __forceinline__ void rowwise_store_staged(const EncodeArgs& a, uint8_t* st, int r,
                                                     int b0, int tm, int tn, int lane,
                                                     const uint32_t (&w)[NBOX][TileGeo<T>::BOXC / 8],
                                                     const uint32_t (&sc)[NBOX]) {
  using G = TileGeo<T>;
  using RS = RowStage<T, NBOX>;
  constexpr int NB = RS::NB, UB = RS::UB, NR = RS::NR, RP = RS::RP;
  static_assert(UB % 16 == 0, "code bytes of a row per box: a multiple of 16");
  uint8_t* sst = st + NR * RP;
  const int64_t gc0 = (int64_t)tn * G::TILEC + b0 * G::BOXC;
  const uint64_t keep = policy_evict_last();
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    const int bi = NBOX == 2 ? p : 0;
    if (NBOX == 2 || (lane >> 4) == p) {
      const int j = NBOX == 2 ? lane : (lane & 15);
#pragma unroll
      for (int q = 0; q < UB / 16; ++q)
        sts_v4(st + j * RP + 16 * q, w[bi][4 * q], w[bi][4 * q + 1], w[bi][4 * q + 2],
               w[bi][4 * q + 3]);
      if constexpr (NB == 4) *reinterpret_cast<uint32_t*>(sst + j * 4) = sc[bi];
      else *reinterpret_cast<uint16_t*>(sst + j * 2) = (uint16_t)sc[bi];
    }
    __syncwarp();
    const int64_t gr0 = (int64_t)tm * kTileRows + (r - lane) + (NBOX == 2 ? 0 : 16 * p);
    const int64_t gc = gc0 + (NBOX == 2 ? p * G::BOXC : 0);
    uint8_t* crow = a.row_codes + gr0 * a.row_cpitch + gc / 2;
    uint8_t* srow = a.row_scales + gr0 * a.row_spitch + gc / 16;
    if (a.rc_g >= 16) staged_rows_out<NR, UB, RP, 16, false>(crow, a.row_cpitch, st, lane, keep);
    else if (a.rc_g >= 8) staged_rows_out<NR, UB, RP, 8, false>(crow, a.row_cpitch, st, lane, keep);
    else staged_rows_out<NR, UB, RP, 4, false>(crow, a.row_cpitch, st, lane, keep);
    constexpr int SW4 = NB >= 4 ? 4 : 1;
    if (NB >= 4 && a.rs_g >= 4) staged_rows_out<NR, NB, NB, SW4, true>(srow, a.row_spitch, sst, lane, keep);
    else if (a.rs_g >= 2) staged_rows_out<NR, NB, NB, 2, true>(srow, a.row_spitch, sst, lane, keep);
    else staged_rows_out<NR, NB, NB, 1, true>(srow, a.row_spitch, sst, lane, keep);
    __syncwarp();  // the staging is read before the next phase overwrites it
  }
}

// Scales only (the codes went out through the TMA store).
template <typename T, int NBOX>
__device__ __forceinline__ void rowwise_store_scales(const EncodeArgs& a, int r, int b0, int tm,
                                                     int tn, const uint32_t (&sc)[NBOX],
                                                     bool fast) {
  using G = TileGeo<T>;
  constexpr int NB = G::BOXC / 16;
  const int64_t gr = (int64_t)tm * kTileRows + r;
  if (gr >= a.M) return;
  const int64_t gc0 = (int64_t)tn * G::TILEC + b0 * G::BOXC;
  uint8_t* sp = a.row_scales + gr * a.row_spitch + gc0 / 16;
  if (fast) {
    const uint64_t keep = policy_evict_last();
    if constexpr (NBOX == 2 && NB == 4) stg_v2_keep(sp, sc[0], sc[1], keep);
    else if constexpr (NBOX == 1 && NB == 4) stg_u32_keep(sp, sc[0], keep);
    else {
#pragma unroll
      for (int bi = 0; bi < NBOX; ++bi) stg_u16_keep(sp + 2 * bi, sc[bi], keep);
    }
  } else {
#pragma unroll
    for (int bi = 0; bi < NBOX; ++bi) {
      const int64_t rem = a.K - (gc0 + bi * G::BOXC);
      if (rem <= 0) return;
      const int ncols = rem < G::BOXC ? (int)rem : G::BOXC;
      store_tail(sp + bi * NB, (ncols + 15) / 16, sc[bi], 0, 0, 0, 0, 0, 0, 0);
    }
  }
}

// ---------------------------------------------------------------- columnwise

// Codes and scales of column pair (cl, cl + 1) over rows [rb0, rb0 + RG).
// RHT_PAIR: the two columns' transforms as packed pairs (fewer instructions, more
// registers: used where the register budget allows, the columnwise-only kernels).
// The exact four-over-six choice of one column's 16-row block (column c of the pair
// at base, row i at base + i * 128 + coff[i & 7]), read again from the stage: codes in
// x, y, scale byte in z.  For the blocks the bound left open; out of line.
template <typename T>
__device__ __noinline__ uint3 col_block_exact(const uint8_t* base, int4 ca, int4 cb, int c,
                                              float S, float A, float F_inv, float negz) {
  const int32_t coff[8] = {ca.x, ca.y, ca.z, ca.w, cb.x, cb.y, cb.z, cb.w};
  float x[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    if constexpr (sizeof(T) == 2) {
      const uint32_t v = *reinterpret_cast<const uint32_t*>(base + i * 128 + coff[i & 7]);
      x[i] = c ? bf16_hi(v) : bf16_lo(v);
    } else {
      const float2 v = *reinterpret_cast<const float2*>(base + i * 128 + coff[i & 7]);
      x[i] = c ? v.y : v.x;
    }
  }
  const float b = absmax16_f32(x);
  uint3 r;
  r.z = quantize16_exact<sizeof(T) == 2>(x, b, S, A, F_inv, negz, r.x, r.y);
  return r;
}

template <typename T, int RG, bool FOS, bool B2D, bool RHT = false, bool RHT_PAIR = false,
          typename M>
__device__ __forceinline__ void colwise_compute(const uint8_t* stage, const M& m,
                                                const EncodeArgs& a, int cl, int rb0,
                                                const int32_t (&coff)[8], float S_t, float A_t,
                                                uint32_t (&w0)[RG / 8], uint32_t (&w1)[RG / 8],
                                                uint32_t& sc0, uint32_t& sc1) {
  using G = TileGeo<T>;
  constexpr int NB = RG / 16;
  const float S0 = a.row_scaled ? m.colS[cl] : S_t;
  const float S1 = a.row_scaled ? m.colS[cl + 1] : S_t;
  const float A0 = a.row_scaled ? m.colA(cl) : A_t;
  const float A1 = a.row_scaled ? m.colA(cl + 1) : A_t;
  // four-over-six: the blocks the bound leaves open are redone after the loop
  constexpr bool DEFER = FOS && !B2D && !RHT;
  uint32_t open_mask = 0;
  sc0 = sc1 = 0;
#pragma unroll
  for (int jb = 0; jb < NB; ++jb) {
    const uint8_t* base = stage + (rb0 + 16 * jb) * 128;
    float x0[16], x1[16];
    float b0 = 0.0f, b1 = 0.0f;
    if constexpr (sizeof(T) == 2) {
      uint32_t v[16];
#pragma unroll
      for (int i = 0; i < 16; ++i)
        v[i] = *reinterpret_cast<const uint32_t*>(base + i * 128 + coff[i & 7]);
      if constexpr (!B2D) {
        uint32_t t8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) t8[i] = absmax_bf16x2(v[2 * i], v[2 * i + 1]);
        uint32_t mm =
            absmax_bf16x2(absmax_bf16x2(absmax_bf16x2(t8[0], t8[1]), absmax_bf16x2(t8[2], t8[3])),
                          absmax_bf16x2(absmax_bf16x2(t8[4], t8[5]), absmax_bf16x2(t8[6], t8[7])));
        mm &= 0x7fff7fffu;
        b0 = __uint_as_float(mm << 16);
        b1 = __uint_as_float(mm & 0xffff0000u);
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        x0[i] = bf16_lo(v[i]);
        x1[i] = bf16_hi(v[i]);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float2 v = *reinterpret_cast<const float2*>(base + i * 128 + coff[i & 7]);
        x0[i] = v.x;
        x1[i] = v.y;
      }
      if constexpr (!B2D) {
        b0 = absmax16_f32(x0);
        b1 = absmax16_f32(x1);
      }
    }
    if constexpr (RHT) {
      // the block of each column replaced by its transform; its max from the result
      if constexpr (RHT_PAIR) {
        rht16_block2(x0, x1, a.rht_mask);
      } else {
        rht16_block(x0, a.rht_mask);
        rht16_block(x1, a.rht_mask);
      }
      b0 = absmax16_f32(x0);
      b1 = absmax16_f32(x1);
    }
    uint32_t s2 = 0;
    float e2 = 0.0f;
    if constexpr (B2D) {
      const int sub = ((rb0 >> 4) + jb) * (G::TILEC / 16) + cl / 16;
      s2 = m.s2d(sub);
      e2 = m.e2d(sub);
    }
    // SHORT (the BF16 block-max division shortcut) holds only for BF16 block maxima
    constexpr bool SHORT = sizeof(T) == 2 && !RHT;
    if constexpr (DEFER) {
      bool o0, o1;
      sc0 |= quantize16_est<SHORT>(x0, b0, S0, A0, a.F_inv, w0[2 * jb], w0[2 * jb + 1], o0)
             << (8 * jb);
      sc1 |= quantize16_est<SHORT>(x1, b1, S1, A1, a.F_inv, w1[2 * jb], w1[2 * jb + 1], o1)
             << (8 * jb);
      open_mask |= ((uint32_t)o0 | ((uint32_t)o1 << 1)) << (2 * jb);
    } else {
      sc0 |= encode_block<FOS, B2D, SHORT>(x0, b0, S0, A0, a.F_inv, a.neg_zero, s2, e2,
                                           w0[2 * jb], w0[2 * jb + 1])
             << (8 * jb);
      sc1 |= encode_block<FOS, B2D, SHORT>(x1, b1, S1, A1, a.F_inv, a.neg_zero, s2, e2,
                                           w1[2 * jb], w1[2 * jb + 1])
             << (8 * jb);
    }
  }
  if constexpr (DEFER) {
    if (open_mask != 0) {
      const int4 ca = make_int4(coff[0], coff[1], coff[2], coff[3]);
      const int4 cb = make_int4(coff[4], coff[5], coff[6], coff[7]);
#pragma unroll
      for (int jb = 0; jb < NB; ++jb) {
        const uint8_t* base = stage + (rb0 + 16 * jb) * 128;
        if (open_mask & (1u << (2 * jb))) {
          const uint3 e = col_block_exact<T>(base, ca, cb, 0, S0, A0, a.F_inv, a.neg_zero);
          w0[2 * jb] = e.x;
          w0[2 * jb + 1] = e.y;
          sc0 = (sc0 & ~(0xffu << (8 * jb))) | (e.z << (8 * jb));
        }
        if (open_mask & (2u << (2 * jb))) {
          const uint3 e = col_block_exact<T>(base, ca, cb, 1, S1, A1, a.F_inv, a.neg_zero);
          w1[2 * jb] = e.x;
          w1[2 * jb + 1] = e.y;
          sc1 = (sc1 & ~(0xffu << (8 * jb))) | (e.z << (8 * jb));
        }
      }
    }
  }
}

// Scales of a column pair (and, unless the codes went out through TMA, codes).
template <typename T, int RG, bool CODES>
__device__ __forceinline__ void colwise_store(const EncodeArgs& a, int cl, int rb0, int tm, int tn,
                                              const uint32_t (&w0)[RG / 8],
                                              const uint32_t (&w1)[RG / 8], uint32_t sc0,
                                              uint32_t sc1, bool interior) {
  using G = TileGeo<T>;
  constexpr int NB = RG / 16;
  const int64_t gc = (int64_t)tn * G::TILEC + cl;
  const int64_t gr0 = (int64_t)tm * kTileRows + rb0;
  if (gc >= a.K || gr0 >= a.M) return;
  const bool has1 = gc + 1 < a.K;
  uint8_t* c0p = a.col_codes + gc * a.col_cpitch + gr0 / 2;
  uint8_t* s0p = a.col_scales + gc * a.col_spitch + gr0 / 16;
  if (interior) {
    if constexpr (CODES) {
      store_words_g<2 * NB>(c0p, w0, a.cc_g);
      store_words_g<2 * NB>(c0p + a.col_cpitch, w1, a.cc_g);
    }
    const uint64_t keep = policy_evict_last();
    store_scales_g<NB>(s0p, sc0, a.cs_g, keep);
    store_scales_g<NB>(s0p + a.col_spitch, sc1, a.cs_g, keep);
  } else {
    const int64_t rem = a.M - gr0;
    const int nrows = rem < RG ? (int)rem : RG;
    const int nbytes = (nrows + 1) / 2, nsc = (nrows + 15) / 16;
    if constexpr (CODES) store_tail_words<2 * NB>(c0p, w0, nbytes);
    store_tail(s0p, nsc, sc0, 0, 0, 0, 0, 0, 0, 0);
    if (has1) {
      if constexpr (CODES) store_tail_words<2 * NB>(c0p + a.col_cpitch, w1, nbytes);
      store_tail(s0p + a.col_spitch, nsc, sc1, 0, 0, 0, 0, 0, 0, 0);
    }
  }
}

// ---------------------------------------------------------------- 16x16 sub-tiles

// One consumer thread per 16x16 sub-tile picks its scale (with four-over-six:
// its target, by the error summed in row-major order inside the sub-tile).
template <typename T, bool FOS, typename M>
__device__ __forceinline__ void subtile_scales(const uint8_t* stage, M& m, float S,
                                               float amax, float F_inv, float negz, int t) {
  using G = TileGeo<T>;
  constexpr int SUBC = G::TILEC / 16, NSUB = (kTileRows / 16) * SUBC;
  if (t >= NSUB) return;
  const int sr = t / SUBC, sc = t % SUBC;
  constexpr int CH = (int)sizeof(T);  // 16-byte chunks per 16 values (2 or 4)
  const int box = (sc * 16) / G::BOXC;
  const int cb = ((sc * 16) % G::BOXC) * (int)sizeof(T) / 16;
  auto load_row = [&](int i, float* x) {
    const int r = sr * 16 + i;
    const uint8_t* rowp = stage + box * kBoxBytes + r * 128;
#pragma unroll
    for (int k = 0; k < CH; ++k) {
      const uint4 v = lds128(rowp + ((((cb + k) ^ (r & 7))) << 4));
      const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if constexpr (sizeof(T) == 2) {
          x[8 * k + 2 * q] = bf16_lo(u[q]);
          x[8 * k + 2 * q + 1] = bf16_hi(u[q]);
        } else {
          x[4 * k + q] = __uint_as_float(u[q]);
        }
      }
    }
  };
  float b = 0.0f;
  for (int i = 0; i < 16; ++i) {
    float x[16];
    load_row(i, x);
    b = fmaxf(b, absmax16_f32(x));
  }
  BlockEnc e6 = block_encode<6, sizeof(T) == 2>(b, S);
  if constexpr (FOS) {
    BlockEnc e4 = block_encode<4>(b, S);
    const float D6 = dequant_factor(e6.sd, amax, F_inv);
    const float D4 = dequant_factor(e4.sd, amax, F_inv);
    float err6 = 0.0f, err4 = 0.0f;
    for (int i = 0; i < 16; ++i) {
      float x[16];
      load_row(i, x);
      uint32_t c0, c1, d0, d1;
      codes16(x, e6.e, c0, c1);
      codes16(x, e4.e, d0, d1);
      err6 = sse16_magnitudes(err6, x, c0, c1, D6, negz);
      err4 = sse16_signed(err4, x, d0, d1, D4, negz);
    }
    if (err4 < err6) e6 = e4;
  }
  m.set_2d(t, e6.s8, e6.e);
}

// 16x16 sub-tile scales without four-over-six (BF16): the scale needs only the
// sub-tile's max, so all 256 consumer threads take part.  Thread (row r, box h)
// reads its 128-byte box row (the rowwise access pattern: conflict free), takes
// the max of each of its 4 blocks of 16 values, and the 16 rows of a sub-tile --
// lanes 0-15 or 16-31 of the warp -- combine theirs with 4 shuffle steps; the
// first lane of the 16 encodes the 4 sub-tile scales.
template <typename M>
__device__ __forceinline__ void subtile_scales_max(const uint8_t* stage, M& m, float S, int t) {
  const int r = t & (kTileRows - 1), h = t >> 7;
  const uint8_t* rowp = stage + h * kBoxBytes + r * 128;
  const int sw = r & 7;
  float bmax[4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
    bmax[j] = absmax8_bf16(lds128(rowp + (((2 * j) ^ sw) << 4)),
                           lds128(rowp + (((2 * j + 1) ^ sw) << 4)));
#pragma unroll
  for (int o = 1; o < 16; o <<= 1)
#pragma unroll
    for (int j = 0; j < 4; ++j) bmax[j] = fmaxf(bmax[j], __shfl_xor_sync(0xffffffffu, bmax[j], o));
  if ((r & 15) == 0) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const BlockEnc e = block_encode<6, true>(bmax[j], S);
      m.set_2d((r >> 4) * (TileGeo<uint16_t>::TILEC / 16) + h * 4 + j, e.s8, e.e);
    }
  }
}

// x row of the tile's first row and how many of its rows hold data: tile row tm of
// the output, through the padded layout when x is ragged.
__device__ __forceinline__ void tile_source(const EncodeArgs& a, int tm, int64_t& src_row0,
                                            int& nvalid) {
  const int64_t p0 = (int64_t)tm * kTileRows;
  if (a.pad_ends == nullptr) {
    src_row0 = p0;
    nvalid = (int)(a.M - p0 < kTileRows ? a.M - p0 : kTileRows);
    return;
  }
  int lo = 0, hi = a.G;  // group: the first whose padded end lies beyond p0
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (a.pad_ends[mid] <= p0) lo = mid + 1;
    else hi = mid;
  }
  const int64_t pstart = lo ? a.pad_ends[lo - 1] : 0, rstart = lo ? a.rag_ends[lo - 1] : 0;
  const int64_t have = a.rag_ends[lo] - rstart - (p0 - pstart);
  src_row0 = rstart + (p0 - pstart);
  nvalid = (int)(have < 0 ? 0 : have < kTileRows ? have : kTileRows);
}

// ---------------------------------------------------------------- the kernel

// Staging bytes per consumer warp for the TMA stores of its codes, per buffer.
constexpr int kStagingPerWarp = 2048;
#ifndef NVFP4_STAGING_BUFFERS
#define NVFP4_STAGING_BUFFERS 2
#endif
// Each consumer warp alternates between kStagingBuffers staging buffers, so a
// tile's codes can be written while the previous tile's TMA store is still
// reading its buffer.
constexpr int kStagingBuffers = NVFP4_STAGING_BUFFERS;

// Output paths for the codes: kOutDirect = 16-byte stores from registers (any
// alignment, edge tiles), kOutTma = per-warp shared-memory staging and TMA tensor
// stores, kOutSector = one 32-byte sector per thread with 256-bit stores.
enum OutMode : int { kOutDirect = 0, kOutTma = 1, kOutSector = 2 };

// Rowwise staging of the direct path (RowStage), used with both directions and
// without four-over-six: the 4 rowwise warps' 1664 bytes each.  (With four-over-six
// or rowwise only, the extra steps cost more than the whole rows save: measured on
// the MoE rowwise encode, 0.527 -> 0.549 ms per step.)
constexpr int kRowStageWarps = 4;
constexpr int kRowStagePerWarp = 1664;

template <int OUTM>
struct EncodeSmem {
  static constexpr int kStagesUsed = OUTM == kOutTma ? 2 : 3;
  static constexpr int kBytes =
      kStagesUsed * kTileBytes +
      (OUTM == kOutTma ? kConsumerWarps * kStagingPerWarp * kStagingBuffers : 0) +
      (OUTM == kOutDirect ? kRowStageWarps * kRowStagePerWarp : 0) + 1024;
};

// TOUT: codes leave through per-warp shared-memory staging and TMA tensor stores
// (full lines instead of one 16-byte partial sector per thread); the ring then
// has 2 stages so that 2 CTAs still fit on an SM.
template <typename T, bool ROW, bool COL, bool FOS, bool B2D, bool TMA, int OUTM,
          bool RHT = false>
__global__ void __launch_bounds__(kPipeThreads, 2)
    k_encode(const __grid_constant__ CUtensorMap tmap, const __grid_constant__ CUtensorMap map_rc,
             const __grid_constant__ CUtensorMap map_cc, EncodeArgs a) {
  using G = TileGeo<T>;
  constexpr int NS = EncodeSmem<OUTM>::kStagesUsed;
  constexpr bool TOUT = OUTM == kOutTma;
  constexpr bool SECT = OUTM == kOutSector;
  constexpr bool STAGED_ROWS = OUTM == kOutDirect && ROW && COL && !FOS;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full[NS];
  __shared__ __align__(8) uint64_t empty[NS];
  __shared__ StageMetaT<FOS || B2D> meta[NS];
  // Columnwise scale bytes of the first three tile rows of a column's 32-byte
  // scale sector, per tile of the super-strip row and column, held until the CTA
  // reaches the fourth (4 tiles apart in its walk): [tile][column][visit][row half].
  __shared__ uint32_t csb[SECT && ROW && COL && sizeof(T) == 2 && !FOS && !B2D ? TileGrid::kGroup : 1]
                         [SECT && ROW && COL && sizeof(T) == 2 && !FOS && !B2D ? 128 : 1][3][2];
  __shared__ volatile int abort_flag;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  if (noop_set(a.noop)) return;
  if constexpr (ROW && !COL) {
    if (a.pad_ends != nullptr) {
      if (!pad_layout_valid(a.rag_ends, a.pad_ends, a.G, a.in_rows, a.M)) return;
    } else if (a.ends != nullptr && !groups_valid(a.ends, a.G, a.M)) {
      return;
    }
  } else if (a.ends != nullptr && !groups_valid(a.ends, a.G, a.M)) {
    return;
  }
  if constexpr (COL && !ROW) {
    if (a.col_grouped && !ends_aligned(a.ends, a.G, kTileRows)) return;
  }
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int begin, end;
  a.grid.chunk(blockIdx.x, gridDim.x, begin, end);
  const int count = end - begin;
  // the amax kernel walks this chunk the other way (a second encode pass: the same way)
  const bool fwd = ((blockIdx.x & 1) != 0) != (a.reverse_walk != 0);
  if (TMA && warp == kConsumerWarps && lane == 0) prefetch_tmap(&tmap);  // while barriers are set up
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 2);  // producer: TMA arrival (with bytes) + staged-meta arrival
      mbar_init(&empty[s], kConsumerWarps);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  pdl_launch_dependents();
  if (count <= 0) return;

  if (warp == kConsumerWarps) {
    // ---------------- producer warp
    // x's tiles at the normal L2 priority (both directions, x larger than L2): the
    // evict-first output lines then leave L2 (written back) first, during this pass,
    // and fewer dirty lines are left to the next kernel; else evict-first
    const uint64_t policy = a.load_normal ? policy_evict_normal() : policy_evict_first();
    // tiles are issued in order k = 0, 1, ...: one cursor steps along with them
    TileCursor ci;
    ci.seek(a.grid, a.grid.walk(begin, end, 0, fwd));
    uint32_t no_load = 0;  // stages whose tile is all padding: nothing loaded
    // the source of the last tile row looked up (the 4 tiles of a super-strip row share it)
    int src_tm = -1, src_n = 0;
    int64_t src_row = 0;
    auto issue = [&](int k) {
      const int tm = ci.tm, tn = ci.tn();
      ci.step(a.grid, fwd);
      const int s = k % NS;
      uint8_t* stage = smem + s * kTileBytes;
      int64_t src0 = (int64_t)tm * kTileRows;
      int nvalid = kTileRows;
      if constexpr (ROW && !COL) {  // a ragged x is quantized rowwise only
        if (tm != src_tm) {
          tile_source(a, tm, src_row, src_n);
          src_tm = tm;
        }
        src0 = src_row;
        nvalid = src_n;
        if (lane == 0) meta[s].nrows = nvalid;
        if (nvalid == 0) {
          no_load |= 1u << s;
          return;
        }
        no_load &= ~(1u << s);
      } else if constexpr (!TMA) {
        tile_source(a, tm, src0, nvalid);
      }
      if constexpr (TMA) {
        if (lane == 0) issue_tile<T>(stage, &tmap, &full[s], (int)src0, tn, policy);
      } else {
        plain_load_tile<T>(stage, static_cast<const T*>(a.x), a.K, src0, nvalid, tn, lane);
      }
    };
    // the ring starts empty: fill it before waiting for the amax values
    for (int k = 0; k < NS && k < count; ++k) issue(k);
    pdl_wait();  // the amax values come from the preceding kernel
    constexpr int RPL = kTileRows / 32, CPL = G::TILEC / 32;  // rows / columns per lane
    const bool rs = a.row_scaled != 0;
    // amax of a tile's rows and columns, loaded one tile ahead so that their L2
    // latency overlaps the wait for the next free stage
    float ra[RPL], ca[CPL];
    // the amax of tile k are loaded in order k = 0, 1, ... as well
    int grp_tm = -1, grp = 0;  // grouped columns: group of tile row grp_tm
    TileCursor cm;
    cm.seek(a.grid, a.grid.walk(begin, end, 0, fwd));
    auto load_amax = [&](int k, float (&r_)[RPL], float (&c_)[CPL]) {
      (void)k;
      const int tm = cm.tm, tn = cm.tn();
      cm.step(a.grid, fwd);
      if (ROW) {
#pragma unroll
        for (int i = 0; i < RPL; ++i) {
          const int64_t gr = (int64_t)tm * kTileRows + lane + 32 * i;
          r_[i] = gr < a.M ? a.row_amax[gr] : 0.0f;
        }
      }
      if (COL) {
        const float* cam = a.col_amax;
        bool one = false;  // one amax for the whole tile (a group's tensor amax)
        if constexpr (COL && !ROW) {
          if (a.col_grouped) {
            if (tm != grp_tm) {  // the group of this tile row (ends are whole tiles)
              int lo = 0, hi = a.G;
              while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (a.ends[mid] <= (int64_t)tm * kTileRows) lo = mid + 1;
                else hi = mid;
              }
              grp = lo;
              grp_tm = tm;
            }
            cam += a.col_grouped_pt ? (int64_t)grp : (int64_t)grp * a.K;
            one = a.col_grouped_pt != 0;
          }
        }
#pragma unroll
        for (int i = 0; i < CPL; ++i) {
          const int64_t gc = (int64_t)tn * G::TILEC + lane + 32 * i;
          c_[i] = gc < a.K ? cam[one ? 0 : gc] : 0.0f;
        }
      }
    };
    if (rs) load_amax(0, ra, ca);
    int issued = count < NS ? count : NS;
    for (int k = 0; k < count; ++k) {
      const int s = k % NS;
      if (k >= NS) {
        const bool ok = mbar_wait_bounded(&empty[s], (uint32_t)(((k / NS) - 1) & 1));
        if (!ok || abort_flag) {
          if (lane == 0 && !ok) {
            abort_flag = 1;
            raise_status(a.status, kStatusTimeout);
          }
          break;
        }
        issue(k);
        issued = k + 1;
      }
      if (rs) {
        float rn[RPL], cn[CPL];
        if (k + 1 < count) load_amax(k + 1, rn, cn);
        auto& m = meta[s];
        if (ROW) {
#pragma unroll
          for (int i = 0; i < RPL; ++i) {
            m.set_rowA(lane + 32 * i, ra[i]);
            m.rowS[lane + 32 * i] = global_scale(ra[i], a.F);
          }
        }
        if (COL) {
#pragma unroll
          for (int i = 0; i < CPL; ++i) {
            m.set_colA(lane + 32 * i, ca[i]);
            m.colS[lane + 32 * i] = global_scale(ca[i], a.F);
          }
        }
        if (k + 1 < count) {
#pragma unroll
          for (int i = 0; i < RPL; ++i) ra[i] = rn[i];
#pragma unroll
          for (int i = 0; i < CPL; ++i) ca[i] = cn[i];
        }
      }
      __syncwarp();
      if (lane == 0) {
        // stands in for the TMA arrival when nothing was loaded by TMA
        if (!TMA || (ROW && !COL && (no_load >> s & 1u))) mbar_arrive(&full[s]);
        mbar_arrive(&full[s]);
      }
    }
    // let copies still in flight land before the CTA's shared memory is released
    if (abort_flag && lane == 0)
      for (int k = issued - NS > 0 ? issued - NS : 0; k < issued; ++k)
        (void)mbar_wait_bounded(&full[k % NS], (uint32_t)((k / NS) & 1));
    return;
  }

  // ---------------- consumer warps
  pdl_wait();
  float S_r = 1.0f, A_r = 0.0f, S_c = 1.0f, A_c = 0.0f;
  if (!a.row_scaled) {
    if (ROW) {
      A_r = a.row_amax[0];
      S_r = global_scale(A_r, a.F);
    }
    if (COL) {
      A_c = a.col_amax[0];
      S_c = global_scale(A_c, a.F);
    }
    if (blockIdx.x == 0 && tid == 0 && a.copy_dst != nullptr) *a.copy_dst = *a.copy_src;
  }
  constexpr bool BOTH = ROW && COL;
  constexpr int NBOX = BOTH ? 2 : 1;          // boxes per rowwise thread
  constexpr int NP = G::TILEC / 2;            // column pairs per tile
  constexpr int NCT = BOTH ? 128 : 256;       // columnwise threads
  constexpr int RG = kTileRows / (NCT / NP);  // rows per columnwise thread
  constexpr int RWB = NBOX * G::BOXC / 2;     // code bytes per rowwise thread (TMA box width)
  constexpr int CWB = RG / 2;                 // code bytes per column (TMA box width)
  const bool is_row = ROW && (!BOTH || tid < 128);
  const int ct = BOTH ? tid - 128 : tid;      // columnwise thread index
  // Columnwise thread mapping.  PAIRED (sector stores, both directions, 1x16,
  // no four-over-six): lane bit 0 selects the row half and the other lane bits
  // the column pair, so the two 32-byte halves of a column's 64 code bytes of a
  // tile, and its two 4-byte scale halves, sit in neighbouring lanes and leave
  // in one coalesced request.  The odd lanes visit the rows of each 16-row block
  // in the order i ^ 4, which puts the two halves on disjoint shared-memory
  // banks; their code words are put back in row order afterwards.  Otherwise
  // consecutive threads take consecutive column pairs.
  // With the transform each thread needs its 16-row blocks in natural row order: the
  // odd lanes then read them in that order too (PERM off) and take the 2-way bank
  // conflict between the two halves.
  constexpr bool PAIRED = SECT && BOTH && sizeof(T) == 2 && !FOS && !B2D;
  constexpr bool PERM = PAIRED && !RHT;
  // CPAIR (sector stores, columnwise only, BF16, 1x16): a thread holds 32 rows of a
  // column pair, and neighbouring lanes hold the two 32-row halves of the same 64-row
  // run, so that after one exchange each lane stores one column's 32 code bytes (a
  // whole sector) and 4 scale bytes.  The rows are read in natural order (the 2-way
  // bank conflict between the two halves costs nothing next to the encode).
  constexpr bool CPAIR = SECT && COL && !ROW && sizeof(T) == 2 && !B2D;
  const int hh = (PAIRED || CPAIR) ? (lane & 1) : 0;
  const int cl = PAIRED  ? 2 * (((ct >> 5) << 4) + (lane >> 1))
                 : CPAIR ? 2 * ((((ct >> 5) & 3) << 4) + (lane >> 1))
                         : 2 * (ct % NP);
  const int rb0 = PAIRED ? hh * RG : CPAIR ? 64 * (ct >> 7) + 32 * hh : (ct / NP) * RG;
  const int r = BOTH ? tid : (tid & 127), b0 = BOTH ? 0 : (tid >> 7);
  // byte offset of row i of a 16-row block: i * 128 + coff[i & 7] (signed: with
  // the i ^ 4 row order an entry can be negative, the sum never is)
  int32_t coff[8];
  {
    const int box = cl / G::BOXC, byte = (cl % G::BOXC) * (int)sizeof(T);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int kk = k ^ (PERM ? 4 * hh : 0);  // the row actually read, mod 8
      coff[k] = box * kBoxBytes + ((((byte >> 4) ^ kk)) << 4) + (byte & 15) + (kk - k) * 128;
    }
  }
  const uint32_t word_sel = hh ? 0x1032u : 0x3210u;  // swaps the halves of a code word
  uint8_t* staging0 = smem + NS * kTileBytes + warp * kStagingPerWarp * kStagingBuffers;
  uint32_t rsg[TileGrid::kGroup][2];  // rowwise scale bytes of the current super-strip row
  const uint64_t out_policy = policy_evict_first();
  TileCursor cur;
  cur.seek(a.grid, a.grid.walk(begin, end, 0, fwd));
  for (int k = 0; k < count; ++k, cur.step(a.grid, fwd)) {
    const int s = k % NS;
    const int tm = cur.tm, tn = cur.tn();
    const bool ok = mbar_wait_bounded(&full[s], (uint32_t)((k / NS) & 1));
    if (!ok) {
      abort_flag = 1;
      if (lane == 0) raise_status(a.status, kStatusTimeout);
    }
    if constexpr (B2D) consumer_sync();  // every consumer sees the same abort decision
    if (abort_flag) break;
    const uint8_t* stage = smem + s * kTileBytes;
    auto& m = meta[s];
    const bool interior = tm < a.full_m && tn < a.full_n;
    const bool fast = a.vec_ok && interior;
    uint8_t* staging = staging0 + (k % kStagingBuffers) * kStagingPerWarp;
    if constexpr (B2D) {
      if constexpr (!FOS && sizeof(T) == 2)
        subtile_scales_max(stage, m, ROW ? S_r : S_c, tid);
      else
        subtile_scales<T, FOS>(stage, m, ROW ? S_r : S_c, ROW ? A_r : A_c, a.F_inv, a.neg_zero,
                               tid);
      consumer_sync();
    }
    if (PAIRED && is_row) {
      if constexpr (PAIRED) {
        // Two rows r1, r1 + 16 of box hb = lane & 1: the two lanes of a pair write the
        // two 32-byte halves of a row's 64 code bytes of the tile in one request.
        // The box-1 lanes read the blocks in the order 2, 3, 0, 1 (rot = 4): the
        // two boxes of a row then sit on disjoint shared-memory banks.
        const int hb = lane & 1, r1 = 32 * warp + (lane >> 1);
        const uint32_t bsel = hb ? 0x1032u : 0x3210u;
        uint32_t sa[1], sb[1];
        // codes of one row: computed, put back in block order 0, 1, 2, 3, stored
        // (each row on its own keeps 8 code words live instead of 16)
        auto row_codes = [&](int rr, uint32_t (&sx)[1]) {
          uint32_t wx[1][8];
          rowwise_compute<T, 1, FOS, B2D>(stage, m, a, rr, hb, S_r, A_r, wx, sx, 4 * hb);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint32_t lo = wx[0][q], hi = wx[0][q + 4];
            wx[0][q] = hb ? hi : lo;
            wx[0][q + 4] = hb ? lo : hi;
          }
          sx[0] = __byte_perm(sx[0], 0, bsel);
          if (fast)
            stg_v8_cs(a.row_codes + ((int64_t)tm * kTileRows + rr) * a.row_cpitch +
                          (int64_t)tn * (G::TILEC / 2) + hb * 32,
                      wx[0]);
          else
            rowwise_store<T, 1>(a, rr, hb, tm, tn, wx, sx, false);
        };
        row_codes(r1, sa);
        row_codes(r1 + 16, sb);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);  // this warp is done reading the stage
        if (fast) {
          const int64_t gr1 = (int64_t)tm * kTileRows + r1;
          const int ss = cur.ss, jt = cur.jt, wdt = cur.wdt;
          const int g0 = ss * a.grid.tiles_m * TileGrid::kGroup + tm * wdt;
          const bool grouped = a.row_scale_groups && wdt == TileGrid::kGroup && g0 >= begin &&
                               g0 + wdt <= end;
          if (grouped) {
            // a row's 4 x 8 scale bytes of the super-strip row: one 32-byte sector,
            // its first half written by the box-0 lane, the second by the box-1 lane
#pragma unroll
            for (int jj = 0; jj < TileGrid::kGroup; ++jj)
              if (jj == jt) {
                rsg[jj][0] = sa[0];
                rsg[jj][1] = sb[0];
              }
            if (jt == (fwd ? TileGrid::kGroup - 1 : 0)) {
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                const uint32_t x1 = __shfl_xor_sync(0xffffffffu, hb ? rsg[0][h] : rsg[2][h], 1);
                const uint32_t x2 = __shfl_xor_sync(0xffffffffu, hb ? rsg[1][h] : rsg[3][h], 1);
                const uint4 v = hb ? make_uint4(x1, rsg[2][h], x2, rsg[3][h])
                                   : make_uint4(rsg[0][h], x1, rsg[1][h], x2);
                stg_v4_cs(a.row_scales + (gr1 + 16 * h) * a.row_spitch + ss * 32 + hb * 16, v);
              }
            }
          } else {
            rowwise_store_scales<T, 1>(a, r1, hb, tm, tn, sa, true);
            rowwise_store_scales<T, 1>(a, r1 + 16, hb, tm, tn, sb, true);
          }
        }
      }
    } else if (is_row) {
      uint32_t w[NBOX][G::BOXC / 8];
      uint32_t sc[NBOX];
      rowwise_compute<T, NBOX, FOS, B2D>(stage, m, a, r, b0, S_r, A_r, w, sc);
      if (ROW && !COL && a.pad_ends != nullptr && r >= m.nrows) {
        // a padding row: zero codes and scales (what a zero row encodes to)
#pragma unroll
        for (int bi = 0; bi < NBOX; ++bi) {
          sc[bi] = 0;
#pragma unroll
          for (int q = 0; q < G::BOXC / 8; ++q) w[bi][q] = 0;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);  // this warp is done reading the stage
      auto store_row_scales = [&]() {
        if constexpr (BOTH && sizeof(T) == 2) {
          // A super-strip row of 4 tiles carries 4 x 8 scale bytes per row: one
          // 32-byte sector.  When the whole group lies in this CTA's chunk, the
          // thread collects it in registers and writes the sector at once.
          const int ss = cur.ss, jt = cur.jt, wdt = cur.wdt;
          const int g0 = ss * a.grid.tiles_m * TileGrid::kGroup + tm * wdt;
          const bool grouped = a.row_scale_groups && wdt == TileGrid::kGroup && g0 >= begin &&
                               g0 + wdt <= end;
          if (grouped) {
#pragma unroll
            for (int jj = 0; jj < TileGrid::kGroup; ++jj)
              if (jj == jt) {
                rsg[jj][0] = sc[0];
                rsg[jj][1] = sc[1];
              }
            const int last = fwd ? TileGrid::kGroup - 1 : 0;
            const int64_t gr = (int64_t)tm * kTileRows + r;
            if (jt == last && gr < a.M) {
              uint8_t* sp = a.row_scales + gr * a.row_spitch + ss * 32;
              stg_v4_cs(sp, make_uint4(rsg[0][0], rsg[0][1], rsg[1][0], rsg[1][1]));
              stg_v4_cs(sp + 16, make_uint4(rsg[2][0], rsg[2][1], rsg[3][0], rsg[3][1]));
            }
            return;
          }
        }
        rowwise_store_scales<T, NBOX>(a, r, b0, tm, tn, sc, fast);
      };
      if constexpr (TOUT) {
        // the store that last used this buffer has finished reading it
        if (lane == 0) bulk_wait_read_allow<kStagingBuffers - 1>();
        __syncwarp();
        uint8_t* dst = staging + lane * RWB;
#pragma unroll
        for (int bi = 0; bi < NBOX; ++bi)
#pragma unroll
          for (int q = 0; q < G::BOXC / 32; ++q)
            sts_v4(dst + bi * (G::BOXC / 2) + 16 * q, w[bi][4 * q], w[bi][4 * q + 1],
                   w[bi][4 * q + 2], w[bi][4 * q + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&map_rc, staging, tn * (G::TILEC / 2) + b0 * (G::BOXC / 2),
                       tm * kTileRows + (r & ~31), out_policy);
          bulk_commit();
        }
        store_row_scales();
      } else if constexpr (SECT) {
        if (fast) {
          uint8_t* cp = a.row_codes + ((int64_t)tm * kTileRows + r) * a.row_cpitch +
                        (int64_t)tn * (G::TILEC / 2);
#pragma unroll
          for (int bi = 0; bi < NBOX; ++bi) stg_v8_cs(cp + bi * 32 + b0 * 32, w[bi]);
          store_row_scales();
        } else {
          rowwise_store<T, NBOX>(a, r, b0, tm, tn, w, sc, false);
        }
      } else if (STAGED_ROWS && interior && a.rc_g >= 4) {
        static_assert(!STAGED_ROWS || kRowStageWarps * RowStage<T, NBOX>::kBytes <=
                                          kRowStageWarps * kRowStagePerWarp,
                      "rowwise staging does not fit");
        rowwise_store_staged<T, NBOX>(a, smem + NS * kTileBytes + warp * RowStage<T, NBOX>::kBytes,
                                      r, b0, tm, tn, lane, w, sc);
      } else {
        rowwise_store<T, NBOX>(a, r, b0, tm, tn, w, sc, interior);
      }
    } else if (COL) {
      uint32_t w0[RG / 8], w1[RG / 8];
      uint32_t sc0, sc1;
      colwise_compute<T, RG, FOS, B2D, RHT, RHT && !ROW>(stage, m, a, cl, rb0, coff, S_c, A_c,
                                                         w0, w1, sc0, sc1);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      if constexpr (PERM) {
#pragma unroll
        for (int q = 0; q < RG / 8; ++q) {
          w0[q] = __byte_perm(w0[q], 0, word_sel);
          w1[q] = __byte_perm(w1[q], 0, word_sel);
        }
      }
      if constexpr (TOUT) {
        if (lane == 0) bulk_wait_read_allow<kStagingBuffers - 1>();
        __syncwarp();
        uint8_t* dst = staging + lane * 2 * CWB;
#pragma unroll
        for (int q = 0; q < CWB / 16; ++q) {
          sts_v4(dst + 16 * q, w0[4 * q], w0[4 * q + 1], w0[4 * q + 2], w0[4 * q + 3]);
          sts_v4(dst + CWB + 16 * q, w1[4 * q], w1[4 * q + 1], w1[4 * q + 2], w1[4 * q + 3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&map_cc, staging, (tm * kTileRows + rb0) / 2,
                       tn * G::TILEC + (cl & ~63), out_policy);
          bulk_commit();
        }
      }
      if constexpr (SECT && CPAIR) {
        if (fast) {
          // lane hh = 0 takes column cl (its own rows 0-31 of the run, the partner's
          // 32-63), lane hh = 1 column cl + 1 (the partner's rows 0-31, its own 32-63)
          uint32_t cw[RG / 4];
#pragma unroll
          for (int q = 0; q < RG / 8; ++q) {
            const uint32_t got = __shfl_xor_sync(0xffffffffu, hh ? w0[q] : w1[q], 1);
            cw[q] = hh ? got : w0[q];
            cw[RG / 8 + q] = hh ? w1[q] : got;
          }
          const uint32_t gs = __shfl_xor_sync(0xffffffffu, hh ? sc0 : sc1, 1);
          const uint32_t scw = hh ? (gs | (sc1 << 16)) : (sc0 | (gs << 16));
          const int64_t gcol = (int64_t)tn * G::TILEC + cl + hh;
          const int64_t grun = (int64_t)tm * kTileRows + rb0 - 32 * hh;
          stg_v8_cs(a.col_codes + gcol * a.col_cpitch + grun / 2, cw);
          stg_u32_keep(a.col_scales + gcol * a.col_spitch + grun / 16, scw, policy_evict_last());
        } else {
          colwise_store<T, RG, true>(a, cl, rb0, tm, tn, w0, w1, sc0, sc1, false);
        }
      } else if constexpr (SECT) {
        if (fast) {
          uint8_t* c0p = a.col_codes + ((int64_t)tn * G::TILEC + cl) * a.col_cpitch +
                         ((int64_t)tm * kTileRows + rb0) / 2;
          stg_v8_cs(c0p, w0);
          stg_v8_cs(c0p + a.col_cpitch, w1);
          bool sector_scales = false;
          if constexpr (PAIRED) {
            // Tile rows 4p .. 4p + 3 of this tile column make up one 32-byte sector of
            // each column's scale row and are 4 tiles apart in the walk.  When all four
            // are full tiles of this CTA's chunk, the first three visited park their
            // scale bytes in csb and the last writes the column's sector in one
            // coalesced request: lane hh = 0 bytes 0-15 (tile rows 4p, 4p + 1),
            // lane hh = 1 bytes 16-31 (tile rows 4p + 2, 4p + 3).
            const int q0 = tm & ~3, q = tm & 3;
            const int L0 = cur.ss * a.grid.tiles_m * TileGrid::kGroup + q0 * cur.wdt + cur.jt;
            sector_scales = a.col_scale_sectors && q0 + 3 < a.full_m && L0 >= begin &&
                            L0 + 3 * cur.wdt < end;
            if (sector_scales) {
              const int v = fwd ? q : 3 - q;  // visit index inside the sector
              if (v < 3) {
                csb[cur.jt][cl][v][hh] = sc0;
                csb[cur.jt][cl + 1][v][hh] = sc1;
              } else {
                const uint32_t o0 = __shfl_xor_sync(0xffffffffu, sc0, 1);
                const uint32_t o1 = __shfl_xor_sync(0xffffffffu, sc1, 1);
                // this tile's 8 bytes of each column: row half 0, then row half 1
                const uint2 t0 = hh ? make_uint2(o0, sc0) : make_uint2(sc0, o0);
                const uint2 t1 = hh ? make_uint2(o1, sc1) : make_uint2(sc1, o1);
                uint2 r0[2], r1[2];
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                  const int qq = 2 * hh + i;  // tile row q0 + qq
                  const int vv = fwd ? qq : 3 - qq;
                  const bool here = qq == q;
                  const int vs = here ? 0 : vv;
                  r0[i] = here ? t0 : make_uint2(csb[cur.jt][cl][vs][0], csb[cur.jt][cl][vs][1]);
                  r1[i] = here ? t1
                               : make_uint2(csb[cur.jt][cl + 1][vs][0], csb[cur.jt][cl + 1][vs][1]);
                }
                uint8_t* s0p = a.col_scales + ((int64_t)tn * G::TILEC + cl) * a.col_spitch +
                               (int64_t)q0 * (kTileRows / 16) + 16 * hh;
                stg_v4_cs(s0p, make_uint4(r0[0].x, r0[0].y, r0[1].x, r0[1].y));
                stg_v4_cs(s0p + a.col_spitch, make_uint4(r1[0].x, r1[0].y, r1[1].x, r1[1].y));
              }
            }
          }
          if (!sector_scales)
            colwise_store<T, RG, false>(a, cl, rb0, tm, tn, w0, w1, sc0, sc1, true);
        } else {
          colwise_store<T, RG, true>(a, cl, rb0, tm, tn, w0, w1, sc0, sc1, false);
        }
      } else {
        colwise_store<T, RG, !TOUT>(a, cl, rb0, tm, tn, w0, w1, sc0, sc1, interior);
      }
    } else {
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
  }
  if constexpr (TOUT) {
    if (lane == 0) bulk_wait_all();
  }
}

using EncodeFn = void (*)(const CUtensorMap, const CUtensorMap, const CUtensorMap, EncodeArgs);

template <typename T, bool ROW, bool COL, bool FOS, bool B2D>
EncodeFn pick_io(bool tma, int outm) {
  if constexpr (sizeof(T) == 2 && ROW && COL) {
    if (tma && outm == kOutTma) return k_encode<T, ROW, COL, FOS, B2D, true, kOutTma>;
    if (tma && outm == kOutSector) return k_encode<T, ROW, COL, FOS, B2D, true, kOutSector>;
  }
  if constexpr (sizeof(T) == 2 && !ROW && COL && !B2D) {
    if (tma && outm == kOutSector) return k_encode<T, ROW, COL, FOS, B2D, true, kOutSector>;
  }
  return tma ? k_encode<T, ROW, COL, FOS, B2D, true, kOutDirect>
             : k_encode<T, ROW, COL, FOS, B2D, false, kOutDirect>;
}

template <typename T, bool ROW, bool COL>
EncodeFn pick_mode(bool fos, bool b2d, bool tma, int outm) {
  if (b2d)
    return fos ? pick_io<T, ROW, COL, true, true>(tma, outm) : pick_io<T, ROW, COL, false, true>(tma, outm);
  if constexpr (ROW && COL) {
    // four-over-six with 1x16 blocks and both directions runs as two passes
    return fos ? nullptr : pick_io<T, ROW, COL, false, false>(tma, outm);
  } else {
    return fos ? pick_io<T, ROW, COL, true, false>(tma, outm)
               : pick_io<T, ROW, COL, false, false>(tma, outm);
  }
}

// Columnwise only, 1x16 blocks, each block transformed first.
template <typename T>
EncodeFn pick_rht(bool fos, bool tma, int outm) {
  if constexpr (sizeof(T) == 2) {
    if (tma && outm == kOutSector)
      return fos ? k_encode<T, false, true, true, false, true, kOutSector, true>
                 : k_encode<T, false, true, false, false, true, kOutSector, true>;
  }
  if (fos)
    return tma ? k_encode<T, false, true, true, false, true, kOutDirect, true>
               : k_encode<T, false, true, true, false, false, kOutDirect, true>;
  return tma ? k_encode<T, false, true, false, false, true, kOutDirect, true>
             : k_encode<T, false, true, false, false, false, kOutDirect, true>;
}

// Both directions, 1x16 blocks, the columnwise blocks transformed first (TMA loads).
template <typename T>
EncodeFn pick_rht_both(bool fos, int outm) {
  if (fos) return nullptr;  // four-over-six: two single-direction passes
  if constexpr (sizeof(T) == 2) {
    if (outm == kOutSector) return k_encode<T, true, true, false, false, true, kOutSector, true>;
  }
  return k_encode<T, true, true, false, false, true, kOutDirect, true>;
}

template <typename T>
EncodeFn pick_dir(bool row, bool col, bool fos, bool b2d, bool tma, int outm) {
  if (row && col) return pick_mode<T, true, true>(fos, b2d, tma, outm);
  if (row) return pick_mode<T, true, false>(fos, b2d, tma, outm);
  return pick_mode<T, false, true>(fos, b2d, tma, outm);
}

bool aligned(const void* p, int n) { return reinterpret_cast<uintptr_t>(p) % n == 0; }

}  // namespace

int pipe_grid_size(int64_t num_tiles, int num_sms) {
  return (int)std::min<int64_t>(num_tiles, 2LL * num_sms);
}

cudaError_t launch_quantize(const QuantArgs& q, const DeviceInfo& dev, cudaStream_t stream) {
  const bool row = q.row_codes != nullptr, col = q.col_codes != nullptr;
  if (!row && !col) return cudaSuccess;
  if (row && col && (q.block_2d ? q.row_amax != q.col_amax : q.four_over_six)) {
    // Both directions as two single-direction passes: rows, then columns walked the
    // other way (starting on the tiles the first pass left in L2).  16x16 tiles share
    // one scale per tile, so two different per-tensor amax need two passes; and
    // four-over-six with 1x16 blocks is faster so: a two-direction kernel would hold
    // both directions' block routines and spill at the 96 registers that two CTAs per
    // SM allow (measured with given amax, BF16: X 16384 x 8192 215.7 -> 194.2 us, dY
    // 16384 x 28672 725.7 -> 625.2 us, although x is read twice).
    QuantArgs qr = q, qc = q;
    qr.col_codes = nullptr;
    qr.rht = false;  // the transform belongs to the columnwise side
    qc.row_codes = nullptr;
    qc.copy_dst = nullptr;
    qc.reverse_walk = !q.reverse_walk;
    const cudaError_t e = launch_quantize(qr, dev, stream);
    return e != cudaSuccess ? e : launch_quantize(qc, dev, stream);
  }
  const bool bf16 = q.in == InType::BF16;
  const int box_cols = bf16 ? TileGeo<uint16_t>::BOXC : TileGeo<float>::BOXC;
  const int tile_cols = 2 * box_cols;
  EncodeArgs a{};
  a.x = q.x;
  a.M = q.M;
  a.K = q.K;
  a.grid.tiles_m = (int)((q.M + kTileRows - 1) / kTileRows);
  a.grid.tiles_n = (int)((q.K + tile_cols - 1) / tile_cols);
  a.grid.num_tiles = a.grid.tiles_m * a.grid.tiles_n;
  a.full_m = (int)(q.M / kTileRows);
  a.full_n = (int)(q.K / tile_cols);
  a.row_codes = q.row_codes;
  a.row_scales = q.row_scales;
  a.row_amax = q.row_amax;
  a.col_codes = q.col_codes;
  a.col_scales = q.col_scales;
  a.col_amax = q.col_amax;
  a.row_cpitch = (q.K + 1) / 2;
  a.row_spitch = (q.K + 15) / 16;
  a.col_cpitch = (q.M + 1) / 2;
  a.col_spitch = (q.M + 15) / 16;
  a.row_scaled = q.row_scaled ? 1 : 0;
  a.F = q.bound * 6.0f;
  a.F_inv = 1.0f / a.F;  // correctly rounded IEEE division on the host
  a.neg_zero = -0.0f;
  a.copy_dst = q.copy_dst;
  a.copy_src = q.copy_src;
  a.noop = q.noop;
  a.status = dev.status;
  a.ends = q.group_ends;
  a.G = q.num_groups;
  a.pad_ends = q.pad_ends;
  a.rag_ends = q.rag_ends;
  a.col_grouped = q.col_grouped ? 1 : 0;
  a.col_grouped_pt = q.col_grouped_per_tensor ? 1 : 0;
  a.in_rows = q.pad_ends != nullptr ? q.in_rows : q.M;
  a.rht_mask = q.rht_mask;
  a.reverse_walk = q.reverse_walk ? 1 : 0;
  // measured: the normal priority helps the two-direction pass over an x larger than
  // L2 (16384 x 28672 BF16: the next amax pass 160.3 -> 157.8 us) and costs the
  // columnwise-only and the L2-resident cases 1-3 %
  a.load_normal = row && col && a.in_rows * q.K * (bf16 ? 2 : 4) > dev.l2_bytes ? 1 : 0;
  if (a.grid.num_tiles == 0) return cudaSuccess;
  if (q.rht && (q.block_2d || q.pad_ends != nullptr || (q.col_grouped && row)))
    return cudaErrorInvalidValue;  // the transform is built for the 1x16 paths

  CUtensorMap map, map_rc, map_cc;
  memset(&map_rc, 0, sizeof(map_rc));
  memset(&map_cc, 0, sizeof(map_cc));
  const bool tma = a.in_rows > 0 && make_tile_map(&map, q.x, q.in, a.in_rows, q.K, box_cols, kTileRows);
  if (!tma) memset(&map, 0, sizeof(map));
  // Output path for the codes of BF16 input with both directions: 32-byte sector
  // stores when the code pitches allow them, else TMA stores from staging.
  const bool both = row && col;
  int outm = kOutDirect;
  if (bf16 && tma && both) {
    if (a.row_cpitch % 32 == 0 && a.col_cpitch % 32 == 0 && aligned(q.row_codes, 32) &&
        aligned(q.col_codes, 32))
      outm = kOutSector;
    else if (make_byte_map(&map_rc, q.row_codes, q.M, a.row_cpitch, 64, 32) &&
             make_byte_map(&map_cc, q.col_codes, q.K, a.col_cpitch, 32, 64))
      outm = kOutTma;
  }
  // the transform with both directions: sector or direct stores only
  if (q.rht && both && outm == kOutTma) outm = kOutDirect;
  if (q.rht && both && !tma) return cudaErrorInvalidValue;  // rows of x not TMA-aligned
  // columnwise only (BF16, 1x16): whole-sector code stores from lane pairs
  if (bf16 && tma && col && !row && !q.block_2d && a.col_cpitch % 32 == 0 &&
      aligned(q.col_codes, 32) && a.col_spitch % 4 == 0 && aligned(q.col_scales, 4))
    outm = kOutSector;
  const bool tout = outm != kOutDirect;
  // aligned vector stores on interior tiles
  const int rows_per_col_thread = bf16 ? (both ? 64 : 32) : (both ? 32 : 16);
  const int row_scale_bytes = (bf16 ? 4 : 2) * ((tout && both) ? 2 : 1);
  bool vec = true;
  if (row)
    vec = vec && (tout || (a.row_cpitch % 16 == 0 && aligned(q.row_codes, 16))) &&
          a.row_spitch % row_scale_bytes == 0 && aligned(q.row_scales, row_scale_bytes);
  if (col) {
    const int cs = std::max(1, rows_per_col_thread / 16);
    vec = vec && (tout || (a.col_cpitch % 16 == 0 && aligned(q.col_codes, 16))) &&
          a.col_spitch % cs == 0 && aligned(q.col_scales, cs);
  }
  a.vec_ok = vec ? 1 : 0;
  auto gran = [](const void* base, int64_t pitch) {
    int g = 16;
    while (g > 1 && (reinterpret_cast<uintptr_t>(base) % g != 0 || pitch % g != 0)) g >>= 1;
    return g;
  };
  a.rc_g = row ? gran(q.row_codes, a.row_cpitch) : 1;
  a.rs_g = row ? gran(q.row_scales, a.row_spitch) : 1;
  a.cc_g = col ? gran(q.col_codes, a.col_cpitch) : 1;
  a.cs_g = col ? gran(q.col_scales, a.col_spitch) : 1;
  a.col_scale_sectors = (both && bf16 && a.col_spitch % 32 == 0 && aligned(q.col_scales, 32)) ? 1 : 0;
  a.row_scale_groups = (tout && both && bf16 && a.row_spitch % 32 == 0 &&
                        aligned(q.row_scales, 32)) ? 1 : 0;

  EncodeFn fn = q.rht ? (both ? (bf16 ? pick_rht_both<uint16_t>(q.four_over_six, outm)
                                     : pick_rht_both<float>(q.four_over_six, outm))
                              : bf16 ? pick_rht<uint16_t>(q.four_over_six, tma, outm)
                                     : pick_rht<float>(q.four_over_six, tma, outm))
               : bf16 ? pick_dir<uint16_t>(row, col, q.four_over_six, q.block_2d, tma, outm)
                      : pick_dir<float>(row, col, q.four_over_six, q.block_2d, tma, outm);
  if (fn == nullptr) return cudaErrorInvalidValue;  // split into two passes above
  const int smem = outm == kOutTma ? EncodeSmem<kOutTma>::kBytes
                   : outm == kOutSector ? EncodeSmem<kOutSector>::kBytes
                                        : EncodeSmem<kOutDirect>::kBytes;
  cudaError_t err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  // two CTAs per SM need nearly all of the SM's shared memory
  err = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)pipe_grid_size(a.grid.num_tiles, dev.num_sms));
  cfg.blockDim = dim3(kPipeThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fn, map, map_rc, map_cc, a);
}

}  // namespace nvfp4
