// kernels_amax.cu -- exact amax kernels.
//
// One pass over x computes the per-row, per-column and/or per-tensor maxima of
// |x| ("row-scaled nvfp4 path: fuse row/col amax into a single TMA-tiled kernel",
// TransformerEngine PR #3454, description: both directions in one kernel; amax
// is an exact max, so the result is byte-identical to separate reductions).
//
// Kernels:
//   k_amax_tma      the pass for x whose rows TMA can describe: persistent, a ring of
//                   128-row x 256-byte tiles in the encode kernel's tile order
//                   (tile_pipeline.cuh), walked the other way so the encode pass
//                   finds the tail in L2; row, column (per tensor or per row group)
//                   and tensor maxima.
//   k_amax_bf16 / k_amax_f32
//                   the same maxima for any x with plain 128-bit loads (below).
//   k_grouped_amax  per-group maxima with plain loads (no per-row output to use).
//   k_group_reduce  per-group maxima from per-row maxima, written back to the rows.
//   k_group_check   validates group ends and clears or copies the outputs.
//   k_prep          clears or copies the outputs after the noop check.
// Every kernel checks the noop flag first.
//
// k_amax_bf16 / k_amax_f32: a CTA owns an item of RB rows x CW columns.  Each thread
// owns 16 bytes of columns (8 BF16 or 4 FP32) and walks down its rows with 8
// independent 128-bit loads in flight; its column maxima stay in registers for
// the whole item.  Row maxima are reduced across the warp with a transposing
// shuffle reduction (8 rows at a time), across the CTA in shared memory, and
// published once per row and item.  Column maxima are combined across the CTA's
// row groups in shared memory and published once per column and item.
// Publishing uses atomicMax on the FP32 bit pattern, valid because every value
// is >= 0, and exact and order-independent.
#include <algorithm>
#include <type_traits>

#include "device_common.cuh"
#include "internal.h"
#include "tile_pipeline.cuh"

namespace nvfp4 {

namespace {

constexpr int kThreads = 256;
constexpr int kColWarps = 2;  // warps side by side along the columns
constexpr int kRowGroups = 4; // warps stacked along the rows

__device__ __forceinline__ void atomic_max_nonneg(float* p, float v) {
  if (v > 0.0f) atomicMax(reinterpret_cast<unsigned int*>(p), __float_as_uint(v));
}

// ---------------------------------------------------------------- prep

// The next kernel (the amax pass, launched for programmatic dependent launch) may
// start its prologue and its loads of x at once: it waits for this grid before it
// touches the outputs cleared here.
__global__ void k_prep(PrepArgs a) {
  pdl_launch_dependents();
  if (noop_set(a.noop)) return;
  const int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t step = (int64_t)gridDim.x * blockDim.x;
#pragma unroll
  for (int k = 0; k < 4; ++k)
    if (a.zero_ptr[k] != nullptr)
      for (int64_t i = i0; i < a.zero_n[k]; i += step) a.zero_ptr[k][i] = 0.0f;
#pragma unroll
  for (int k = 0; k < 2; ++k)
    if (a.copy_dst[k] != nullptr)
      for (int64_t i = i0; i < a.copy_n[k]; i += step) a.copy_dst[k][i] = a.copy_src[k][i];
}

// ---------------------------------------------------------------- loads

// 8 BF16 values (as 4 packed pairs) of row r starting at column c; elements
// outside the matrix read as +0, which never changes a maximum.
template <bool VEC>
__device__ __forceinline__ uint4 load_bf16x8(const uint16_t* x, int64_t M, int64_t K, int64_t r,
                                             int64_t c, uint64_t policy) {
  if (r >= M || c >= K) return make_uint4(0, 0, 0, 0);
  const uint16_t* p = x + r * K + c;
  if constexpr (VEC) {
    return ldg_v4_policy(p, policy);
  } else {
    uint32_t w[4] = {0, 0, 0, 0};
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (c + j < K) w[j >> 1] |= (uint32_t)p[j] << (16 * (j & 1));
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
}

template <bool VEC>
__device__ __forceinline__ float4 load_f32x4(const float* x, int64_t M, int64_t K, int64_t r,
                                             int64_t c, uint64_t policy) {
  if (r >= M || c >= K) return make_float4(0.f, 0.f, 0.f, 0.f);
  const float* p = x + r * K + c;
  if constexpr (VEC) {
    uint4 u = ldg_v4_policy(p, policy);
    return make_float4(__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z),
                       __uint_as_float(u.w));
  } else {
    float w[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (c + j < K) w[j] = p[j];
    return make_float4(w[0], w[1], w[2], w[3]);
  }
}

// ---------------------------------------------------------------- warp reductions

// Eight row partials held as four packed BF16 pairs P[k] = (row 2k, row 2k+1).
// After the call every lane holds, in one packed pair, the warp-wide maxima of
// rows 4*bit4 + 2*bit3 + {0, 1} of its lane index.  Sign bits are garbage.
__device__ __forceinline__ uint32_t warp_rowmax8_bf16(const uint32_t P[4], int lane) {
  const bool up16 = lane & 16;
  uint32_t s0 = up16 ? P[0] : P[2], s1 = up16 ? P[1] : P[3];
  uint32_t k0 = up16 ? P[2] : P[0], k1 = up16 ? P[3] : P[1];
  k0 = absmax_bf16x2(k0, __shfl_xor_sync(0xffffffffu, s0, 16));
  k1 = absmax_bf16x2(k1, __shfl_xor_sync(0xffffffffu, s1, 16));
  const bool up8 = lane & 8;
  uint32_t s = up8 ? k0 : k1, k = up8 ? k1 : k0;
  k = absmax_bf16x2(k, __shfl_xor_sync(0xffffffffu, s, 8));
  k = absmax_bf16x2(k, __shfl_xor_sync(0xffffffffu, k, 4));
  k = absmax_bf16x2(k, __shfl_xor_sync(0xffffffffu, k, 2));
  k = absmax_bf16x2(k, __shfl_xor_sync(0xffffffffu, k, 1));
  return k;
}

// Same for eight FP32 row partials; afterwards lane holds row
// 4*bit4 + 2*bit3 + bit2 of its lane index.
__device__ __forceinline__ float warp_rowmax8_f32(const float v[8], int lane) {
  const bool up16 = lane & 16, up8 = lane & 8, up4 = lane & 4;
  float a[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float send = up16 ? v[j] : v[4 + j];
    float keep = up16 ? v[4 + j] : v[j];
    a[j] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, 16));
  }
  float b[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    float send = up8 ? a[j] : a[2 + j];
    float keep = up8 ? a[2 + j] : a[j];
    b[j] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, 8));
  }
  float send = up4 ? b[0] : b[1];
  float keep = up4 ? b[1] : b[0];
  float c = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, 4));
  c = fmaxf(c, __shfl_xor_sync(0xffffffffu, c, 2));
  c = fmaxf(c, __shfl_xor_sync(0xffffffffu, c, 1));
  return c;
}

__device__ __forceinline__ float block_max(float v, float* red) {
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[w] = v;
  __syncthreads();
  float m = 0.0f;
  if (threadIdx.x == 0)
    for (int i = 0; i < kThreads / 32; ++i) m = fmaxf(m, red[i]);
  return m;  // valid in thread 0
}

// ---------------------------------------------------------------- amax kernels

struct AmaxKernelArgs {
  const void* x;
  int64_t M, K;
  float* row_amax;
  float* col_amax;
  float* tensor_amax;
  const float* noop;
  const int64_t* ends;
  int G;
  const int64_t* pad_ends;  // with ends: also require this padded layout (pad_rows rows)
  int64_t pad_rows;
  int64_t rows_per_item;  // multiple of 8 * kRowGroups
  int64_t keep_from_row;  // rows >= this are loaded with an L2 evict_last hint
  int num_col_items;
};

// BF16 input: thread = 8 columns, CTA item = rows_per_item x 512 columns.
template <bool ROW, bool COL, bool TEN, bool VEC>
__global__ void __launch_bounds__(kThreads) k_amax_bf16(AmaxKernelArgs a) {
  constexpr int VE = 8, CW = kColWarps * 32 * VE;
  __shared__ float row_red[kColWarps][512];
  __shared__ float col_red[kRowGroups][CW];
  __shared__ float red[kThreads / 32];
  if (noop_set(a.noop)) return;
  if (a.ends != nullptr && (!groups_valid(a.ends, a.G, a.M) ||
                            (a.pad_ends != nullptr &&
                             !pad_layout_valid(a.ends, a.pad_ends, a.G, a.M, a.pad_rows))))
    return;
  const uint16_t* x = static_cast<const uint16_t*>(a.x);
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int cw = w % kColWarps, rg = w / kColWarps;
  const int64_t item = blockIdx.x;
  const int64_t band = item / a.num_col_items, cr = item % a.num_col_items;
  const int64_t r0 = band * a.rows_per_item;
  const int64_t c = cr * CW + cw * 32 * VE + lane * VE;
  const uint64_t pol_first = policy_evict_first(), pol_last = policy_evict_last();

  uint32_t cm[4] = {0, 0, 0, 0};
  uint32_t tm = 0;
  const int chunks = (int)(a.rows_per_item / (8 * kRowGroups));
  for (int k = 0; k < chunks; ++k) {
    const int64_t rr = r0 + (int64_t)(k * kRowGroups + rg) * 8;
    const uint64_t pol = rr >= a.keep_from_row ? pol_last : pol_first;
    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = load_bf16x8<VEC>(x, a.M, a.K, rr + i, c, pol);
    uint32_t rp[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (COL) {
        cm[0] = absmax_bf16x2(cm[0], v[i].x);
        cm[1] = absmax_bf16x2(cm[1], v[i].y);
        cm[2] = absmax_bf16x2(cm[2], v[i].z);
        cm[3] = absmax_bf16x2(cm[3], v[i].w);
      }
      rp[i] = absmax_bf16x2(absmax_bf16x2(v[i].x, v[i].y), absmax_bf16x2(v[i].z, v[i].w));
    }
    if (TEN) {
#pragma unroll
      for (int i = 0; i < 8; ++i) tm = absmax_bf16x2(tm, rp[i]);
    }
    if (ROW) {
      // fold each pair to its max in both halves, then pack two rows per word
      uint32_t P[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t f0 = absmax_bf16x2(rp[2 * j], __byte_perm(rp[2 * j], 0, 0x1032));
        uint32_t f1 = absmax_bf16x2(rp[2 * j + 1], __byte_perm(rp[2 * j + 1], 0, 0x1032));
        P[j] = __byte_perm(f0, f1, 0x7610);
      }
      uint32_t R = warp_rowmax8_bf16(P, lane) & 0x7fff7fffu;
      if ((lane & 7) == 0) {
        const int rl = (k * kRowGroups + rg) * 8 + ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2;
        row_red[cw][rl] = __uint_as_float(R << 16);
        row_red[cw][rl + 1] = __uint_as_float(R & 0xffff0000u);
      }
    }
  }
  if (ROW || COL) {
    if (COL) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t m = cm[j] & 0x7fff7fffu;
        col_red[rg][cw * 32 * VE + lane * VE + 2 * j] = __uint_as_float(m << 16);
        col_red[rg][cw * 32 * VE + lane * VE + 2 * j + 1] = __uint_as_float(m & 0xffff0000u);
      }
    }
    __syncthreads();
    if (ROW) {
      for (int t = tid; t < a.rows_per_item; t += kThreads) {
        const int64_t r = r0 + t;
        if (r < a.M) atomic_max_nonneg(&a.row_amax[r], fmaxf(row_red[0][t], row_red[1][t]));
      }
    }
    if (COL) {
      for (int t = tid; t < CW; t += kThreads) {
        const int64_t col = cr * CW + t;
        float m = fmaxf(fmaxf(col_red[0][t], col_red[1][t]), fmaxf(col_red[2][t], col_red[3][t]));
        if (col < a.K) atomic_max_nonneg(&a.col_amax[col], m);
      }
    }
  }
  if (TEN) {
    float m = block_max(bf16x2_hmax_f32(tm), red);
    if (tid == 0) atomic_max_nonneg(a.tensor_amax, m);
  }
}

// FP32 input: thread = 4 columns, CTA item = rows_per_item x 256 columns.
template <bool ROW, bool COL, bool TEN, bool VEC>
__global__ void __launch_bounds__(kThreads) k_amax_f32(AmaxKernelArgs a) {
  constexpr int VE = 4, CW = kColWarps * 32 * VE;
  __shared__ float row_red[kColWarps][512];
  __shared__ float col_red[kRowGroups][CW];
  __shared__ float red[kThreads / 32];
  if (noop_set(a.noop)) return;
  if (a.ends != nullptr && (!groups_valid(a.ends, a.G, a.M) ||
                            (a.pad_ends != nullptr &&
                             !pad_layout_valid(a.ends, a.pad_ends, a.G, a.M, a.pad_rows))))
    return;
  const float* x = static_cast<const float*>(a.x);
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int cw = w % kColWarps, rg = w / kColWarps;
  const int64_t item = blockIdx.x;
  const int64_t band = item / a.num_col_items, cr = item % a.num_col_items;
  const int64_t r0 = band * a.rows_per_item;
  const int64_t c = cr * CW + cw * 32 * VE + lane * VE;
  const uint64_t pol_first = policy_evict_first(), pol_last = policy_evict_last();

  float cm[4] = {0.f, 0.f, 0.f, 0.f};
  float tm = 0.f;
  const int chunks = (int)(a.rows_per_item / (8 * kRowGroups));
  for (int k = 0; k < chunks; ++k) {
    const int64_t rr = r0 + (int64_t)(k * kRowGroups + rg) * 8;
    const uint64_t pol = rr >= a.keep_from_row ? pol_last : pol_first;
    float4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = load_f32x4<VEC>(x, a.M, a.K, rr + i, c, pol);
    float rp[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float e0 = fabsf(v[i].x), e1 = fabsf(v[i].y), e2 = fabsf(v[i].z), e3 = fabsf(v[i].w);
      if (COL) {
        cm[0] = fmaxf(cm[0], e0);
        cm[1] = fmaxf(cm[1], e1);
        cm[2] = fmaxf(cm[2], e2);
        cm[3] = fmaxf(cm[3], e3);
      }
      rp[i] = fmaxf(fmaxf(e0, e1), fmaxf(e2, e3));
      if (TEN) tm = fmaxf(tm, rp[i]);
    }
    if (ROW) {
      const float R = warp_rowmax8_f32(rp, lane);
      if ((lane & 3) == 0) {
        const int rl = (k * kRowGroups + rg) * 8 + ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 +
                       ((lane >> 2) & 1);
        row_red[cw][rl] = R;
      }
    }
  }
  if (ROW || COL) {
    if (COL) {
#pragma unroll
      for (int j = 0; j < 4; ++j) col_red[rg][cw * 32 * VE + lane * VE + j] = cm[j];
    }
    __syncthreads();
    if (ROW) {
      for (int t = tid; t < a.rows_per_item; t += kThreads) {
        const int64_t r = r0 + t;
        if (r < a.M) atomic_max_nonneg(&a.row_amax[r], fmaxf(row_red[0][t], row_red[1][t]));
      }
    }
    if (COL) {
      for (int t = tid; t < CW; t += kThreads) {
        const int64_t col = cr * CW + t;
        float m = fmaxf(fmaxf(col_red[0][t], col_red[1][t]), fmaxf(col_red[2][t], col_red[3][t]));
        if (col < a.K) atomic_max_nonneg(&a.col_amax[col], m);
      }
    }
  }
  if (TEN) {
    float m = block_max(tm, red);
    if (tid == 0) atomic_max_nonneg(a.tensor_amax, m);
  }
}

using AmaxFn = void (*)(AmaxKernelArgs);

template <bool ROW, bool COL, bool TEN>
AmaxFn pick_amax(InType in, bool vec) {
  if (in == InType::BF16)
    return vec ? k_amax_bf16<ROW, COL, TEN, true> : k_amax_bf16<ROW, COL, TEN, false>;
  return vec ? k_amax_f32<ROW, COL, TEN, true> : k_amax_f32<ROW, COL, TEN, false>;
}

AmaxFn pick_amax(InType in, bool vec, bool row, bool col, bool ten) {
  const int key = (row ? 4 : 0) | (col ? 2 : 0) | (ten ? 1 : 0);
  switch (key) {
    case 1: return pick_amax<false, false, true>(in, vec);
    case 2: return pick_amax<false, true, false>(in, vec);
    case 3: return pick_amax<false, true, true>(in, vec);
    case 4: return pick_amax<true, false, false>(in, vec);
    case 5: return pick_amax<true, false, true>(in, vec);
    case 6: return pick_amax<true, true, false>(in, vec);
    case 7: return pick_amax<true, true, true>(in, vec);
    default: return nullptr;
  }
}

// ---------------------------------------------------------------- TMA amax kernel

// The same tiles, tile order and grid size as the encode kernel (see
// tile_pipeline.cuh): CTA j walks its chunk in the direction opposite to the
// encode kernel's CTA j, so that kernel finds the tail of the walk in L2 (the
// last tiles of each walk are loaded with an L2 evict_last policy).
//
// Consumer warp w reads box (w & 1), rows 32 * (w >> 1) .. +32; lane l owns the
// 16-byte column chunk (l & 7) of rows (l >> 3) + 4 i.  Column maxima of the
// super-strip's kGroup tile columns stay in registers while the CTA walks down
// the super-strip and are published when it moves to another one; row maxima are
// reduced over the 8 lanes that share a row with a transposing shuffle reduction
// and published per tile.
struct AmaxTmaArgs {
  int64_t M, K;
  TileGrid grid;
  float* row_amax;
  float* col_amax;
  float* tensor_amax;
  const float* noop;
  const int64_t* ends;
  int G;
  const int64_t* pad_ends;  // with ends: also require this padded layout (pad_rows rows)
  int64_t pad_rows;
  int keep_tiles;  // the last keep_tiles tiles of a chunk are loaded with evict_last
  int* status;
  // grouped columns: col_amax is [G][K], the column maxima of each group's rows (the
  // group ends, multiples of kTileRows, are ends / G)
  int col_grouped;
};

// group of tile row tm (group ends are multiples of kTileRows): a binary search
// over the ends in global memory
__device__ __forceinline__ int group_of_tile_row(const int64_t* ends, int G, int tm) {
  const int64_t r = (int64_t)tm * kTileRows;
  int lo = 0, hi = G;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(ends + mid) <= r) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

template <typename T, bool ROW, bool COL, bool TEN>
__global__ void __launch_bounds__(kPipeThreads, 2)
    k_amax_tma(const __grid_constant__ CUtensorMap tmap, AmaxTmaArgs a) {
  using Geo = TileGeo<T>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full[kStages];
  __shared__ __align__(8) uint64_t empty[kStages];
  __shared__ volatile int abort_flag;
  // column maxima of a super-strip, combined over the four row groups of warps
  // before one global atomic per column (two buffers, used by alternate flushes)
  constexpr int kSpan = TileGrid::kGroup * Geo::TILEC;
  __shared__ uint32_t col_buf[COL ? 2 : 1][COL ? kSpan : 1];
  __shared__ __align__(8) uint64_t col_bar[2];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  if (noop_set(a.noop)) return;
  if (a.ends != nullptr && (!groups_valid(a.ends, a.G, a.M) ||
                            (a.col_grouped && !ends_aligned(a.ends, a.G, kTileRows)) ||
                            (a.pad_ends != nullptr &&
                             !pad_layout_valid(a.ends, a.pad_ends, a.G, a.M, a.pad_rows))))
    return;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int begin, end;
  a.grid.chunk(blockIdx.x, gridDim.x, begin, end);
  const int count = end - begin;
  const bool fwd = (blockIdx.x & 1) == 0;  // the encode kernel walks this chunk the other way
  if (warp == kConsumerWarps && lane == 0) prefetch_tmap(&tmap);  // while the barriers are set up
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    mbar_init(&col_bar[0], kConsumerWarps);
    mbar_init(&col_bar[1], kConsumerWarps);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (COL)
    for (int i = tid; i < 2 * kSpan; i += kPipeThreads) col_buf[i / kSpan][i % kSpan] = 0;
  __syncthreads();
  pdl_launch_dependents();
  if (count <= 0) return;

  if (warp == kConsumerWarps) {
    if (lane != 0) return;
    const uint64_t pol_first = policy_evict_first(), pol_last = policy_evict_last();
    TileCursor cur;
    cur.seek(a.grid, a.grid.walk(begin, end, 0, fwd));
    int issued = 0;
    for (int k = 0; k < count; ++k) {
      const int s = k % kStages;
      if (k >= kStages &&
          !mbar_wait_bounded(&empty[s], (uint32_t)(((k / kStages) - 1) & 1))) {
        abort_flag = 1;
        raise_status(a.status, kStatusTimeout);
        break;
      }
      if (abort_flag) break;
      issue_tile<T>(smem + s * kTileBytes, &tmap, &full[s], cur.tm * kTileRows, cur.tn(),
                    k >= count - a.keep_tiles ? pol_last : pol_first);
      cur.step(a.grid, fwd);
      issued = k + 1;
    }
    if (abort_flag)
      for (int k = issued - kStages > 0 ? issued - kStages : 0; k < issued; ++k)
        (void)mbar_wait_bounded(&full[k % kStages], (uint32_t)((k / kStages) & 1));
    return;
  }

  // consumers: the preceding kernel zeroes the outputs
  pdl_wait();
  const int box = warp & 1, rg = warp >> 1;
  const int c = lane & 7, ro = lane >> 3;
  const uint32_t offA = box * kBoxBytes + ((c ^ (ro & 7)) << 4);
  const uint32_t offB = box * kBoxBytes + ((c ^ ((ro + 4) & 7)) << 4);
  constexpr bool BF16 = sizeof(T) == 2;
  constexpr int NG = TileGrid::kGroup;
  using Acc = typename std::conditional<BF16, uint32_t, float>::type;
  Acc cm[NG][4];
#pragma unroll
  for (int g = 0; g < NG; ++g)
#pragma unroll
    for (int j = 0; j < 4; ++j) cm[g][j] = 0;
  Acc tmx = 0;
  int cur_ss = -1;

  int cur_g = 0, grp_tm = -1, grp = 0;  // grouped columns: group of the partials / of tile row grp_tm
  int n_col_flush = 0;
  // Publish the column maxima of super-strip ss: reduce over the 4 row lanes of
  // the warp, combine the 4 row-group warps in shared memory, then one global
  // atomic per column.  Returns false when the wait for the other warps ran out.
  auto flush_cols = [&](int ss) -> bool {
    const int b = n_col_flush & 1;
    const uint32_t parity = (uint32_t)((n_col_flush >> 1) & 1);
    ++n_col_flush;
    uint32_t* const buf = col_buf[b];
#pragma unroll
    for (int g = 0; g < NG; ++g) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if constexpr (BF16) {
          cm[g][j] = absmax_bf16x2(cm[g][j], __shfl_xor_sync(0xffffffffu, cm[g][j], 8));
          cm[g][j] = absmax_bf16x2(cm[g][j], __shfl_xor_sync(0xffffffffu, cm[g][j], 16));
        } else {
          cm[g][j] = fmaxf(cm[g][j], __shfl_xor_sync(0xffffffffu, cm[g][j], 8));
          cm[g][j] = fmaxf(cm[g][j], __shfl_xor_sync(0xffffffffu, cm[g][j], 16));
        }
      }
      if (ro == 0) {
        const int c0 = g * Geo::TILEC + box * Geo::BOXC + c * (16 / (int)sizeof(T));
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if constexpr (BF16) {
            const uint32_t mv = cm[g][j] & 0x7fff7fffu;
            if (mv & 0xffffu) atomicMax(&buf[c0 + 2 * j], mv << 16);
            if (mv >> 16) atomicMax(&buf[c0 + 2 * j + 1], mv & 0xffff0000u);
          } else {
            if (cm[g][j] > 0.0f) atomicMax(&buf[c0 + j], __float_as_uint(cm[g][j]));
          }
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) cm[g][j] = 0;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&col_bar[b]);
    if (!mbar_wait_bounded(&col_bar[b], parity)) return false;
    float* const cbase = a.col_amax + (a.col_grouped ? (int64_t)cur_g * a.K : 0);
    const int64_t span0 = (int64_t)ss * kSpan;
    for (int i = tid; i < kSpan; i += kConsumerWarps * 32) {
      const uint32_t v = buf[i];
      if (v == 0) continue;
      buf[i] = 0;  // free for the flush after next (ordered by the next flush's barrier)
      if (span0 + i < a.K) atomicMax(reinterpret_cast<unsigned int*>(cbase + span0 + i), v);
    }
    return true;
  };

  Acc rpa[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) rpa[i] = 0;
  int cur_tm = -1;
  // Row maxima of tile row tm_ accumulated over consecutive tiles of that row:
  // reduce over the 8 lanes that share a row, publish, reset.
  auto flush_rows = [&](int tm_) {
    const int64_t row0 = (int64_t)tm_ * kTileRows + rg * 32 + ro;
    if constexpr (BF16) {
      // fold each pair, pack two rows per word, reduce over the 8 lanes of the row
      uint32_t P[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t f0 = absmax_bf16x2(rpa[2 * j], __byte_perm(rpa[2 * j], 0, 0x1032));
        const uint32_t f1 = absmax_bf16x2(rpa[2 * j + 1], __byte_perm(rpa[2 * j + 1], 0, 0x1032));
        P[j] = __byte_perm(f0, f1, 0x7610);
      }
      const bool u4 = lane & 4, u2 = lane & 2;
      uint32_t q0 = absmax_bf16x2(u4 ? P[2] : P[0], __shfl_xor_sync(0xffffffffu, u4 ? P[0] : P[2], 4));
      uint32_t q1 = absmax_bf16x2(u4 ? P[3] : P[1], __shfl_xor_sync(0xffffffffu, u4 ? P[1] : P[3], 4));
      uint32_t rr = absmax_bf16x2(u2 ? q1 : q0, __shfl_xor_sync(0xffffffffu, u2 ? q0 : q1, 2));
      rr = absmax_bf16x2(rr, __shfl_xor_sync(0xffffffffu, rr, 1)) & 0x7fff7fffu;
      if ((lane & 1) == 0) {
        const int i0 = (u4 ? 4 : 0) + (u2 ? 2 : 0);
        const int64_t r0 = row0 + 4 * i0, r1 = r0 + 4;
        if (r0 < a.M) atomic_max_nonneg(&a.row_amax[r0], __uint_as_float(rr << 16));
        if (r1 < a.M) atomic_max_nonneg(&a.row_amax[r1], __uint_as_float(rr & 0xffff0000u));
      }
    } else {
      const bool u4 = lane & 4, u2 = lane & 2, u1 = lane & 1;
      float q[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        q[j] = fmaxf(u4 ? rpa[4 + j] : rpa[j], __shfl_xor_sync(0xffffffffu, u4 ? rpa[j] : rpa[4 + j], 4));
      float h[2];
#pragma unroll
      for (int j = 0; j < 2; ++j)
        h[j] = fmaxf(u2 ? q[2 + j] : q[j], __shfl_xor_sync(0xffffffffu, u2 ? q[j] : q[2 + j], 2));
      const float g = fmaxf(u1 ? h[1] : h[0], __shfl_xor_sync(0xffffffffu, u1 ? h[0] : h[1], 1));
      const int i0 = (u4 ? 4 : 0) + (u2 ? 2 : 0) + (u1 ? 1 : 0);
      const int64_t r0 = row0 + 4 * i0;
      if (r0 < a.M) atomic_max_nonneg(&a.row_amax[r0], g);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) rpa[i] = 0;
  };

  TileCursor cur;
  cur.seek(a.grid, a.grid.walk(begin, end, 0, fwd));
  for (int k = 0; k < count; ++k, cur.step(a.grid, fwd)) {
    const int s = k % kStages;
    const int tm = cur.tm, ss = cur.ss, gsel = cur.jt;
    if (COL) {
      // a new super-strip, or (grouped columns) a new group: publish the partials
      if (a.col_grouped && tm != grp_tm) {
        grp = group_of_tile_row(a.ends, a.G, tm);
        grp_tm = tm;
      }
      const int g_now = a.col_grouped ? grp : 0;
      if (ss != cur_ss || g_now != cur_g) {
        if (cur_ss >= 0 && !flush_cols(cur_ss)) {
          abort_flag = 1;
          if (lane == 0) raise_status(a.status, kStatusTimeout);
          break;
        }
        cur_ss = ss;
        cur_g = g_now;
      }
    }
    if (!mbar_wait_bounded(&full[s], (uint32_t)((k / kStages) & 1))) {
      abort_flag = 1;
      if (lane == 0) raise_status(a.status, kStatusTimeout);
      break;
    }
    if (abort_flag) break;
    const uint8_t* stage = smem + s * kTileBytes + (rg * 32 + ro) * 128;
    Acc rp[8], ct[4] = {0, 0, 0, 0};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint4 v = *reinterpret_cast<const uint4*>(stage + i * 4 * 128 + ((i & 1) ? offB : offA));
      if constexpr (BF16) {
        if (COL) {
          ct[0] = absmax_bf16x2(ct[0], v.x);
          ct[1] = absmax_bf16x2(ct[1], v.y);
          ct[2] = absmax_bf16x2(ct[2], v.z);
          ct[3] = absmax_bf16x2(ct[3], v.w);
        }
        rp[i] = absmax_bf16x2(absmax_bf16x2(v.x, v.y), absmax_bf16x2(v.z, v.w));
      } else {
        const float e0 = fabsf(__uint_as_float(v.x)), e1 = fabsf(__uint_as_float(v.y));
        const float e2 = fabsf(__uint_as_float(v.z)), e3 = fabsf(__uint_as_float(v.w));
        if (COL) {
          ct[0] = fmaxf(ct[0], e0);
          ct[1] = fmaxf(ct[1], e1);
          ct[2] = fmaxf(ct[2], e2);
          ct[3] = fmaxf(ct[3], e3);
        }
        rp[i] = fmaxf(fmaxf(e0, e1), fmaxf(e2, e3));
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);  // the tile is in registers now
    if (COL) {
      // merge into the partials of this tile's column strip (register arrays
      // cannot be indexed at run time: select)
#pragma unroll
      for (int g = 0; g < NG; ++g) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          Acc mv;
          if constexpr (BF16) mv = absmax_bf16x2(cm[g][j], ct[j]);
          else mv = fmaxf(cm[g][j], ct[j]);
          cm[g][j] = (g == gsel) ? mv : cm[g][j];
        }
      }
    }
    if (TEN) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if constexpr (BF16) tmx = absmax_bf16x2(tmx, rp[i]);
        else tmx = fmaxf(tmx, rp[i]);
      }
    }
    if (ROW) {
      if (tm != cur_tm) {
        if (cur_tm >= 0) flush_rows(cur_tm);
        cur_tm = tm;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if constexpr (BF16) rpa[i] = absmax_bf16x2(rpa[i], rp[i]);
        else rpa[i] = fmaxf(rpa[i], rp[i]);
      }
    }
  }
  if (COL && cur_ss >= 0 && !abort_flag && !flush_cols(cur_ss)) {
    abort_flag = 1;
    if (lane == 0) raise_status(a.status, kStatusTimeout);
  }
  if (ROW && cur_tm >= 0 && !abort_flag) flush_rows(cur_tm);
  if (TEN) {
    float m;
    if constexpr (BF16) m = bf16x2_hmax_f32(tmx);
    else m = tmx;
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) atomic_max_nonneg(a.tensor_amax, m);
  }
}

using AmaxTmaFn = void (*)(const CUtensorMap, AmaxTmaArgs);

template <typename T>
AmaxTmaFn pick_amax_tma(bool row, bool col, bool ten) {
  const int key = (row ? 4 : 0) | (col ? 2 : 0) | (ten ? 1 : 0);
  switch (key) {
    case 1: return k_amax_tma<T, false, false, true>;
    case 2: return k_amax_tma<T, false, true, false>;
    case 3: return k_amax_tma<T, false, true, true>;
    case 4: return k_amax_tma<T, true, false, false>;
    case 5: return k_amax_tma<T, true, false, true>;
    case 6: return k_amax_tma<T, true, true, false>;
    case 7: return k_amax_tma<T, true, true, true>;
    default: return nullptr;
  }
}

// ---------------------------------------------------------------- grouped

constexpr int kMaxGroups = 4096;

// Loads the group ends into shared memory and checks them.  Returns false when
// invalid.  Every thread of the block must call it.
__device__ bool load_group_ends(const int64_t* ends, int G, int64_t M, int64_t* s_ends) {
  for (int g = threadIdx.x; g < G; g += blockDim.x) s_ends[g] = ends[g];
  return groups_valid(ends, G, M);
}

// group of row r = number of ends <= r (ends non-decreasing)
__device__ __forceinline__ int group_of(const int64_t* s_ends, int G, int64_t r) {
  int lo = 0, hi = G;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (s_ends[mid] <= r) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

struct GroupedKernelArgs {
  const void* x;
  int64_t M, K;
  const int64_t* ends;
  int G;
  float* group_amax;
  const float* noop;
  int* status;
  int64_t rows_per_item;
  int num_col_items;
  const int64_t* pad_ends;  // optional: also require this padded layout of the groups
  int64_t pad_rows;
  int tile_aligned;  // also require every group end to be a multiple of kTileRows
};

// Per-group amax: like the tensor reduction, but a CTA item is split at group
// boundaries; each row adds its maximum to its group's running maximum.
template <bool BF16, bool VEC>
__global__ void __launch_bounds__(kThreads) k_grouped_amax(GroupedKernelArgs a) {
  constexpr int VE = BF16 ? 8 : 4, CW = kColWarps * 32 * VE;
  __shared__ int64_t s_ends[kMaxGroups];
  __shared__ float row_red[kColWarps][512];
  if (noop_set(a.noop)) return;
  const bool ok = load_group_ends(a.ends, a.G, a.M, s_ends);
  if (!ok ||
      (a.pad_ends != nullptr && !pad_layout_valid(a.ends, a.pad_ends, a.G, a.M, a.pad_rows)) ||
      (a.tile_aligned && !ends_aligned(a.ends, a.G, kTileRows))) {
    if (blockIdx.x == 0 && threadIdx.x == 0) raise_status(a.status, kStatusBadGroups);
    return;
  }
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int cw = w % kColWarps, rg = w / kColWarps;
  const int64_t band = blockIdx.x / a.num_col_items, cr = blockIdx.x % a.num_col_items;
  const int64_t r0 = band * a.rows_per_item;
  const int64_t c = cr * CW + cw * 32 * VE + lane * VE;
  const uint64_t pol = policy_evict_normal();
  const int chunks = (int)(a.rows_per_item / (8 * kRowGroups));
  for (int k = 0; k < chunks; ++k) {
    const int64_t rr = r0 + (int64_t)(k * kRowGroups + rg) * 8;
    float rp[8];
    if constexpr (BF16) {
      const uint16_t* x = static_cast<const uint16_t*>(a.x);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        uint4 v = load_bf16x8<VEC>(x, a.M, a.K, rr + i, c, pol);
        rp[i] = bf16x2_hmax_f32(absmax_bf16x2(absmax_bf16x2(v.x, v.y), absmax_bf16x2(v.z, v.w)));
      }
    } else {
      const float* x = static_cast<const float*>(a.x);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        float4 v = load_f32x4<VEC>(x, a.M, a.K, rr + i, c, pol);
        rp[i] = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
      }
    }
    const float R = warp_rowmax8_f32(rp, lane);
    if ((lane & 3) == 0) {
      const int rl = (k * kRowGroups + rg) * 8 + ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 +
                     ((lane >> 2) & 1);
      row_red[cw][rl] = R;
    }
  }
  __syncthreads();
  // one thread per row of the item; combine consecutive rows of the same group
  // through a warp segment-max before the atomic
  for (int t = tid; t < a.rows_per_item; t += kThreads) {
    const int64_t r = r0 + t;
    float m = (r < a.M) ? fmaxf(row_red[0][t], row_red[1][t]) : 0.0f;
    const int g = (r < a.M) ? group_of(s_ends, a.G, r) : -1;
    // segmented max over lanes with the same group (groups are contiguous)
    for (int o = 1; o < 32; o <<= 1) {
      const float mo = __shfl_down_sync(0xffffffffu, m, o);
      const int go = __shfl_down_sync(0xffffffffu, g, o);
      if ((lane + o) < 32 && go == g) m = fmaxf(m, mo);
    }
    const int gp = __shfl_up_sync(0xffffffffu, g, 1);
    if (g >= 0 && (lane == 0 || gp != g)) atomic_max_nonneg(&a.group_amax[g], m);
  }
}

// Group maxima from per-row maxima: group_amax[g] = max of row_max over the rows of
// group g, and with `expand` every row of group g then takes that value (row_max is
// the per-row amax output of the grouped quantize).  A CTA owns whole groups
// (g = blockIdx.x, += gridDim.x): it reads a group's rows before it writes them, and
// no other CTA touches them.  Nothing is written unless the ends are valid.
__global__ void __launch_bounds__(kThreads) k_group_reduce(GroupReduceArgs a) {
  __shared__ int64_t s_ends[kMaxGroups];
  __shared__ float red[kThreads / 32];
  __shared__ float s_m;
  if (noop_set(a.noop)) return;
  if (!load_group_ends(a.group_ends, a.num_groups, a.M, s_ends)) return;
  if (a.pad_ends != nullptr &&
      !pad_layout_valid(a.group_ends, a.pad_ends, a.num_groups, a.M, a.pad_rows))
    return;
  const int tid = threadIdx.x;
  for (int g = blockIdx.x; g < a.num_groups; g += gridDim.x) {
    const int64_t r0 = g ? s_ends[g - 1] : 0, r1 = s_ends[g];
    float m = 0.0f;
    for (int64_t r = r0 + tid; r < r1; r += kThreads) m = fmaxf(m, a.row_max[r]);
    m = block_max(m, red);
    if (tid == 0) {
      a.group_amax[g] = m;
      s_m = m;
    }
    __syncthreads();
    if (a.expand) {
      const float v = s_m;
      for (int64_t r = r0 + tid; r < r1; r += kThreads) a.row_max[r] = v;
    }
    __syncthreads();  // s_m and red are reused by the next group
  }
}

__global__ void k_group_check(GroupCheckArgs a, int* status, bool expand_pass) {
  __shared__ int64_t s_ends[kMaxGroups];
  pdl_launch_dependents();  // as k_prep: the next kernel waits before it reads our outputs
  if (noop_set(a.noop)) return;
  const bool ok = load_group_ends(a.group_ends, a.num_groups, a.M, s_ends);
  // padded layout: group_ends are the padded ends (M output rows), rag_ends the
  // ragged ends of x (in_rows rows)
  if (!ok ||
      (a.rag_ends != nullptr &&
       !pad_layout_valid(a.rag_ends, a.group_ends, a.num_groups, a.in_rows, a.M)) ||
      (a.tile_aligned && !ends_aligned(a.group_ends, a.num_groups, kTileRows))) {
    if (blockIdx.x == 0 && threadIdx.x == 0) raise_status(status, kStatusBadGroups);
    return;
  }
  const int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t step = (int64_t)gridDim.x * blockDim.x;
#pragma unroll
  for (int k = 0; k < 4; ++k)
    if (a.prep.zero_ptr[k] != nullptr)
      for (int64_t i = i0; i < a.prep.zero_n[k]; i += step) a.prep.zero_ptr[k][i] = 0.0f;
#pragma unroll
  for (int k = 0; k < 2; ++k)
    if (a.prep.copy_dst[k] != nullptr)
      for (int64_t i = i0; i < a.prep.copy_n[k]; i += step)
        a.prep.copy_dst[k][i] = a.prep.copy_src[k][i];
  if (!expand_pass || a.expand == nullptr) return;
  for (int64_t r = i0; r < a.M; r += step)
    a.expand[r] = a.group_amax[group_of(s_ends, a.num_groups, r)];
}

int pick_rows_per_item(int64_t M, int64_t col_items, int num_sms) {
  // Largest power of two in [32, 512] that still gives >= 8 items per SM
  // (fewer atomics per element, enough CTAs to balance the SMs).
  int rb = 512;
  while (rb > 32 && ((M + rb - 1) / rb) * col_items < 8LL * num_sms) rb >>= 1;
  return rb;
}

}  // namespace

cudaError_t launch_prep(const PrepArgs& a, const DeviceInfo& dev, cudaStream_t stream) {
  int64_t n = 1;
  for (int k = 0; k < 4; ++k) n = std::max(n, a.zero_n[k]);
  for (int k = 0; k < 2; ++k) n = std::max(n, a.copy_n[k]);
  const int64_t blocks = std::min<int64_t>((n + 255) / 256, 4LL * dev.num_sms);
  k_prep<<<(unsigned)blocks, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_amax(const AmaxArgs& a, const DeviceInfo& dev, cudaStream_t stream) {
  if (a.M == 0 || a.K == 0) return cudaSuccess;
  {
    const bool bf16 = a.in == InType::BF16;
    const int box_cols = bf16 ? TileGeo<uint16_t>::BOXC : TileGeo<float>::BOXC;
    CUtensorMap map;
    if (make_tile_map(&map, a.x, a.in, a.M, a.K, box_cols, kTileRows)) {
      AmaxTmaArgs k{};
      k.M = a.M;
      k.K = a.K;
      k.grid.tiles_m = (int)((a.M + kTileRows - 1) / kTileRows);
      k.grid.tiles_n = (int)((a.K + 2 * box_cols - 1) / (2 * box_cols));
      k.grid.num_tiles = k.grid.tiles_m * k.grid.tiles_n;
      k.row_amax = a.row_amax;
      k.col_amax = a.col_amax;
      k.tensor_amax = a.tensor_amax;
      k.noop = a.noop;
      k.ends = a.group_ends;
      k.G = a.num_groups;
      k.pad_ends = a.pad_ends;
      k.pad_rows = a.pad_rows;
      k.status = dev.status;
      k.col_grouped = a.col_grouped ? 1 : 0;
      const int grid = pipe_grid_size(k.grid.num_tiles, dev.num_sms);
      // keep about 80 MB of the tail of the walk in L2 for the encode pass
      k.keep_tiles = (int)std::max<int64_t>(1, (80LL << 20) / ((int64_t)grid * kTileBytes));
      AmaxTmaFn fn = bf16 ? pick_amax_tma<uint16_t>(a.row_amax, a.col_amax, a.tensor_amax)
                          : pick_amax_tma<float>(a.row_amax, a.col_amax, a.tensor_amax);
      if (fn == nullptr) return cudaSuccess;
      constexpr int smem = kStages * kTileBytes + 1024;
      cudaError_t err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (err != cudaSuccess) return err;
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((unsigned)grid);
      cfg.blockDim = dim3(kPipeThreads);
      cfg.dynamicSmemBytes = smem;
      cfg.stream = stream;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[0].val.programmaticStreamSerializationAllowed = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      return cudaLaunchKernelEx(&cfg, fn, map, k);
    }
  }
  // x rows not 16-byte aligned: plain 128-bit (or scalar) loads
  const int elem = a.in == InType::BF16 ? 2 : 4;
  const int VE = 16 / elem;
  const int CW = kColWarps * 32 * VE;
  const bool vec = (a.K % VE == 0) && (reinterpret_cast<uintptr_t>(a.x) % 16 == 0);
  AmaxKernelArgs k{};
  k.x = a.x;
  k.M = a.M;
  k.K = a.K;
  k.row_amax = a.row_amax;
  k.col_amax = a.col_amax;
  k.tensor_amax = a.tensor_amax;
  k.noop = a.noop;
  k.ends = a.group_ends;
  k.G = a.num_groups;
  k.pad_ends = a.pad_ends;
  k.pad_rows = a.pad_rows;
  k.num_col_items = (int)((a.K + CW - 1) / CW);
  k.rows_per_item = pick_rows_per_item(a.M, k.num_col_items, dev.num_sms);
  // keep the last ~80 MB of x in L2 for the encode pass, which walks x backwards
  const int64_t row_bytes = a.K * elem;
  const int64_t keep_rows = std::max<int64_t>(0, (80LL << 20) / std::max<int64_t>(row_bytes, 1));
  k.keep_from_row = std::max<int64_t>(0, a.M - keep_rows);
  AmaxFn fn = pick_amax(a.in, vec, a.row_amax != nullptr, a.col_amax != nullptr,
                        a.tensor_amax != nullptr);
  if (fn == nullptr) return cudaSuccess;
  const int64_t items = ((a.M + k.rows_per_item - 1) / k.rows_per_item) * k.num_col_items;
  fn<<<(unsigned)items, kThreads, 0, stream>>>(k);
  return cudaGetLastError();
}

cudaError_t launch_grouped_amax(const GroupedAmaxArgs& a, const DeviceInfo& dev,
                                cudaStream_t stream) {
  if (a.M == 0 || a.K == 0) return cudaSuccess;
  const int elem = a.in == InType::BF16 ? 2 : 4;
  const int VE = 16 / elem;
  const int CW = kColWarps * 32 * VE;
  const bool vec = (a.K % VE == 0) && (reinterpret_cast<uintptr_t>(a.x) % 16 == 0);
  GroupedKernelArgs k{};
  k.x = a.x;
  k.M = a.M;
  k.K = a.K;
  k.ends = a.group_ends;
  k.G = a.num_groups;
  k.group_amax = a.group_amax;
  k.noop = a.noop;
  k.status = dev.status;
  k.pad_ends = a.pad_ends;
  k.pad_rows = a.pad_rows;
  k.tile_aligned = a.tile_aligned ? 1 : 0;
  k.num_col_items = (int)((a.K + CW - 1) / CW);
  k.rows_per_item = pick_rows_per_item(a.M, k.num_col_items, dev.num_sms);
  const int64_t items = ((a.M + k.rows_per_item - 1) / k.rows_per_item) * k.num_col_items;
  void (*fn)(GroupedKernelArgs);
  if (a.in == InType::BF16) fn = vec ? k_grouped_amax<true, true> : k_grouped_amax<true, false>;
  else fn = vec ? k_grouped_amax<false, true> : k_grouped_amax<false, false>;
  fn<<<(unsigned)items, kThreads, 0, stream>>>(k);
  return cudaGetLastError();
}

cudaError_t launch_group_reduce(const GroupReduceArgs& a, const DeviceInfo& dev,
                                cudaStream_t stream) {
  const int blocks = std::min(a.num_groups, 2 * dev.num_sms);
  if (blocks < 1) return cudaSuccess;
  k_group_reduce<<<(unsigned)blocks, kThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_group_check(const GroupCheckArgs& a, const DeviceInfo& dev,
                               cudaStream_t stream, bool expand_pass) {
  int64_t n = expand_pass ? a.M : 0;
  for (int k = 0; k < 4; ++k) n = std::max(n, a.prep.zero_n[k]);
  for (int k = 0; k < 2; ++k) n = std::max(n, a.prep.copy_n[k]);
  const int64_t blocks = std::max<int64_t>(1, std::min<int64_t>((n + 255) / 256, 2LL * dev.num_sms));
  k_group_check<<<(unsigned)blocks, 256, 0, stream>>>(a, dev.status, expand_pass);
  return cudaGetLastError();
}

}  // namespace nvfp4
