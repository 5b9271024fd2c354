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
// Design (sm_103a): a persistent grid of 2 CTAs per SM walks 128-row tiles of x
// (128 BF16 or 64 FP32 columns = two 128-byte TMA boxes with the 128-byte
// swizzle) through a 3-stage shared-memory ring filled by cp.async.bulk.tensor
// and tracked by mbarriers.  Rowwise blocks are read as 16-byte rows of a box;
// columnwise blocks are read down a column pair; both access patterns are
// bank-conflict free under the swizzle.  Tiles are visited in reverse order so
// that the tail of x, which the amax pass read last, is re-read from L2.
#include <algorithm>

#include "device_common.cuh"
#include "internal.h"

namespace nvfp4 {

namespace {

constexpr int kThreads = 256;
constexpr int kTileRows = 128;
constexpr int kStages = 3;
constexpr int kBoxBytes = 128 * 128;       // 128 rows x 128 bytes
constexpr int kStageBytes = 2 * kBoxBytes;  // two boxes per tile
constexpr int kSmemBytes = kStages * kStageBytes + 1024;

template <typename T>
struct Geo {
  static constexpr int ELEM = sizeof(T);
  static constexpr int BOXC = 128 / ELEM;  // columns per box (64 BF16 / 32 FP32)
  static constexpr int TILEC = 2 * BOXC;   // columns per tile
  static constexpr int NB_R = BOXC / 16;   // rowwise blocks per thread
  static constexpr int NP = TILEC / 2;     // column pairs per tile
  static constexpr int NQ = kThreads / NP; // row groups of the columnwise threads
  static constexpr int RQ = kTileRows / NQ;// rows per columnwise thread
  static constexpr int NB_C = RQ / 16;     // columnwise blocks per column per thread
  static constexpr int SUBC = TILEC / 16;  // 16x16 sub-tiles across a tile
  static constexpr int NSUB = (kTileRows / 16) * SUBC;
};

// Byte offset of element (r, c) of a tile in its stage buffer (128-byte swizzle:
// the 16-byte chunk index inside each 128-byte row is XORed with r mod 8).
template <typename T>
__device__ __forceinline__ uint32_t soff(int r, int c) {
  constexpr int BOXC = Geo<T>::BOXC;
  const int box = c / BOXC;
  const int byte = (c % BOXC) * (int)sizeof(T);
  return box * kBoxBytes + r * 128 + ((((byte >> 4) ^ (r & 7))) << 4) + (byte & 15);
}

__device__ __forceinline__ uint4 lds128(const uint8_t* p) {
  return *reinterpret_cast<const uint4*>(p);
}

struct QuantKernelArgs {
  const void* x;
  int64_t M, K;
  int64_t tiles_n, num_tiles;
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
};

// ---------------------------------------------------------------- per-thread work

// Unpack 16 values of a rowwise block from two 16-byte chunks.
template <typename T>
__device__ __forceinline__ void unpack16(const uint4& v0, const uint4& v1, const uint4& v2,
                                         const uint4& v3, float* x) {
  if constexpr (sizeof(T) == 2) {
    const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      x[2 * i] = bf16_lo(w[i]);
      x[2 * i + 1] = bf16_hi(w[i]);
    }
  } else {
    const uint32_t w[16] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w,
                            v2.x, v2.y, v2.z, v2.w, v3.x, v3.y, v3.z, v3.w};
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = __uint_as_float(w[i]);
  }
}

template <typename T, bool B2D>
__device__ __forceinline__ uint32_t encode_block(const float* x, float S, float a, float F_inv,
                                                 bool fos, uint32_t s2d, float e2d, uint32_t& c0,
                                                 uint32_t& c1) {
  if constexpr (B2D) {
    c0 = e2m1x8(__fmul_rn(x[0], e2d), __fmul_rn(x[1], e2d), __fmul_rn(x[2], e2d),
                __fmul_rn(x[3], e2d), __fmul_rn(x[4], e2d), __fmul_rn(x[5], e2d),
                __fmul_rn(x[6], e2d), __fmul_rn(x[7], e2d));
    c1 = e2m1x8(__fmul_rn(x[8], e2d), __fmul_rn(x[9], e2d), __fmul_rn(x[10], e2d),
                __fmul_rn(x[11], e2d), __fmul_rn(x[12], e2d), __fmul_rn(x[13], e2d),
                __fmul_rn(x[14], e2d), __fmul_rn(x[15], e2d));
    return s2d;
  } else {
    if (fos) return quantize16<true>(x, S, a, F_inv, c0, c1);
    return quantize16<false>(x, S, a, F_inv, c0, c1);
  }
}

// Rowwise: thread = one row of one box (NB_R blocks of 16).
template <typename T, bool FOS, bool B2D>
__device__ __forceinline__ void rowwise_tile(const uint8_t* stage, const QuantKernelArgs& a,
                                             int64_t tm, int64_t tn, float S_tensor,
                                             const uint32_t* s2d_s8, const float* s2d_e) {
  using G = Geo<T>;
  const int tid = threadIdx.x;
  const int r = tid & (kTileRows - 1), box = tid >> 7;
  const int64_t gr = tm * kTileRows + r;
  const int64_t gc0 = tn * G::TILEC + box * G::BOXC;
  if (gr >= a.M || gc0 >= a.K) return;
  const float amax = a.row_amax[a.row_scaled ? gr : 0];
  const float S = a.row_scaled ? global_scale(amax, a.F) : S_tensor;
  uint32_t w[2 * G::NB_R];
  uint32_t sc = 0;
  const uint8_t* rowp = stage + box * kBoxBytes + r * 128;
#pragma unroll
  for (int j = 0; j < G::NB_R; ++j) {
    float x[16];
    constexpr int CH = 16 * (int)sizeof(T) / 16;  // 16-byte chunks per block (2 or 4)
    uint4 v[4];
#pragma unroll
    for (int k = 0; k < CH; ++k) v[k] = lds128(rowp + ((((CH * j + k) ^ (r & 7))) << 4));
    unpack16<T>(v[0], v[1], CH > 2 ? v[2] : v[0], CH > 2 ? v[3] : v[0], x);
    uint32_t s8s = 0;
    float e2 = 0.f;
    if constexpr (B2D) {
      const int sub = (r >> 4) * G::SUBC + (box * G::BOXC) / 16 + j;
      s8s = s2d_s8[sub];
      e2 = s2d_e[sub];
    }
    const uint32_t s8 = encode_block<T, B2D>(x, S, amax, a.F_inv, FOS, s8s, e2, w[2 * j],
                                             w[2 * j + 1]);
    sc |= s8 << (8 * j);
  }
  const int64_t rem_c = a.K - gc0;
  const int ncols = rem_c < G::BOXC ? (int)rem_c : G::BOXC;
  const int nbytes = (int)((ncols + 1) / 2);
  const int nsc = (int)((ncols + 15) / 16);
  uint8_t* cp = a.row_codes + gr * a.row_cpitch + gc0 / 2;
  store_bytes(cp, w, nbytes < 16 ? nbytes : 16);
  if (nbytes > 16) store_bytes(cp + 16, w + 4, nbytes - 16);
  store_bytes(a.row_scales + gr * a.row_spitch + gc0 / 16, &sc, nsc);
}

// Columnwise: thread = a column pair over RQ rows (NB_C blocks per column).
template <typename T, bool FOS, bool B2D>
__device__ __forceinline__ void colwise_tile(const uint8_t* stage, const QuantKernelArgs& a,
                                             int64_t tm, int64_t tn, float S_tensor,
                                             const uint32_t* s2d_s8, const float* s2d_e) {
  using G = Geo<T>;
  const int tid = threadIdx.x;
  const int p = tid % G::NP, q = tid / G::NP;
  const int cl = 2 * p;
  const int64_t gc = tn * G::TILEC + cl;
  const int64_t gr0 = tm * kTileRows + q * G::RQ;
  if (gc >= a.K || gr0 >= a.M) return;
  const bool has1 = gc + 1 < a.K;
  const float a0 = a.row_scaled ? a.col_amax[gc] : a.col_amax[0];
  const float a1 = has1 ? (a.row_scaled ? a.col_amax[gc + 1] : a.col_amax[0]) : 0.0f;
  const float S0 = a.row_scaled ? global_scale(a0, a.F) : S_tensor;
  const float S1 = a.row_scaled ? global_scale(a1, a.F) : S_tensor;
  uint32_t w0[2 * G::NB_C], w1[2 * G::NB_C];
  uint32_t sc0 = 0, sc1 = 0;
#pragma unroll
  for (int jb = 0; jb < G::NB_C; ++jb) {
    const int rb = q * G::RQ + 16 * jb;
    float x0[16], x1[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if constexpr (sizeof(T) == 2) {
        const uint32_t v = *reinterpret_cast<const uint32_t*>(stage + soff<T>(rb + i, cl));
        x0[i] = bf16_lo(v);
        x1[i] = bf16_hi(v);
      } else {
        const float2 v = *reinterpret_cast<const float2*>(stage + soff<T>(rb + i, cl));
        x0[i] = v.x;
        x1[i] = v.y;
      }
    }
    uint32_t s8s = 0;
    float e2 = 0.f;
    if constexpr (B2D) {
      const int sub = (rb >> 4) * G::SUBC + cl / 16;
      s8s = s2d_s8[sub];
      e2 = s2d_e[sub];
    }
    sc0 |= encode_block<T, B2D>(x0, S0, a0, a.F_inv, FOS, s8s, e2, w0[2 * jb], w0[2 * jb + 1])
           << (8 * jb);
    sc1 |= encode_block<T, B2D>(x1, S1, a1, a.F_inv, FOS, s8s, e2, w1[2 * jb], w1[2 * jb + 1])
           << (8 * jb);
  }
  const int64_t rem_r = a.M - gr0;
  const int nrows = rem_r < G::RQ ? (int)rem_r : G::RQ;
  const int nbytes = (int)((nrows + 1) / 2);
  const int nsc = (int)((nrows + 15) / 16);
  store_bytes(a.col_codes + gc * a.col_cpitch + gr0 / 2, w0, nbytes);
  store_bytes(a.col_scales + gc * a.col_spitch + gr0 / 16, &sc0, nsc);
  if (has1) {
    store_bytes(a.col_codes + (gc + 1) * a.col_cpitch + gr0 / 2, w1, nbytes);
    store_bytes(a.col_scales + (gc + 1) * a.col_spitch + gr0 / 16, &sc1, nsc);
  }
}

// 16x16 blocks: one thread per sub-tile picks its scale (and, with
// four-over-six, its target by the error summed in row-major order).
template <typename T, bool FOS>
__device__ __forceinline__ void subtile_scales(const uint8_t* stage, const QuantKernelArgs& a,
                                               float S, float amax, uint32_t* s2d_s8,
                                               float* s2d_e) {
  using G = Geo<T>;
  const int tid = threadIdx.x;
  if (tid >= G::NSUB) return;
  const int sr = tid / G::SUBC, sc = tid % G::SUBC;
  constexpr int CH = 16 * (int)sizeof(T) / 16;
  auto load_row = [&](int i, float* x) {
    const int r = sr * 16 + i;
    const uint8_t* rowp = stage + ((sc * 16) / G::BOXC) * kBoxBytes + r * 128;
    const int cb = ((sc * 16) % G::BOXC) * (int)sizeof(T) / 16;  // first chunk in the box row
    uint4 v[4];
#pragma unroll
    for (int k = 0; k < CH; ++k) v[k] = lds128(rowp + ((((cb + k) ^ (r & 7))) << 4));
    unpack16<T>(v[0], v[1], CH > 2 ? v[2] : v[0], CH > 2 ? v[3] : v[0], x);
  };
  float b = 0.0f;
  for (int i = 0; i < 16; ++i) {
    float x[16];
    load_row(i, x);
#pragma unroll
    for (int k = 0; k < 16; ++k) b = fmaxf(b, fabsf(x[k]));
  }
  BlockEnc e6 = block_encode<6>(b, S);
  if constexpr (FOS) {
    BlockEnc e4 = block_encode<4>(b, S);
    const float D6 = dequant_factor(e6.sd, amax, a.F_inv);
    const float D4 = dequant_factor(e4.sd, amax, a.F_inv);
    float err6 = 0.0f, err4 = 0.0f;
    for (int i = 0; i < 16; ++i) {
      float x[16];
      load_row(i, x);
      uint32_t c[4];
      c[0] = e2m1x8(__fmul_rn(x[0], e6.e), __fmul_rn(x[1], e6.e), __fmul_rn(x[2], e6.e),
                    __fmul_rn(x[3], e6.e), __fmul_rn(x[4], e6.e), __fmul_rn(x[5], e6.e),
                    __fmul_rn(x[6], e6.e), __fmul_rn(x[7], e6.e));
      c[1] = e2m1x8(__fmul_rn(x[8], e6.e), __fmul_rn(x[9], e6.e), __fmul_rn(x[10], e6.e),
                    __fmul_rn(x[11], e6.e), __fmul_rn(x[12], e6.e), __fmul_rn(x[13], e6.e),
                    __fmul_rn(x[14], e6.e), __fmul_rn(x[15], e6.e));
      c[2] = e2m1x8(__fmul_rn(x[0], e4.e), __fmul_rn(x[1], e4.e), __fmul_rn(x[2], e4.e),
                    __fmul_rn(x[3], e4.e), __fmul_rn(x[4], e4.e), __fmul_rn(x[5], e4.e),
                    __fmul_rn(x[6], e4.e), __fmul_rn(x[7], e4.e));
      c[3] = e2m1x8(__fmul_rn(x[8], e4.e), __fmul_rn(x[9], e4.e), __fmul_rn(x[10], e4.e),
                    __fmul_rn(x[11], e4.e), __fmul_rn(x[12], e4.e), __fmul_rn(x[13], e4.e),
                    __fmul_rn(x[14], e4.e), __fmul_rn(x[15], e4.e));
      err6 = sse8(sse8(err6, x, c[0], D6), x + 8, c[1], D6);
      err4 = sse8(sse8(err4, x, c[2], D4), x + 8, c[3], D4);
    }
    if (err4 < err6) e6 = e4;
  }
  s2d_s8[tid] = e6.s8;
  s2d_e[tid] = e6.e;
}

// ---------------------------------------------------------------- the kernel

template <typename T, bool ROW, bool COL, bool FOS, bool B2D, bool TMA>
__global__ void __launch_bounds__(kThreads, 2)
    k_quantize(const __grid_constant__ CUtensorMap tmap, QuantKernelArgs a) {
  using G = Geo<T>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full[kStages];
  __shared__ uint32_t s2d_s8[B2D ? G::NSUB : 1];
  __shared__ float s2d_e[B2D ? G::NSUB : 1];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  if (noop_set(a.noop)) return;
  if (a.ends != nullptr && !groups_valid(a.ends, a.G, a.M)) return;
  const int tid = threadIdx.x;
  if (blockIdx.x == 0 && tid == 0 && a.copy_dst != nullptr) *a.copy_dst = *a.copy_src;

  const int64_t G_ = gridDim.x;
  const int64_t first = blockIdx.x;
  if (first >= a.num_tiles) return;
  const int64_t count = (a.num_tiles - first + G_ - 1) / G_;
  auto tile_of = [&](int64_t k) { return a.num_tiles - 1 - (first + k * G_); };

  // per-tensor scales, one per direction (16x16 blocks share the rowwise one:
  // the host launches the directions separately when their amax sources differ)
  const float amax_r = (ROW && !a.row_scaled) ? a.row_amax[0] : 0.0f;
  const float amax_c = (COL && !a.row_scaled) ? a.col_amax[0] : 0.0f;
  const float S_row = a.row_scaled ? 1.0f : global_scale(amax_r, a.F);
  const float S_col = a.row_scaled ? 1.0f : global_scale(amax_c, a.F);
  const float amax_2d = ROW ? amax_r : amax_c;
  const float S_2d = ROW ? S_row : S_col;

  uint64_t policy = 0;
  if constexpr (TMA) {
    policy = policy_evict_first();
    if (tid == 0) {
      prefetch_tmap(&tmap);
      for (int s = 0; s < kStages; ++s) mbar_init(&full[s], 1);
      fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) {
      for (int s = 0; s < kStages && s < count; ++s) {
        const int64_t t = tile_of(s);
        const int32_t y = (int32_t)((t / a.tiles_n) * kTileRows);
        const int32_t x0 = (int32_t)((t % a.tiles_n) * G::TILEC);
        uint8_t* dst = smem + s * kStageBytes;
        mbar_expect_tx(&full[s], kStageBytes);
        tma_load_2d(dst, &tmap, &full[s], x0, y, policy);
        tma_load_2d(dst + kBoxBytes, &tmap, &full[s], x0 + G::BOXC, y, policy);
      }
    }
  }

  for (int64_t k = 0; k < count; ++k) {
    const int s = (int)(k % kStages);
    const int64_t t = tile_of(k);
    const int64_t tm = t / a.tiles_n, tn = t % a.tiles_n;
    uint8_t* stage = smem + s * kStageBytes;
    if constexpr (TMA) {
      const bool ok = mbar_wait_bounded(&full[s], (uint32_t)((k / kStages) & 1));
      if (__syncthreads_or(!ok)) {
        if (tid == 0) {
          raise_status(a.status, kStatusTimeout);
          // let the copies already issued land before this CTA's memory is released
          for (int64_t j = k + 1; j < count && j < k + kStages; ++j)
            (void)mbar_wait_bounded(&full[j % kStages], (uint32_t)((j / kStages) & 1));
        }
        __syncthreads();
        return;
      }
    } else {
      // plain loads into the same swizzled layout (x rows not 16-byte aligned)
      const T* x = static_cast<const T*>(a.x);
      for (int idx = tid; idx < kTileRows * G::TILEC; idx += kThreads) {
        const int r = idx / G::TILEC, c = idx % G::TILEC;
        const int64_t gr = tm * kTileRows + r, gc = tn * G::TILEC + c;
        T v = T(0);
        if (gr < a.M && gc < a.K) v = x[gr * a.K + gc];
        *reinterpret_cast<T*>(stage + soff<T>(r, c)) = v;
      }
      __syncthreads();
    }
    if constexpr (B2D) {
      subtile_scales<T, FOS>(stage, a, S_2d, amax_2d, s2d_s8, s2d_e);
      __syncthreads();
    }
    if constexpr (ROW) rowwise_tile<T, FOS, B2D>(stage, a, tm, tn, S_row, s2d_s8, s2d_e);
    if constexpr (COL) colwise_tile<T, FOS, B2D>(stage, a, tm, tn, S_col, s2d_s8, s2d_e);
    __syncthreads();  // stage s is free again
    if constexpr (TMA) {
      if (tid == 0 && k + kStages < count) {
        const int64_t t2 = tile_of(k + kStages);
        const int32_t y = (int32_t)((t2 / a.tiles_n) * kTileRows);
        const int32_t x0 = (int32_t)((t2 % a.tiles_n) * G::TILEC);
        mbar_expect_tx(&full[s], kStageBytes);
        tma_load_2d(stage, &tmap, &full[s], x0, y, policy);
        tma_load_2d(stage + kBoxBytes, &tmap, &full[s], x0 + G::BOXC, y, policy);
      }
    }
  }
}

using QuantFn = void (*)(const CUtensorMap, QuantKernelArgs);

template <typename T, bool ROW, bool COL, bool FOS, bool B2D>
QuantFn pick_tma(bool tma) {
  return tma ? k_quantize<T, ROW, COL, FOS, B2D, true> : k_quantize<T, ROW, COL, FOS, B2D, false>;
}

template <typename T, bool ROW, bool COL>
QuantFn pick_mode(bool fos, bool b2d, bool tma) {
  if (b2d) return fos ? pick_tma<T, ROW, COL, true, true>(tma) : pick_tma<T, ROW, COL, false, true>(tma);
  return fos ? pick_tma<T, ROW, COL, true, false>(tma) : pick_tma<T, ROW, COL, false, false>(tma);
}

template <typename T>
QuantFn pick_dir(bool row, bool col, bool fos, bool b2d, bool tma) {
  if (row && col) return pick_mode<T, true, true>(fos, b2d, tma);
  if (row) return pick_mode<T, true, false>(fos, b2d, tma);
  return pick_mode<T, false, true>(fos, b2d, tma);
}

}  // namespace

cudaError_t launch_quantize(const QuantArgs& q, const DeviceInfo& dev, cudaStream_t stream) {
  const bool row = q.row_codes != nullptr, col = q.col_codes != nullptr;
  if (!row && !col) return cudaSuccess;
  const bool bf16 = q.in == InType::BF16;
  const int box_cols = bf16 ? Geo<uint16_t>::BOXC : Geo<float>::BOXC;
  const int tile_cols = 2 * box_cols;
  QuantKernelArgs a{};
  a.x = q.x;
  a.M = q.M;
  a.K = q.K;
  a.tiles_n = (q.K + tile_cols - 1) / tile_cols;
  a.num_tiles = ((q.M + kTileRows - 1) / kTileRows) * a.tiles_n;
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
  a.copy_dst = q.copy_dst;
  a.copy_src = q.copy_src;
  a.noop = q.noop;
  a.status = dev.status;
  a.ends = q.group_ends;
  a.G = q.num_groups;
  if (a.num_tiles == 0) return cudaSuccess;

  CUtensorMap map;
  const bool tma = make_tile_map(&map, q.x, q.in, q.M, q.K, box_cols, kTileRows);
  if (!tma) memset(&map, 0, sizeof(map));
  QuantFn fn = bf16 ? pick_dir<uint16_t>(row, col, q.four_over_six, q.block_2d, tma)
                    : pick_dir<float>(row, col, q.four_over_six, q.block_2d, tma);
  cudaError_t err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemBytes);
  if (err != cudaSuccess) return err;
  const int64_t grid = std::min<int64_t>(a.num_tiles, 2LL * dev.num_sms);
  fn<<<(unsigned)grid, kThreads, kSmemBytes, stream>>>(map, a);
  return cudaGetLastError();
}

}  // namespace nvfp4
