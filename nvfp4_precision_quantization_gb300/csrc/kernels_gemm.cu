// kernels_gemm.cu -- the GEMM that consumes two NVFP4 operands, on the
// fifth-generation tensor cores (tcgen05, sm_103a).
//
// What it computes ("NVFP4: enable row-scaled transpose quantization for
// backward", TransformerEngine PR #3206, sequence diagram): the fprop GEMM scales
// its output by the activation's per-row amax and the weight's amax, the wgrad
// GEMM by the outer product of both operands' per-line amax.  As a definition:
//   D[i][j] = sum_k value_A(i,k) * value_B(j,k),
//   value = code * decode(scale) * amax / (bound * 6)
// with both operands K-major (a rowwise output, or a columnwise output when the
// operand is the transpose).  The block part code * decode(scale) is exact in the
// tensor core's block-scaled MMA (kind::mxf4nvf4, one E4M3 scale per 16 values),
// which accumulates in FP32 in TMEM; the per-line factors alpha_i = amax_A[i] *
// fl(1/F_A) and beta_j = amax_B[j] * fl(1/F_B) are applied in the epilogue as
// D = fl(fl(acc * alpha_i) * beta_j) -- the bilateral post-scale, fused, so the
// accumulator never goes to HBM.
//
// Structure (one CTA per 128 x 256 output tile, 1 CTA per SM):
//   warp 0   producer: TMA loads of the A and B code tiles (128 B of K per row,
//            128B swizzle) and 1D bulk copies of their scale chunks, into a
//            4-stage shared-memory ring guarded by mbarriers;
//   warp 1   allocates TMEM (512 columns) and, from one thread, copies each
//            stage's scales to TMEM (tcgen05.cp) and issues the MMAs (M = 128,
//            N = 128, K = 64; two per K step for the 256 columns), releasing each
//            stage with tcgen05.commit;
//   warps 2-5 epilogue: read the accumulator (tcgen05.ld, one lane quarter per
//            warp), apply alpha_i * beta_j, convert and store D.
// Scales reach the kernel in the tensor core's chunk layout: a pre-pass
// (k_sf_block) rewrites the compact [lines][k/16] scales into 512-byte chunks of
// 128 lines x 4 scales, byte (l % 32) * 16 + (l / 32) * 4 + s, which one
// tcgen05.cp .32x128b.warpx4 moves into four TMEM columns.
//
// Every wait is bounded (about 2 s): on a timeout the kernel records
// NVFP4_DEVICE_TIMEOUT, stops issuing work, waits (bounded) for what it already
// issued, writes no output, frees its TMEM and returns.
#include <cuda_bf16.h>

#include <algorithm>

#include "device_common.cuh"
#include "internal.h"

namespace nvfp4 {
namespace {

constexpr int kBM = 128;                   // tile rows of A = MMA M
constexpr int kBN = 256;                   // tile rows of B = output columns per tile
constexpr int kUmmaN = 128;                // N of one MMA instruction
constexpr int kHalves = kBN / kUmmaN;      // MMAs per K step
constexpr int kBKBytes = 128;              // K bytes per stage and row: 256 E2M1 values
constexpr int kUmmaKBytes = 32;            // K = 64 values per MMA
constexpr int kKSteps = kBKBytes / kUmmaKBytes;  // 4
constexpr int kStages = 4;
constexpr int kABytes = kBM * kBKBytes;    // 16 KB
constexpr int kBBytes = kBN * kBKBytes;    // 32 KB
constexpr int kSfChunk = 512;              // 128 lines x 4 scales
constexpr int kSfaBytes = kKSteps * kSfChunk;            // 2 KB
constexpr int kSfbBytes = kHalves * kKSteps * kSfChunk;  // 4 KB
constexpr int kStageBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes;
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr int kSfCol0 = kBN;                            // scale columns follow the accumulator
constexpr int kSfColsPerStage = kKSteps * 4 * (1 + kHalves);
constexpr int kMetaBytes = 2048;  // barriers, TMEM address, error flag, beta of the tile
constexpr int kSmemBytes = kStages * kStageBytes + kMetaBytes + 1024 /* alignment */;
static_assert(kSfCol0 + kStages * kSfColsPerStage <= (int)kTmemCols, "TMEM columns");
static_assert(kStageBytes % 1024 == 0, "stages stay 1024-byte aligned for the 128B swizzle");

// ---------------------------------------------------------------- tcgen05 wrappers

__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Arrive on `bar` once every tcgen05 operation this thread issued so far is done.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_addr(bar))
               : "memory");
}
// 32 lanes x 128 bits from shared memory, replicated into all four lane quarters.
__device__ __forceinline__ void tc_cp_sf(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}
// D (+)= (A x scaleA) * (B x scaleB)^T, E2M1 operands with one E4M3 scale per 16 values.
__device__ __forceinline__ void tc_mma_nvf4(uint32_t d_taddr, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t sfa_taddr,
                                            uint32_t sfb_taddr, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X"
      " [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d_taddr),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_taddr), "r"(sfb_taddr)
      : "memory");
}
// This warp's lane quarter, 32 consecutive FP32 columns: v[j] = column col + j of
// lane (quarter base + lane id).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* v) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32"
      " {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15,"
      " %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31},"
      " [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
        "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
        "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major operand tile with 128-byte rows in
// the 128B swizzle: 8-row groups 1024 bytes apart (stride byte offset), the
// leading byte offset unused for this layout, bits 46-48 = 0b001, swizzle mode 2.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) |
         ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Descriptor of one 512-byte scale chunk read as 32 rows of 16 bytes, no swizzle:
// 8-row core matrices 128 bytes apart, one core matrix along the 16-byte width.
__device__ __forceinline__ uint64_t desc_sf_chunk(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(128 >> 4) << 32) |
         ((uint64_t)1 << 46);
}

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// ---------------------------------------------------------------- scale pre-pass

// Compact scales [rows][k16] -> chunks [n_rb][n_kc][512 bytes]: chunk (rb, kc)
// holds lines rb*128 .. +127 and scales kc*4 .. +3, line l at byte
// (l % 32) * 16 + (l / 32) * 4, scale s at + s.  Lines and scales past the
// operand are zero (a zero scale times the zero-filled codes there adds 0).
__global__ void __launch_bounds__(256) k_sf_block(const uint8_t* __restrict__ sc, int64_t rows,
                                                  int64_t k16, int64_t n_kc, int64_t n_words,
                                                  uint32_t* __restrict__ out) {
  for (int64_t w = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; w < n_words;
       w += (int64_t)gridDim.x * blockDim.x) {
    const int64_t chunk = w >> 7;
    const int inner = (int)(w & 127);
    const int64_t rb = chunk / n_kc, kc = chunk - rb * n_kc;
    const int64_t line = rb * 128 + (inner & 3) * 32 + (inner >> 2);
    uint32_t word = 0;
    if (line < rows) {
      const uint8_t* p = sc + line * k16;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int64_t s = kc * 4 + b;
        if (s < k16) word |= (uint32_t)p[s] << (8 * b);
      }
    }
    out[w] = word;
  }
}

// ---------------------------------------------------------------- the GEMM

struct GemmParams {
  const uint8_t* sfa;  // chunked scales of A, n_kc chunks per 128-line block
  const uint8_t* sfb;
  const float* a_amax;
  const float* b_amax;
  int a_amax_stride;  // 1 (per line) or 0 (per tensor)
  int b_amax_stride;
  float a_finv, b_finv;  // fl(1 / (bound * 6)) of each operand
  int M, N;
  int k_tiles;  // ceil(K / 256)
  int n_kc;     // 4 * k_tiles
  int tiles_m, tiles_n;
  void* d;
  bool d_bf16;
  uint32_t idesc;
  int* status;
};

constexpr int kRasterGroup = 16;  // M tiles walked together so their A tiles stay in L2

__global__ void __launch_bounds__(kThreads, 1)
    k_gemm_nvf4(const __grid_constant__ CUtensorMap map_a,
                const __grid_constant__ CUtensorMap map_b, const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  uint64_t* empty = full + kStages;
  uint64_t* acc_full = empty + kStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);
  int* err = reinterpret_cast<int*>(tmem_slot + 1);
  float* s_beta = reinterpret_cast<float*>(smem + kStages * kStageBytes + 1024);  // [kBN]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // tile of this CTA: groups of kRasterGroup M tiles, M fastest inside a group
  const int idx = blockIdx.x;
  const int group = idx / (kRasterGroup * p.tiles_n);
  const int first_m = group * kRasterGroup;
  const int gm = min(p.tiles_m - first_m, kRasterGroup);
  const int rem = idx - group * kRasterGroup * p.tiles_n;
  const int tm = first_m + rem % gm, tn = rem / gm;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    *err = 0;
    fence_mbar_init();
    prefetch_tmap(&map_a);
    prefetch_tmap(&map_b);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ---------------- producer
    const uint64_t pol_a = policy_evict_last();
    const uint64_t pol_b = policy_evict_normal();
    int issued = 0;
    for (int kt = 0; kt < p.k_tiles; ++kt) {
      const int s = kt % kStages;
      if (kt >= kStages && !mbar_wait_bounded(&empty[s], ((kt / kStages) - 1) & 1)) {
        *err = 1;
        break;
      }
      if (*(volatile int*)err) break;
      uint8_t* st = smem + s * kStageBytes;
      mbar_expect_tx(&full[s], kStageBytes);
      tma_load_2d(st, &map_a, &full[s], kt * kBKBytes, tm * kBM, pol_a);
      tma_load_2d(st + kABytes, &map_b, &full[s], kt * kBKBytes, tn * kBN, pol_b);
      const uint8_t* sa = p.sfa + ((int64_t)tm * p.n_kc + kt * kKSteps) * kSfChunk;
      bulk_load(st + kABytes + kBBytes, sa, kSfaBytes, &full[s], pol_a);
      for (int h = 0; h < kHalves; ++h) {
        const uint8_t* sb =
            p.sfb + ((int64_t)(tn * kHalves + h) * p.n_kc + kt * kKSteps) * kSfChunk;
        bulk_load(st + kABytes + kBBytes + kSfaBytes + h * kKSteps * kSfChunk, sb,
                  kKSteps * kSfChunk, &full[s], pol_b);
      }
      issued = kt + 1;
    }
    // drain: every copy issued must have landed before the CTA may exit
    for (int kt = max(0, issued - kStages); kt < issued; ++kt)
      if (!mbar_wait_bounded(&full[kt % kStages], (kt / kStages) & 1)) *err = 1;
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer
    int issued = 0;
    for (int kt = 0; kt < p.k_tiles; ++kt) {
      const int s = kt % kStages;
      if (!mbar_wait_bounded(&full[s], (kt / kStages) & 1)) {
        *err = 1;
        break;
      }
      if (*(volatile int*)err) break;
      tc_fence_after();
      const uint32_t st = smem_addr(smem + s * kStageBytes);
      const uint32_t st_sfa = st + kABytes + kBBytes;
      const uint32_t st_sfb = st_sfa + kSfaBytes;
      const uint32_t sf_col = tmem + kSfCol0 + s * kSfColsPerStage;
#pragma unroll
      for (int ks = 0; ks < kKSteps; ++ks) {
        tc_cp_sf(sf_col + ks * 4, desc_sf_chunk(st_sfa + ks * kSfChunk));
#pragma unroll
        for (int h = 0; h < kHalves; ++h)
          tc_cp_sf(sf_col + kKSteps * 4 + (ks * kHalves + h) * 4,
                   desc_sf_chunk(st_sfb + (h * kKSteps + ks) * kSfChunk));
      }
#pragma unroll
      for (int ks = 0; ks < kKSteps; ++ks) {
        const uint64_t adesc = desc_sw128(st + ks * kUmmaKBytes);
#pragma unroll
        for (int h = 0; h < kHalves; ++h) {
          const uint64_t bdesc = desc_sw128(st + kABytes + h * kUmmaN * kBKBytes + ks * kUmmaKBytes);
          tc_mma_nvf4(tmem + h * kUmmaN, adesc, bdesc, p.idesc, sf_col + ks * 4,
                      sf_col + kKSteps * 4 + (ks * kHalves + h) * 4, (kt | ks) != 0);
        }
      }
      tc_commit(&empty[s]);
      issued = kt + 1;
    }
    // the accumulator is complete (or abandoned) once everything issued is done
    if (issued > 0) tc_commit(acc_full);
    else asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(acc_full)) : "memory");
    if (!mbar_wait_bounded(acc_full, 0)) *err = 1;
  } else if (warp >= 2) {
    // ---------------- epilogue: lane quarter q = rows 32q .. 32q+31 of the tile
    const int q = warp & 3;
    for (int t = threadIdx.x - 64; t < kBN; t += 128) {
      const int col = tn * kBN + t;
      s_beta[t] = col < p.N ? __fmul_rn(p.b_amax[(int64_t)col * p.b_amax_stride], p.b_finv) : 0.0f;
    }
    asm volatile("bar.sync 1, 128;" ::: "memory");  // the four epilogue warps
    const bool ready = mbar_wait_bounded(acc_full, 0);
    tc_fence_after();
    const int row = tm * kBM + q * 32 + lane;
    const bool row_ok = row < p.M;
    const float alpha =
        row_ok ? __fmul_rn(p.a_amax[(int64_t)row * p.a_amax_stride], p.a_finv) : 0.0f;
    const bool write = ready && *(volatile int*)err == 0;
    if (!ready) *err = 1;
#pragma unroll 1
    for (int c = 0; c < kBN / 32; ++c) {
      uint32_t v[32];
      tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + c * 32, v);
      tmem_ld_wait();
      const int col0 = tn * kBN + c * 32;
      if (!write || !row_ok || col0 >= p.N) continue;
      float o[32];
#pragma unroll
      for (int j = 0; j < 32; ++j)
        o[j] = __fmul_rn(__fmul_rn(__uint_as_float(v[j]), alpha), s_beta[c * 32 + j]);
      const int64_t off = (int64_t)row * p.N + col0;
      const int nvalid = min(32, p.N - col0);
      if (p.d_bf16) {
        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.d) + off;
        if (nvalid == 32 && (reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
          uint32_t w[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            __nv_bfloat162 h2 = __floats2bfloat162_rn(o[2 * j], o[2 * j + 1]);
            w[j] = *reinterpret_cast<uint32_t*>(&h2);
          }
#pragma unroll
          for (int j = 0; j < 4; ++j)
            *reinterpret_cast<uint4*>(dst + 8 * j) =
                make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j < nvalid) dst[j] = __float2bfloat16_rn(o[j]);
        }
      } else {
        float* dst = static_cast<float*>(p.d) + off;
        if (nvalid == 32 && (reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
#pragma unroll
          for (int j = 0; j < 8; ++j)
            *reinterpret_cast<float4*>(dst + 4 * j) =
                make_float4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j < nvalid) dst[j] = o[j];
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && *(volatile int*)err) raise_status(p.status, kStatusTimeout);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Instruction descriptor of kind::mxf4nvf4 (dense, K = 64): A and B E2M1 (format
// 1) and K-major, UE4M3 scales (bit 23 clear), scale-factor ids 0, N >> 3 at bit
// 17, M >> 4 at bit 24.
constexpr uint32_t make_idesc_nvf4(int m, int n) {
  return (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

GemmLayout gemm_layout(int64_t M, int64_t N, int64_t K) {
  GemmLayout L;
  L.k_tiles = ceil_div(K, 2 * kBKBytes);
  L.n_kc = L.k_tiles * kKSteps;
  L.tiles_m = ceil_div(M, kBM);
  L.tiles_n = ceil_div(N, kBN);
  L.sfa_bytes = L.tiles_m * L.n_kc * kSfChunk;
  L.sfb_bytes = L.tiles_n * kHalves * L.n_kc * kSfChunk;
  L.sfb_offset = (L.sfa_bytes + 255) / 256 * 256;
  L.workspace_bytes = L.sfb_offset + L.sfb_bytes;
  return L;
}

cudaError_t launch_gemm(const GemmArgs& a, const DeviceInfo& dev, cudaStream_t stream) {
  const GemmLayout L = gemm_layout(a.M, a.N, a.K);
  uint8_t* sfa = a.workspace;
  uint8_t* sfb = a.workspace + L.sfb_offset;
  const int64_t words_a = L.sfa_bytes / 4, words_b = L.sfb_bytes / 4;
  const int pre_grid = (int)std::min<int64_t>(ceil_div(words_a + words_b, 256), 8 * dev.num_sms);
  k_sf_block<<<pre_grid, 256, 0, stream>>>(a.a_scales, a.M, a.K / 16, L.n_kc, words_a,
                                           reinterpret_cast<uint32_t*>(sfa));
  k_sf_block<<<pre_grid, 256, 0, stream>>>(a.b_scales, a.N, a.K / 16, L.n_kc, words_b,
                                           reinterpret_cast<uint32_t*>(sfb));
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  CUtensorMap map_a, map_b;
  if (!make_operand_map(&map_a, a.a_codes, a.M, a.K / 2, kBKBytes, kBM) ||
      !make_operand_map(&map_b, a.b_codes, a.N, a.K / 2, kBKBytes, kBN))
    return cudaErrorInvalidValue;

  static bool attr_set[64] = {};
  if (dev.device < 64 && !attr_set[dev.device]) {
    e = cudaFuncSetAttribute(k_gemm_nvf4, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set[dev.device] = true;
  }
  GemmParams p;
  p.sfa = sfa;
  p.sfb = sfb;
  p.a_amax = a.a_amax;
  p.b_amax = a.b_amax;
  p.a_amax_stride = a.a_row_scaled ? 1 : 0;
  p.b_amax_stride = a.b_row_scaled ? 1 : 0;
  p.a_finv = 1.0f / (a.a_bound * 6.0f);
  p.b_finv = 1.0f / (a.b_bound * 6.0f);
  p.M = (int)a.M;
  p.N = (int)a.N;
  p.k_tiles = (int)L.k_tiles;
  p.n_kc = (int)L.n_kc;
  p.tiles_m = (int)L.tiles_m;
  p.tiles_n = (int)L.tiles_n;
  p.d = a.d;
  p.d_bf16 = a.d_bf16;
  p.idesc = make_idesc_nvf4(kBM, kUmmaN);
  p.status = dev.status;
  const int64_t tiles = L.tiles_m * L.tiles_n;
  k_gemm_nvf4<<<(unsigned)tiles, kThreads, kSmemBytes, stream>>>(map_a, map_b, p);
  return cudaGetLastError();
}

}  // namespace nvfp4
