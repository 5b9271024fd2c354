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
// Structure (persistent: one CTA per SM walks 128 x 256 output tiles, tile c,
// c + gridDim.x, ..., groups of 32 M tiles side by side so their A tiles stay in L2):
//   warp 0    producer: TMA loads of the A and B code tiles (128 B of K per row,
//             128B swizzle) and 1D bulk copies of their scales, into a 3-stage
//             shared-memory ring (72 KB a stage) guarded by mbarriers, running on
//             across tile boundaries;
//   warp 1    allocates TMEM (512 columns) and, from one thread, copies each
//             stage's scales to TMEM (tcgen05.cp) and issues the MMAs (M = 128,
//             N = 256, K = 64, four per stage), releasing each stage with
//             tcgen05.commit and the finished accumulator with one more;
//   warps 2-9 epilogue, two per TMEM lane quarter (128 columns each): before the
//             accumulator is ready, load alpha_i and stage the 128 beta_j in shared
//             memory; then copy the accumulator to registers (tcgen05.ld), hand
//             TMEM back to the MMA warp at once (the next tile's MMAs overlap the
//             rest), apply alpha_i * beta_j, convert and store D in whole 32-byte
//             sectors.
// Scales reach the kernel in the layout their TMEM copies want (see SfLayout): a
// pre-pass (k_sf_layout) rewrites the compact [lines][k/16] scales of both operands
// into the caller's workspace.
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
constexpr int kBN = 256;                   // tile rows of B = output columns per tile = MMA N
// K bytes per stage and row: 256 E2M1 values.  (64 -- six stages of 36 KB with the
// 64B swizzle -- is correct too but measured 17 % slower.)
constexpr int kBKBytes = 128;
constexpr int kUmmaKBytes = 32;            // K = 64 values per MMA
constexpr int kKSteps = kBKBytes / kUmmaKBytes;  // MMAs per stage
constexpr int kTileScales = kBKBytes / 8;        // scales per line and K tile
// the operand tiles' shared-memory swizzle: one 8-row atom of kBKBytes-byte rows
constexpr int kSwizzleMode = kBKBytes == 128 ? 2 : 4;  // descriptor code: 128B / 64B
static_assert(kBKBytes == 128 || kBKBytes == 64, "K tile of 128 or 64 bytes per row");
constexpr int kABytes = kBM * kBKBytes;    // 16 KB
constexpr int kBBytes = kBN * kBKBytes;    // 32 KB
constexpr int kEpilogueWarps = 8;                    // two per TMEM lane quarter
constexpr int kEpiCols = kBN / 2;                     // accumulator columns per epilogue warp
constexpr int kThreads = 64 + 32 * kEpilogueWarps;    // producer, MMA, epilogue
constexpr uint32_t kTmemCols = 512;
constexpr int kSfCol0 = kBN;                          // scale columns follow the accumulator
constexpr int kMetaBytes = 1024;                      // barriers, TMEM address, error flag
constexpr int kSmemEnds = 512;                        // group ends staged in shared memory
constexpr int kBetaBytes = kEpilogueWarps * kEpiCols * 4;  // per-warp column factors

// Where the tensor core reads the scales of a block-scaled MMA with M = 128 and
// scale_vec::4X (one 32-bit TMEM word = the four scales of a line for the MMA's
// K = 64; base columns on multiples of 4): A's line l from its accumulator lane l
// at column base + l / 32; B's line n (N = 256) by each lane quarter q of the tensor
// core from its own lanes, lane 32q + n % 32, at column base + n / 32 -- B's scales
// must be present in all four quarters.  They get there by tcgen05.cp .128x256b
// (lane l <- a 32-byte row of shared memory, 8 columns): one copy holds two K steps
// of A (row l: the words of K steps 2c and 2c + 1 at bytes 4q and 16 + 4q, q = l /
// 32, zero elsewhere) or one K step of all 256 lines of B (row l: line 32c + l % 32
// at bytes 4c).  Per K tile of 256: 2 + 4 copies, 8 + 16 KB of shared memory, 16 +
// 32 TMEM columns (A's K step ks at base + 4ks, B's at base + 8ks).
struct SfLayout {
  static constexpr int kStages = kBKBytes == 128 ? 3 : 6;
  static constexpr int kSfaBytes = kKSteps / 2 * 4096;
  static constexpr int kSfbBytes = kKSteps * 4096;
  static constexpr int kSfaCols = 4 * kKSteps, kSfbCols = 8 * kKSteps;
};
template <class SF>
struct GemmGeom {
  static constexpr int kStageBytes = kABytes + kBBytes + SF::kSfaBytes + SF::kSfbBytes;
  static constexpr int kSfColsPerStage = SF::kSfaCols + SF::kSfbCols;
  static constexpr int kSmemBytes = SF::kStages * kStageBytes + kMetaBytes +
                                    kSmemEnds * 8 /* group ends */ + kBetaBytes +
                                    1024 /* alignment */;
  static_assert(kSfCol0 + SF::kStages * kSfColsPerStage <= (int)kTmemCols, "TMEM columns");
  static_assert(kStageBytes % 1024 == 0, "stages stay 1024-byte aligned for the 128B swizzle");
  static_assert(kSmemBytes <= 232448, "shared memory");
};


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
// 128 lanes x 256 bits from shared memory: lane l, column c <- row l, bytes 4c .. 4c+3.
__device__ __forceinline__ void tc_cp_128x256b(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.128x256b [%0], %1;" ::"r"(taddr), "l"(sdesc)
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

// Shared-memory matrix descriptor of a K-major operand tile with kBKBytes-byte rows
// in the matching swizzle: 8-row groups 8 * kBKBytes bytes apart (stride byte
// offset), the leading byte offset unused for this layout, bits 46-48 = 0b001.
__device__ __forceinline__ uint64_t desc_swz(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) |
         ((uint64_t)(8 * kBKBytes >> 4) << 32) | ((uint64_t)1 << 46) |
         ((uint64_t)kSwizzleMode << 61);
}
// Descriptor of a no-swizzle K-major scale matrix: 8-row x 16-byte core matrices
// `sbo` bytes apart along the lines and `lbo` bytes apart along the row.
__device__ __forceinline__ uint64_t desc_plain(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(lbo >> 4) << 16) |
         ((uint64_t)(sbo >> 4) << 32) | ((uint64_t)1 << 46);
}

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// ---------------------------------------------------------------- scale pre-pass

// Scale pre-pass.  Compact scales [rows][k16] -> [n_blk][k_tiles][copies][4096] for
// blocks of 128 * P lines (P = 1: A, two copies per K tile; P = 2: B, four).  In
// copy c, lane l owns a 32-byte row of eight 4-byte words (the four scales of one
// line and K step each, zero where unused):
//   A (P = 1): word 4u + q (q = l / 32) of row l = line blk * 128 + l, K step 2c + u;
//   B (P = 2): word cc of row l = line blk * 256 + 32 cc + l % 32, K step c.
// Stored as one tcgen05.cp .128x256b reads it: 16-byte half u at 2048 u, row l at
// 16 l.  One CTA per (block, K tile): it stages the block's 16 scales per line of
// that K tile in shared memory (16-byte loads where the rows allow), then writes
// the block's copies as coalesced 16-byte stores, one 16-byte row half per thread.
__global__ void __launch_bounds__(256) k_sf_layout(const uint8_t* __restrict__ sc, int64_t rows,
                                                  int64_t k16, int64_t k_tiles, int P,
                                                  uint8_t* __restrict__ out) {
  __shared__ uint32_t cw[256 * kKSteps];  // cw[kKSteps * line + ks]: the line's K step ks
  const int L = 128 * P;
  const int copies = P == 1 ? kKSteps / 2 : kKSteps;
  const int64_t kt = blockIdx.x % k_tiles, blk = blockIdx.x / k_tiles;
  const int64_t s0 = kt * kTileScales;
  const bool vec = k16 % kTileScales == 0 && (reinterpret_cast<uintptr_t>(sc) & 15) == 0;
  for (int i = threadIdx.x; i < L; i += blockDim.x) {
    const int64_t line = blk * L + i;
    uint32_t w[kKSteps];
#pragma unroll
    for (int j = 0; j < kKSteps; ++j) w[j] = 0;
    if (line < rows) {
      const uint8_t* p = sc + line * k16 + s0;
      if (vec) {
#pragma unroll
        for (int j = 0; j < kKSteps; ++j) w[j] = __ldg(reinterpret_cast<const uint32_t*>(p) + j);
      } else {
        for (int j = 0; j < kTileScales && s0 + j < k16; ++j)
          w[j >> 2] |= (uint32_t)p[j] << (8 * (j & 3));
      }
    }
#pragma unroll
    for (int j = 0; j < kKSteps; ++j) cw[kKSteps * i + j] = w[j];
  }
  __syncthreads();
  uint4* dst = reinterpret_cast<uint4*>(out + blockIdx.x * (int64_t)copies * 4096);
  for (int v = threadIdx.x; v < copies * 256; v += blockDim.x) {
    const int c = v >> 8, u = (v >> 7) & 1, l = v & 127;  // copy, half, row
    uint32_t w[4];
    if (P == 1) {  // line l, K step 2c + u, at word l / 32
#pragma unroll
      for (int j = 0; j < 4; ++j) w[j] = j == (l >> 5) ? cw[kKSteps * l + 2 * c + u] : 0u;
    } else {  // words 4u .. 4u + 3: lines 32 (4u + j) + l % 32, K step c
#pragma unroll
      for (int j = 0; j < 4; ++j) w[j] = cw[kKSteps * (32 * (4 * u + j) + (l & 31)) + c];
    }
    dst[u * 128 + l + c * 256] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// ---------------------------------------------------------------- the GEMM

struct GemmParams {
  const uint8_t* sfa;  // A's scales in the kernel's layout
  const uint8_t* sfb;
  const float* a_amax;
  const float* b_amax;
  int a_amax_stride;  // 1 (per line) or 0 (per tensor)
  int b_amax_stride;
  float a_finv, b_finv;  // fl(1 / (bound * 6)) of each operand
  int M, N;
  int k_tiles;  // ceil(K / 256)
  int tiles_m, tiles_n;
  void* d;
  bool d_bf16;
  uint32_t idesc;
  int* status;
  // grouped (per-expert) GEMM: rows of A in groups ending at group_ends (multiples of
  // 128), group g multiplying rows g * b_group_rows .. of B; NULL for one GEMM
  const int64_t* group_ends;
  int num_groups;
  int b_group_rows;         // N in the grouped GEMM, 0 otherwise
  int b_amax_group_stride;  // where group g's amax starts in b_amax (N, 1 or 0)
  // K-grouped (the per-expert wgrad GEMM): group_ends cut K (tokens, multiples of 256)
  // and group g writes its own [M][N] block of d, d + g * M * N
  bool k_grouped;
  int64_t group_total;      // what the last group end must equal (rows of A, or K)
  int a_amax_group_stride;  // where group g's amax starts in a_amax (K-grouped: M, 1)
};

// One output tile of this CTA's walk: its group, tile coordinates and K tiles.
struct TileJob {
  int g, tm, tn, kt0, kt1;
};

// The group of the A tile starting at row r: the first g with group_ends[g] > r
// (empty groups are skipped); 0 when the GEMM is not grouped by rows.
__device__ __forceinline__ int group_of_row(const GemmParams& p, const int64_t* ends, int64_t r) {
  if (p.group_ends == nullptr || p.k_grouped) return 0;
  int lo = 0, hi = p.num_groups - 1;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (ends[mid] > r) hi = mid;
    else lo = mid + 1;
  }
  return lo;
}

constexpr int kRasterGroup = 32;  // M tiles walked together so their A tiles stay in L2

__device__ __forceinline__ void tile_coords(int idx, int tiles_m, int tiles_n, int& tm, int& tn);
__device__ __forceinline__ int group_of_row(const GemmParams& p, const int64_t* ends, int64_t r);

// ends: the group ends (a shared-memory copy when they fit)
__device__ __forceinline__ TileJob tile_job(const GemmParams& p, const int64_t* ends, int tile) {
  TileJob j;
  j.g = 0;
  j.kt0 = 0;
  j.kt1 = p.k_tiles;
  if (p.k_grouped) {
    const int per = p.tiles_m * p.tiles_n;
    j.g = tile / per;
    tile_coords(tile - j.g * per, p.tiles_m, p.tiles_n, j.tm, j.tn);
    j.kt0 = (int)((j.g ? ends[j.g - 1] : 0) / (2 * kBKBytes));
    j.kt1 = (int)(ends[j.g] / (2 * kBKBytes));
  } else {
    tile_coords(tile, p.tiles_m, p.tiles_n, j.tm, j.tn);
    if (p.group_ends != nullptr) j.g = group_of_row(p, ends, (int64_t)j.tm * kBM);
  }
  return j;
}

__device__ __forceinline__ void tile_coords(int idx, int tiles_m, int tiles_n, int& tm, int& tn) {
  const int group = idx / (kRasterGroup * tiles_n);
  const int first_m = group * kRasterGroup;
  const int gm = min(tiles_m - first_m, kRasterGroup);
  const int rem = idx - group * kRasterGroup * tiles_n;
  tm = first_m + rem % gm;
  tn = rem / gm;
}

// Persistent: CTA c computes tiles c, c + gridDim.x, ...  The load ring runs on
// across tile boundaries; the epilogue copies the accumulator to registers,
// hands TMEM back (acc_empty) and stores while the MMAs of the next tile run.
template <class SF>
__global__ void __launch_bounds__(kThreads, 1)
    k_gemm_nvf4(const __grid_constant__ CUtensorMap map_a,
                const __grid_constant__ CUtensorMap map_b, const GemmParams p) {
  using G = GemmGeom<SF>;
  constexpr int S = SF::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * G::kStageBytes);
  uint64_t* empty = full + S;
  uint64_t* acc_full = empty + S;
  uint64_t* acc_empty = acc_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 1);
  int* err = reinterpret_cast<int*>(tmem_slot + 1);
  int64_t* s_ends = reinterpret_cast<int64_t*>(smem + S * G::kStageBytes + kMetaBytes);
  float* s_beta = reinterpret_cast<float*>(s_ends + kSmemEnds);
  // every tile looks its group up: from shared memory when the ends fit
  const int64_t* ends = p.num_groups <= kSmemEnds ? s_ends : p.group_ends;
  if (p.group_ends != nullptr && p.num_groups <= kSmemEnds)
    for (int g = threadIdx.x; g < p.num_groups; g += blockDim.x) s_ends[g] = p.group_ends[g];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int num_tiles = (p.k_grouped ? p.num_groups : 1) * p.tiles_m * p.tiles_n;

  if (p.group_ends != nullptr) {  // every thread takes part; nothing is written if invalid
    const bool ok = groups_valid(p.group_ends, p.num_groups, p.group_total) &&
                    ends_aligned(p.group_ends, p.num_groups, p.k_grouped ? 2 * kBKBytes : kBM);
    if (!ok) {
      if (threadIdx.x == 0) raise_status(p.status, kStatusBadGroups);
      return;
    }
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, kEpilogueWarps);
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
    uint32_t it = 0;  // K tiles issued, over all tiles of this CTA
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
      const TileJob job = tile_job(p, ends, tile);
      const int tm = job.tm, tn = job.tn;
      const int b_tile0 = job.g * (p.b_group_rows / kBN);  // the expert's rows of B
      for (int kt = job.kt0; kt < job.kt1; ++kt, ++it) {
        const uint32_t s = it % S;
        if (it >= (uint32_t)S && !mbar_wait_bounded(&empty[s], ((it / S) - 1) & 1)) {
          *err = 1;
          ok = false;
          break;
        }
        if (*(volatile int*)err) {
          ok = false;
          break;
        }
        uint8_t* st = smem + s * G::kStageBytes;
        uint8_t* st_sf = st + kABytes + kBBytes;
        mbar_expect_tx(&full[s], G::kStageBytes);
        const int bt = b_tile0 + tn;  // B's 256-row tile (of its group)
        tma_load_2d(st, &map_a, &full[s], kt * kBKBytes, tm * kBM, pol_a);
        tma_load_2d(st + kABytes, &map_b, &full[s], kt * kBKBytes, bt * kBN, pol_b);
        bulk_load(st_sf, p.sfa + ((int64_t)tm * p.k_tiles + kt) * SF::kSfaBytes, SF::kSfaBytes,
                  &full[s], pol_a);
        bulk_load(st_sf + SF::kSfaBytes, p.sfb + ((int64_t)bt * p.k_tiles + kt) * SF::kSfbBytes,
                  SF::kSfbBytes, &full[s], pol_b);
      }
    }
    // drain: every copy issued must have landed before the CTA may exit
    for (uint32_t j = it > (uint32_t)S ? it - S : 0; j < it; ++j)
      if (!mbar_wait_bounded(&full[j % S], (j / S) & 1)) *err = 1;
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer: per K tile, the stage's scales to TMEM, then
    // the four MMAs (K = 64 each) that read them
    auto copy_scales = [&](uint32_t j) {
      const uint32_t s = j % S;
      const uint32_t st_sfa = smem_addr(smem + s * G::kStageBytes) + kABytes + kBBytes;
      const uint32_t st_sfb = st_sfa + SF::kSfaBytes;
      const uint32_t sfa_col = tmem + kSfCol0 + s * G::kSfColsPerStage;
      const uint32_t sfb_col = sfa_col + SF::kSfaCols;
      // 128 rows x 32 bytes per copy: 16-byte halves 2048 bytes apart, rows 16 apart
#pragma unroll
      for (int c = 0; c < kKSteps / 2; ++c)
        tc_cp_128x256b(sfa_col + 8 * c, desc_plain(st_sfa + c * 4096, 2048, 128));
#pragma unroll
      for (int ks = 0; ks < kKSteps; ++ks)
        tc_cp_128x256b(sfb_col + 8 * ks, desc_plain(st_sfb + ks * 4096, 2048, 128));
    };
    uint32_t it = 0, t = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x, ++t) {
      // the epilogue of the previous tile has copied the accumulator out
      if (t > 0 && !mbar_wait_bounded(acc_empty, (t - 1) & 1)) {
        *err = 1;
        break;
      }
      tc_fence_after();
      const TileJob job = tile_job(p, ends, tile);
      for (int kt = job.kt0; kt < job.kt1; ++kt, ++it) {
        const uint32_t s = it % S;
        if (!mbar_wait_bounded(&full[s], (it / S) & 1)) {
          *err = 1;
          ok = false;
          break;
        }
        if (*(volatile int*)err) {
          ok = false;
          break;
        }
        tc_fence_after();
        copy_scales(it);
        const uint32_t st = smem_addr(smem + s * G::kStageBytes);
        const uint32_t sfa_col = tmem + kSfCol0 + s * G::kSfColsPerStage;
        const uint32_t sfb_col = sfa_col + SF::kSfaCols;
#pragma unroll
        for (int ks = 0; ks < kKSteps; ++ks)
          tc_mma_nvf4(tmem, desc_swz(st + ks * kUmmaKBytes),
                      desc_swz(st + kABytes + ks * kUmmaKBytes), p.idesc, sfa_col + 4 * ks,
                      sfb_col + 8 * ks, (kt != job.kt0) || ks != 0);
        tc_commit(&empty[s]);
      }
      // the accumulator of this tile is complete (or abandoned) once all issued MMAs are
      tc_commit(acc_full);
    }
    // everything issued must be done before TMEM is freed
    if (t > 0 && !mbar_wait_bounded(acc_full, (t - 1) & 1)) *err = 1;
  } else if (warp >= 2) {
    // ---------------- epilogue: lane quarter q (rows 32q ..), column half `half`
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    const bool b_lines = p.b_amax_stride != 0;  // one amax per line of B
    uint32_t t = 0;
    float* beta = s_beta + (warp - 2) * kEpiCols;  // this warp's column factors
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++t) {
      const TileJob job = tile_job(p, ends, tile);
      const int tm = job.tm, tn = job.tn;
      const int row = tm * kBM + q * 32 + lane;
      const int col_base = tn * kBN + half * kEpiCols;
      const bool live = row < p.M && col_base < p.N;
      // Before the accumulator is ready: alpha = fl(amax_a[row] * fl(1/F_a)) and this
      // warp's 128 column factors beta = fl(amax_b[col] * fl(1/F_b)), lane l computing
      // columns 4l .. 4l+3 into shared memory, so that no global load waits behind
      // the accumulator.
      const float alpha =
          live ? __fmul_rn(p.a_amax[(int64_t)job.g * p.a_amax_group_stride +
                                    (int64_t)row * p.a_amax_stride],
                           p.a_finv)
               : 0.f;
      {
        const float* b_amax = p.b_amax + (int64_t)job.g * p.b_amax_group_stride;
        const int c4 = col_base + 4 * lane;
        float b4[4];
        // 16-byte loads only where this group's amax row is 16-byte aligned
        if (b_lines && (reinterpret_cast<uintptr_t>(b_amax) & 15) == 0 && c4 + 4 <= p.N) {
          const float4 t4 = __ldg(reinterpret_cast<const float4*>(b_amax + c4));
          b4[0] = t4.x, b4[1] = t4.y, b4[2] = t4.z, b4[3] = t4.w;
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            b4[j] = __ldg(b_amax + (int64_t)max(0, min(c4 + j, p.N - 1)) * p.b_amax_stride);
        }
        __syncwarp();  // every lane has read the previous tile's factors
        sts_v4(beta + 4 * lane, __float_as_uint(__fmul_rn(b4[0], p.b_finv)),
               __float_as_uint(__fmul_rn(b4[1], p.b_finv)),
               __float_as_uint(__fmul_rn(b4[2], p.b_finv)),
               __float_as_uint(__fmul_rn(b4[3], p.b_finv)));
        __syncwarp();
      }
      const bool ready = mbar_wait_bounded(acc_full, t & 1);
      if (!ready) *err = 1;
      tc_fence_after();
      uint32_t v[kEpiCols];
#pragma unroll
      for (int c = 0; c < kEpiCols / 32; ++c)
        tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + half * kEpiCols + c * 32, v + c * 32);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty);  // TMEM may take the next tile's MMAs
      if (!ready || *(volatile int*)err) break;
      if (job.kt1 == job.kt0) {  // an empty K range (an empty group): the sum is 0
#pragma unroll
        for (int i = 0; i < kEpiCols; ++i) v[i] = 0u;
      }
      if (!live) continue;
      const int nvalid = min(kEpiCols, p.N - col_base);
      const int64_t off = (p.k_grouped ? (int64_t)job.g * p.M * p.N : 0) +
                          (int64_t)row * p.N + col_base;
      // whole 32-byte sectors per store where the row's run is 32-byte aligned,
      // else 16-byte stores, else (ragged N or odd alignment) element stores
      const uintptr_t d_addr = reinterpret_cast<uintptr_t>(p.d) + off * (p.d_bf16 ? 2 : 4);
      const bool vec = nvalid == kEpiCols && (d_addr & 15) == 0;
      const bool vec32 = vec && (d_addr & 31) == 0;
#pragma unroll
      for (int c = 0; c < kEpiCols / 32; ++c) {
        uint32_t* vc = v + c * 32;
        // d = fl(fl(acc * alpha) * beta)
#pragma unroll
        for (int j4 = 0; j4 < 8; ++j4) {
          const float4 b4 = *reinterpret_cast<const float4*>(beta + c * 32 + 4 * j4);
          const float bj[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
          for (int j = 0; j < 4; ++j)
            vc[4 * j4 + j] =
                __float_as_uint(__fmul_rn(__fmul_rn(__uint_as_float(vc[4 * j4 + j]), alpha), bj[j]));
        }
        if (p.d_bf16) {
          uint16_t* dst = static_cast<uint16_t*>(p.d) + off + c * 32;
          uint32_t w[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(vc[2 * j]),
                                                      __uint_as_float(vc[2 * j + 1]));
            w[j] = *reinterpret_cast<uint32_t*>(&h2);
          }
          if (vec32) {
            stg_v8(dst, w);
            stg_v8(dst + 16, w + 8);
          } else if (vec) {
#pragma unroll
            for (int g = 0; g < 4; ++g)
              *reinterpret_cast<uint4*>(dst + 8 * g) =
                  make_uint4(w[4 * g], w[4 * g + 1], w[4 * g + 2], w[4 * g + 3]);
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (c * 32 + j < nvalid) dst[j] = (uint16_t)(w[j >> 1] >> (16 * (j & 1)));
          }
        } else {
          uint32_t* dst = static_cast<uint32_t*>(p.d) + off + c * 32;
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            if (vec32) {
              if ((g & 1) == 0) stg_v8(dst + 4 * g, vc + 4 * g);
            } else if (vec) {
              *reinterpret_cast<uint4*>(dst + 4 * g) =
                  make_uint4(vc[4 * g], vc[4 * g + 1], vc[4 * g + 2], vc[4 * g + 3]);
            } else {
#pragma unroll
              for (int j = 0; j < 4; ++j)
                if (c * 32 + 4 * g + j < nvalid) dst[4 * g + j] = vc[4 * g + j];
            }
          }
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

GemmLayout gemm_layout(int64_t M, int64_t N, int64_t K, int64_t b_lines) {
  GemmLayout L;
  L.k_tiles = ceil_div(K, 2 * kBKBytes);
  L.tiles_m = ceil_div(M, kBM);
  L.tiles_n = ceil_div(N, kBN);
  L.sfa_bytes = L.tiles_m * L.k_tiles * SfLayout::kSfaBytes;
  L.sfb_bytes = ceil_div(b_lines, kBN) * L.k_tiles * SfLayout::kSfbBytes;
  L.sfb_offset = (L.sfa_bytes + 255) / 256 * 256;
  L.workspace_bytes = L.sfb_offset + L.sfb_bytes;
  return L;
}

template <class SF>
static cudaError_t launch_gemm_t(const GemmArgs& a, const GemmLayout& L, const DeviceInfo& dev,
                                 cudaStream_t stream) {
  using G = GemmGeom<SF>;
  uint8_t* sfa = a.workspace;
  uint8_t* sfb = a.workspace + L.sfb_offset;
  k_sf_layout<<<(unsigned)(L.tiles_m * L.k_tiles), 256, 0, stream>>>(a.a_scales, a.M, a.K / 16,
                                                                     L.k_tiles, 1, sfa);
  const int64_t b_lines = a.group_ends && !a.k_grouped ? (int64_t)a.num_groups * a.N : a.N;
  k_sf_layout<<<(unsigned)(ceil_div(b_lines, kBN) * L.k_tiles), 256, 0, stream>>>(
      a.b_scales, b_lines, a.K / 16, L.k_tiles, 2, sfb);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  CUtensorMap map_a, map_b;
  if (!make_operand_map(&map_a, a.a_codes, a.M, a.K / 2, kBKBytes, kBM) ||
      !make_operand_map(&map_b, a.b_codes, b_lines, a.K / 2, kBKBytes, kBN))
    return cudaErrorInvalidValue;

  static bool attr_set[64] = {};
  if (dev.device < 64 && !attr_set[dev.device]) {
    e = cudaFuncSetAttribute(k_gemm_nvf4<SF>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             G::kSmemBytes);
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
  p.tiles_m = (int)L.tiles_m;
  p.tiles_n = (int)L.tiles_n;
  p.d = a.d;
  p.d_bf16 = a.d_bf16;
  p.idesc = make_idesc_nvf4(kBM, kBN);
  p.status = dev.status;
  p.group_ends = a.group_ends;
  p.num_groups = a.group_ends ? a.num_groups : 0;
  p.k_grouped = a.group_ends != nullptr && a.k_grouped;
  p.b_group_rows = a.group_ends && !a.k_grouped ? (int)a.N : 0;
  p.b_amax_group_stride = a.group_ends ? (a.b_row_scaled ? (int)a.N : 1) : 0;
  p.a_amax_group_stride = p.k_grouped ? (a.a_row_scaled ? (int)a.M : 1) : 0;
  p.group_total = p.k_grouped ? a.K : a.M;
  const int64_t tiles = (a.group_ends && a.k_grouped ? a.num_groups : 1) * L.tiles_m * L.tiles_n;
  const int grid = (int)std::min<int64_t>(tiles, dev.num_sms);
  k_gemm_nvf4<SF><<<grid, kThreads, G::kSmemBytes, stream>>>(map_a, map_b, p);
  return cudaGetLastError();
}

cudaError_t launch_gemm(const GemmArgs& a, const DeviceInfo& dev, cudaStream_t stream) {
  const GemmLayout L = gemm_layout(
      a.M, a.N, a.K, a.group_ends && !a.k_grouped ? (int64_t)a.num_groups * a.N : a.N);
  return launch_gemm_t<SfLayout>(a, L, dev, stream);
}

}  // namespace nvfp4
