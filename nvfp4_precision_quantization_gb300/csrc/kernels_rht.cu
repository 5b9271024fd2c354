// kernels_rht.cu -- random Hadamard transform (RHT) of the columnwise operand.
//
// "NVFP4: enable row-scaled transpose quantization for backward" (TransformerEngine
// PR #3206, description) names an RHT of the transposed path, among what that PR
// leaves out, without defining it.  The reading implemented here: per column and per
// block of 16 consecutive rows (one columnwise 1x16 block), y = (1/4) H16 diag(s) x,
// with H16 the Sylvester Hadamard matrix (entry (i, j) = (-1)^popcount(i & j)) and
// s_j = -1 where bit j of the caller's sign mask is set.  FP32 steps, in this
// order: the signs (exact), the four butterfly stages of the natural-order fast
// Walsh-Hadamard transform (h = 1, 2, 4, 8: rows i and i + h with i & h == 0 become
// u + v and u - v), then the product with 0.25.
//
// Two kernels, both HBM-bound, with 64 FP32 operations per 16 elements:
//   k_rht16       writes the transform to an FP32 buffer: 2 (BF16) or 4 (FP32) bytes
//                 in and 4 bytes out per element.  It serves nvfp4_rht16 and the
//                 16x16-block path of the transformed quantize.
//   k_rht16_amax  reads x once and writes only the exact amax of the transform, per
//                 column or per tensor.  It is the amax pass of the fused transformed
//                 quantize, whose encode pass transforms its blocks in registers
//                 (kernels_quantize.cu).
// A thread works on V adjacent columns: V = 2 where the row pitch and the base
// addresses allow 4- or 8-byte accesses, else 1.  So each of its row loads and
// stores is part of a warp-wide run of 32 V contiguous elements.  Items (row block or
// run of row blocks, column group) are walked with a grid-stride loop, adjacent
// threads on adjacent column groups.  Both kernels return at once when the noop flag
// is set.
#include <algorithm>

#include "device_common.cuh"
#include "internal.h"

namespace nvfp4 {

namespace {

constexpr int kRhtThreads = 256;

struct RhtKernelArgs {
  const void* x;
  float* y;
  int64_t cols;
  int64_t groups;  // column groups per row block
  int64_t items;   // row blocks x column groups
  uint32_t mask;
  const float* noop;
};

template <bool BF16, int V>
__global__ void __launch_bounds__(kRhtThreads) k_rht16(RhtKernelArgs a) {
  if (a.noop != nullptr && *a.noop == 1.0f) return;
  const int64_t stride = (int64_t)gridDim.x * kRhtThreads;
  for (int64_t it = (int64_t)blockIdx.x * kRhtThreads + threadIdx.x; it < a.items;
       it += stride) {
    const int64_t rb = it / a.groups;
    const int64_t c0 = (it - rb * a.groups) * V;
    const int64_t base = rb * 16 * a.cols + c0;  // element (16 rb, c0)
    float v[V][16];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      const int64_t e = base + r * a.cols;
      if constexpr (BF16) {
        const uint16_t* xb = static_cast<const uint16_t*>(a.x);
        if constexpr (V == 2) {
          const uint32_t w = __ldg(reinterpret_cast<const unsigned int*>(xb + e));
          v[0][r] = __uint_as_float(w << 16);
          v[1][r] = __uint_as_float(w & 0xffff0000u);
        } else {
          v[0][r] = __uint_as_float((uint32_t)__ldg(xb + e) << 16);
        }
      } else {
        const float* xf = static_cast<const float*>(a.x);
        if constexpr (V == 2) {
          const float2 t = __ldg(reinterpret_cast<const float2*>(xf + e));
          v[0][r] = t.x;
          v[1][r] = t.y;
        } else {
          v[0][r] = __ldg(xf + e);
        }
      }
    }
#pragma unroll
    if constexpr (V == 2) rht16_block2(v[0], v[1], a.mask);
    else rht16_block(v[0], a.mask);
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      float* yp = a.y + base + r * a.cols;
      if constexpr (V == 2) {
        *reinterpret_cast<float2*>(yp) = make_float2(v[0][r], v[1][r]);
      } else {
        *yp = v[0][r];
      }
    }
  }
}

// Exact amax of the transformed operand without writing it: per column (col_amax,
// [cols]) or over the tensor (tensor_amax, [1]), into buffers the prep step zeroed.
// A thread walks kAmaxBlocks consecutive 16-row blocks of its V columns, keeps the
// running max |y| of each, and ends with one atomic max per column (per-tensor: a
// warp maximum, one atomic per warp).  Non-negative floats order like their bit
// patterns, so the atomic works on the bits; the result is the exact max whatever
// the order.
constexpr int kAmaxBlocks = 16;
constexpr int kMaxRhtGroups = 4096;

struct RhtAmaxKernelArgs {
  const void* x;
  int64_t rows, cols;
  int64_t groups;  // column groups
  int64_t chunks;  // runs of kAmaxBlocks row blocks
  int64_t items;   // chunks x groups
  uint32_t mask;
  float* col_amax;
  float* tensor_amax;
  const float* noop;
  // grouped rows (group ends multiples of 128): col_amax is [G][cols] (each group's
  // column maxima) or tensor_amax is [G] (each group's maximum)
  const int64_t* ends;
  int G;
};

template <bool BF16, int V>
__global__ void __launch_bounds__(kRhtThreads) k_rht16_amax(RhtAmaxKernelArgs a) {
  __shared__ float s_gmax[kMaxRhtGroups];  // grouped per-group maxima of this CTA
  if (a.noop != nullptr && *a.noop == 1.0f) return;
  const bool grouped = a.ends != nullptr;
  const bool group_tensor = grouped && a.tensor_amax != nullptr;
  if (grouped) {
    if (!groups_valid(a.ends, a.G, a.rows) || !ends_aligned(a.ends, a.G, 128)) return;
    if (group_tensor) {
      for (int g = threadIdx.x; g < a.G; g += kRhtThreads) s_gmax[g] = 0.0f;
      __syncthreads();
    }
  }
  const int64_t stride = (int64_t)gridDim.x * kRhtThreads;
  const int64_t row_blocks = a.rows / 16;
  float tmax = 0.0f;  // per-tensor: this thread's max over all its items
  for (int64_t it = (int64_t)blockIdx.x * kRhtThreads + threadIdx.x; it < a.items;
       it += stride) {
    const int64_t ch = it / a.groups;
    const int64_t c0 = (it - ch * a.groups) * V;
    const int64_t rb1 = min(row_blocks, (ch + 1) * kAmaxBlocks);
    float cmax[V];
#pragma unroll
    for (int k = 0; k < V; ++k) cmax[k] = 0.0f;
    // grouped: the group of the current row block, and where it ends
    int g = 0;
    int64_t g_end = a.rows;
    if (grouped) {
      const int64_t r0 = ch * kAmaxBlocks * 16;
      int lo = 0, hi = a.G;  // first group whose end is > r0
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(a.ends + mid) <= r0) lo = mid + 1;
        else hi = mid;
      }
      g = lo;
      g_end = __ldg(a.ends + g);
    }
    // publish the maxima of group g's rows seen so far
    auto flush = [&]() {
      if (group_tensor) {
        float m = cmax[0];
#pragma unroll
        for (int k = 1; k < V; ++k) m = fmaxf(m, cmax[k]);
        if (m > 0.0f) atomicMax(reinterpret_cast<unsigned int*>(s_gmax + g), __float_as_uint(m));
      } else {
#pragma unroll
        for (int k = 0; k < V; ++k)
          if (cmax[k] > 0.0f)
            atomicMax(reinterpret_cast<unsigned int*>(a.col_amax + (int64_t)g * a.cols + c0 + k),
                      __float_as_uint(cmax[k]));
      }
#pragma unroll
      for (int k = 0; k < V; ++k) cmax[k] = 0.0f;
    };
    for (int64_t rb = ch * kAmaxBlocks; rb < rb1; ++rb) {
      if (grouped && rb * 16 >= g_end) {
        flush();
        do {
          g_end = __ldg(a.ends + ++g);
        } while (rb * 16 >= g_end);
      }
      const int64_t base = rb * 16 * a.cols + c0;
      float v[V][16];
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        const int64_t e = base + r * a.cols;
        if constexpr (BF16) {
          const uint16_t* xb = static_cast<const uint16_t*>(a.x);
          if constexpr (V == 2) {
            const uint32_t w = __ldg(reinterpret_cast<const unsigned int*>(xb + e));
            v[0][r] = __uint_as_float(w << 16);
            v[1][r] = __uint_as_float(w & 0xffff0000u);
          } else {
            v[0][r] = __uint_as_float((uint32_t)__ldg(xb + e) << 16);
          }
        } else {
          const float* xf = static_cast<const float*>(a.x);
          if constexpr (V == 2) {
            const float2 t = __ldg(reinterpret_cast<const float2*>(xf + e));
            v[0][r] = t.x;
            v[1][r] = t.y;
          } else {
            v[0][r] = __ldg(xf + e);
          }
        }
      }
      if constexpr (V == 2) rht16_block2(v[0], v[1], a.mask);
      else rht16_block(v[0], a.mask);
#pragma unroll
      for (int k = 0; k < V; ++k) {
#pragma unroll
        for (int r = 0; r < 16; ++r) cmax[k] = fmaxf(cmax[k], fabsf(v[k][r]));
      }
    }
    if (grouped) {
      flush();
      continue;
    }
    if (a.col_amax != nullptr) {
#pragma unroll
      for (int k = 0; k < V; ++k)
        atomicMax(reinterpret_cast<unsigned int*>(a.col_amax + c0 + k), __float_as_uint(cmax[k]));
    }
#pragma unroll
    for (int k = 0; k < V; ++k) tmax = fmaxf(tmax, cmax[k]);
  }
  if (group_tensor) {
    __syncthreads();
    for (int gg = threadIdx.x; gg < a.G; gg += kRhtThreads)
      if (s_gmax[gg] > 0.0f)
        atomicMax(reinterpret_cast<unsigned int*>(a.tensor_amax + gg), __float_as_uint(s_gmax[gg]));
    return;
  }
  if (grouped) return;
  if (a.tensor_amax != nullptr) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
    if ((threadIdx.x & 31) == 0)
      atomicMax(reinterpret_cast<unsigned int*>(a.tensor_amax), __float_as_uint(tmax));
  }
}

// The transform's column maxima and, in the same read of x, x's own row maxima
// (the two-direction transform quantize: rows as they are, columns transformed).
// The CTA's 256 threads take 256 adjacent column groups of one run of kAmaxBlocks row
// blocks (the launcher requires column groups a multiple of 256), so the loop is
// uniform over the CTA.  Per row block a warp reduces its 16 rows' |x| maxima over
// its 32 lanes with a transposing shuffle reduction (16 shuffles, each row ending in
// a lane pair), the 8 warps combine theirs with shared-memory atomics, and after the
// run one global atomic per row (row_max [rows]) or one per CTA and run
// (row_tensor [1]) publishes them.
struct RhtAmaxRowsArgs {
  RhtAmaxKernelArgs k;
  float* row_max;     // [rows] or NULL
  float* row_tensor;  // [1] or NULL
};

template <bool BF16, int V>
__global__ void __launch_bounds__(kRhtThreads) k_rht16_amax_rows(RhtAmaxRowsArgs ra) {
  const RhtAmaxKernelArgs& a = ra.k;
  constexpr int kRunRows = kAmaxBlocks * 16;
  __shared__ float s_rmax[kRunRows];
  __shared__ float s_red[kRhtThreads / 32];
  if (a.noop != nullptr && *a.noop == 1.0f) return;
  const int tid = threadIdx.x, lane = tid & 31;
  const int64_t stride = (int64_t)gridDim.x * kRhtThreads;
  const int64_t row_blocks = a.rows / 16;
  // this lane pair's row of a 16-row block after the transposing reduction
  const int my_row = ((lane >> 4) & 1) * 8 + ((lane >> 3) & 1) * 4 + ((lane >> 2) & 1) * 2 +
                     ((lane >> 1) & 1);
  float tmax = 0.0f;
  for (int64_t base = (int64_t)blockIdx.x * kRhtThreads; base < a.items; base += stride) {
    const int64_t it = base + tid;  // items is a multiple of kRhtThreads
    const int64_t ch = it / a.groups;
    const int64_t c0 = (it - ch * a.groups) * V;
    const int64_t rb0 = ch * kAmaxBlocks, rb1 = min(row_blocks, rb0 + kAmaxBlocks);
    s_rmax[tid] = 0.0f;  // kRunRows == kRhtThreads
    __syncthreads();
    float cmax[V];
#pragma unroll
    for (int k = 0; k < V; ++k) cmax[k] = 0.0f;
    for (int64_t rb = rb0; rb < rb1; ++rb) {
      const int64_t rowbase = rb * 16 * a.cols + c0;
      float v[V][16];
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        const int64_t e = rowbase + r * a.cols;
        if constexpr (BF16) {
          const uint16_t* xb = static_cast<const uint16_t*>(a.x);
          if constexpr (V == 4) {
            const uint2 w = __ldg(reinterpret_cast<const uint2*>(xb + e));
            v[0][r] = __uint_as_float(w.x << 16);
            v[1][r] = __uint_as_float(w.x & 0xffff0000u);
            v[2][r] = __uint_as_float(w.y << 16);
            v[3][r] = __uint_as_float(w.y & 0xffff0000u);
          } else if constexpr (V == 2) {
            const uint32_t w = __ldg(reinterpret_cast<const unsigned int*>(xb + e));
            v[0][r] = __uint_as_float(w << 16);
            v[1][r] = __uint_as_float(w & 0xffff0000u);
          } else {
            v[0][r] = __uint_as_float((uint32_t)__ldg(xb + e) << 16);
          }
        } else {
          static_assert(V <= 2, "four columns per thread: BF16 only");
          const float* xf = static_cast<const float*>(a.x);
          if constexpr (V == 2) {
            const float2 t = __ldg(reinterpret_cast<const float2*>(xf + e));
            v[0][r] = t.x;
            v[1][r] = t.y;
          } else {
            v[0][r] = __ldg(xf + e);
          }
        }
      }
      // x's row maxima over this warp's columns: halve the rows held per lane
      // with each shuffle step (16 -> 8 -> 4 -> 2 -> 1), then the lane pair
      float m[16];
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        m[r] = fabsf(v[0][r]);
#pragma unroll
        for (int k = 1; k < V; ++k) m[r] = fmaxf(m[r], fabsf(v[k][r]));
      }
#pragma unroll
      for (int h = 8; h >= 1; h >>= 1) {
        const bool up = lane & (2 * h);  // this lane keeps the upper half of its rows
#pragma unroll
        for (int j = 0; j < h; ++j) {
          const float send = up ? m[j] : m[j + h];
          const float keep = up ? m[j + h] : m[j];
          m[j] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, 2 * h));
        }
      }
      m[0] = fmaxf(m[0], __shfl_xor_sync(0xffffffffu, m[0], 1));
      if ((lane & 1) == 0 && m[0] > 0.0f)
        atomicMax(reinterpret_cast<unsigned int*>(s_rmax + 16 * (rb - rb0) + my_row),
                  __float_as_uint(m[0]));
      if constexpr (V == 4) {
        rht16_block2(v[0], v[1], a.mask);
        rht16_block2(v[2], v[3], a.mask);
      } else if constexpr (V == 2) {
        rht16_block2(v[0], v[1], a.mask);
      } else {
        rht16_block(v[0], a.mask);
      }
#pragma unroll
      for (int k = 0; k < V; ++k) {
#pragma unroll
        for (int r = 0; r < 16; ++r) cmax[k] = fmaxf(cmax[k], fabsf(v[k][r]));
      }
    }
    if (a.col_amax != nullptr) {
#pragma unroll
      for (int k = 0; k < V; ++k)
        atomicMax(reinterpret_cast<unsigned int*>(a.col_amax + c0 + k), __float_as_uint(cmax[k]));
    }
#pragma unroll
    for (int k = 0; k < V; ++k) tmax = fmaxf(tmax, cmax[k]);
    __syncthreads();  // every warp's row maxima of this run are in s_rmax
    const int64_t r = rb0 * 16 + tid;
    const float rv = s_rmax[tid];
    if (ra.row_max != nullptr && r < a.rows && rv > 0.0f)
      atomicMax(reinterpret_cast<unsigned int*>(ra.row_max + r), __float_as_uint(rv));
    if (ra.row_tensor != nullptr) {
      float w = rv;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) w = fmaxf(w, __shfl_xor_sync(0xffffffffu, w, o));
      if (lane == 0) s_red[tid >> 5] = w;
      __syncthreads();
      if (tid == 0) {
        float t = 0.0f;
        for (int i = 0; i < kRhtThreads / 32; ++i) t = fmaxf(t, s_red[i]);
        if (t > 0.0f) atomicMax(reinterpret_cast<unsigned int*>(ra.row_tensor), __float_as_uint(t));
      }
    }
    __syncthreads();  // s_rmax and s_red are reused by the next run
  }
  if (a.tensor_amax != nullptr) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
    if (lane == 0) atomicMax(reinterpret_cast<unsigned int*>(a.tensor_amax), __float_as_uint(tmax));
  }
}
static_assert(kAmaxBlocks * 16 == kRhtThreads, "one row of a run per thread");

bool pair_ok(const void* x, bool bf16, int64_t cols, const void* y) {
  const int elem = bf16 ? 2 : 4;
  return cols % 2 == 0 && reinterpret_cast<uintptr_t>(x) % (2 * elem) == 0 &&
         (y == nullptr || reinterpret_cast<uintptr_t>(y) % 8 == 0);
}

}  // namespace

// BF16 rows of 4 x 256-column multiples: four columns per thread (the row maxima's
// shuffle reduction then serves twice the elements).
bool quad_ok(const void* x, bool bf16, int64_t cols) {
  return bf16 && cols % (4 * kRhtThreads) == 0 && reinterpret_cast<uintptr_t>(x) % 8 == 0;
}

bool rht16_amax_rows_supported(const void* x, bool bf16, int64_t cols) {
  const int64_t groups = pair_ok(x, bf16, cols, nullptr) ? cols / 2 : cols;
  return quad_ok(x, bf16, cols) || groups % kRhtThreads == 0;
}

cudaError_t launch_rht16_amax_rows(const RhtAmaxArgs& q, float* row_max, float* row_tensor,
                                   const DeviceInfo& dev, cudaStream_t stream) {
  if (q.rows == 0 || q.cols == 0) return cudaSuccess;
  if (!rht16_amax_rows_supported(q.x, q.bf16, q.cols) || q.group_ends != nullptr)
    return cudaErrorInvalidValue;
  const bool quad = quad_ok(q.x, q.bf16, q.cols);
  const bool pair = pair_ok(q.x, q.bf16, q.cols, nullptr);
  RhtAmaxRowsArgs ra{};
  RhtAmaxKernelArgs& a = ra.k;
  a.x = q.x;
  a.rows = q.rows;
  a.cols = q.cols;
  a.groups = quad ? q.cols / 4 : pair ? q.cols / 2 : q.cols;
  a.chunks = (q.rows / 16 + kAmaxBlocks - 1) / kAmaxBlocks;
  a.items = a.chunks * a.groups;
  a.mask = q.sign_mask;
  a.col_amax = q.col_amax;
  a.tensor_amax = q.tensor_amax;
  a.noop = q.noop;
  ra.row_max = row_max;
  ra.row_tensor = row_tensor;
  const int64_t blocks = std::min<int64_t>(a.items / kRhtThreads, 8LL * dev.num_sms);
  void (*fn)(RhtAmaxRowsArgs);
  if (q.bf16)
    fn = quad ? k_rht16_amax_rows<true, 4>
              : pair ? k_rht16_amax_rows<true, 2> : k_rht16_amax_rows<true, 1>;
  else
    fn = pair ? k_rht16_amax_rows<false, 2> : k_rht16_amax_rows<false, 1>;
  fn<<<(unsigned)blocks, kRhtThreads, 0, stream>>>(ra);
  return cudaGetLastError();
}

cudaError_t launch_rht16_amax(const RhtAmaxArgs& q, const DeviceInfo& dev, cudaStream_t stream) {
  if (q.rows == 0 || q.cols == 0) return cudaSuccess;
  const bool pair = pair_ok(q.x, q.bf16, q.cols, nullptr);
  RhtAmaxKernelArgs a{};
  a.x = q.x;
  a.rows = q.rows;
  a.cols = q.cols;
  a.groups = pair ? q.cols / 2 : q.cols;
  a.chunks = (q.rows / 16 + kAmaxBlocks - 1) / kAmaxBlocks;
  a.items = a.chunks * a.groups;
  a.mask = q.sign_mask;
  a.col_amax = q.col_amax;
  a.tensor_amax = q.tensor_amax;
  a.noop = q.noop;
  a.ends = q.group_ends;
  a.G = q.num_groups;
  if (a.ends != nullptr && (a.G < 1 || a.G > kMaxRhtGroups)) return cudaErrorInvalidValue;
  const int64_t blocks =
      std::min<int64_t>((a.items + kRhtThreads - 1) / kRhtThreads, 8LL * dev.num_sms);
  void (*fn)(RhtAmaxKernelArgs);
  if (q.bf16) fn = pair ? k_rht16_amax<true, 2> : k_rht16_amax<true, 1>;
  else fn = pair ? k_rht16_amax<false, 2> : k_rht16_amax<false, 1>;
  fn<<<(unsigned)blocks, kRhtThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_rht16(const RhtArgs& q, const DeviceInfo& dev, cudaStream_t stream) {
  if (q.rows == 0 || q.cols == 0) return cudaSuccess;
  // two columns per thread: even row pitch, and bases aligned for 2-element accesses
  const bool pair = pair_ok(q.x, q.bf16, q.cols, q.y);
  RhtKernelArgs a{};
  a.x = q.x;
  a.y = q.y;
  a.cols = q.cols;
  a.groups = pair ? q.cols / 2 : q.cols;
  a.items = (q.rows / 16) * a.groups;
  a.mask = q.sign_mask;
  a.noop = q.noop;
  const int64_t blocks =
      std::min<int64_t>((a.items + kRhtThreads - 1) / kRhtThreads, 8LL * dev.num_sms);
  void (*fn)(RhtKernelArgs);
  if (q.bf16) fn = pair ? k_rht16<true, 2> : k_rht16<true, 1>;
  else fn = pair ? k_rht16<false, 2> : k_rht16<false, 1>;
  fn<<<(unsigned)blocks, kRhtThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace nvfp4
