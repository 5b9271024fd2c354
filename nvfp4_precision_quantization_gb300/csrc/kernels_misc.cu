// kernels_misc.cu -- NVFP4 dequantize and the self-tests (conversions, the division
// by a block scale, a bounded wait that runs out).
//
// Dequantize follows "Add backward overrides and 1x16 weights to NVFP4
// four-over-six" (torchao PR #8, description): value = code * ((scale * amax) *
// factor_inv), factor_inv a correctly rounded FP32 reciprocal of bound * 6, with
// BF16 output rounded to nearest even from the FP32 value.
//
// The kernel is write-bound (0.5625 bytes in, 2 or 4 bytes out per element): a
// thread expands 8 consecutive values (4 code bytes and their block's scale) into
// 16 (BF16) or 32 (FP32) contiguous output bytes, so one store instruction of a
// warp writes 512 B or 1 KB of contiguous output.  A CTA works on 2048-value
// segments of one row at a time (the row index is computed once per segment).
#include <algorithm>

#include <cuda_bf16.h>

#include "device_common.cuh"
#include "internal.h"

namespace nvfp4 {

namespace {

struct DequantKernelArgs {
  const uint8_t* codes;
  const uint8_t* scales;
  const float* amax;
  int row_scaled;
  int64_t rows, cols;
  int64_t cpitch, spitch;
  float F_inv;
  void* out;
};

constexpr int kDqThreads = 256;
constexpr int kDqPerThread = 8;
constexpr int kDqSegment = kDqThreads * kDqPerThread;  // values of a row per CTA item

template <bool BF16, bool VEC>
__global__ void __launch_bounds__(kDqThreads) k_dequantize(DequantKernelArgs a) {
  const int64_t per_row = (a.cols + kDqSegment - 1) / kDqSegment;
  const int64_t items = a.rows * per_row;
  for (int64_t it = blockIdx.x; it < items; it += gridDim.x) {
    const int64_t r = it / per_row;
    const int64_t c0 = (it - r * per_row) * kDqSegment + (int64_t)threadIdx.x * kDqPerThread;
    if (c0 >= a.cols) continue;
    const int n = (a.cols - c0) < kDqPerThread ? (int)(a.cols - c0) : kDqPerThread;
    const float amax = a.amax[a.row_scaled ? r : 0];
    const float D = dequant_factor(e4m3_value(a.scales[r * a.spitch + c0 / 16]), amax, a.F_inv);
    const uint8_t* cp = a.codes + r * a.cpitch + c0 / 2;
    uint32_t w;
    if (VEC && n == kDqPerThread) {
      w = *reinterpret_cast<const uint32_t*>(cp);
    } else {
      w = 0;
      for (int b = 0; b < (n + 1) / 2; ++b) w |= (uint32_t)cp[b] << (8 * b);
    }
    float v[kDqPerThread];
#pragma unroll
    for (int b = 0; b < kDqPerThread / 2; ++b) {
      float lo, hi;
      e2m1x2_values(w >> (8 * b), lo, hi);
      v[2 * b] = __fmul_rn(lo, D);
      v[2 * b + 1] = __fmul_rn(hi, D);
    }
    if constexpr (BF16) {
      __nv_bfloat16* o = static_cast<__nv_bfloat16*>(a.out) + r * a.cols + c0;
      if (VEC && n == kDqPerThread) {
        uint32_t p[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * k], v[2 * k + 1]);
          p[k] = *reinterpret_cast<uint32_t*>(&h);
        }
        stg_v4_cs(o, make_uint4(p[0], p[1], p[2], p[3]));
      } else {
#pragma unroll
        for (int k = 0; k < kDqPerThread; ++k)
          if (k < n) o[k] = __float2bfloat16_rn(v[k]);
      }
    } else {
      float* o = static_cast<float*>(a.out) + r * a.cols + c0;
      if (VEC && n == kDqPerThread) {
        uint32_t p[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) p[k] = __float_as_uint(v[k]);
        stg_v8_cs(o, p);
      } else {
#pragma unroll
        for (int k = 0; k < kDqPerThread; ++k)
          if (k < n) o[k] = v[k];
      }
    }
  }
}

// One code (and one scale byte) per input value, through the same conversion
// helpers the kernels use: 8 inputs are packed by e2m1x8 and split again, so
// a wrong nibble order shows up as permuted codes.
__global__ void k_selftest_convert(const float* in, int64_t n, uint8_t* e2m1, uint8_t* e4m3) {
  for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g * 8 < n;
       g += (int64_t)gridDim.x * blockDim.x) {
    float v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) v[k] = (g * 8 + k < n) ? in[g * 8 + k] : 0.0f;
    const uint32_t w = e2m1x8(v[0], v[1], v[2], v[3], v[4], v[5], v[6], v[7]);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int64_t i = g * 8 + k;
      if (i < n) {
        if (e2m1 != nullptr) e2m1[i] = (uint8_t)((w >> (4 * k)) & 15u);
        if (e4m3 != nullptr) e4m3[i] = (uint8_t)e4m3_byte(v[k]);
      }
    }
  }
}

// The encode factor e = fl(S / decode(s8)) as the encode kernels compute it (0 when
// the scale decodes to 0), for each S[i] and each E4M3 byte s8 = 0 .. 126:
// e[i * 127 + s8].
__global__ void k_selftest_scale_division(const float* S, int64_t n, float* e) {
  for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < n * 127;
       g += (int64_t)gridDim.x * blockDim.x) {
    const float sd = e4m3_value((uint32_t)(g % 127));
    e[g] = sd == 0.0f ? 0.0f : div_by_scale(S[g / 127], sd);
  }
}

// A bounded wait that runs out: thread 0 initialises a shared-memory mbarrier that
// expects one arrival, and no thread ever arrives on it.  Every thread of the warp
// waits on its first phase through the same bounded wait the pipelines use, with
// the caller's limit.  When the wait gives up, the kernel sets the timeout bit of
// the status word and returns without writing *out.  Had the wait completed, *out
// would be set to 1.  Nothing is in flight (no copy, no TMEM), so returning leaves
// the context clean.
__global__ void k_selftest_wait_timeout(uint64_t limit_ns, uint32_t* out, int* status) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  const bool ok = mbar_wait_bounded(&bar, 0, limit_ns);
  if (__all_sync(0xffffffffu, ok)) {
    if (threadIdx.x == 0) *out = 1u;
  } else if (threadIdx.x == 0) {
    raise_status(status, kStatusTimeout);
  }
}

}  // namespace

cudaError_t launch_selftest_scale_division(const float* S, int64_t n, float* e,
                                           cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>((n * 127 + 255) / 256, 4096);
  k_selftest_scale_division<<<(unsigned)blocks, 256, 0, stream>>>(S, n, e);
  return cudaGetLastError();
}

cudaError_t launch_selftest_wait_timeout(uint64_t limit_ns, uint32_t* out, const DeviceInfo& dev,
                                         cudaStream_t stream) {
  k_selftest_wait_timeout<<<1, 32, 0, stream>>>(limit_ns, out, dev.status);
  return cudaGetLastError();
}

cudaError_t launch_dequantize(const DequantArgs& q, const DeviceInfo& dev, cudaStream_t stream) {
  DequantKernelArgs a{};
  a.codes = q.codes;
  a.scales = q.scales;
  a.amax = q.amax;
  a.row_scaled = q.row_scaled ? 1 : 0;
  a.rows = q.rows;
  a.cols = q.cols;
  a.cpitch = (q.cols + 1) / 2;
  a.spitch = (q.cols + 15) / 16;
  a.F_inv = 1.0f / (q.bound * 6.0f);
  a.out = q.out;
  if (a.rows == 0 || a.cols == 0) return cudaSuccess;
  // whole 8-value groups: 4-byte code loads and 16-byte (BF16) / 32-byte (FP32)
  // stores, which need the row pitches and bases aligned to those sizes
  const int elem = q.out_bf16 ? 2 : 4;
  const bool vec = (q.cols % 8 == 0) && (reinterpret_cast<uintptr_t>(q.codes) % 4 == 0) &&
                   (reinterpret_cast<uintptr_t>(q.out) % (8 * elem) == 0);
  const int64_t items = a.rows * ((a.cols + kDqSegment - 1) / kDqSegment);
  const int64_t blocks = std::min<int64_t>(items, 8LL * dev.num_sms);
  void (*fn)(DequantKernelArgs);
  if (q.out_bf16) fn = vec ? k_dequantize<true, true> : k_dequantize<true, false>;
  else fn = vec ? k_dequantize<false, true> : k_dequantize<false, false>;
  fn<<<(unsigned)blocks, kDqThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_selftest_convert(const float* in, int64_t n, uint8_t* e2m1, uint8_t* e4m3,
                                    cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  const int64_t groups = (n + 7) / 8;
  const int64_t blocks = std::min<int64_t>((groups + 255) / 256, 4096);
  k_selftest_convert<<<(unsigned)blocks, 256, 0, stream>>>(in, n, e2m1, e4m3);
  return cudaGetLastError();
}

}  // namespace nvfp4
