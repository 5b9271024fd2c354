// api.cu -- the C ABI of libnvfp4 (declared in include/nvfp4.h).
//
// Host side only: argument validation with a per-thread message (in the style of
// the checks quoted in "NVFP4: enable row-scaled transpose quantization for
// backward", TransformerEngine PR #3206, review of the grouped GEMM draft, and
// "row-scaled nvfp4 path: fuse row/col amax into a single TMA-tiled kernel",
// PR #3454, review of compute_fused_amax), the per-device cache (SM count and the
// status word, for the *current* device -- the draft reviewed in PR #3206
// hard-coded device 0), and the stream-ordered launch sequences.  Nothing here
// allocates device memory, synchronizes, or reads device data, except
// nvfp4_device_status, which exists to do exactly that.
//
// Unlike the wrapper reviewed in PR #3454, amax buffers are never cleared by a
// host-side memset: clearing happens in a kernel that first checks the noop
// flag, so a skipped call leaves existing amax metadata untouched.
#include <cstring>
#include <mutex>
#include <string>

#include "../../include/nvfp4.h"
#include "internal.h"

namespace nvfp4 {

// The library's one piece of device state: sticky error bits that kernels set
// when they find invalid device-resident input or give up a bounded wait.
__device__ int g_status_word;

// Workspace of nvfp4_gemm_static_ws: file-scope device memory reserved when the module
// loads, so that call allocates nothing.
static __device__ __align__(256) uint8_t g_gemm_static_ws[NVFP4_GEMM_STATIC_WS_BYTES];

namespace {

thread_local std::string g_last_error;

nvfp4_status fail(nvfp4_status st, const std::string& msg) {
  g_last_error = msg;
  return st;
}

nvfp4_status cuda_fail(cudaError_t e, const char* what) {
  return fail(NVFP4_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

// Whether the byte ranges [a, a + na) and [b, b + nb) share a byte (empty ranges and
// NULL pointers share none).
bool bytes_overlap(const void* a, uint64_t na, const void* b, uint64_t nb) {
  if (a == nullptr || b == nullptr || na == 0 || nb == 0) return false;
  const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
  return pa < pb + nb && pb < pa + na;
}

struct DevCacheEntry {
  bool ready = false;
  int num_sms = 0;
  int64_t l2_bytes = 0;
  int* status = nullptr;
  uint8_t* gemm_static_ws = nullptr;  // device address of g_gemm_static_ws
};
constexpr int kMaxDevices = 64;
std::mutex g_mu;
DevCacheEntry g_dev[kMaxDevices];

nvfp4_status current_device(DeviceInfo* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(NVFP4_ERR_UNSUPPORTED, "device index too large");
  std::lock_guard<std::mutex> lock(g_mu);
  DevCacheEntry& c = g_dev[dev];
  if (!c.ready) {
    int sms = 0, l2 = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    e = cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_status_word);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status word)");
    void* ws = nullptr;
    e = cudaGetSymbolAddress(&ws, g_gemm_static_ws);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static GEMM workspace)");
    c.num_sms = sms;
    c.l2_bytes = l2;
    c.status = static_cast<int*>(p);
    c.gemm_static_ws = static_cast<uint8_t*>(ws);
    c.ready = true;
  }
  out->device = dev;
  out->num_sms = c.num_sms;
  out->l2_bytes = c.l2_bytes;
  out->status = c.status;
  out->gemm_static_ws = c.gemm_static_ws;
  return NVFP4_OK;
}

bool valid_in_dtype(int32_t d) { return d == NVFP4_IN_BF16 || d == NVFP4_IN_FP32; }

nvfp4_status check_sizes(int64_t rows, int64_t cols) {
  if (rows < 0 || cols < 0) return fail(NVFP4_ERR_INVALID, "rows and cols must be >= 0");
  if (rows >= (1LL << 31) || cols >= (1LL << 31))
    return fail(NVFP4_ERR_INVALID, "rows and cols must be < 2^31");
  return NVFP4_OK;
}

nvfp4_status check_config(const nvfp4_config* cfg) {
  if (cfg == nullptr) return fail(NVFP4_ERR_INVALID, "cfg is NULL");
  if (cfg->mode != NVFP4_PER_TENSOR && cfg->mode != NVFP4_ROW_SCALED)
    return fail(NVFP4_ERR_INVALID, "cfg->mode must be NVFP4_PER_TENSOR or NVFP4_ROW_SCALED");
  if (!(cfg->bound == 448.0f || cfg->bound == 256.0f))
    return fail(NVFP4_ERR_INVALID, "cfg->bound must be 448 or 256");
  if (cfg->four_over_six != 0 && cfg->four_over_six != 1)
    return fail(NVFP4_ERR_INVALID, "cfg->four_over_six must be 0 or 1");
  if (cfg->block_2d != 0 && cfg->block_2d != 1)
    return fail(NVFP4_ERR_INVALID, "cfg->block_2d must be 0 or 1");
  if (cfg->block_2d && cfg->mode == NVFP4_ROW_SCALED)
    return fail(NVFP4_ERR_INVALID, "16x16 blocks are per-tensor only");
  return NVFP4_OK;
}

nvfp4_status check_out(const nvfp4_out* o, const char* name, int64_t lines, int64_t n,
                       int64_t amax_len) {
  if (o == nullptr) return fail(NVFP4_ERR_INVALID, std::string(name) + " is NULL");
  if (o->amax == nullptr && amax_len > 0)
    return fail(NVFP4_ERR_INVALID, std::string(name) + "->amax is NULL");
  if (lines * n > 0 && (o->codes == nullptr || o->scales == nullptr))
    return fail(NVFP4_ERR_INVALID, std::string(name) + "->codes / ->scales is NULL");
  return NVFP4_OK;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// One sequence of launches for any quantize direction set (row and/or col may be NULL).
nvfp4_status quantize_impl(const void* x, int32_t in_dtype, int64_t rows, int64_t cols,
                           const nvfp4_config* cfg, const nvfp4_out* row, const nvfp4_out* col,
                           const float* noop, cudaStream_t stream,
                           const int64_t* group_ends = nullptr, int num_groups = 0,
                           bool rht = false, uint32_t rht_mask = 0) {
  nvfp4_status st;
  if (!valid_in_dtype(in_dtype)) return fail(NVFP4_ERR_INVALID, "unknown in_dtype");
  if ((st = check_sizes(rows, cols)) != NVFP4_OK) return st;
  if ((st = check_config(cfg)) != NVFP4_OK) return st;
  const bool rs_mode = cfg->mode == NVFP4_ROW_SCALED;
  if (row && (st = check_out(row, "row", rows, cols, rs_mode ? rows : 1)) != NVFP4_OK) return st;
  if (col && (st = check_out(col, "col", cols, rows, rs_mode ? cols : 1)) != NVFP4_OK) return st;
  if (x == nullptr && rows * cols > 0) return fail(NVFP4_ERR_INVALID, "x is NULL");
  DeviceInfo dev;
  if ((st = current_device(&dev)) != NVFP4_OK) return st;

  const bool rs = cfg->mode == NVFP4_ROW_SCALED;
  const bool need_r = row && row->amax_in == nullptr;
  const bool need_c = col && col->amax_in == nullptr;
  const InType in = in_dtype == NVFP4_IN_BF16 ? InType::BF16 : InType::FP32;

  PrepArgs prep{};
  AmaxArgs am{};
  am.x = x;
  am.in = in;
  am.M = rows;
  am.K = cols;
  am.noop = noop;
  am.group_ends = group_ends;
  am.num_groups = num_groups;
  QuantArgs q{};
  q.x = x;
  q.in = in;
  q.M = rows;
  q.K = cols;
  q.row_scaled = rs;
  q.four_over_six = cfg->four_over_six != 0;
  q.block_2d = cfg->block_2d != 0;
  q.bound = cfg->bound;
  q.noop = noop;
  q.group_ends = group_ends;
  q.num_groups = num_groups;
  q.rht = rht;
  q.rht_mask = rht_mask;
  if (row) {
    q.row_codes = row->codes;
    q.row_scales = row->scales;
    q.row_amax = row->amax;
  }
  if (col) {
    q.col_codes = col->codes;
    q.col_scales = col->scales;
    q.col_amax = col->amax;
  }
  int nz = 0, nc = 0;
  auto add_zero = [&](float* p, int64_t n) {
    prep.zero_ptr[nz] = p;
    prep.zero_n[nz++] = n;
  };
  auto add_copy = [&](float* d, const float* s, int64_t n) {
    if (d == s) return;
    prep.copy_dst[nc] = d;
    prep.copy_src[nc] = s;
    prep.copy_n[nc++] = n;
  };
  if (rs) {
    if (need_r) {
      add_zero(row->amax, rows);
      am.row_amax = row->amax;
    } else if (row) {
      add_copy(row->amax, row->amax_in, rows);
    }
    if (need_c) {
      add_zero(col->amax, cols);
      am.col_amax = col->amax;
    } else if (col) {
      add_copy(col->amax, col->amax_in, cols);
    }
  } else {
    float* target = need_r ? row->amax : (need_c ? col->amax : nullptr);
    if (target) {
      add_zero(target, 1);
      am.tensor_amax = target;
    }
    if (row && !need_r) add_copy(row->amax, row->amax_in, 1);
    if (col && !need_c) add_copy(col->amax, col->amax_in, 1);
    if (need_r && need_c) {
      // both directions use the one tensor amax computed into row->amax; the
      // quantize kernel copies it to col->amax (zeroed here for empty inputs)
      add_zero(col->amax, 1);
      q.col_amax = row->amax;
      q.copy_dst = col->amax;
      q.copy_src = row->amax;
    }
  }
  cudaError_t e;
  prep.noop = noop;
  if (nz + nc > 0) {
    if (group_ends) {
      // grouped calls: the prep step must also refuse invalid group ends
      GroupCheckArgs g{};
      g.M = rows;
      g.group_ends = group_ends;
      g.num_groups = num_groups;
      g.noop = noop;
      g.prep = prep;
      if ((e = launch_group_check(g, dev, stream, false)) != cudaSuccess)
        return cuda_fail(e, "group check launch");
    } else if ((e = launch_prep(prep, dev, stream)) != cudaSuccess) {
      return cuda_fail(e, "prep launch");
    }
  }
  if (rht && (am.col_amax || am.tensor_amax)) {
    // the amax of the transformed columns, computed from x without writing them
    RhtAmaxArgs ra{x, in == InType::BF16, rows, cols, rht_mask, am.col_amax, am.tensor_amax,
                   noop};
    if ((e = launch_rht16_amax(ra, dev, stream)) != cudaSuccess)
      return cuda_fail(e, "transform amax launch");
  } else if (am.row_amax || am.col_amax || am.tensor_amax) {
    if ((e = launch_amax(am, dev, stream)) != cudaSuccess) return cuda_fail(e, "amax launch");
  }
  if ((e = launch_quantize(q, dev, stream)) != cudaSuccess) return cuda_fail(e, "quantize launch");
  return NVFP4_OK;
}

}  // namespace

bool make_tile_map(CUtensorMap* map, const void* base, InType in, int64_t rows, int64_t cols,
                   int box_cols, int box_rows) {
  const int elem = in == InType::BF16 ? 2 : 4;
  if (rows <= 0 || cols <= 0) return false;
  if (reinterpret_cast<uintptr_t>(base) % 16 != 0) return false;
  if ((cols * elem) % 16 != 0) return false;
  EncodeTiledFn fn = encode_tiled();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)(cols * elem)};
  const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  const cuuint32_t estride[2] = {1, 1};
  const CUresult r =
      fn(map, in == InType::BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
         2, const_cast<void*>(base), dims, strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_byte_map(CUtensorMap* map, const void* base, int64_t rows, int64_t pitch,
                   int box_bytes, int box_rows) {
  if (rows <= 0 || pitch <= 0) return false;
  if (reinterpret_cast<uintptr_t>(base) % 16 != 0 || pitch % 16 != 0) return false;
  if (rows >= (1LL << 31) || pitch >= (1LL << 31)) return false;
  EncodeTiledFn fn = encode_tiled();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)pitch, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)pitch};
  const cuuint32_t box[2] = {(cuuint32_t)box_bytes, (cuuint32_t)box_rows};
  const cuuint32_t estride[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
                        strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_operand_map(CUtensorMap* map, const void* base, int64_t rows, int64_t pitch,
                      int box_bytes, int box_rows) {
  if (rows <= 0 || pitch <= 0) return false;
  if (box_bytes != 128 && box_bytes != 64) return false;
  if (reinterpret_cast<uintptr_t>(base) % 16 != 0 || pitch % 16 != 0) return false;
  if (rows >= (1LL << 31) || pitch >= (1LL << 31)) return false;
  EncodeTiledFn fn = encode_tiled();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)pitch, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)pitch};
  const cuuint32_t box[2] = {(cuuint32_t)box_bytes, (cuuint32_t)box_rows};
  const cuuint32_t estride[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
                        strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        box_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace nvfp4

using namespace nvfp4;

extern "C" {

nvfp4_status nvfp4_amax(const void* x, int32_t in_dtype, int64_t rows, int64_t cols,
                        float* row_amax, float* col_amax, float* tensor_amax, const float* noop,
                        nvfp4_stream_t stream) {
  nvfp4_status st;
  if (!valid_in_dtype(in_dtype)) return fail(NVFP4_ERR_INVALID, "unknown in_dtype");
  if ((st = check_sizes(rows, cols)) != NVFP4_OK) return st;
  if (!row_amax && !col_amax && !tensor_amax)
    return fail(NVFP4_ERR_INVALID, "no amax output given");
  if (x == nullptr && rows * cols > 0) return fail(NVFP4_ERR_INVALID, "x is NULL");
  DeviceInfo dev;
  if ((st = current_device(&dev)) != NVFP4_OK) return st;
  PrepArgs prep{};
  int nz = 0;
  if (row_amax) { prep.zero_ptr[nz] = row_amax; prep.zero_n[nz++] = rows; }
  if (col_amax) { prep.zero_ptr[nz] = col_amax; prep.zero_n[nz++] = cols; }
  if (tensor_amax) { prep.zero_ptr[nz] = tensor_amax; prep.zero_n[nz++] = 1; }
  prep.noop = noop;
  cudaError_t e = launch_prep(prep, dev, stream);
  if (e != cudaSuccess) return cuda_fail(e, "prep launch");
  AmaxArgs am{};
  am.x = x;
  am.in = in_dtype == NVFP4_IN_BF16 ? InType::BF16 : InType::FP32;
  am.M = rows;
  am.K = cols;
  am.row_amax = row_amax;
  am.col_amax = col_amax;
  am.tensor_amax = tensor_amax;
  am.noop = noop;
  if ((e = launch_amax(am, dev, stream)) != cudaSuccess) return cuda_fail(e, "amax launch");
  return NVFP4_OK;
}

nvfp4_status nvfp4_quantize_rowwise(const void* x, int32_t in_dtype, int64_t rows, int64_t cols,
                                    const nvfp4_config* cfg, const nvfp4_out* row,
                                    const float* noop, nvfp4_stream_t stream) {
  if (row == nullptr) return fail(NVFP4_ERR_INVALID, "row is NULL");
  return quantize_impl(x, in_dtype, rows, cols, cfg, row, nullptr, noop, stream);
}

nvfp4_status nvfp4_quantize_columnwise(const void* x, int32_t in_dtype, int64_t rows,
                                       int64_t cols, const nvfp4_config* cfg,
                                       const nvfp4_out* col, const float* noop,
                                       nvfp4_stream_t stream) {
  if (col == nullptr) return fail(NVFP4_ERR_INVALID, "col is NULL");
  return quantize_impl(x, in_dtype, rows, cols, cfg, nullptr, col, noop, stream);
}

nvfp4_status nvfp4_quantize_both(const void* x, int32_t in_dtype, int64_t rows, int64_t cols,
                                 const nvfp4_config* cfg, const nvfp4_out* row,
                                 const nvfp4_out* col, const float* noop, nvfp4_stream_t stream) {
  if (row == nullptr || col == nullptr) return fail(NVFP4_ERR_INVALID, "row or col is NULL");
  return quantize_impl(x, in_dtype, rows, cols, cfg, row, col, noop, stream);
}

namespace {

nvfp4_status check_rht(const void* x, int32_t in_dtype, int64_t rows, int64_t cols,
                       uint32_t sign_mask) {
  nvfp4_status st = check_sizes(rows, cols);
  if (st != NVFP4_OK) return st;
  if (!valid_in_dtype(in_dtype)) return fail(NVFP4_ERR_INVALID, "unknown in_dtype");
  if (sign_mask > 0xFFFFu) return fail(NVFP4_ERR_INVALID, "sign_mask must be < 2^16");
  if (rows % 16 != 0)
    return fail(NVFP4_ERR_UNSUPPORTED, "the transform needs rows a multiple of 16");
  if (rows * cols > 0 && x == nullptr) return fail(NVFP4_ERR_INVALID, "x is NULL");
  return NVFP4_OK;
}

}  // namespace

nvfp4_status nvfp4_rht16(const void* x, int32_t in_dtype, int64_t rows, int64_t cols,
                         uint32_t sign_mask, float* y, nvfp4_stream_t stream) {
  nvfp4_status st = check_rht(x, in_dtype, rows, cols, sign_mask);
  if (st != NVFP4_OK) return st;
  if (rows * cols > 0 && y == nullptr) return fail(NVFP4_ERR_INVALID, "y is NULL");
  const uint64_t n = (uint64_t)rows * (uint64_t)cols;
  const uint64_t x_bytes = n * (in_dtype == NVFP4_IN_FP32 ? 4u : 2u);
  // a thread reads its 16-row block before writing it, but a neighbouring block of a
  // partly overlapping y may already have been overwritten: only y == x (FP32) is safe
  const bool same = static_cast<const void*>(y) == x && in_dtype == NVFP4_IN_FP32;
  if (!same && bytes_overlap(x, x_bytes, y, 4 * n))
    return fail(NVFP4_ERR_INVALID, "y overlaps x (only y == x, for FP32 input, is allowed)");
  DeviceInfo dev{};
  st = current_device(&dev);
  if (st != NVFP4_OK) return st;
  RhtArgs a{x, in_dtype == NVFP4_IN_BF16, rows, cols, sign_mask, y, nullptr};
  cudaError_t e = launch_rht16(a, dev, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? NVFP4_OK : cuda_fail(e, "transform launch");
}

nvfp4_status nvfp4_quantize_columnwise_rht(const void* x, int32_t in_dtype, int64_t rows,
                                           int64_t cols, uint32_t sign_mask,
                                           const nvfp4_config* cfg, const nvfp4_out* col,
                                           float* workspace, uint64_t ws_bytes,
                                           const float* noop, nvfp4_stream_t stream) {
  // every argument is checked before the first launch, so a rejected call enqueues nothing
  nvfp4_status st = check_rht(x, in_dtype, rows, cols, sign_mask);
  if (st != NVFP4_OK) return st;
  st = check_config(cfg);
  if (st != NVFP4_OK) return st;
  st = check_out(col, "col", cols, rows, cfg->mode == NVFP4_ROW_SCALED ? cols : 1);
  if (st != NVFP4_OK) return st;
  if (!cfg->block_2d) {
    // fused: the amax pass and the encode pass each transform the blocks they read
    return quantize_impl(x, in_dtype, rows, cols, cfg, nullptr, col, noop, stream, nullptr, 0,
                         true, sign_mask);
  }
  // 16x16 blocks: the transformed operand is written to the workspace and quantized
  const uint64_t need = 4ull * (uint64_t)rows * (uint64_t)cols;
  if (need > 0 && (workspace == nullptr || ws_bytes < need))
    return fail(NVFP4_ERR_INVALID, "workspace must hold rows * cols FP32 values");
  const uint64_t n = (uint64_t)rows * (uint64_t)cols;
  const uint64_t na = cfg->mode == NVFP4_ROW_SCALED ? (uint64_t)cols : 1u;
  if (bytes_overlap(workspace, need, x, n * (in_dtype == NVFP4_IN_FP32 ? 4u : 2u)) ||
      bytes_overlap(workspace, need, col->codes, (uint64_t)cols * (((uint64_t)rows + 1) / 2)) ||
      bytes_overlap(workspace, need, col->scales, (uint64_t)cols * (((uint64_t)rows + 15) / 16)) ||
      bytes_overlap(workspace, need, col->amax, 4 * na) ||
      bytes_overlap(workspace, need, col->amax_in, col->amax_in ? 4 * na : 0))
    return fail(NVFP4_ERR_INVALID, "workspace overlaps x or an output");
  DeviceInfo dev{};
  st = current_device(&dev);
  if (st != NVFP4_OK) return st;
  RhtArgs a{x, in_dtype == NVFP4_IN_BF16, rows, cols, sign_mask, workspace, noop};
  cudaError_t e = launch_rht16(a, dev, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "transform launch");
  return quantize_impl(workspace, NVFP4_IN_FP32, rows, cols, cfg, nullptr, col, noop, stream);
}

nvfp4_status nvfp4_quantize_both_rht(const void* x, int32_t in_dtype, int64_t rows, int64_t cols,
                                     uint32_t sign_mask, const nvfp4_config* cfg,
                                     const nvfp4_out* row, const nvfp4_out* col,
                                     const float* noop, nvfp4_stream_t stream) {
  // every argument is checked before the first launch, so a rejected call enqueues nothing
  nvfp4_status st = check_rht(x, in_dtype, rows, cols, sign_mask);
  if (st != NVFP4_OK) return st;
  if ((st = check_config(cfg)) != NVFP4_OK) return st;
  if (cfg->block_2d)
    return fail(NVFP4_ERR_UNSUPPORTED, "the two-direction transform quantize uses 1x16 blocks");
  if (row == nullptr || col == nullptr) return fail(NVFP4_ERR_INVALID, "row and col must be non-NULL");
  const bool rs = cfg->mode == NVFP4_ROW_SCALED;
  const int64_t n_r = rs ? rows : 1, n_c = rs ? cols : 1;
  if ((st = check_out(row, "row", rows, cols, n_r)) != NVFP4_OK) return st;
  if ((st = check_out(col, "col", cols, rows, n_c)) != NVFP4_OK) return st;
  const int elem = in_dtype == NVFP4_IN_FP32 ? 4 : 2;
  if (rows * cols > 0 &&
      ((cols * elem) % 16 != 0 || reinterpret_cast<uintptr_t>(x) % 16 != 0))
    return fail(NVFP4_ERR_UNSUPPORTED, "x rows must be 16-byte aligned");
  DeviceInfo dev{};
  if ((st = current_device(&dev)) != NVFP4_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const InType in = in_dtype == NVFP4_IN_BF16 ? InType::BF16 : InType::FP32;
  const bool need_r = row->amax_in == nullptr, need_c = col->amax_in == nullptr;
  // 1. clear the amax outputs (or copy the given ones), after the noop check
  PrepArgs prep{};
  int nz = 0, nc = 0;
  if (need_r) {
    prep.zero_ptr[nz] = row->amax;
    prep.zero_n[nz++] = n_r;
  } else if (row->amax != row->amax_in) {
    prep.copy_dst[nc] = row->amax;
    prep.copy_src[nc] = row->amax_in;
    prep.copy_n[nc++] = n_r;
  }
  if (need_c) {
    prep.zero_ptr[nz] = col->amax;
    prep.zero_n[nz++] = n_c;
  } else if (col->amax != col->amax_in) {
    prep.copy_dst[nc] = col->amax;
    prep.copy_src[nc] = col->amax_in;
    prep.copy_n[nc++] = n_c;
  }
  prep.noop = noop;
  cudaError_t e;
  if (nz + nc > 0 && (e = launch_prep(prep, dev, s)) != cudaSuccess)
    return cuda_fail(e, "prep launch");
  // 2. the transposed side's amax is the transform's; the rowwise side's is x's --
  //    both from one read of x where the column count allows
  if (need_c && need_r && rht16_amax_rows_supported(x, in == InType::BF16, cols)) {
    RhtAmaxArgs ra{x, in == InType::BF16, rows, cols, sign_mask, rs ? col->amax : nullptr,
                   rs ? nullptr : col->amax, noop};
    if ((e = launch_rht16_amax_rows(ra, rs ? row->amax : nullptr, rs ? nullptr : row->amax, dev,
                                    s)) != cudaSuccess)
      return cuda_fail(e, "transform and row amax launch");
  } else {
    if (need_c) {
      RhtAmaxArgs ra{x, in == InType::BF16, rows, cols, sign_mask, rs ? col->amax : nullptr,
                     rs ? nullptr : col->amax, noop};
      if ((e = launch_rht16_amax(ra, dev, s)) != cudaSuccess)
        return cuda_fail(e, "transform amax launch");
    }
    if (need_r) {
      AmaxArgs am{};
      am.x = x;
      am.in = in;
      am.M = rows;
      am.K = cols;
      am.row_amax = rs ? row->amax : nullptr;
      am.tensor_amax = rs ? nullptr : row->amax;
      am.noop = noop;
      if ((e = launch_amax(am, dev, s)) != cudaSuccess) return cuda_fail(e, "amax launch");
    }
  }
  // 3. one encode pass: rows as they are, columns transformed block by block
  QuantArgs q{};
  q.x = x;
  q.in = in;
  q.M = rows;
  q.K = cols;
  q.row_scaled = rs;
  q.four_over_six = cfg->four_over_six != 0;
  q.block_2d = false;
  q.bound = cfg->bound;
  q.noop = noop;
  q.rht = true;
  q.rht_mask = sign_mask;
  q.row_codes = row->codes;
  q.row_scales = row->scales;
  q.row_amax = row->amax;
  q.col_codes = col->codes;
  q.col_scales = col->scales;
  q.col_amax = col->amax;
  if ((e = launch_quantize(q, dev, s)) != cudaSuccess) return cuda_fail(e, "quantize launch");
  return NVFP4_OK;
}

nvfp4_status nvfp4_dequantize(const uint8_t* codes, const uint8_t* scales, const float* amax,
                              int32_t mode, int64_t rows, int64_t cols, float bound, void* out,
                              int32_t out_dtype, nvfp4_stream_t stream) {
  nvfp4_status st;
  if ((st = check_sizes(rows, cols)) != NVFP4_OK) return st;
  if (mode != NVFP4_PER_TENSOR && mode != NVFP4_ROW_SCALED)
    return fail(NVFP4_ERR_INVALID, "mode must be NVFP4_PER_TENSOR or NVFP4_ROW_SCALED");
  if (!(bound == 448.0f || bound == 256.0f)) return fail(NVFP4_ERR_INVALID, "bound must be 448 or 256");
  if (out_dtype != NVFP4_OUT_BF16 && out_dtype != NVFP4_OUT_FP32)
    return fail(NVFP4_ERR_INVALID, "unknown out_dtype");
  if (rows * cols > 0 && (!codes || !scales || !amax || !out))
    return fail(NVFP4_ERR_INVALID, "codes, scales, amax and out must be non-NULL");
  DeviceInfo dev;
  if ((st = current_device(&dev)) != NVFP4_OK) return st;
  DequantArgs d{};
  d.codes = codes;
  d.scales = scales;
  d.amax = amax;
  d.row_scaled = mode == NVFP4_ROW_SCALED;
  d.rows = rows;
  d.cols = cols;
  d.bound = bound;
  d.out = out;
  d.out_bf16 = out_dtype == NVFP4_OUT_BF16;
  cudaError_t e = launch_dequantize(d, dev, stream);
  if (e != cudaSuccess) return cuda_fail(e, "dequantize launch");
  return NVFP4_OK;
}

nvfp4_status nvfp4_gemm_workspace_size(int64_t m, int64_t n, int64_t k, uint64_t* bytes) {
  if (bytes == nullptr) return fail(NVFP4_ERR_INVALID, "bytes is NULL");
  nvfp4_status st;
  if ((st = check_sizes(m, n)) != NVFP4_OK) return st;
  if ((st = check_sizes(k, 0)) != NVFP4_OK) return st;
  *bytes = (m == 0 || n == 0 || k == 0) ? 0 : (uint64_t)gemm_layout(m, n, k, n).workspace_bytes;
  return NVFP4_OK;
}

namespace {
// workspace == NULL: the static workspace of the current device (nvfp4_gemm_static_ws)
// group_ends != NULL: the grouped GEMM (num_groups groups of A's rows, B = [groups*n][k])
nvfp4_status gemm_impl(const nvfp4_operand* a, const nvfp4_operand* b, const int64_t* group_ends,
                       int32_t num_groups, int64_t m, int64_t n, int64_t k, void* d,
                       int32_t out_dtype, void* workspace, uint64_t workspace_bytes,
                       nvfp4_stream_t stream, bool static_ws, bool k_grouped = false) {
  nvfp4_status st;
  if ((st = check_sizes(m, n)) != NVFP4_OK) return st;
  if ((st = check_sizes(k, 0)) != NVFP4_OK) return st;
  if (a == nullptr || b == nullptr) return fail(NVFP4_ERR_INVALID, "a or b is NULL");
  if (out_dtype != NVFP4_OUT_BF16 && out_dtype != NVFP4_OUT_FP32)
    return fail(NVFP4_ERR_INVALID, "unknown out_dtype");
  for (const nvfp4_operand* o : {a, b}) {
    if (o->mode != NVFP4_PER_TENSOR && o->mode != NVFP4_ROW_SCALED)
      return fail(NVFP4_ERR_INVALID, "operand mode must be NVFP4_PER_TENSOR or NVFP4_ROW_SCALED");
    if (!(o->bound == 448.0f || o->bound == 256.0f))
      return fail(NVFP4_ERR_INVALID, "operand bound must be 448 or 256");
  }
  if (m == 0 || n == 0) return NVFP4_OK;
  if (d == nullptr) return fail(NVFP4_ERR_INVALID, "d is NULL");
  const size_t esize = out_dtype == NVFP4_OUT_BF16 ? 2 : 4;
  if (k == 0) {  // the empty sum
    const size_t blocks = k_grouped ? (size_t)num_groups : 1;
    cudaError_t e = cudaMemsetAsync(d, 0, blocks * (size_t)m * (size_t)n * esize, stream);
    return e == cudaSuccess ? NVFP4_OK : cuda_fail(e, "cudaMemsetAsync");
  }
  if (k % 32 != 0) return fail(NVFP4_ERR_UNSUPPORTED, "k must be a multiple of 32");
  for (const nvfp4_operand* o : {a, b}) {
    if (!o->codes || !o->scales || !o->amax)
      return fail(NVFP4_ERR_INVALID, "operand codes, scales and amax must be non-NULL");
    if (reinterpret_cast<uintptr_t>(o->codes) % 16 != 0)
      return fail(NVFP4_ERR_UNSUPPORTED, "operand codes must be 16-byte aligned");
  }
  if (group_ends != nullptr && !k_grouped && n % 256 != 0)
    return fail(NVFP4_ERR_UNSUPPORTED, "grouped GEMM: n must be a multiple of 256");
  if (k_grouped && k % 256 != 0)
    return fail(NVFP4_ERR_UNSUPPORTED, "grouped wgrad GEMM: tokens must be a multiple of 256");
  const GemmLayout L =
      gemm_layout(m, n, k, group_ends && !k_grouped ? (int64_t)num_groups * n : n);
  if (L.tiles_m * L.tiles_n >= (1LL << 31)) return fail(NVFP4_ERR_UNSUPPORTED, "too many tiles");
  if (static_ws) {
    if ((uint64_t)L.workspace_bytes > (uint64_t)NVFP4_GEMM_STATIC_WS_BYTES)
      return fail(NVFP4_ERR_UNSUPPORTED,
                  "the shape needs " + std::to_string(L.workspace_bytes) +
                      " bytes of workspace, more than the static workspace holds");
  } else {
    if (workspace == nullptr || reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
      return fail(NVFP4_ERR_INVALID, "workspace must be non-NULL and 256-byte aligned");
    if (workspace_bytes < (uint64_t)L.workspace_bytes)
      return fail(NVFP4_ERR_INVALID, "workspace smaller than nvfp4_gemm_workspace_size");
  }
  DeviceInfo dev;
  if ((st = current_device(&dev)) != NVFP4_OK) return st;
  GemmArgs g{};
  g.a_codes = a->codes;
  g.a_scales = a->scales;
  g.a_amax = a->amax;
  g.a_row_scaled = a->mode == NVFP4_ROW_SCALED;
  g.a_bound = a->bound;
  g.b_codes = b->codes;
  g.b_scales = b->scales;
  g.b_amax = b->amax;
  g.b_row_scaled = b->mode == NVFP4_ROW_SCALED;
  g.b_bound = b->bound;
  g.M = m;
  g.N = n;
  g.K = k;
  g.d = d;
  g.d_bf16 = out_dtype == NVFP4_OUT_BF16;
  g.workspace = static_ws ? dev.gemm_static_ws : static_cast<uint8_t*>(workspace);
  g.group_ends = group_ends;
  g.num_groups = num_groups;
  g.k_grouped = k_grouped;
  cudaError_t e = launch_gemm(g, dev, stream);
  if (e != cudaSuccess) return cuda_fail(e, "gemm launch");
  return NVFP4_OK;
}
}  // namespace

nvfp4_status nvfp4_gemm(const nvfp4_operand* a, const nvfp4_operand* b, int64_t m, int64_t n,
                        int64_t k, void* d, int32_t out_dtype, void* workspace,
                        uint64_t workspace_bytes, nvfp4_stream_t stream) {
  return gemm_impl(a, b, nullptr, 0, m, n, k, d, out_dtype, workspace, workspace_bytes, stream,
                   false);
}

nvfp4_status nvfp4_grouped_gemm_workspace_size(int64_t rows, int64_t n, int64_t k,
                                               int32_t num_groups, uint64_t* bytes) {
  if (bytes == nullptr) return fail(NVFP4_ERR_INVALID, "bytes is NULL");
  nvfp4_status st;
  if ((st = check_sizes(rows, n)) != NVFP4_OK) return st;
  if ((st = check_sizes(k, 0)) != NVFP4_OK) return st;
  if (num_groups < 1 || num_groups > 4096)
    return fail(NVFP4_ERR_INVALID, "num_groups must be in [1, 4096]");
  *bytes = (rows == 0 || n == 0 || k == 0)
               ? 0
               : (uint64_t)gemm_layout(rows, n, k, (int64_t)num_groups * n).workspace_bytes;
  return NVFP4_OK;
}

nvfp4_status nvfp4_grouped_gemm(const nvfp4_operand* a, const nvfp4_operand* b,
                                const int64_t* group_ends, int32_t num_groups, int64_t rows,
                                int64_t n, int64_t k, void* d, int32_t out_dtype, void* workspace,
                                uint64_t workspace_bytes, nvfp4_stream_t stream) {
  if (group_ends == nullptr) return fail(NVFP4_ERR_INVALID, "group_ends is NULL");
  if (num_groups < 1 || num_groups > 4096)
    return fail(NVFP4_ERR_INVALID, "num_groups must be in [1, 4096]");
  return gemm_impl(a, b, group_ends, num_groups, rows, n, k, d, out_dtype, workspace,
                   workspace_bytes, stream, false);
}

nvfp4_status nvfp4_grouped_gemm_wgrad(const nvfp4_operand* a, const nvfp4_operand* b,
                                      const int64_t* group_ends, int32_t num_groups, int64_t m,
                                      int64_t n, int64_t tokens, void* d, int32_t out_dtype,
                                      void* workspace, uint64_t workspace_bytes,
                                      nvfp4_stream_t stream) {
  if (group_ends == nullptr) return fail(NVFP4_ERR_INVALID, "group_ends is NULL");
  if (num_groups < 1 || num_groups > 4096)
    return fail(NVFP4_ERR_INVALID, "num_groups must be in [1, 4096]");
  return gemm_impl(a, b, group_ends, num_groups, m, n, tokens, d, out_dtype, workspace,
                   workspace_bytes, stream, false, true);
}

nvfp4_status nvfp4_gemm_static_ws(const nvfp4_operand* a, const nvfp4_operand* b, int64_t m,
                                  int64_t n, int64_t k, void* d, int32_t out_dtype,
                                  nvfp4_stream_t stream) {
  return gemm_impl(a, b, nullptr, 0, m, n, k, d, out_dtype, nullptr, 0, stream, true);
}

nvfp4_status nvfp4_grouped_amax(const void* x, int32_t in_dtype, int64_t rows, int64_t cols,
                                const int64_t* group_ends, int32_t num_groups, float* group_amax,
                                float* row_amax_expanded, const float* noop,
                                nvfp4_stream_t stream) {
  nvfp4_status st;
  if (!valid_in_dtype(in_dtype)) return fail(NVFP4_ERR_INVALID, "unknown in_dtype");
  if ((st = check_sizes(rows, cols)) != NVFP4_OK) return st;
  if (num_groups < 1 || num_groups > 4096)
    return fail(NVFP4_ERR_INVALID, "num_groups must be in [1, 4096]");
  if (group_ends == nullptr || group_amax == nullptr)
    return fail(NVFP4_ERR_INVALID, "group_ends and group_amax must be non-NULL");
  if (x == nullptr && rows * cols > 0) return fail(NVFP4_ERR_INVALID, "x is NULL");
  DeviceInfo dev;
  if ((st = current_device(&dev)) != NVFP4_OK) return st;
  GroupCheckArgs g{};
  g.M = rows;
  g.group_ends = group_ends;
  g.num_groups = num_groups;
  g.noop = noop;
  g.prep.zero_ptr[0] = group_amax;
  g.prep.zero_n[0] = num_groups;
  g.prep.noop = noop;
  const InType in = in_dtype == NVFP4_IN_BF16 ? InType::BF16 : InType::FP32;
  if (row_amax_expanded) {
    // With a per-row output to work in: the row maxima from the tiled amax pass,
    // then each group's maximum over its rows, written back to its rows.
    g.prep.zero_ptr[1] = row_amax_expanded;
    g.prep.zero_n[1] = rows;
    cudaError_t e = launch_group_check(g, dev, stream, false);
    if (e != cudaSuccess) return cuda_fail(e, "group check launch");
    AmaxArgs am{};
    am.x = x;
    am.in = in;
    am.M = rows;
    am.K = cols;
    am.row_amax = row_amax_expanded;
    am.noop = noop;
    am.group_ends = group_ends;
    am.num_groups = num_groups;
    if ((e = launch_amax(am, dev, stream)) != cudaSuccess) return cuda_fail(e, "amax launch");
    GroupReduceArgs r{};
    r.group_ends = group_ends;
    r.num_groups = num_groups;
    r.M = rows;
    r.row_max = row_amax_expanded;
    r.group_amax = group_amax;
    r.noop = noop;
    r.expand = 1;
    if ((e = launch_group_reduce(r, dev, stream)) != cudaSuccess)
      return cuda_fail(e, "group reduce launch");
    return NVFP4_OK;
  }
  cudaError_t e = launch_group_check(g, dev, stream, false);
  if (e != cudaSuccess) return cuda_fail(e, "group check launch");
  GroupedAmaxArgs a{};
  a.x = x;
  a.in = in;
  a.M = rows;
  a.K = cols;
  a.group_ends = group_ends;
  a.num_groups = num_groups;
  a.group_amax = group_amax;
  a.noop = noop;
  if ((e = launch_grouped_amax(a, dev, stream)) != cudaSuccess)
    return cuda_fail(e, "grouped amax launch");
  if (row_amax_expanded) {
    g.prep = PrepArgs{};
    g.group_amax = group_amax;
    g.expand = row_amax_expanded;
    if ((e = launch_group_check(g, dev, stream, true)) != cudaSuccess)
      return cuda_fail(e, "group expand launch");
  }
  return NVFP4_OK;
}

nvfp4_status nvfp4_grouped_quantize_rowwise(const void* x, int32_t in_dtype, int64_t rows,
                                            int64_t cols, const int64_t* group_ends,
                                            int32_t num_groups, const nvfp4_config* cfg,
                                            const nvfp4_out* row, float* group_amax,
                                            const float* noop, nvfp4_stream_t stream) {
  nvfp4_status st;
  if ((st = check_config(cfg)) != NVFP4_OK) return st;
  if (cfg->block_2d) return fail(NVFP4_ERR_INVALID, "grouped quantize uses 1x16 blocks");
  if (row == nullptr) return fail(NVFP4_ERR_INVALID, "row is NULL");
  if (row->amax_in != nullptr)
    return fail(NVFP4_ERR_INVALID, "grouped quantize computes its amax: row->amax_in must be NULL");
  if (num_groups < 1 || num_groups > 4096)
    return fail(NVFP4_ERR_INVALID, "num_groups must be in [1, 4096]");
  if (group_ends == nullptr) return fail(NVFP4_ERR_INVALID, "group_ends is NULL");
  if (cfg->mode == NVFP4_PER_TENSOR && group_amax == nullptr)
    return fail(NVFP4_ERR_INVALID, "group_amax is required with NVFP4_PER_TENSOR");
  nvfp4_config rcfg = *cfg;
  rcfg.mode = NVFP4_ROW_SCALED;
  if (cfg->mode == NVFP4_ROW_SCALED) {
    if (group_amax) {
      st = nvfp4_grouped_amax(x, in_dtype, rows, cols, group_ends, num_groups, group_amax,
                              nullptr, noop, stream);
      if (st != NVFP4_OK) return st;
    }
    return quantize_impl(x, in_dtype, rows, cols, &rcfg, row, nullptr, noop, stream, group_ends,
                         num_groups);
  }
  st = nvfp4_grouped_amax(x, in_dtype, rows, cols, group_ends, num_groups, group_amax, row->amax,
                          noop, stream);
  if (st != NVFP4_OK) return st;
  nvfp4_out r = *row;
  r.amax_in = row->amax;  // the expanded per-row amax is already in place
  return quantize_impl(x, in_dtype, rows, cols, &rcfg, &r, nullptr, noop, stream, group_ends,
                       num_groups);
}

nvfp4_status nvfp4_grouped_quantize_rowwise_padded(
    const void* x, int32_t in_dtype, int64_t tokens, int64_t cols, const int64_t* ragged_ends,
    const int64_t* padded_ends, int32_t num_groups, int64_t padded_rows, const nvfp4_config* cfg,
    const nvfp4_out* row, float* group_amax, const float* noop, nvfp4_stream_t stream) {
  nvfp4_status st;
  if (!valid_in_dtype(in_dtype)) return fail(NVFP4_ERR_INVALID, "unknown in_dtype");
  if ((st = check_sizes(tokens, cols)) != NVFP4_OK) return st;
  if ((st = check_sizes(padded_rows, cols)) != NVFP4_OK) return st;
  if ((st = check_config(cfg)) != NVFP4_OK) return st;
  if (cfg->mode != NVFP4_PER_TENSOR)
    return fail(NVFP4_ERR_UNSUPPORTED,
                "padded grouped quantize uses each group's amax (cfg->mode NVFP4_PER_TENSOR)");
  if (num_groups < 1 || num_groups > 4096)
    return fail(NVFP4_ERR_INVALID, "num_groups must be in [1, 4096]");
  if (ragged_ends == nullptr || padded_ends == nullptr || group_amax == nullptr)
    return fail(NVFP4_ERR_INVALID, "ragged_ends, padded_ends and group_amax must be non-NULL");
  if (row == nullptr) return fail(NVFP4_ERR_INVALID, "row is NULL");
  if (row->amax_in != nullptr)
    return fail(NVFP4_ERR_INVALID, "grouped quantize computes its amax: row->amax_in must be NULL");
  if ((st = check_out(row, "row", padded_rows, cols, padded_rows)) != NVFP4_OK) return st;
  if (x == nullptr && tokens * cols > 0) return fail(NVFP4_ERR_INVALID, "x is NULL");
  DeviceInfo dev;
  if ((st = current_device(&dev)) != NVFP4_OK) return st;
  const InType in = in_dtype == NVFP4_IN_BF16 ? InType::BF16 : InType::FP32;
  // 1. both layouts valid?  zero the group maxima
  GroupCheckArgs g{};
  g.M = padded_rows;
  g.group_ends = padded_ends;
  g.num_groups = num_groups;
  g.noop = noop;
  g.rag_ends = ragged_ends;
  g.in_rows = tokens;
  g.prep.zero_ptr[0] = group_amax;
  g.prep.zero_n[0] = num_groups;
  // row->amax [padded_rows >= tokens] holds the ragged rows' maxima until step 3
  g.prep.zero_ptr[1] = row->amax;
  g.prep.zero_n[1] = tokens;
  g.prep.noop = noop;
  cudaError_t e = launch_group_check(g, dev, stream, false);
  if (e != cudaSuccess) return cuda_fail(e, "group check launch");
  // 2. group maxima over the ragged rows: the tiled row amax pass, then each
  //    group's max over its rows
  AmaxArgs am{};
  am.x = x;
  am.in = in;
  am.M = tokens;
  am.K = cols;
  am.row_amax = row->amax;
  am.noop = noop;
  am.group_ends = ragged_ends;
  am.num_groups = num_groups;
  am.pad_ends = padded_ends;
  am.pad_rows = padded_rows;
  if ((e = launch_amax(am, dev, stream)) != cudaSuccess) return cuda_fail(e, "amax launch");
  GroupReduceArgs rd{};
  rd.group_ends = ragged_ends;
  rd.num_groups = num_groups;
  rd.M = tokens;
  rd.row_max = row->amax;
  rd.group_amax = group_amax;
  rd.noop = noop;
  rd.expand = 0;
  rd.pad_ends = padded_ends;
  rd.pad_rows = padded_rows;
  if ((e = launch_group_reduce(rd, dev, stream)) != cudaSuccess)
    return cuda_fail(e, "group reduce launch");
  // 3. every padded row (padding included) takes its group's amax
  g.prep = PrepArgs{};
  g.group_amax = group_amax;
  g.expand = row->amax;
  if ((e = launch_group_check(g, dev, stream, true)) != cudaSuccess)
    return cuda_fail(e, "group expand launch");
  // 4. rowwise encode of the padded rows, reading only the ragged rows of x
  QuantArgs q{};
  q.x = x;
  q.in = in;
  q.M = padded_rows;
  q.K = cols;
  q.row_scaled = true;
  q.four_over_six = cfg->four_over_six != 0;
  q.block_2d = false;
  q.bound = cfg->bound;
  q.noop = noop;
  q.num_groups = num_groups;
  q.row_codes = row->codes;
  q.row_scales = row->scales;
  q.row_amax = row->amax;
  q.pad_ends = padded_ends;
  q.rag_ends = ragged_ends;
  q.in_rows = tokens;
  if ((e = launch_quantize(q, dev, stream)) != cudaSuccess) return cuda_fail(e, "quantize");
  return NVFP4_OK;
}

namespace {
// The grouped columnwise quantize, of x or (rht) of its transform.
nvfp4_status grouped_columnwise_impl(const void* x, int32_t in_dtype, int64_t rows, int64_t cols,
                                     const int64_t* group_ends, int32_t num_groups,
                                     const nvfp4_config* cfg, const nvfp4_out* col,
                                     const float* noop, nvfp4_stream_t stream, bool rht,
                                     uint32_t sign_mask) {
  nvfp4_status st;
  if (rht && (st = check_rht(x, in_dtype, rows, cols, sign_mask)) != NVFP4_OK) return st;
  if (!valid_in_dtype(in_dtype)) return fail(NVFP4_ERR_INVALID, "unknown in_dtype");
  if ((st = check_sizes(rows, cols)) != NVFP4_OK) return st;
  if ((st = check_config(cfg)) != NVFP4_OK) return st;
  if (cfg->block_2d) return fail(NVFP4_ERR_INVALID, "grouped quantize uses 1x16 blocks");
  if (num_groups < 1 || num_groups > 4096)
    return fail(NVFP4_ERR_INVALID, "num_groups must be in [1, 4096]");
  if (group_ends == nullptr) return fail(NVFP4_ERR_INVALID, "group_ends is NULL");
  const bool rs = cfg->mode == NVFP4_ROW_SCALED;
  const int64_t namax = rs ? (int64_t)num_groups * cols : num_groups;
  if ((st = check_out(col, "col", cols, rows, namax)) != NVFP4_OK) return st;
  if (x == nullptr && rows * cols > 0) return fail(NVFP4_ERR_INVALID, "x is NULL");
  const int elem = in_dtype == NVFP4_IN_BF16 ? 2 : 4;
  if (rows * cols > 0 &&
      ((cols * elem) % 16 != 0 || reinterpret_cast<uintptr_t>(x) % 16 != 0))
    return fail(NVFP4_ERR_UNSUPPORTED,
                "grouped columnwise quantize needs 16-byte aligned rows of x (TMA tiles)");
  DeviceInfo dev;
  if ((st = current_device(&dev)) != NVFP4_OK) return st;
  const InType in = in_dtype == NVFP4_IN_BF16 ? InType::BF16 : InType::FP32;
  // validate the ends (whole 128-row tiles) and clear (or copy in) the maxima
  GroupCheckArgs g{};
  g.M = rows;
  g.group_ends = group_ends;
  g.num_groups = num_groups;
  g.noop = noop;
  g.tile_aligned = true;
  g.prep.noop = noop;
  if (col->amax_in == nullptr) {
    g.prep.zero_ptr[0] = col->amax;
    g.prep.zero_n[0] = namax;
  } else if (col->amax_in != col->amax) {
    g.prep.copy_dst[0] = col->amax;
    g.prep.copy_src[0] = col->amax_in;
    g.prep.copy_n[0] = namax;
  }
  cudaError_t e = launch_group_check(g, dev, stream, false);
  if (e != cudaSuccess) return cuda_fail(e, "group check launch");
  if (col->amax_in == nullptr && rht) {
    // each group's column maxima (or maximum) of the transform, read-only
    RhtAmaxArgs ra{x, in == InType::BF16, rows, cols, sign_mask, rs ? col->amax : nullptr,
                   rs ? nullptr : col->amax, noop};
    ra.group_ends = group_ends;
    ra.num_groups = num_groups;
    if ((e = launch_rht16_amax(ra, dev, stream)) != cudaSuccess)
      return cuda_fail(e, "transform amax launch");
  } else if (col->amax_in == nullptr) {
    if (rs) {
      // each group's column maxima: the TMA amax pass publishing per group
      AmaxArgs am{};
      am.x = x;
      am.in = in;
      am.M = rows;
      am.K = cols;
      am.col_amax = col->amax;
      am.noop = noop;
      am.group_ends = group_ends;
      am.num_groups = num_groups;
      am.col_grouped = true;
      if ((e = launch_amax(am, dev, stream)) != cudaSuccess)
        return cuda_fail(e, "amax launch");
    } else {
      GroupedAmaxArgs ga{};
      ga.x = x;
      ga.in = in;
      ga.M = rows;
      ga.K = cols;
      ga.group_ends = group_ends;
      ga.num_groups = num_groups;
      ga.group_amax = col->amax;
      ga.noop = noop;
      ga.tile_aligned = true;
      if ((e = launch_grouped_amax(ga, dev, stream)) != cudaSuccess)
        return cuda_fail(e, "grouped amax launch");
    }
  }
  QuantArgs q{};
  q.x = x;
  q.in = in;
  q.M = rows;
  q.K = cols;
  q.row_scaled = true;  // the producer stages each tile's column scales from its group's amax
  q.four_over_six = cfg->four_over_six != 0;
  q.block_2d = false;
  q.bound = cfg->bound;
  q.noop = noop;
  q.col_codes = col->codes;
  q.col_scales = col->scales;
  q.col_amax = col->amax;
  q.group_ends = group_ends;
  q.num_groups = num_groups;
  q.col_grouped = true;
  q.col_grouped_per_tensor = !rs;
  q.rht = rht;
  q.rht_mask = sign_mask;
  if ((e = launch_quantize(q, dev, stream)) != cudaSuccess) return cuda_fail(e, "quantize");
  return NVFP4_OK;
}
}  // namespace

nvfp4_status nvfp4_grouped_quantize_columnwise(const void* x, int32_t in_dtype, int64_t rows,
                                               int64_t cols, const int64_t* group_ends,
                                               int32_t num_groups, const nvfp4_config* cfg,
                                               const nvfp4_out* col, const float* noop,
                                               nvfp4_stream_t stream) {
  return grouped_columnwise_impl(x, in_dtype, rows, cols, group_ends, num_groups, cfg, col, noop,
                                 stream, false, 0);
}

nvfp4_status nvfp4_grouped_quantize_columnwise_rht(const void* x, int32_t in_dtype, int64_t rows,
                                                   int64_t cols, const int64_t* group_ends,
                                                   int32_t num_groups, uint32_t sign_mask,
                                                   const nvfp4_config* cfg, const nvfp4_out* col,
                                                   const float* noop, nvfp4_stream_t stream) {
  return grouped_columnwise_impl(x, in_dtype, rows, cols, group_ends, num_groups, cfg, col, noop,
                                 stream, true, sign_mask);
}

const char* nvfp4_last_error(void) { return g_last_error.c_str(); }

nvfp4_status nvfp4_device_status(int32_t* status, int32_t reset) {
  if (status == nullptr) return fail(NVFP4_ERR_INVALID, "status is NULL");
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  int v = 0;
  if ((e = cudaMemcpyFromSymbol(&v, g_status_word, sizeof(int))) != cudaSuccess)
    return cuda_fail(e, "read status word");
  *status = v;
  if (reset) {
    const int zero = 0;
    if ((e = cudaMemcpyToSymbol(g_status_word, &zero, sizeof(int))) != cudaSuccess)
      return cuda_fail(e, "reset status word");
  }
  if (v & NVFP4_DEVICE_TIMEOUT)
    return fail(NVFP4_ERR_TIMEOUT, "a kernel gave up a bounded wait; its outputs are incomplete");
  return NVFP4_OK;
}

nvfp4_status nvfp4_selftest_scale_division(const float* S, int64_t n, float* e_out,
                                          nvfp4_stream_t stream) {
  if (n < 0) return fail(NVFP4_ERR_INVALID, "n must be >= 0");
  if (n > (int64_t(1) << 40)) return fail(NVFP4_ERR_INVALID, "n too large");
  if (n > 0 && (S == nullptr || e_out == nullptr))
    return fail(NVFP4_ERR_INVALID, "S and e_out must be non-NULL");
  cudaError_t e = launch_selftest_scale_division(S, n, e_out, stream);
  if (e != cudaSuccess) return cuda_fail(e, "selftest launch");
  return NVFP4_OK;
}

nvfp4_status nvfp4_selftest_wait_timeout(int64_t limit_ns, uint32_t* out, nvfp4_stream_t stream) {
  if (limit_ns < 0 || limit_ns > 1000000000LL)
    return fail(NVFP4_ERR_INVALID, "limit_ns must lie in [0, 1e9]");
  if (out == nullptr) return fail(NVFP4_ERR_INVALID, "out is NULL");
  DeviceInfo dev;
  nvfp4_status st = current_device(&dev);
  if (st != NVFP4_OK) return st;
  cudaError_t e = launch_selftest_wait_timeout((uint64_t)limit_ns, out, dev, stream);
  if (e != cudaSuccess) return cuda_fail(e, "selftest launch");
  return NVFP4_OK;
}

nvfp4_status nvfp4_selftest_convert(const float* in, int64_t n, uint8_t* e2m1_out,
                                    uint8_t* e4m3_out, nvfp4_stream_t stream) {
  if (n < 0) return fail(NVFP4_ERR_INVALID, "n must be >= 0");
  if (n > 0 && (in == nullptr || (e2m1_out == nullptr && e4m3_out == nullptr)))
    return fail(NVFP4_ERR_INVALID, "in and one output must be non-NULL");
  cudaError_t e = launch_selftest_convert(in, n, e2m1_out, e4m3_out, stream);
  if (e != cudaSuccess) return cuda_fail(e, "selftest launch");
  return NVFP4_OK;
}

}  // extern "C"
