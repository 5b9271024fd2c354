// internal.h -- host-side launch interface between the C ABI (api.cu) and the
// kernel translation units.  Not installed; not part of the ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace nvfp4 {

enum class InType : int { BF16 = 0, FP32 = 1 };

struct DeviceInfo {
  int device;
  int num_sms;
  int64_t l2_bytes;  // the device's L2 size
  int* status;  // device address of the library status word
  uint8_t* gemm_static_ws;  // device address of the static GEMM workspace
};

// Zero up to four float arrays and copy up to two (dst <- src), unless noop.
struct PrepArgs {
  float* zero_ptr[4];
  int64_t zero_n[4];
  float* copy_dst[2];
  const float* copy_src[2];
  int64_t copy_n[2];
  const float* noop;
};
cudaError_t launch_prep(const PrepArgs& a, const DeviceInfo& dev, cudaStream_t stream);

// Fused exact amax over x [M][K].  Outputs must be zeroed first (launch_prep)
// unless they are NULL.  Maxima are published with atomicMax on the FP32 bit
// pattern (valid for non-negative values).
struct AmaxArgs {
  const void* x;
  InType in;
  int64_t M, K;
  float* row_amax;     // [M] or NULL
  float* col_amax;     // [K] or NULL
  float* tensor_amax;  // [1] or NULL
  const float* noop;
  const int64_t* group_ends;  // optional: do nothing unless these group ends are valid
  int num_groups;
  const int64_t* pad_ends;  // optional, with group_ends: and this padded layout of them
  int64_t pad_rows;
  // grouped columns (TMA path): col_amax is [num_groups][K], each group's column maxima;
  // the group ends must be multiples of 128
  bool col_grouped;
};
cudaError_t launch_amax(const AmaxArgs& a, const DeviceInfo& dev, cudaStream_t stream);

// Grouped amax: group_amax[g] = max over rows of group g (must be zeroed first).
struct GroupedAmaxArgs {
  const void* x;
  InType in;
  int64_t M, K;
  const int64_t* group_ends;
  int num_groups;
  float* group_amax;
  const float* noop;
  const int64_t* pad_ends;  // optional: do nothing unless this padded layout is valid too
  int64_t pad_rows;
  bool tile_aligned;  // also require every group end to be a multiple of 128
};
cudaError_t launch_grouped_amax(const GroupedAmaxArgs& a, const DeviceInfo& dev,
                                cudaStream_t stream);

// Validates group ends (sets the status word and returns early if invalid),
// then performs `prep` (zero / copy) and, in the expand pass, writes
// expand[r] = group_amax[group of r].
struct GroupCheckArgs {
  int64_t M;
  const int64_t* group_ends;
  int num_groups;
  const float* group_amax;
  float* expand;
  const float* noop;
  PrepArgs prep;
  // optional: group_ends are padded ends of ragged x (ragged ends rag_ends, in_rows rows)
  const int64_t* rag_ends;
  int64_t in_rows;
  bool tile_aligned;  // also require every group end to be a multiple of 128
};
cudaError_t launch_group_check(const GroupCheckArgs& a, const DeviceInfo& dev,
                               cudaStream_t stream, bool expand_pass);

// Group maxima from per-row maxima (row_max [M], computed before), optionally
// written back to every row of the group.  Writes nothing unless the ends are valid.
struct GroupReduceArgs {
  const int64_t* group_ends;
  int num_groups;
  int64_t M;
  float* row_max;
  float* group_amax;
  const float* noop;
  int expand;
  const int64_t* pad_ends;  // optional: also require this padded layout of the groups
  int64_t pad_rows;
};
cudaError_t launch_group_reduce(const GroupReduceArgs& a, const DeviceInfo& dev,
                                cudaStream_t stream);

// Tile quantize of x [M][K] into the rowwise and/or columnwise outputs.
struct QuantArgs {
  const void* x;
  InType in;
  int64_t M, K;
  bool row_scaled;
  bool four_over_six;
  bool block_2d;
  float bound;
  // rowwise output (codes == NULL to skip)
  uint8_t* row_codes;
  uint8_t* row_scales;
  const float* row_amax;  // [M] or [1] (read)
  // columnwise output (codes == NULL to skip)
  uint8_t* col_codes;
  uint8_t* col_scales;
  const float* col_amax;  // [K] or [1] (read)
  // per-tensor: copy *copy_src to *copy_dst once (the second direction's amax)
  float* copy_dst;
  const float* copy_src;
  const float* noop;
  const int64_t* group_ends;  // optional: do nothing unless these group ends are valid
  int num_groups;
  // optional: x is ragged (in_rows rows) and the output padded: group g's output rows
  // [pad_ends[g-1], pad_ends[g]) take x rows from rag_ends[g-1] on (rowwise only)
  const int64_t* pad_ends;
  const int64_t* rag_ends;
  int64_t in_rows;
  // optional, columnwise only: each group (ends multiples of 128) is quantized with its
  // own amax -- col_amax [num_groups][K] (per column) or [num_groups] (per tensor)
  bool col_grouped;
  bool col_grouped_per_tensor;
  // optional, columnwise only (1x16 blocks): each 16-row block of a column is
  // replaced by its random Hadamard transform with this sign mask before encoding
  bool rht;
  uint32_t rht_mask;
  // walk each CTA's tiles the other way (a second pass over x then starts on the tiles
  // that the first one read last, still in L2)
  bool reverse_walk;
};
cudaError_t launch_quantize(const QuantArgs& a, const DeviceInfo& dev, cudaStream_t stream);

struct DequantArgs {
  const uint8_t* codes;
  const uint8_t* scales;
  const float* amax;
  bool row_scaled;
  int64_t rows, cols;
  float bound;
  void* out;
  bool out_bf16;
};
cudaError_t launch_dequantize(const DequantArgs& a, const DeviceInfo& dev, cudaStream_t stream);

cudaError_t launch_selftest_convert(const float* in, int64_t n, uint8_t* e2m1, uint8_t* e4m3,
                                    cudaStream_t stream);
cudaError_t launch_selftest_scale_division(const float* S, int64_t n, float* e,
                                           cudaStream_t stream);
cudaError_t launch_selftest_wait_timeout(uint64_t limit_ns, uint32_t* out, const DeviceInfo& dev,
                                         cudaStream_t stream);

// GEMM consumer of two NVFP4 operands (kernels_gemm.cu): D [M][N] = A [M][K] x B [N][K]^T
// on the dequantized values, K-major codes [lines][K/2] and compact scales [lines][K/16].
// Random Hadamard transform of x along its rows, per column and per 16-row block,
// into the FP32 y (kernels_rht.cu); rows a multiple of 16.
struct RhtArgs {
  const void* x;
  bool bf16;
  int64_t rows, cols;
  uint32_t sign_mask;
  float* y;
  const float* noop;
};
cudaError_t launch_rht16(const RhtArgs& a, const DeviceInfo& dev, cudaStream_t stream);
// Exact amax of the transformed x (never written): col_amax [cols] and / or
// tensor_amax [1], accumulated by atomic max into zeroed buffers.
struct RhtAmaxArgs {
  const void* x;
  bool bf16;
  int64_t rows, cols;
  uint32_t sign_mask;
  float* col_amax;
  float* tensor_amax;
  const float* noop;
  // optional grouped rows (ends multiples of 128): col_amax [G][cols] or tensor_amax [G]
  const int64_t* group_ends = nullptr;
  int num_groups = 0;
};
cudaError_t launch_rht16_amax(const RhtAmaxArgs& a, const DeviceInfo& dev, cudaStream_t stream);
// The transform's column maxima (a.col_amax / a.tensor_amax) and x's row maxima
// (row_max [rows] or row_tensor [1]) in one read of x; for column counts whose
// thread groups fill whole CTAs (rht16_amax_rows_supported), no group ends.
bool rht16_amax_rows_supported(const void* x, bool bf16, int64_t cols);
cudaError_t launch_rht16_amax_rows(const RhtAmaxArgs& a, float* row_max, float* row_tensor,
                                   const DeviceInfo& dev, cudaStream_t stream);

struct GemmArgs {
  const uint8_t* a_codes;
  const uint8_t* a_scales;
  const float* a_amax;  // [M] (a_row_scaled) or [1]
  bool a_row_scaled;
  float a_bound;
  const uint8_t* b_codes;
  const uint8_t* b_scales;
  const float* b_amax;  // [N] or [1]
  bool b_row_scaled;
  float b_bound;
  int64_t M, N, K;  // M, N >= 1; K >= 32 and a multiple of 32
  void* d;
  bool d_bf16;
  uint8_t* workspace;  // >= gemm_layout(M, N, K, b_lines).workspace_bytes, 256-byte aligned
  // grouped GEMM (NULL otherwise): A's rows in num_groups groups ending at group_ends
  // (device, multiples of 128); group g multiplies B's rows [g*N, (g+1)*N), N a
  // multiple of 256; b_amax [num_groups*N] (row-scaled) or [num_groups]
  const int64_t* group_ends;
  int num_groups;
  // with group_ends: false -- groups of A's rows (per-expert fprop); true -- groups of
  // K (tokens, ends multiples of 256): group g writes d + g*M*N from its K range,
  // a_amax [num_groups*M] or [num_groups], b_amax [num_groups*N] or [num_groups]
  bool k_grouped;
};
struct GemmLayout {
  int64_t k_tiles, tiles_m, tiles_n;
  int64_t sfa_bytes, sfb_bytes, sfb_offset, workspace_bytes;
};
// b_lines: rows of B (N, or num_groups * N for the grouped GEMM)
GemmLayout gemm_layout(int64_t M, int64_t N, int64_t K, int64_t b_lines);
cudaError_t launch_gemm(const GemmArgs& a, const DeviceInfo& dev, cudaStream_t stream);

// Grid size shared by the TMA amax and encode kernels (same tile -> CTA mapping).
int pipe_grid_size(int64_t num_tiles, int num_sms);

// Host helpers (api.cu): encode 2D tiled tensor maps; false if TMA cannot be used.
bool make_tile_map(CUtensorMap* map, const void* base, InType in, int64_t rows, int64_t cols,
                   int box_cols, int box_rows);
// K-major code matrix [rows][pitch] read by the GEMM: box of box_bytes (128 or 64) x
// box_rows, the swizzle of that width (128B / 64B), zero fill outside the matrix
bool make_operand_map(CUtensorMap* map, const void* base, int64_t rows, int64_t pitch,
                      int box_bytes, int box_rows);
// byte matrix [rows][pitch] (an output of codes), box of box_bytes x box_rows
bool make_byte_map(CUtensorMap* map, const void* base, int64_t rows, int64_t pitch,
                   int box_bytes, int box_rows);

}  // namespace nvfp4
