// tile_pipeline.cuh -- tile geometry, work split and the producer/consumer
// plumbing shared by the TMA amax kernel and the encode kernel.
//
// A tile is 128 rows x 256 bytes of x (128 BF16 or 64 FP32 columns), loaded as
// two 128-row x 128-byte TMA boxes with the 128-byte swizzle.  Tiles are numbered
// in super-strips of kGroup tile columns: inside a super-strip, row tile tm, then
// the kGroup tiles of that row (so one CTA writes the 4 x 8 scale bytes that make
// up a 32-byte sector of a rowwise scale row within 4 consecutive tiles).  The
// numbering is cut into G contiguous, equal chunks, one per CTA.  The amax kernel
// walks each chunk one way and the encode kernel, launched with the same G, the
// other way, so each CTA starts on the tiles its twin in the amax grid loaded
// last, which are still in L2.  Even and odd CTAs walk in opposite directions so
// that the two CTAs on either side of a chunk boundary reach it at about the same
// time (they share the scale sectors there).
#pragma once

#include "device_common.cuh"

namespace nvfp4 {

constexpr int kTileRows = 128;
constexpr int kBoxBytes = 128 * 128;        // one box: 128 rows x 128 bytes
constexpr int kTileBytes = 2 * kBoxBytes;   // two boxes side by side
constexpr int kStages = 3;                  // shared-memory ring depth
constexpr int kConsumerWarps = 8;
constexpr int kPipeThreads = (kConsumerWarps + 1) * 32;  // + one producer warp

template <typename T>
struct TileGeo {
  static constexpr int ELEM = sizeof(T);
  static constexpr int BOXC = 128 / ELEM;  // columns per box
  static constexpr int TILEC = 2 * BOXC;   // columns per tile
};

struct TileGrid {
  static constexpr int kGroup = 4;  // tile columns per super-strip
  int tiles_m, tiles_n, num_tiles;

  // contiguous chunk [begin, end) of the tile order for CTA `cta`
  __device__ __forceinline__ void chunk(int cta, int G, int& begin, int& end) const {
    begin = (int)(((long long)cta * num_tiles) / G);
    end = (int)(((long long)(cta + 1) * num_tiles) / G);
  }
  __device__ __forceinline__ void coords(int L, int& tm, int& tn) const {
    const int per_ss = tiles_m * kGroup;
    const int ss = L / per_ss;
    const int rem = L - ss * per_ss;
    const int wdt = (tiles_n - ss * kGroup) < kGroup ? (tiles_n - ss * kGroup) : kGroup;
    tm = rem / wdt;
    tn = ss * kGroup + (rem - tm * wdt);
  }
  // k-th tile of a chunk walked forwards (fwd) or backwards
  __device__ __forceinline__ int walk(int begin, int end, int k, bool fwd) const {
    return fwd ? begin + k : end - 1 - k;
  }
};

// A position in the tile order that moves one tile at a time without integer
// divisions: row tile tm, super-strip ss, tile jt inside the super-strip row, and
// that row's width wdt (kGroup, or less in the last super-strip).
struct TileCursor {
  int tm, ss, jt, wdt;
  __device__ __forceinline__ int tn() const { return ss * TileGrid::kGroup + jt; }

  __device__ __forceinline__ void seek(const TileGrid& g, int L) {
    const int per_ss = g.tiles_m * TileGrid::kGroup;
    ss = L / per_ss;
    const int rem = L - ss * per_ss;
    wdt = min(TileGrid::kGroup, g.tiles_n - ss * TileGrid::kGroup);
    tm = rem / wdt;
    jt = rem - tm * wdt;
  }
  // the next tile of the order (fwd) or the previous one
  __device__ __forceinline__ void step(const TileGrid& g, bool fwd) {
    if (fwd) {
      if (++jt < wdt) return;
      jt = 0;
      if (++tm < g.tiles_m) return;
      tm = 0;
      ++ss;
      wdt = min(TileGrid::kGroup, g.tiles_n - ss * TileGrid::kGroup);
    } else {
      if (jt > 0) {
        --jt;
      } else if (tm > 0) {
        --tm;
        jt = wdt - 1;
      } else {
        --ss;
        wdt = min(TileGrid::kGroup, g.tiles_n - ss * TileGrid::kGroup);
        tm = g.tiles_m - 1;
        jt = wdt - 1;
      }
    }
  }
};

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Programmatic dependent launch: wait for the preceding grid's results /
// allow the next grid to start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Barrier among the consumer warps only (named barrier 1).
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}

// Issue the two TMA boxes of tile (tm, tn) into `dst`, completing on `bar`; the
// tile's rows start at x row src_row0 (tm * kTileRows unless x is ragged).
template <typename T>
__device__ __forceinline__ void issue_tile(uint8_t* dst, const CUtensorMap* map, uint64_t* bar,
                                           int src_row0, int tn, uint64_t policy) {
  using G = TileGeo<T>;
  mbar_expect_tx(bar, kTileBytes);
  tma_load_2d(dst, map, bar, tn * G::TILEC, src_row0, policy);
  tma_load_2d(dst + kBoxBytes, map, bar, tn * G::TILEC + G::BOXC, src_row0, policy);
}

// Byte offset of element (r, c) of a tile in its stage buffer: the 16-byte
// chunk index inside each 128-byte row is XORed with r mod 8 (128-byte swizzle).
template <typename T>
__device__ __forceinline__ uint32_t swz_off(int r, int c) {
  constexpr int BOXC = TileGeo<T>::BOXC;
  const int box = c / BOXC;
  const int byte = (c % BOXC) * (int)sizeof(T);
  return box * kBoxBytes + r * 128 + ((((byte >> 4) ^ (r & 7))) << 4) + (byte & 15);
}

// Fallback when x cannot be described by a tensor map (rows not 16-byte aligned):
// the 32 lanes of the producer warp copy the tile with plain loads into the same
// swizzled layout.  Tile row r comes from x row src_row0 + r for r < nvalid and is
// zero otherwise (zero outside the matrix too).
template <typename T>
__device__ __forceinline__ void plain_load_tile(uint8_t* dst, const T* x, int64_t K,
                                                int64_t src_row0, int nvalid, int tn, int lane) {
  using G = TileGeo<T>;
  for (int idx = lane; idx < kTileRows * G::TILEC; idx += 32) {
    const int r = idx / G::TILEC, c = idx % G::TILEC;
    const int64_t gc = (int64_t)tn * G::TILEC + c;
    T v = T(0);
    if (r < nvalid && gc < K) v = x[(src_row0 + r) * K + gc];
    *reinterpret_cast<T*>(dst + swz_off<T>(r, c)) = v;
  }
}

}  // namespace nvfp4
