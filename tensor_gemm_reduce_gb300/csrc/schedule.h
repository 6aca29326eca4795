// schedule.h -- tile order of the over-decomposed GEMM and of the reduce units.
//
// Over-decomposition and tile-coordinate swizzling follow the FLUX page
// (abstract: split communication and computation into fine-grained pieces and
// fuse them into one kernel; TL;DR: tile coordinate swizzling), applied to the
// row-parallel layer of the problem page "A fused GEMM + reduce-scatter kernel
// hiding 90% of communication on 8 H100 GPUs" ("What is asked": split into
// tiles, send each when done).
//
// Work is indexed by an order position.  The output is cut into regions of
// BM x BN (128 x 256) elements; each region has 8 rank tiles (one per virtual
// rank), placed next to each other in the order (rank innermost) so the 8
// partials of one region are produced at the same time and its reduction can
// start while later regions are still being multiplied.  Regions are ordered
// in horizontal bands of `band` tile rows; inside a band the order walks down
// a column of regions before moving right, so the band's rows of A stay in L2
// while each column block of W is read once per band.
//
// Shared by host code (tests, plan) and device code.
#pragma once
#include <stdint.h>

#if defined(__CUDACC__)
#define GRS_HD __host__ __device__ __forceinline__
#else
#define GRS_HD inline
#endif

namespace grs {

constexpr int kWorld = 8;
constexpr int kBM = 128;  // rows of a tile (MMA M)
constexpr int kBN = 256;  // columns of a tile (MMA N)
constexpr int kBK = 64;   // K per pipeline stage (one 128-byte swizzle row of bf16)

struct Region {
  int mt, nt;
};

// Region at order position p (0 <= p < mt_count*nt_count).  The plan keeps
// every tile count below 2^30, so the divisions are 32-bit (a 64-bit division
// is a long software routine on the GPU, paid once per tile by the threads
// that walk the order).
GRS_HD Region region_at(int64_t p, int mt_count, int nt_count, int band) {
  const uint32_t band_regions = (uint32_t)band * (uint32_t)nt_count;
  const uint32_t pp = (uint32_t)p;
  const uint32_t b = pp / band_regions;
  const uint32_t rem = pp - b * band_regions;
  const int mt0 = (int)b * band;
  const int h = (mt_count - mt0) < band ? (mt_count - mt0) : band;  // last band may be short
  const uint32_t q = rem / (uint32_t)h;
  Region r;
  r.nt = (int)q;
  r.mt = mt0 + (int)(rem - q * (uint32_t)h);
  return r;
}

struct TileCoord {
  int rank, mt, nt;
  int half;  // -1: the whole tile; 0 / 1: its left / right half (columns [0, 128) / [128, 256))
};

// Optionally the last regions of the order are computed in half-width tiles
// (2 per rank tile, so 16 per region): a final wave of tiles half as long
// halves the spread of the CTAs' finishing times and the last tile's
// epilogue, after which only the last regions' reduction is left.
// Rank tiles before region half_region: 8 per region, ranks 0..7; from
// half_region on: 16 per region, the left halves of ranks 0..7, then the
// right halves.  Tile count of an order with `regions` regions:
GRS_HD int64_t tiles_of(int64_t regions, int64_t half_region) {
  return (int64_t)kWorld * half_region + 2 * (int64_t)kWorld * (regions - half_region);
}

// Rank tile at order position idx (0 <= idx < tiles_of(mt_count*nt_count, half_region)).
GRS_HD TileCoord tile_at(int64_t idx, int mt_count, int nt_count, int band, int64_t half_region) {
  static_assert(kWorld == 8, "rank = low 3 bits of the order position");
  const uint32_t i = (uint32_t)idx;
  const uint32_t full = (uint32_t)kWorld * (uint32_t)half_region;
  uint32_t g;
  TileCoord t;
  if (i < full) {
    g = i >> 3;
    t.rank = (int)(i & 7u);
    t.half = -1;
  } else {
    const uint32_t q = i - full;
    g = (uint32_t)half_region + (q >> 4);
    t.half = (int)((q >> 3) & 1u);
    t.rank = (int)(q & 7u);
  }
  const Region r = region_at(g, mt_count, nt_count, band);
  t.mt = r.mt;
  t.nt = r.nt;
  return t;
}

// First region in half-width tiles for a request of `half_regions` regions
// (0 or negative: none), clamped to the regions there are.  None is the
// default: measured with 1 to 9 half-width regions, the shorter final wave
// did not pay for the half-width tiles' lower throughput (they load 24 KiB
// per 256-cycle k-step instead of 32 KiB per 512) on o_proj-sized shapes.
GRS_HD int64_t half_region_of(int64_t regions, int half_regions) {
  const int64_t want = half_regions < 0 ? 0 : half_regions;
  return want >= regions ? 0 : regions - want;
}

// AllGather + GEMM (mKernel page, section 4: the local shard first, then
// the other shards, in the order they arrive).  Ranks one after the other
// (one rank's gathered A and its column shard of W are what L2 keeps);
// inside a rank, the tile rows are taken from the first tile row of its own
// shard onwards (wrapping around), in bands of `band` tile rows whose column
// tiles are walked band by band as in region_at.  The copies bring rank r the
// shards (r + 1) mod 8, (r + 2) mod 8, ... in the same order.
GRS_HD TileCoord ag_tile_at(int64_t idx, int mt_count, int nt_count, int shard_rows,
                            int tile_rows, int band) {
  const uint32_t per_rank = (uint32_t)mt_count * (uint32_t)nt_count;
  TileCoord t;
  t.half = -1;
  t.rank = (int)((uint32_t)idx / per_rank);
  const Region g = region_at((uint32_t)idx - (uint32_t)t.rank * per_rank, mt_count, nt_count, band);
  const int start = (int)(((uint32_t)t.rank * (uint32_t)shard_rows) / (uint32_t)tile_rows);
  const int mt = start + g.mt;
  t.mt = mt >= mt_count ? mt - mt_count : mt;
  t.nt = g.nt;
  return t;
}

// Automatic band height, in tile rows of tile_rows output rows: keep the
// band's rows of A (all ranks, full K) at or under ~32 MiB of the 126 MiB L2,
// and no taller than the output.
GRS_HD int auto_band(int64_t M, int64_t K, int tile_rows = kBM) {
  const int64_t mt_count = (M + tile_rows - 1) / tile_rows;
  const int64_t per_tile_row = (int64_t)tile_rows * K * 2;  // bytes of A per band row
  int64_t b = per_tile_row > 0 ? ((int64_t)32 << 20) / per_tile_row : mt_count;
  if (b < 1) b = 1;
  if (b > mt_count) b = mt_count;
  if (b < 1) b = 1;
  return (int)b;
}

}  // namespace grs
