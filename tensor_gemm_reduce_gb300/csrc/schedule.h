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

// Region at order position p (0 <= p < mt_count*nt_count).
GRS_HD Region region_at(int64_t p, int mt_count, int nt_count, int band) {
  const int64_t band_regions = (int64_t)band * nt_count;
  const int64_t b = p / band_regions;
  const int64_t rem = p - b * band_regions;
  const int mt0 = (int)(b * band);
  const int h = (mt_count - mt0) < band ? (mt_count - mt0) : band;  // last band may be short
  Region r;
  r.nt = (int)(rem / h);
  r.mt = mt0 + (int)(rem % h);
  return r;
}

struct TileCoord {
  int rank, mt, nt;
};

// Rank tile at order position idx (0 <= idx < 8*mt_count*nt_count).
GRS_HD TileCoord tile_at(int64_t idx, int mt_count, int nt_count, int band) {
  const Region g = region_at(idx / kWorld, mt_count, nt_count, band);
  TileCoord t;
  t.rank = (int)(idx % kWorld);
  t.mt = g.mt;
  t.nt = g.nt;
  return t;
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
  const int64_t per_rank = (int64_t)mt_count * nt_count;
  TileCoord t;
  t.rank = (int)(idx / per_rank);
  const Region g = region_at(idx - t.rank * per_rank, mt_count, nt_count, band);
  const int start = (int)(((int64_t)t.rank * shard_rows) / tile_rows);
  t.mt = (int)((start + g.mt) % mt_count);
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
