// kernels.cuh -- the device side: the fused GEMM + reduce-scatter (also
// all-reduce), the fused all-gather + GEMM, and the standalone kernels of the
// unfused paths.
//
// Problem page "A fused GEMM + reduce-scatter kernel hiding 90% of
// communication on 8 H100 GPUs": "What is asked" (partials summed across the
// 8 ranks, each rank keeps one slice), the step list (split into tiles, send
// each when done, one fused kernel overlaps both jobs) and "Bottlenecks" #1
// (tile completion signals and remote writes through low-overhead flags,
// without slowing the GEMM).  FLUX page, TL;DR: reduce-scatter as a GEMM
// epilogue.  mKernel page, abstract and section 3.2: a persistent kernel whose
// SMs (here: warps) take compute and communication roles, and blocks that run
// out of compute work help with communication.
//
// One persistent CTA per SM; with kPair = 2 the CTAs of a 2-CTA cluster (two
// SMs) share each MMA: a 256 x 256 tile, rows split between the CTAs (128
// each, in each CTA's TMEM), B's columns split between their shared memories.
// Warp roles (per CTA):
//   warp 0        A loader: its CTA's rows of A_r, one k-block per stage of
//                 the smem ring (and, in the cluster's first CTA, the tile
//                 claims published to the tile ring)
//   warp 1        MMA issuer (the pair's first CTA only): tcgen05.mma
//                 (bf16 in, fp32 in TMEM, two 256-column accumulators);
//                 TMEM allocation in every CTA
//   W loader      one warp after the epilogue warps (warp 9 from 3
//                 communication warps on): its CTA's columns of W_r for the
//                 same stages; a stage is full once both loaders' copies landed
//   warps 2..5    epilogue: TMEM -> registers (one row per lane) -> bf16
//                 (RNE) -> the warp's 32 x 64 block written into a shared
//                 buffer in the 128-byte swizzle -> one TMA store of the
//                 block into the rank's staging region; then
//                 (fused kernel) each warp publishes its 32 rows with a release
//                 add on the 128-row block's completion count (8 ranks x 4
//                 warps = 32 adds per block and run)
//   the others    reducers (fused reduce-scatter): take the next reduce item
//                 in the order the tiles complete (one atomic ticket), wait
//                 (acquire) until its block's count is complete, add the 8
//                 bf16 partials in fp32 in rank order, write bf16 output (to
//                 every rank's copy for the all-reduce).  The epilogue warps,
//                 both loaders and the MMA issuer join them when the CTA's
//                 tiles are done (fused o_proj -0.3%, 2048 x 6144 x 6144 -2.7%,
//                 512 x 8192 x 28672 -2...4%); optionally a
//                 controller sets how many of them take items (adaptive share).
//                 In the fused all-gather the same warps are copy warps that
//                 gather A's row shards into each rank's buffer, and the
//                 A loader waits for a shard's copies before loading its rows.
// Every wait is bounded by p.timeout_ns; on expiry the kernel records an error
// word, stops its loops, lets its in-flight copies land, frees TMEM and returns.
#pragma once
#include "ptx.cuh"
#include "schedule.h"

namespace grs {

// What a launch of gemm_rs_kernel does besides the tile GEMM.
enum Kind : int {
  kKindGemm = 0,  // only the GEMM (unfused paths)
  kKindRS = 1,    // + completion publication and reducer warps (fused reduce-scatter)
  kKindAG = 2,    // + copy warps gathering A's row shards (fused all-gather + GEMM)
};

constexpr int kEpiWarps = 4;
constexpr int kTmemCols = 2 * kBN;      // two fp32 accumulators of 256 columns
constexpr int kGemmWarps = 2 + kEpiWarps;
constexpr int kMaxReducerWarps = 5;

// Warp roles: 0 loads A (and claims the tiles in the cluster's first CTA),
// 1 issues the MMAs, 2-5 run the epilogue; then one warp loads W and the
// communication warps (reducers or copy warps) follow.  The operand loads are
// split over two threads because one thread issuing both operands' copies
// could not keep up with the tensor pipe: a 64-wide K step is 512 tensor
// cycles, and the single loader spent ~365 cycles of it blocked in its TMA
// issues plus its waits and bookkeeping (GEMM alone, o_proj: 713 cycles per
// K step with one loader, 625 with two).  Warp w runs on the SM
// sub-partition w % 4; a reducer beside the MMA warp (warp 1) slows the MMA
// stream it shares issue slots with (no-load fused runs: 167 cycles per
// 256x256x16 MMA with a reducer on that sub-partition, 153 without), so from
// 3 communication warps on the W loader, which mostly waits, takes warp 9.
__host__ __device__ constexpr int w_loader_warp(int comm_warps) {
  return kGemmWarps + (comm_warps >= 3 ? 3 : comm_warps);
}
__host__ __device__ constexpr int cta_warps(int comm_warps) { return kGemmWarps + 1 + comm_warps; }

// Epilogue buffers: each epilogue warp stages 32 rows x 64 columns of bf16
// (4 KiB, 128-byte swizzle) in shared memory for a TMA store, two buffers
// per warp so one can fill while the other's store reads it.
constexpr int kEpiBufBytes = 32 * 64 * 2;
constexpr int kEpiSmem = kEpiWarps * 2 * kEpiBufBytes;

// Shared-memory plan of one CTA.  kCtas = CTAs of the cluster that share a
// tile: 1 (one-CTA MMA) or 2 (one 2-CTA MMA).  Every CTA loads its own
// operands; no load is shared between CTAs.  6 operand stages of 32 KiB (4 of
// 48 KiB with one CTA) and 32 KiB of epilogue buffers.  Fewer stages in
// flight also queue less in front of the reducers' loads (fused o_proj: 7
// stages 206 us, 6 stages 203 us).
template <int kKind, int kCtas>
struct TileCfg {
  static_assert(kCtas == 1 || kCtas == 2, "one CTA or a CTA pair per tile");
  static constexpr int kPair = kCtas;                  // CTAs per MMA
  static constexpr int kStages = kCtas == 1 ? 4 : 6;
  static constexpr int kTileRows = kBM * kCtas;        // output rows of one cluster tile
  static constexpr int kBCols = kBN / kPair;           // W columns held by one CTA
  static constexpr int kBBoxes = kBCols / 64;          // 64-column TMA boxes per stage
  static constexpr int kBBoxBytes = kBK * 64 * 2;      // 8 KiB: 64 k-rows x 64 n, N-major
  static constexpr int kAStage = kBM * kBK * 2;        // 16 KiB: 128 rows x 64 k, K-major
  static constexpr int kBStage = kBK * kBCols * 2;     // 32 KiB (one CTA) / 16 KiB (pair)
  static constexpr int kStage = kAStage + kBStage;     // bytes one CTA loads per stage
  static constexpr int kSmemA = 0;
  static constexpr int kSmemB = kSmemA + kStages * kAStage;
  static constexpr int kSmemEpi = kSmemB + kStages * kBStage;  // 1024-byte aligned
  static constexpr int kSmemBar = kSmemEpi + kEpiSmem;
  // full[S], empty[S], acc_full[2], acc_empty[2], drain, tile ring full[4], empty[4]
  static constexpr int kNumBars = 2 * kStages + 5 + 2 * 4;
  static constexpr int kSmemMisc = kSmemBar + kNumBars * 8;
  // tmem addr, abort, items reduced, pad, ring slots[4]
  static constexpr int kSmemBytes = kSmemMisc + 16 + 4 * 4;
  static constexpr int kSmemAlloc = kSmemBytes + 1024;  // slack to align the base to 1024 bytes
  static_assert(kSmemAlloc <= 232448, "shared memory per CTA");
};

// control words in the workspace
enum CtrlWord : int {
  kCtrlReduced = 0,  // reduce items finished in this run (checked by the last CTA)
  kCtrlQueueTail = 7,  // unused (kept zero)
  kCtrlQueueHead = 8,  // next reduce item to take (a position in the item order)
  kCtrlDone = 1,     // CTAs finished (the last one resets the words above and below)
  kCtrlAbort = 2,    // set when some warp gave up waiting
  kCtrlError = 3,    // error bits (kErr*), cleared by the host
  kCtrlErrWhere = 4, // which wait gave up
  kCtrlErrWhat = 5,  // region / tile index of that wait
  kCtrlTileTicket = 6, // next GEMM tile to claim
  kCtrlCopyTicket = 9, // next all-gather copy item to take
  kCtrlTarget = 10,    // adaptive: reducer warps per CTA that take items (0 = all)
  kCtrlCount = 16
};
// Every control word, completion count and item stamp slot sits in its own part of
// a cache line, so atomics and polls on one do not queue behind another's.
constexpr int kCtrlStride = 32;   // words: one 128-byte line per control word
constexpr int kCtrlWords = kCtrlCount * kCtrlStride;
constexpr int kFlagStride = 32;   // words: one 128-byte line per block count
constexpr int kQueueStride = 4;   // 8-byte words per item's debug stamps (one 32-byte sector)
enum ErrBits : uint32_t { kErrFlagTimeout = 1u, kErrPipeTimeout = 2u, kErrIncomplete = 4u };
enum ErrWhere : uint32_t {
  kWhereTma = 1, kWhereMma = 2, kWhereEpi = 3, kWhereReducer = 4, kWhereShard = 5, kWhereRing = 6
};

struct GemmParams {
  CUtensorMap tmap_a;   // A  [8][M][Kr] : dims {Kr, M, 8}, box {64, 128, 1}
  CUtensorMap tmap_b;   // W  [8][Kr][N] : dims {N, Kr, 8}, box {64, 64, 1}
  // Epilogue stores: the staging [8][M][N] (all-gather: the output
  // [8][M][N/8]) : dims {N, M, 8}, box {64, 32, 1}, 128-byte swizzle.
  CUtensorMap tmap_s;
  // All-gather + GEMM (kKindAG): tmap_a covers the input's row shards
  // [8][M/8][K] (dims {K, M/8, 8}), tmap_g the gather buffers [8][M][K]
  // (dims {K, M, 8}; rank r's copy of every shard).  Kr is then the full K and
  // N the rank's N/8 columns.
  CUtensorMap tmap_g;
  // W again as 4-D {64 columns, rows, column blocks of 64, 8 ranks}, box {64,
  // 64, columns per CTA / 64, 1}: a CTA's whole stage of W in one copy
  // instead of one per 64-column block.  Set (w4 = 1) when the W rows hold a
  // whole number of 64-column blocks.
  CUtensorMap tmap_w4;
  int w4;
  const uint16_t* ag_src;  // input row shards, [8][M/8][K]
  uint16_t* gather;        // gather buffers, [8][M][K]
  uint32_t* ag_flags;      // copied chunks of shard s in rank r's buffer: ag_flags[(r*8+s)*kFlagStride]
  uint32_t ag_target;      // chunks per shard x fused all-gather runs so far
  int shard_rows;          // M / 8
  int ag_direct;           // own shard read from the input (shard_rows % tile_rows == 0)
  int chunks_per_shard;
  int first_round;         // 1 when the own shards are not copied
  int ag_order;            // tiles in the all-gather order (ag_tile_at), also when unfused
  long long copy_items;    // copy items of a run
  long long copy_chunk;    // elements per copy item
  int copy_paced;          // copy rank r's shards only once rank r - 1's tiles are claimed
  uint16_t* stage;   // rank r's partial of output element (i, j): stage[r * plane + i * N + j]
  long long plane;   // elements from one rank's staging region to the next
  uint16_t* out;
  int replicas;          // copies of the output: 1 (reduce-scatter) or 8 (all-reduce)
  long long out_stride;  // elements from one output copy to the next
  // Completion count per 128-row block of the output (a region's blocks are
  // consecutive, one per CTA of the pair): each of the 4 epilogue warps of
  // every rank's tile adds 1 per fused run, so a run's target is
  // 32 * (runs so far) and the add that reaches it completes the block.
  uint32_t* flags;
  uint32_t* ctrl;   // kCtrlWords words (kCtrlCount words, kCtrlStride apart)
  int M, N, Kr;
  int mt_count, nt_count, band;  // mt_count and band count tile rows of kTileRows rows
  int num_kb;
  int unit_rows;          // rows per reduce item: 8, 16 or 32
  int splits;             // reduce items per 128-row block (128 / unit_rows)
  int blocks_per_region;  // tile_rows / 128
  // Reduce items are taken in the order the regions complete (the tile order
  // of schedule.h, region after region).  Regions from order position
  // tail_region on are completed by the last waves of tiles: their blocks are
  // cut into 4-row items so the reduction after the last tile is spread over
  // many warps.  Item positions: tail_region * blocks_per_region * splits
  // unit_rows-row items, then 32 4-row items per block of the tail regions.
  int tail_region;
  // Regions from order position half_region on are computed in half-width
  // tiles (tile_at); each of their blocks then receives 64 release adds per
  // run instead of 32.  The number of regions if none.
  int half_region;
  long long num_tiles;
  long long num_items;    // reduce items of a run
  // Debug stamps of each item (GEMM_RS_DEBUG_TRACE only), kQueueStride words
  // per item position: (epoch << 32) | item, queued, taken, done.
  unsigned long long* queue;
  uint32_t epoch;         // fused runs on this workspace so far, this one included
  uint32_t flag_target;
  uint32_t debug_flags;
  // Fused kernel only: staging tiles are stored with an L2 evict-last hint so
  // they are still in L2 when reduced, and each reduced staging line is
  // discarded from L2 (never written back).  Needs N % 64 == 0 and a staging
  // base on a 128-byte boundary, so that no 128-byte line holds data of two
  // reduce units.
  uint32_t staging_in_l2;
  // Adaptive reducer share (mKernel page, section 3.2): a controller thread
  // publishes how many of each CTA's reducer warps take items; the others wait.
  int adaptive;
  int reducer_warps;
  int tile_rows;  // rows of a region: 128 (one CTA per MMA) or 256 (a CTA pair)
  unsigned long long timeout_ns;
  // Debug timeline (null unless asked for): per CTA, global-timer stamps
  // [start, epilogue done with its tiles, MMA issue drained, last warp done].
  unsigned long long* trace;
};
constexpr int kTraceWords = 4;
constexpr int kMaxTraceCtas = 1024;

// ---------------------------------------------------------------------------

__device__ __forceinline__ void record_error(const GemmParams& p, uint32_t bit, uint32_t where,
                                             uint32_t what) {
  atomicOr(p.ctrl + kCtrlError * kCtrlStride, bit);
  atomicExch(p.ctrl + kCtrlErrWhere * kCtrlStride, where);
  atomicExch(p.ctrl + kCtrlErrWhat * kCtrlStride, what);
  atomicExch(p.ctrl + kCtrlAbort * kCtrlStride, 1u);
}

// Bounded mbarrier wait; false if the limit passed or the CTA is aborting.
// kCluster: acquire at cluster scope (arrivals come from the peer CTA).
template <bool kCluster = false>
__device__ __forceinline__ bool bar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                         volatile uint32_t* cta_abort) {
  auto probe = [&]() {
    return kCluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
  };
  if (probe()) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 128; ++i)
      if (probe()) return true;
    if (*cta_abort) return false;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

// Sum of the 8 rank partials for 8 consecutive bf16 elements (16 bytes), in
// fp32, rank order 0..7, rounded to bf16.
__device__ __forceinline__ uint4 reduce8(const uint4 (&v)[kWorld]) {
  float a[8];
  a[0] = bf16lo_to_f32(v[0].x); a[1] = bf16hi_to_f32(v[0].x);
  a[2] = bf16lo_to_f32(v[0].y); a[3] = bf16hi_to_f32(v[0].y);
  a[4] = bf16lo_to_f32(v[0].z); a[5] = bf16hi_to_f32(v[0].z);
  a[6] = bf16lo_to_f32(v[0].w); a[7] = bf16hi_to_f32(v[0].w);
#pragma unroll
  for (int r = 1; r < kWorld; ++r) {
    a[0] = __fadd_rn(a[0], bf16lo_to_f32(v[r].x)); a[1] = __fadd_rn(a[1], bf16hi_to_f32(v[r].x));
    a[2] = __fadd_rn(a[2], bf16lo_to_f32(v[r].y)); a[3] = __fadd_rn(a[3], bf16hi_to_f32(v[r].y));
    a[4] = __fadd_rn(a[4], bf16lo_to_f32(v[r].z)); a[5] = __fadd_rn(a[5], bf16hi_to_f32(v[r].z));
    a[6] = __fadd_rn(a[6], bf16lo_to_f32(v[r].w)); a[7] = __fadd_rn(a[7], bf16hi_to_f32(v[r].w));
  }
  uint4 o;
  o.x = pack_bf16x2(a[0], a[1]);
  o.y = pack_bf16x2(a[2], a[3]);
  o.z = pack_bf16x2(a[4], a[5]);
  o.w = pack_bf16x2(a[6], a[7]);
  return o;
}

// A reduce item: rows [row_begin, row_begin + rows) of a 128-row block.
struct Item {
  int block;  // 128-row block: (physical region) * blocks_per_region + CTA of the pair
  int part;   // which rows of the block
  int rows;   // unit_rows, or 4 in the tail regions
  int g;      // the region's position in the order
};

// Release adds a block receives per run: 8 ranks x 4 epilogue warps, twice
// that in the regions computed in half-width tiles.
__device__ __forceinline__ uint32_t adds_per_run(const GemmParams& p, long long g) {
  return (uint32_t)(kWorld * kEpiWarps) * (g >= p.half_region ? 2u : 1u);
}

// The item at order position pos (0 <= pos < num_items): regions in the order
// the tiles complete them (tile_at's region order), each region's blocks in
// turn, each block's parts in turn.
__device__ __forceinline__ Item item_at(const GemmParams& p, long long pos) {
  const long long per_region = (long long)p.blocks_per_region * p.splits;
  const long long tail_start = (long long)p.tail_region * per_region;
  long long g, r;
  int per_block;
  Item it;
  if (pos < tail_start) {
    g = pos / per_region;
    r = pos - g * per_region;
    per_block = p.splits;
    it.rows = p.unit_rows;
  } else {
    const long long q = pos - tail_start;
    const long long per_tail_region = (long long)p.blocks_per_region * (kBM / 4);
    g = p.tail_region + q / per_tail_region;
    r = q - (g - p.tail_region) * per_tail_region;
    per_block = kBM / 4;
    it.rows = 4;
  }
  const Region reg = region_at(g, p.mt_count, p.nt_count, p.band);
  it.g = (int)g;
  it.block = (reg.mt * p.nt_count + reg.nt) * p.blocks_per_region + (int)(r / per_block);
  it.part = (int)(r % per_block);
  return it;
}

// First order position of a block's items, and how many it has (the inverse
// of item_at; used only to stamp the debug timeline).
__device__ __forceinline__ long long first_item_of(const GemmParams& p, int block, int* count,
                                                   long long* g_out) {
  const int phys = block / p.blocks_per_region;
  const int rb = block - phys * p.blocks_per_region;
  const int mt = phys / p.nt_count, nt = phys - (phys / p.nt_count) * p.nt_count;
  const int b = mt / p.band, mt0 = b * p.band;
  const int h = (p.mt_count - mt0) < p.band ? (p.mt_count - mt0) : p.band;
  const long long g = (long long)b * p.band * p.nt_count + (long long)nt * h + (mt - mt0);
  *g_out = g;
  const long long per_region = (long long)p.blocks_per_region * p.splits;
  if (g < p.tail_region) {
    *count = p.splits;
    return g * per_region + (long long)rb * p.splits;
  }
  *count = kBM / 4;
  return (long long)p.tail_region * per_region +
         (g - p.tail_region) * p.blocks_per_region * (kBM / 4) + (long long)rb * (kBM / 4);
}

// Take the next item position and wait until its block is complete (all 32
// release adds of this run): 1 with *it and *pos set, 0 when every item of
// the run is taken, -1 if the wait gave up.  Lane 0 polls with acquire loads
// (the reducers read the staging through L2 only, so the L1 invalidation of
// an acquire costs nothing); the warp barrier after the successful poll
// orders every lane's staging loads after lane 0's acquire, and so after the
// releases that completed the block.
__device__ __forceinline__ int item_pop(const GemmParams& p, int lane, Item* it, long long* pos_out) {
  uint32_t pos = 0;
  if (lane == 0) pos = atomicAdd(p.ctrl + kCtrlQueueHead * kCtrlStride, 1u);
  pos = __shfl_sync(0xffffffffu, pos, 0);
  if ((long long)pos >= p.num_items) return 0;
  *it = item_at(p, pos);
  *pos_out = pos;
  const uint32_t* cnt = p.flags + (size_t)it->block * kFlagStride;
  const uint32_t target = adds_per_run(p, it->g) * p.epoch;  // this run's adds, counted since clearing
  uint64_t t0 = 0;
  if (lane == 0) t0 = globaltimer_ns();
  uint32_t sleep_ns = 32;
  while (true) {
    int ready = 0;
    if (lane == 0) ready = (int)(ld_acquire_gpu(cnt) - target) >= 0;
    if (__shfl_sync(0xffffffffu, ready, 0)) {
      __syncwarp();
      return 1;
    }
    int give_up = 0;
    if (lane == 0)
      give_up = (globaltimer_ns() - t0 > p.timeout_ns) || ld_volatile_u32(p.ctrl + kCtrlAbort * kCtrlStride);
    if (__shfl_sync(0xffffffffu, give_up, 0)) return -1;
    __nanosleep(sleep_ns);
    sleep_ns = sleep_ns < 256 ? sleep_ns * 2 : 256;
  }
}

// Rows [row, row + R) of one reduce item: 8R loads of 16 bytes in flight per
// lane, then the rank-order sums and the stores.
template <int R>
__device__ __forceinline__ void reduce_rows(const GemmParams& p, size_t plane, int row, int col,
                                            bool active, bool drop, int lane, int col0) {
  const size_t off = (size_t)row * p.N + col;
  if (active) {
    uint4 v[R][kWorld];
#pragma unroll
    for (int i = 0; i < R; ++i)
#pragma unroll
      for (int r = 0; r < kWorld; ++r)
        v[i][r] = __ldcg(reinterpret_cast<const uint4*>(p.stage + r * plane + off + (size_t)i * p.N));
#pragma unroll
    for (int i = 0; i < R; ++i) {
      const uint4 o = reduce8(v[i]);
#pragma unroll 1
      for (int c = 0; c < p.replicas; ++c)  // all-reduce: every rank's copy
        *reinterpret_cast<uint4*>(p.out + (size_t)c * p.out_stride + off + (size_t)i * p.N) = o;
    }
  }
  if (p.staging_in_l2) {
    __syncwarp();  // every lane has consumed its loads (its stores depend on them)
    // R rows x 8 ranks x 4 lines of 128 bytes: spread over the 32 lanes (R
    // lines each) rather than issued by the 4 lanes that start a line, which
    // serialised 8 * R discards on each of them
    if (drop) {
#pragma unroll
      for (int i = 0; i < R; ++i) {
        const int line = lane + 32 * i;       // (rank, row, 128-byte segment) of the R rows
        const int seg = line & 3, r = (line >> 2) & 7, ri = line >> 5;
        if (col0 + seg * 64 < p.N)
          discard_l2_line(p.stage + r * plane + (size_t)(row + ri) * p.N + col0 + seg * 64);
      }
    }
  }
}

// Reduce one item of a completed 128-row block (lane l covers columns
// [8l, 8l+8) of the block's 256).  With p.staging_in_l2 the staging lines
// just read are dropped from L2.
__device__ __forceinline__ void reduce_item(const GemmParams& p, const Item& it, int lane) {
  const size_t plane = (size_t)p.plane;
  const int region = it.block / p.blocks_per_region;
  const int rb = it.block - region * p.blocks_per_region;
  const int mt = region / p.nt_count;
  const int nt = region - mt * p.nt_count;
  const int rows = it.rows;
  const int row_begin = mt * p.tile_rows + rb * kBM + it.part * rows;
  if (row_begin >= p.M) return;  // rows of a ragged last tile that do not exist
  int row_end = row_begin + rows;
  if (row_end > p.M) row_end = p.M;
  const int col0 = nt * kBN;
  const int col = col0 + lane * 8;
  const bool active = col < p.N;
  const bool drop = p.staging_in_l2;
  int row = row_begin;
#pragma unroll 1
  for (; row + 3 < row_end; row += 4) reduce_rows<4>(p, plane, row, col, active, drop, lane, col0);
  if (row + 1 < row_end) {
    reduce_rows<2>(p, plane, row, col, active, drop, lane, col0);
    row += 2;
  }
  if (row < row_end) reduce_rows<1>(p, plane, row, col, active, drop, lane, col0);
}

// Adaptive reducer share (mKernel page, section 3.2: a controller estimates
// the roles' costs from cycle counters and sets the number of communication
// workers so that the predicted completion times are equal).  Run by one
// thread (CTA 0's first reducer warp) after each of its items: with tau its
// own cycles per item (moving average), rate the tiles claimed per cycle
// (moving average of the ticket's advance), W the items not yet taken and T
// the tiles not yet claimed, the reduction keeps pace with the GEMM if each
// CTA runs w >= W * tau * rate / (grid * T) reducer warps; one more is added
// as margin, and all of them once every tile is claimed.
struct Controller {
  float tau = 0.f, rate = 0.f;
  long long last_clock = 0;
  uint32_t last_ticket = 0;
  __device__ void update(const GemmParams& p, long long item_cycles) {
    const long long now = clock64();
    const uint32_t ticket = ld_volatile_u32(p.ctrl + kCtrlTileTicket * kCtrlStride);
    const uint32_t head = ld_volatile_u32(p.ctrl + kCtrlQueueHead * kCtrlStride);
    tau = tau == 0.f ? (float)item_cycles : 0.8f * tau + 0.2f * (float)item_cycles;
    if (last_clock != 0 && now > last_clock && ticket >= last_ticket) {
      const float r = (float)(ticket - last_ticket) / (float)(now - last_clock);
      rate = rate == 0.f ? r : 0.8f * rate + 0.2f * r;
    }
    last_clock = now;
    last_ticket = ticket;
    const long long tiles_left = p.num_tiles - (long long)ticket;
    int w = p.reducer_warps;
    if (tiles_left > 0 && rate > 0.f) {
      const float items_left = (float)(p.num_items - (long long)head);
      const float need = items_left * tau * rate / ((float)gridDim.x * (float)tiles_left);
      w = (int)ceilf(need) + 1;
      if (w < 1) w = 1;
      if (w > p.reducer_warps) w = p.reducer_warps;
    }
    atomicExch(p.ctrl + kCtrlTarget * kCtrlStride, (uint32_t)w);
  }
};

// A reducer warp above the published share waits here (bounded): false once
// every item is taken or the run is aborting, so the warp can stop.
__device__ __forceinline__ bool wait_for_share(const GemmParams& p, int my_idx, int lane) {
  int go = 1;
  if (lane == 0) {
    const uint64_t t0 = globaltimer_ns();
    while (true) {
      const uint32_t target = ld_volatile_u32(p.ctrl + kCtrlTarget * kCtrlStride);
      if (target == 0 || my_idx < (int)target) break;
      if ((long long)ld_volatile_u32(p.ctrl + kCtrlQueueHead * kCtrlStride) >= p.num_items ||
          ld_volatile_u32(p.ctrl + kCtrlAbort * kCtrlStride) || globaltimer_ns() - t0 > p.timeout_ns) {
        go = 0;
        break;
      }
      __nanosleep(1000);
    }
  }
  return __shfl_sync(0xffffffffu, go, 0) != 0;
}

// Reducer role: take item positions until every item of the run is taken.
// Items done are counted in the CTA's shared counter (added to the run's
// total once, when the CTA ends).  my_idx: the warp's index among the CTA's
// reducer warps (-1 for epilogue warps that joined: never held back).
__device__ __noinline__ void reducer_loop(const GemmParams& p, int lane, uint32_t* cta_reduced,
                                          int my_idx) {
  const bool controller = p.adaptive && my_idx == 0 && blockIdx.x == 0 && lane == 0;
  Controller ctl;
  while (true) {
    if (p.adaptive && my_idx > 0 && !wait_for_share(p, my_idx, lane)) break;
    Item it;
    long long pos = 0;
    const int got = item_pop(p, lane, &it, &pos);
    if (got == 0) break;
    if (got < 0) {
      if (lane == 0 && !ld_volatile_u32(p.ctrl + kCtrlAbort * kCtrlStride))
        record_error(p, kErrFlagTimeout, kWhereReducer, (uint32_t)it.block);
      break;
    }
    const long long c0 = controller ? clock64() : 0;
    const uint64_t t_take = (p.trace && lane == 0) ? globaltimer_ns() : 0;
    reduce_item(p, it, lane);
    __syncwarp();
    if (lane == 0) atomicAdd(cta_reduced, 1u);
    if (controller) ctl.update(p, clock64() - c0);
    if (p.trace && lane == 0) {  // debug timeline: item, taken, done (words 0, 2 and 3)
      unsigned long long* slot = p.queue + (size_t)pos * kQueueStride;
      st_relaxed_gpu_u64(slot, ((uint64_t)p.epoch << 32) | (uint32_t)((it.block << 5) | it.part));
      st_relaxed_gpu_u64(slot + 2, t_take);
      st_relaxed_gpu_u64(slot + 3, globaltimer_ns());
    }
  }
}

// One epilogue warp's 32 rows of a rank tile are stored (and ordered before
// this thread by __syncwarp): count them with a release add on the 128-row
// block's completion count.  The add returns nothing, so the warp does not
// wait for a reply; the reducers poll the count.  With the debug timeline the
// add returns the old count, and the add that completes the block stamps the
// time its items became ready.
__device__ __forceinline__ void publish_rows(const GemmParams& p, int block, bool skip) {
  if (skip) return;  // debug: this completion never arrives
  uint32_t* cnt = p.flags + (size_t)block * kFlagStride;
  if (!p.trace) {
    red_release_gpu_add(cnt, 1u);
    return;
  }
  int n = 0;
  long long g = 0;
  const long long first = first_item_of(p, block, &n, &g);
  if (atom_add_release_gpu(cnt, 1u) == adds_per_run(p, g) * p.epoch - 1u) {
    const uint64_t now = globaltimer_ns();
    for (int i = 0; i < n; ++i) st_relaxed_gpu_u64(p.queue + (size_t)(first + i) * kQueueStride + 1, now);
  }
}

// ---------------------------------------------------------------------------
// All-gather role (kKindAG): copy warps take copy items from one atomic
// ticket, in order, rank after rank like the tiles: with R = 8 - first_round
// rounds per rank, item i is rank r = i / (R * chunks), round k = (i / chunks)
// mod R + first_round, chunk c: chunk c of shard (r + k) mod 8 into rank r's
// gather buffer.
// Copies depend on nothing, so every item is taken by some running warp.
// After an item, lane 0 publishes it with a release add on (r, s)'s count.
__device__ __noinline__ void copy_loop(const GemmParams& p, int lane) {
  const long long shard_elems = (long long)p.shard_rows * p.Kr;
  const long long per_rank = (long long)(kWorld - p.first_round) * p.chunks_per_shard;
  while (true) {
    uint32_t i = 0;
    if (lane == 0) i = atomicAdd(p.ctrl + kCtrlCopyTicket * kCtrlStride, 1u);
    i = __shfl_sync(0xffffffffu, i, 0);
    if ((long long)i >= p.copy_items) break;
    const int r = (int)(i / per_rank);
    if (p.copy_paced && r > 1) {
      // Paced copies: rank r's shards are written only once the GEMM has begun
      // claiming rank r - 1's tiles, so they are still in L2 when rank r's
      // tiles read them (copied all at once, the 8 buffers outgrow L2 and are
      // read back from DRAM).  Bounded; a late copy only delays its tiles.
      if (lane == 0) {
        const long long need = (long long)(r - 1) * p.mt_count * p.nt_count;
        const uint64_t t0 = globaltimer_ns();
        while ((long long)ld_volatile_u32(p.ctrl + kCtrlTileTicket * kCtrlStride) < need &&
               !ld_volatile_u32(p.ctrl + kCtrlAbort * kCtrlStride) &&
               globaltimer_ns() - t0 < p.timeout_ns)
          __nanosleep(500);
      }
      __syncwarp();
    }
    const long long rem = i % per_rank;
    const int k = (int)(rem / p.chunks_per_shard) + p.first_round;
    const long long c = rem % p.chunks_per_shard;
    const int s = (r + k) % kWorld;
    const long long e0 = c * p.copy_chunk;
    long long n = shard_elems - e0;
    if (n > p.copy_chunk) n = p.copy_chunk;
    const uint4* src = reinterpret_cast<const uint4*>(p.ag_src + s * shard_elems + e0);
    uint4* dst = reinterpret_cast<uint4*>(p.gather + (long long)r * p.M * p.Kr + s * shard_elems + e0);
    // 16 loads of 16 bytes in flight per lane (8 KiB per warp): a copy warp
    // is latency-bound, and the copies must stay ahead of the tiles
    constexpr int kU = 16;
    const long long nv = n / 8;
    long long v = lane;
#pragma unroll 1
    for (; v + 32 * (kU - 1) < nv; v += 32 * kU) {
      uint4 t[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) t[u] = __ldg(src + v + 32 * u);
#pragma unroll
      for (int u = 0; u < kU; ++u) dst[v + 32 * u] = t[u];
    }
#pragma unroll 1
    for (; v < nv; v += 32) dst[v] = __ldg(src + v);
    __syncwarp();  // the warp's stores are ordered before lane 0's release
    if (lane == 0 && !((p.debug_flags & 1u) && i == 0)) {  // debug: item 0 never published
      fence_proxy_async_global();
      red_release_gpu_add(p.ag_flags + (size_t)(r * kWorld + s) * kFlagStride, 1u);
    }
  }
}

// Producer side of the all-gather: wait (acquire, bounded) until every shard
// that rows [row_lo, row_hi] of rank r's tile come from is in r's gather
// buffer; then order the TMA (async proxy) reads after the copies.
__device__ __forceinline__ bool wait_shards(const GemmParams& p, int r, int row_lo, int row_hi,
                                            uint64_t limit, volatile uint32_t* abort) {
  const int s_lo = row_lo / p.shard_rows, s_hi = row_hi / p.shard_rows;
  for (int s = s_lo; s <= s_hi; ++s) {
    if (p.ag_direct && s == r) continue;  // read from the input
    const uint32_t* f = p.ag_flags + (size_t)(r * kWorld + s) * kFlagStride;
    if ((int)(ld_acquire_gpu(f) - p.ag_target) >= 0) continue;
    const uint64_t t0 = globaltimer_ns();
    uint32_t sleep_ns = 32;
    while ((int)(ld_acquire_gpu(f) - p.ag_target) < 0) {
      if (*abort || globaltimer_ns() - t0 > limit) return false;
      __nanosleep(sleep_ns);
      sleep_ns = sleep_ns < 512 ? sleep_ns * 2 : 512;
    }
  }
  fence_proxy_async_global();
  return true;
}

// ---------------------------------------------------------------------------
// Tile ring: the cluster's first CTA claims tiles from one atomic ticket (so
// no tile waits for a CTA that is not running) and hands each tile index to
// every consumer through a small ring in shared memory, mirrored into the
// other CTAs of the cluster.  Consumers: the MMA thread of each MMA leader,
// the 4 epilogue warps and the W loader of each CTA, and the A loader of
// every other CTA.
// Index -1 ends the stream.  The copies in the other CTAs are written with
// st.async, which completes their full barrier's transaction bytes; readers
// arrive on their own CTA's barrier, and one thread of each other CTA passes
// the slot's release on to CTA 0 at cluster scope (TileRing::forward).
template <int kCtas>
struct TileRing {
  static constexpr int kDepth = 4;
  // Readers of a slot in each CTA: the W loader, the epilogue warps, and the
  // MMA issuer in CTA 0 (whose A loader writes the slots) or the A loader in
  // the other CTA.
  static constexpr uint32_t kLocalConsumers = 2 + kEpiWarps;
  uint32_t slots;   // shared address of int32 slot[kDepth]
  uint32_t full;    // shared address of mbarrier full[kDepth]
  uint32_t empty;   // shared address of mbarrier empty[kDepth]
  bool owner;       // this CTA is CTA 0, which claims the tiles
  int slot = 0;
  uint32_t phase = 0;

  // Arrivals that free a slot: the CTA's own readers, and in CTA 0 of a pair
  // one more, forwarded by the other CTA once all of its readers are done.
  static __device__ __forceinline__ uint32_t empty_count(bool is_owner) {
    return kLocalConsumers + ((kCtas > 1 && is_owner) ? 1u : 0u);
  }
  __device__ __forceinline__ void advance() {
    if (++slot == kDepth) {
      slot = 0;
      phase ^= 1u;
    }
  }
  // Producer (CTA 0's TMA thread): publish the next claimed tile, or -1.
  __device__ __forceinline__ bool put(int tile, uint64_t limit, volatile uint32_t* abort) {
    // cluster-scope acquire: pairs with the other CTA's forwarded release
    if (!bar_wait<(kCtas > 1)>(empty + 8 * slot, phase ^ 1u, limit, abort)) return false;
    st_shared_u32(slots + 4 * slot, (uint32_t)tile);
    mbar_arrive(full + 8 * slot);
#pragma unroll
    for (uint32_t r = 1; r < (uint32_t)kCtas; ++r) {
      const uint32_t remote_full = mapa_shared(full + 8 * slot, r);
      mbar_arrive_expect_tx_remote(remote_full, 4);
      st_async_u32(mapa_shared(slots + 4 * slot, r), (uint32_t)tile, remote_full);
    }
    advance();
    return true;
  }
  // Consumer: next tile index (-1 at the end); false if the wait gave up.
  // The arrival is local (CTA-scope release after the read) in every CTA.
  // In the other CTA the slot is written by CTA 0's st.async, and the slot's
  // barrier there completes only once those 4 bytes have landed in this CTA's
  // shared memory (its transaction count), so the wait is a local one.
  __device__ __forceinline__ bool get(int* tile, uint64_t limit, volatile uint32_t* abort) {
    if (!bar_wait(full + 8 * slot, phase, limit, abort)) return false;
    *tile = (int)ld_shared_u32(slots + 4 * slot);
    mbar_arrive(empty + 8 * slot);
    advance();
    return true;
  }
  // Forwarder (one otherwise idle thread of the other CTA): once every reader
  // of this CTA has arrived on a slot's local barrier, pass one arrival on to
  // CTA 0's barrier of that slot, with release at cluster scope, so that all
  // those reads are performed before CTA 0 may rewrite the slot.  (A remote
  // arrival of CTA scope from each reader let the rewrite overtake a read now
  // and then: a reader then took a tile twice and skipped another.  A
  // cluster-scope release from each reader closed that too, but cost 2-7% of
  // the GEMM's time.)  Ends after forwarding the -1 slot.
  __device__ __forceinline__ bool forward(uint64_t limit, volatile uint32_t* abort) {
    while (true) {
      if (!bar_wait<true>(full + 8 * slot, phase, limit, abort)) return false;
      const int tile = (int)ld_shared_u32(slots + 4 * slot);
      if (!bar_wait(empty + 8 * slot, phase, limit, abort)) return false;
      mbar_arrive_remote_release_cluster(mapa_shared(empty + 8 * slot, 0));
      advance();
      if (tile < 0) return true;
    }
  }
};

// ---------------------------------------------------------------------------
// The persistent GEMM kernel.  kKind adds the fused communication role (see
// Kind); kCtas selects the tile shape (see TileCfg).
template <int kKind, int kCtas>
__global__ void __launch_bounds__(32 * cta_warps(kKind == kKindGemm ? 0 : kMaxReducerWarps), 1)
    gemm_rs_kernel(const __grid_constant__ GemmParams p) {
  constexpr bool kFused = kKind == kKindRS;  // reduce-scatter (or all-reduce) fused
  constexpr bool kAG = kKind == kKindAG;     // all-gather fused
  using C = TileCfg<kKind, kCtas>;
  using Ring = TileRing<kCtas>;
  constexpr int kPair = C::kPair;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t cta_rank = kCtas > 1 ? cluster_ctarank() : 0u;
  const bool first_cta = cta_rank == 0;                  // claims the cluster's tiles
  const uint32_t half = cta_rank % kPair;                // which CTA of its MMA pair
  const uint32_t mma_leader_rank = cta_rank - half;      // issues the pair's MMAs
  const bool mma_leader = half == 0;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_full = sbase + C::kSmemBar;
  const uint32_t bar_empty = bar_full + 8 * C::kStages;
  const uint32_t bar_acc_full = bar_empty + 8 * C::kStages;
  const uint32_t bar_acc_empty = bar_acc_full + 16;
  const uint32_t bar_drain = bar_acc_empty + 16;
  const uint32_t bar_ring_full = bar_drain + 8;
  const uint32_t bar_ring_empty = bar_ring_full + 8 * Ring::kDepth;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kSmemMisc);
  volatile uint32_t* cta_abort = reinterpret_cast<volatile uint32_t*>(smem + C::kSmemMisc + 4);
  uint32_t* cta_reduced = reinterpret_cast<uint32_t*>(smem + C::kSmemMisc + 8);
  const uint32_t ring_slots = sbase + C::kSmemMisc + 16;
  const uint64_t limit = p.timeout_ns;
  auto coord = [&](int idx) {
    return (kAG || p.ag_order)
               ? ag_tile_at(idx, p.mt_count, p.nt_count, p.shard_rows, C::kTileRows, p.band)
               : tile_at(idx, p.mt_count, p.nt_count, p.band, p.half_region);
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      // the MMA leader's two loaders' expect-tx arrivals (+ the bytes landing
      // in its pair)
      mbar_init(bar_full + 8 * s, 2);
      // one MMA commit frees the stage
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_acc_full + 8 * b, 1);
      mbar_init(bar_acc_empty + 8 * b, kEpiWarps * kPair);  // every epilogue warp of the pair
    }
    mbar_init(bar_drain, 1);
    for (int s = 0; s < Ring::kDepth; ++s) {
      mbar_init(bar_ring_full + 8 * s, 1);
      mbar_init(bar_ring_empty + 8 * s, Ring::empty_count(first_cta));
    }
    *cta_abort = 0;
    *cta_reduced = 0;
    fence_mbar_init();
    fence_proxy_async_shared();
    tma_prefetch_desc(&p.tmap_a);
    tma_prefetch_desc(p.w4 ? &p.tmap_w4 : &p.tmap_b);
    if (kAG) tma_prefetch_desc(&p.tmap_g);
  }
  if (warp == 1) {
    tmem_alloc<kPair>(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish<kPair>();
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (kCtas > 1) cluster_sync();  // every CTA's barriers exist before any remote use
  tc_fence_after();
  // The set-up above touches only this CTA's own shared memory and TMEM, so
  // with programmatic dependent launch it overlaps the previous grid's last
  // CTAs; nothing below runs before that grid (which may use the same
  // workspace, counts and output) has completed.  Each CTA lets the next grid
  // be scheduled as soon as it is running: that grid's CTAs then take the SMs
  // this grid leaves, and none of this grid's CTAs waits for an SM.
  griddep_wait();
  if (threadIdx.x == 0) griddep_launch_dependents();
  const uint32_t tmem_base = *tmem_slot;
  unsigned long long* trace =
      (p.trace && blockIdx.x < kMaxTraceCtas) ? p.trace + blockIdx.x * kTraceWords : nullptr;
  if (trace && threadIdx.x == 0) trace[0] = globaltimer_ns();
  Ring ring{ring_slots, bar_ring_full, bar_ring_empty, first_cta};

  if (warp == 0) {
    // ------------------------------------------------------------ A loader
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, issued_mask = 0, issued_par = 0;
      // The cluster's tiles come from one atomic ticket.  The next ticket is
      // taken as soon as a tile is published, so the atomic's round trip
      // overlaps this tile's loads instead of stalling the next tile's.
      uint32_t* const ticket = p.ctrl + kCtrlTileTicket * kCtrlStride;
      uint32_t next = first_cta ? atomicAdd(ticket, 1u) : 0u;
      while (true) {
        int idx = -1;
        bool ok;
        if (first_cta) {  // publish the claimed tile to the cluster, claim the one after
          idx = (long long)next < p.num_tiles ? (int)next : -1;
          ok = ring.put(idx, limit, cta_abort);
          if (ok && idx >= 0) next = atomicAdd(ticket, 1u);
        } else {
          ok = ring.get(&idx, limit, cta_abort);
        }
        if (!ok) {
          if (!*cta_abort) {
            record_error(p, kErrPipeTimeout, kWhereTma, 0xFFFFFFFFu);
            *cta_abort = 1;
          }
          break;
        }
        if (idx < 0) break;
        const TileCoord tc = coord(idx);
        const int m0 = tc.mt * C::kTileRows + (int)cta_rank * kBM;
        const CUtensorMap* amap = &p.tmap_a;
        int arow = m0;
        if constexpr (kAG) {
          // own rows come from the input; the others once their shards are gathered
          if (m0 < p.M && p.ag_direct && m0 / p.shard_rows == tc.rank) {
            arow = m0 - tc.rank * p.shard_rows;
          } else {
            amap = &p.tmap_g;
            if (m0 < p.M &&
                !wait_shards(p, tc.rank, m0, (m0 + kBM < p.M ? m0 + kBM : p.M) - 1, limit,
                             cta_abort)) {
              if (!*cta_abort) {
                record_error(p, kErrFlagTimeout, kWhereShard, (uint32_t)idx);
                *cta_abort = 1;
              }
              break;
            }
          }
        }
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!bar_wait(bar_empty + 8 * stage, phase ^ 1u, limit, cta_abort)) {
            if (!*cta_abort) {
              record_error(p, kErrPipeTimeout, kWhereTma, (uint32_t)idx);
              *cta_abort = 1;
            }
            ok = false;
            break;
          }
          const uint32_t fb = bar_full + 8 * stage;
          const uint32_t sa = sbase + C::kSmemA + stage * C::kAStage;
          if constexpr (kCtas == 1) {
            mbar_arrive_expect_tx(fb, C::kAStage);
            tma_load_3d(sa, amap, fb, kb * kBK, arow, tc.rank);
          } else {
            // both CTAs' bytes are counted on the leader's barrier
            if (mma_leader) mbar_arrive_expect_tx(fb, kPair * C::kAStage);
            tma_load_3d_pair(sa, amap, mapa_shared(fb, 0), kb * kBK, arow, tc.rank);
          }
          issued_mask |= 1u << stage;
          issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
      }
      // Let every copy this CTA started (or expects) land before it can exit
      // (with a 2-CTA MMA the leader's barriers also count the peer's bytes;
      // a stage's barrier completes only once the W loader's copies landed
      // too, and the W loader walks the same stages).
      if (kCtas == 1 || mma_leader)
        for (int s = 0; s < C::kStages; ++s)
          if (issued_mask & (1u << s))
            bar_wait(bar_full + 8 * s, (issued_par >> s) & 1u, limit, cta_abort);
    }
    __syncwarp();
    // out of tiles: help with the reduction of the last regions
    if (kFused) reducer_loop(p, lane, cta_reduced, -1);
  } else if (warp == 1) {
    if (lane == 0 && mma_leader) {
      // ---------------------------------------------------------- MMA issuer
      constexpr uint32_t idesc_full = idesc_bf16_f32(kBM * kPair, kBN, /*b_mn_major=*/1);
      constexpr uint32_t idesc_half = idesc_bf16_f32(kBM * kPair, kBN / 2, /*b_mn_major=*/1);
      // Operand descriptors of stage 0, split in halves; a stage or K step
      // only moves the start address (low half, 16-byte units), so the loop
      // adds constants instead of rebuilding 64-bit descriptors.
      // A: K-major rows of 128 bytes, 8-row groups 1024 bytes apart; a
      // 16-element K step moves 32 bytes inside the swizzled row.
      // B: N-major; 64-column boxes 8 KiB apart (leading), 8-k-row groups
      // 1024 bytes apart (stride); a 16-row K step moves 2 KiB.
      const uint64_t a_desc0 = smem_desc_sw128(sbase + C::kSmemA, 16, 1024);
      const uint64_t b_desc0 = smem_desc_sw128(sbase + C::kSmemB, C::kBBoxBytes, 1024);
      const uint32_t a_lo0 = (uint32_t)a_desc0, a_hi = (uint32_t)(a_desc0 >> 32);
      const uint32_t b_lo0 = (uint32_t)b_desc0, b_hi = (uint32_t)(b_desc0 >> 32);
      // order positions from here on are half-width tiles (tile_at)
      const long long first_half = (kAG || p.ag_order) ? p.num_tiles : (long long)kWorld * p.half_region;
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      while (ok) {
        int idx = -1;
        if (!ring.get(&idx, limit, cta_abort)) {
          if (!*cta_abort) {
            record_error(p, kErrPipeTimeout, kWhereMma, 0xFFFFFFFFu);
            *cta_abort = 1;
          }
          break;
        }
        if (idx < 0) break;
        if (!bar_wait(bar_acc_empty + 8 * acc, acc_phase ^ 1u, limit, cta_abort)) {
          if (!*cta_abort) {
            record_error(p, kErrPipeTimeout, kWhereMma, (uint32_t)idx);
            *cta_abort = 1;
          }
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * kBN);
        const uint32_t idesc = (long long)idx >= first_half ? idesc_half : idesc_full;
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!bar_wait(bar_full + 8 * stage, phase, limit, cta_abort)) {
            if (!*cta_abort) {
              record_error(p, kErrPipeTimeout, kWhereMma, (uint32_t)idx);
              *cta_abort = 1;
            }
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_lo = a_lo0 + (uint32_t)stage * (uint32_t)(C::kAStage >> 4);
          const uint32_t b_lo = b_lo0 + (uint32_t)stage * (uint32_t)(C::kBStage >> 4);
#pragma unroll
          for (int s = 0; s < kBK / 16; ++s)
            mma_bf16<kPair>(d_tmem, desc_join(a_lo + 2u * s, a_hi), desc_join(b_lo + 128u * s, b_hi),
                            idesc, (kb | s) != 0 ? 1u : 0u);
          // frees the smem stage (in both CTAs of the pair) when these MMAs finish
          if constexpr (kCtas == 1)
            mma_commit<1>(bar_empty + 8 * stage);
          else
            mma_commit_pair_multicast(bar_empty + 8 * stage, 0x3);
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        // accumulator ready for the epilogue warps (of both CTAs of the pair)
        if constexpr (kCtas == 1)
          mma_commit<1>(bar_acc_full + 8 * acc);
        else
          mma_commit_pair_multicast(bar_acc_full + 8 * acc, 0x3);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      // All MMAs of this thread complete before TMEM can be released.
      mma_commit<kPair>(bar_drain);
      bar_wait(bar_drain, 0, limit, cta_abort);
      if (trace) trace[2] = globaltimer_ns();
    }
    if constexpr (kCtas > 1) {
      if (lane == 0 && !first_cta && !ring.forward(limit, cta_abort) && !*cta_abort) {
        record_error(p, kErrPipeTimeout, kWhereRing, 0xFFFFFFFFu);
        *cta_abort = 1;
      }
    }
    __syncwarp();
    if (kFused) reducer_loop(p, lane, cta_reduced, -1);  // MMA issuer or forwarder: out of tiles
  } else if (warp < kGemmWarps) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;     // TMEM lane quadrant this warp can read
    const int ew = warp - 2;
    const bool hint = kFused && p.staging_in_l2;
    const uint64_t keep_policy = hint ? policy_evict_last() : 0;
    // this warp's two shared buffers; lane l writes row l of a 32 x 64 block,
    // its 16-byte granule j at position j ^ (l % 8) (the 128-byte swizzle the
    // store's tensor map expects), so a warp's 16-byte writes fill 4 whole
    // 128-byte shared-memory wavefronts
    const uint32_t ebuf = sbase + C::kSmemEpi + (uint32_t)ew * 2 * kEpiBufBytes;
    const uint32_t lane_row = ebuf + (uint32_t)lane * 128;
    int acc = 0, nbuf = 0;
    uint32_t acc_phase = 0;
    while (true) {
      int idx = -1, got = 0;
      if (lane == 0) {
        got = ring.get(&idx, limit, cta_abort) ? 1 : 0;
        if (got && idx >= 0)
          got = bar_wait(bar_acc_full + 8 * acc, acc_phase, limit, cta_abort) ? 1 : 0;
      }
      got = __shfl_sync(0xffffffffu, got, 0);
      idx = __shfl_sync(0xffffffffu, idx, 0);
      if (lane != 0) ring.advance();  // keep every lane's ring position in step
      if (!got) {
        if (lane == 0 && !*cta_abort) {
          record_error(p, kErrPipeTimeout, kWhereEpi, (uint32_t)idx);
          *cta_abort = 1;
        }
        break;
      }
      if (idx < 0) break;
      const TileCoord tc = coord(idx);
      tc_fence_after();
      const int row0 = tc.mt * C::kTileRows + (int)cta_rank * kBM + q * 32;  // the warp's first row
      const int nchunks = tc.half >= 0 ? kBN / 128 : kBN / 64;  // 64-column chunks of the tile
      const int col0 = tc.nt * kBN + (tc.half >= 0 ? tc.half * (kBN / 2) : 0);
#pragma unroll 1
      // chunk c + 1's TMEM loads are in flight while chunk c is packed,
      // written to shared memory and stored
      uint32_t v0[32], v1[32];
      {
        const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * kBN);
        tmem_ld_32x32b_x32(taddr, v0);
        tmem_ld_32x32b_x32(taddr + 32, v1);
      }
      for (int c = 0; c < nchunks; ++c) {
        tmem_ld_wait(v0);
        tmem_ld_wait(v1);
        uint32_t w[32];  // the chunk's 64 columns of the lane's row as bf16 pairs
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          w[i] = pack_bf16x2(__uint_as_float(v0[2 * i]), __uint_as_float(v0[2 * i + 1]));
          w[16 + i] = pack_bf16x2(__uint_as_float(v1[2 * i]), __uint_as_float(v1[2 * i + 1]));
        }
        if (c == nchunks - 1) {
          // accumulator fully read: hand it back to the (leader's) MMA warp
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            if (kPair == 1 || mma_leader)
              mbar_arrive(bar_acc_empty + 8 * acc);
            else
              mbar_arrive_remote(mapa_shared(bar_acc_empty + 8 * acc, mma_leader_rank));
          }
        } else {
          const uint32_t taddr =
              tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * kBN + (c + 1) * 64);
          tmem_ld_32x32b_x32(taddr, v0);
          tmem_ld_32x32b_x32(taddr + 32, v1);
        }
        const int col = col0 + c * 64;
        if (row0 < p.M && col < p.N) {  // warp-uniform; the store clips ragged edges
          const uint32_t buf = lane_row + (uint32_t)nbuf * kEpiBufBytes;
          if (lane == 0) bulk_wait_group_read<1>();  // this buffer's previous store has read it
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 8; ++j)  // granule j = columns [8j, 8j + 8) of the lane's row
            st_shared_v4(buf + (uint32_t)((j ^ (lane & 7)) << 4), w[4 * j], w[4 * j + 1], w[4 * j + 2],
                         w[4 * j + 3]);
          fence_proxy_async_shared();  // the writes, before the async proxy reads them
          __syncwarp();
          if (lane == 0) {
            const uint32_t block_src = ebuf + (uint32_t)nbuf * kEpiBufBytes;
            if (hint)
              tma_store_3d_hint(&p.tmap_s, block_src, col, row0, tc.rank, keep_policy);
            else
              tma_store_3d(&p.tmap_s, block_src, col, row0, tc.rank);
            bulk_commit_group();
          }
          nbuf ^= 1;
        }
      }
      if (kFused) {
        if (lane == 0) {
          // the warp's rows of this tile are in the staging (async proxy),
          // ordered before the release that publishes them
          bulk_wait_group<0>();
          fence_proxy_async_global();
          const int block =
              ((int)(tc.mt * p.nt_count + tc.nt)) * p.blocks_per_region + (int)cta_rank;
          publish_rows(p, block, (p.debug_flags & 1u) && idx == 0 && first_cta && ew == 0);
        }
        __syncwarp();
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (lane == 0) bulk_wait_group<0>();  // the last stores have read their buffers and landed
    __syncwarp();
    if (trace && ew == 0 && lane == 0) trace[1] = globaltimer_ns();
    if (kFused) reducer_loop(p, lane, cta_reduced, -1);  // out of tiles: help with the reduction
  } else if (warp == w_loader_warp((int)(blockDim.x >> 5) - cta_warps(0))) {
    // ------------------------------------------------------------ W loader
    // Walks the same tiles and stages as the A loader; each stage's barrier
    // takes both loaders' arrivals and bytes.
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      while (true) {
        int idx = -1;
        if (!ring.get(&idx, limit, cta_abort)) {
          if (!*cta_abort) {
            record_error(p, kErrPipeTimeout, kWhereTma, 0xFFFFFFFFu);
            *cta_abort = 1;
          }
          break;
        }
        if (idx < 0) break;
        const TileCoord tc = coord(idx);
        // a half-width tile is the left or right 128 of the 256 columns: each
        // CTA loads half as many columns of W
        const bool half_tile = tc.half >= 0;
        const int cta_cols = (half_tile ? kBN / 2 : kBN) / kPair;
        const int n0 = tc.nt * kBN + (half_tile ? tc.half * (kBN / 2) : 0) + (int)half * cta_cols;
        const int nboxes = cta_cols / 64;
        const bool one_copy = p.w4 && nboxes == C::kBBoxes;
        bool ok = true;
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!bar_wait(bar_empty + 8 * stage, phase ^ 1u, limit, cta_abort)) {
            if (!*cta_abort) {
              record_error(p, kErrPipeTimeout, kWhereTma, (uint32_t)idx);
              *cta_abort = 1;
            }
            ok = false;
            break;
          }
          const uint32_t fb = bar_full + 8 * stage;
          const uint32_t sb = sbase + C::kSmemB + stage * C::kBStage;
          const uint32_t bytes = (uint32_t)(nboxes * C::kBBoxBytes);
          if constexpr (kCtas == 1) {
            mbar_arrive_expect_tx(fb, bytes);
            if (one_copy)
              tma_load_4d(sb, &p.tmap_w4, fb, 0, kb * kBK, n0 >> 6, tc.rank);
            else
              for (int j = 0; j < nboxes; ++j)
                tma_load_3d(sb + j * C::kBBoxBytes, &p.tmap_b, fb, n0 + 64 * j, kb * kBK, tc.rank);
          } else {
            if (mma_leader) mbar_arrive_expect_tx(fb, kPair * bytes);
            const uint32_t fb_leader = mapa_shared(fb, 0);
            if (one_copy)
              tma_load_4d_pair(sb, &p.tmap_w4, fb_leader, 0, kb * kBK, n0 >> 6, tc.rank);
            else
              for (int j = 0; j < nboxes; ++j)
                tma_load_3d_pair(sb + j * C::kBBoxBytes, &p.tmap_b, fb_leader, n0 + 64 * j,
                                 kb * kBK, tc.rank);
          }
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
      }
    }
    __syncwarp();
    if (kFused) reducer_loop(p, lane, cta_reduced, -1);
  } else {
    // ------------------------------------------------- reducers / copy warps
    const int wl = w_loader_warp((int)(blockDim.x >> 5) - cta_warps(0));
    const int comm_idx = warp - kGemmWarps - (warp > wl ? 1 : 0);
    if (kFused) reducer_loop(p, lane, cta_reduced, comm_idx);
    if (kAG) copy_loop(p, lane);
  }

  if (trace && lane == 0) atomicMax(trace + 3, (unsigned long long)globaltimer_ns());
  tc_fence_before();
  __syncthreads();
  if constexpr (kCtas > 1) cluster_sync();  // no MMA or remote arrive targets this CTA any more
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<kPair>(tmem_base, kTmemCols);
  }
  if (threadIdx.x == 0) {
    if (kFused) atomicAdd(p.ctrl + kCtrlReduced * kCtrlStride, *cta_reduced);
    __threadfence();
    const uint32_t prev = atomicAdd(p.ctrl + kCtrlDone * kCtrlStride, 1u);
    if (prev == gridDim.x - 1) {  // last CTA: check the run, reset the per-run counters
      __threadfence();
      if (kFused && (long long)atomicExch(p.ctrl + kCtrlReduced * kCtrlStride, 0u) != p.num_items)
        atomicOr(p.ctrl + kCtrlError * kCtrlStride, (uint32_t)kErrIncomplete);
      atomicExch(p.ctrl + kCtrlQueueTail * kCtrlStride, 0u);
      atomicExch(p.ctrl + kCtrlQueueHead * kCtrlStride, 0u);
      atomicExch(p.ctrl + kCtrlTileTicket * kCtrlStride, 0u);
      atomicExch(p.ctrl + kCtrlCopyTicket * kCtrlStride, 0u);
      atomicExch(p.ctrl + kCtrlTarget * kCtrlStride, 0u);
      atomicExch(p.ctrl + kCtrlAbort * kCtrlStride, 0u);
      atomicExch(p.ctrl + kCtrlDone * kCtrlStride, 0u);
      __threadfence();
    }
  }
}

// ---------------------------------------------------------------------------
// Standalone reduce-scatter kernel of the unfused and chunked paths: the same
// arithmetic (reduce8) over `elems` consecutive output elements, one 16-byte
// vector per thread and step.  stage points at rank 0's first element; rank
// r's partial of the same element is `plane` elements further per rank.  The
// sum goes to `replicas` copies of the output, `out_stride` elements apart
// (8 for the all-reduce).
__device__ __forceinline__ void store_replicas(uint16_t* out, long long v, uint4 o, int replicas,
                                               long long out_stride) {
#pragma unroll 1
  for (int c = 0; c < replicas; ++c) reinterpret_cast<uint4*>(out + c * out_stride)[v] = o;
}

__global__ void __launch_bounds__(256) rs_reduce_kernel(const uint16_t* __restrict__ stage,
                                                        uint16_t* __restrict__ out,
                                                        long long elems, long long plane,
                                                        int replicas, long long out_stride) {
  const long long nvec = elems / 8;
  const long long stride = (long long)gridDim.x * blockDim.x;
  long long v = (long long)blockIdx.x * blockDim.x + threadIdx.x;
#pragma unroll 1
  for (; v + stride < nvec; v += 2 * stride) {
    uint4 a[kWorld], b[kWorld];
#pragma unroll
    for (int r = 0; r < kWorld; ++r) {
      a[r] = __ldcg(reinterpret_cast<const uint4*>(stage + r * plane) + v);
      b[r] = __ldcg(reinterpret_cast<const uint4*>(stage + r * plane) + v + stride);
    }
    store_replicas(out, v, reduce8(a), replicas, out_stride);
    store_replicas(out, v + stride, reduce8(b), replicas, out_stride);
  }
  if (v < nvec) {
    uint4 a[kWorld];
#pragma unroll
    for (int r = 0; r < kWorld; ++r)
      a[r] = __ldcg(reinterpret_cast<const uint4*>(stage + r * plane) + v);
    store_replicas(out, v, reduce8(a), replicas, out_stride);
  }
}


// Standalone all-gather of the unfused path: every rank's gather buffer gets
// all 8 row shards, its own included.  Rank r's buffer [M][K] is the 8 shards
// one after the other, which is the input's own layout, so it is a copy of
// the whole input; 16-byte vectors, grid-stride.
__global__ void __launch_bounds__(256) ag_gather_kernel(const uint16_t* __restrict__ src,
                                                        uint16_t* __restrict__ gather,
                                                        long long rank_elems) {
  const long long per_rank = rank_elems / 8;  // vectors
  const long long total = (long long)kWorld * per_rank;
  const long long stride = (long long)gridDim.x * blockDim.x;
  const uint4* s = reinterpret_cast<const uint4*>(src);
  uint4* d = reinterpret_cast<uint4*>(gather);
#pragma unroll 1
  for (long long v = (long long)blockIdx.x * blockDim.x + threadIdx.x; v < total; v += stride)
    d[v] = __ldg(s + v % per_rank);
}

// Zero fill (empty contraction, K = 0): n16 16-byte vectors.
__global__ void __launch_bounds__(256) zero_fill_kernel(uint4* __restrict__ p, long long n16) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += stride)
    p[i] = make_uint4(0u, 0u, 0u, 0u);
}

}  // namespace grs
