// kernels.cuh -- the device side of the fused GEMM + reduce-scatter.
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
//   warp 0        TMA producer: its CTA's rows of A_r and columns of W_r, one
//                 k-block per stage of the smem ring
//   warp 1        MMA issuer (the pair's first CTA only): tcgen05.mma
//                 (bf16 in, fp32 in TMEM, two 256-column accumulators);
//                 TMEM allocation in every CTA
//   warps 2..5    epilogue: TMEM -> registers -> bf16 (RNE) -> swizzled smem ->
//                 TMA store into the rank's staging region; then the tile's
//                 flag is raised with a release add (fused kernel only)
//   warps 6..     reducers (fused kernel only): claim reduce units in tile
//                 order, acquire the 8 rank flags of the unit's region, add the
//                 8 bf16 partials in fp32 in rank order, write bf16 output.
//                 The epilogue warps join them when the CTA's tiles are done.
// Every wait is bounded by p.timeout_ns; on expiry the kernel records an error
// word, stops its loops, lets its in-flight copies land, frees TMEM and returns.
#pragma once
#include "ptx.cuh"
#include "schedule.h"

namespace grs {

constexpr int kEpiWarps = 4;
constexpr int kEpiBufBytes = 32 * 128;  // 32 rows x 64 bf16 columns
constexpr int kTmemCols = 2 * kBN;      // two fp32 accumulators of 256 columns
constexpr int kGemmWarps = 2 + kEpiWarps;
constexpr int kMaxReducerWarps = 8;

// Shared-memory plan of one CTA for 1 or 2 CTAs per MMA.
template <int kPair>
struct TileCfg {
  static constexpr int kStages = kPair == 1 ? 4 : 6;
  static constexpr int kTileRows = kBM * kPair;        // output rows of one (pair) tile
  static constexpr int kBCols = kBN / kPair;           // W columns held by one CTA
  static constexpr int kBBoxes = kBCols / 64;          // 64-column TMA boxes per stage
  static constexpr int kBBoxBytes = kBK * 64 * 2;      // 8 KiB: 64 k-rows x 64 n, N-major
  static constexpr int kAStage = kBM * kBK * 2;        // 16 KiB: 128 rows x 64 k, K-major
  static constexpr int kBStage = kBK * kBCols * 2;     // 32 KiB (one CTA) / 16 KiB (pair)
  static constexpr int kStage = kAStage + kBStage;     // bytes one CTA loads per stage
  static constexpr int kSmemA = 0;
  static constexpr int kSmemB = kSmemA + kStages * kAStage;
  static constexpr int kSmemEpi = kSmemB + kStages * kBStage;
  static constexpr int kSmemBar = kSmemEpi + kEpiWarps * 2 * kEpiBufBytes;
  static constexpr int kNumBars = 2 * kStages + 5;   // full, empty, acc_full[2], acc_empty[2], drain
  static constexpr int kSmemMisc = kSmemBar + kNumBars * 8;
  static constexpr int kSmemBytes = kSmemMisc + 16;
  static constexpr int kSmemAlloc = kSmemBytes + 1024;  // slack to align the base to 1024 bytes
  static constexpr uint32_t kFlagAddsPerTile = kEpiWarps * kPair;
  static_assert(kSmemAlloc <= 232448, "shared memory per CTA");
};

// control words in the workspace
enum CtrlWord : int {
  kCtrlTicket = 0,   // next reduce unit to claim
  kCtrlDone = 1,     // CTAs finished (the last one resets the words above and below)
  kCtrlAbort = 2,    // set when some warp gave up waiting
  kCtrlError = 3,    // error bits (kErr*), cleared by the host
  kCtrlErrWhere = 4, // which wait gave up
  kCtrlErrWhat = 5,  // region / tile index of that wait
  kCtrlWords = 16
};
enum ErrBits : uint32_t { kErrFlagTimeout = 1u, kErrPipeTimeout = 2u };
enum ErrWhere : uint32_t { kWhereTma = 1, kWhereMma = 2, kWhereEpi = 3, kWhereReducer = 4 };

struct GemmParams {
  CUtensorMap tmap_a;   // A  [8][M][Kr] : dims {Kr, M, 8}, box {64, 128, 1}
  CUtensorMap tmap_b;   // W  [8][Kr][N] : dims {N, Kr, 8}, box {64, 64, 1}
  CUtensorMap tmap_st;  // staging [8][M][N] : dims {N, M, 8}, box {64, 32, 1}
  const uint16_t* stage;
  uint16_t* out;
  uint32_t* flags;  // [8][mt_count * nt_count]; each tile adds kFlagAddsPerTile per fused run
  uint32_t* ctrl;   // kCtrlWords words
  int M, N, Kr;
  int mt_count, nt_count, band;  // mt_count and band count tile rows of kTileRows rows
  int num_kb;
  int unit_rows, units_per_region;
  long long num_tiles;
  long long num_units;
  uint32_t flag_target;
  uint32_t debug_flags;
  // Fused kernel only: staging tiles are stored with an L2 evict-last hint so
  // they are still in L2 when reduced, and each reduced staging line is
  // discarded from L2 (never written back).  Needs N % 64 == 0 so that no
  // 128-byte line holds data of two reduce units.
  uint32_t staging_in_l2;
  int tile_rows;  // rows of a region: 128 (one CTA per MMA) or 256 (a CTA pair)
  unsigned long long timeout_ns;
};

// ---------------------------------------------------------------------------

__device__ __forceinline__ void record_error(const GemmParams& p, uint32_t bit, uint32_t where,
                                             uint32_t what) {
  atomicOr(p.ctrl + kCtrlError, bit);
  atomicExch(p.ctrl + kCtrlErrWhere, where);
  atomicExch(p.ctrl + kCtrlErrWhat, what);
  atomicExch(p.ctrl + kCtrlAbort, 1u);
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

// Wait (bounded) until the 8 rank tiles of `region` are published for this
// run.  Every lane performs its own acquire loads of all 8 flags, so each
// lane's later staging loads are ordered after the producers' releases.
__device__ __forceinline__ bool wait_region_flags(const GemmParams& p, int region, int lane) {
  const size_t regions = (size_t)p.mt_count * p.nt_count;
  const uint32_t* f = p.flags + region;
  uint64_t t0 = 0;
  if (lane == 0) t0 = globaltimer_ns();
  uint32_t sleep_ns = 64;
  while (true) {
    bool ok = true;
#pragma unroll
    for (int r = 0; r < kWorld; ++r) {
      const uint32_t v = ld_acquire_gpu(f + (size_t)r * regions);
      ok = ok && ((int32_t)(v - p.flag_target) >= 0);
    }
    if (__all_sync(0xffffffffu, ok)) return true;
    int give_up = 0;
    if (lane == 0)
      give_up = (globaltimer_ns() - t0 > p.timeout_ns) || ld_volatile_u32(p.ctrl + kCtrlAbort);
    if (__shfl_sync(0xffffffffu, give_up, 0)) return false;
    __nanosleep(sleep_ns);
    sleep_ns = sleep_ns < 1024 ? sleep_ns * 2 : 1024;
  }
}

// Drop the staging lines of one output row segment from L2 (fused kernel,
// after the whole warp has consumed them).
__device__ __forceinline__ void discard_row(const GemmParams& p, size_t plane, size_t off,
                                            int lane) {
  if ((lane & 7) == 0) {
#pragma unroll
    for (int r = 0; r < kWorld; ++r) discard_l2_line(p.stage + r * plane + off);
  }
}

// Reducer role: claim units until none are left.  A unit is unit_rows rows x
// 256 columns of one region; lane l covers columns [8l, 8l+8) of it.
__device__ __noinline__ void reducer_loop(const GemmParams& p, int lane) {
  const size_t plane = (size_t)p.M * p.N;
  while (true) {
    uint32_t u = 0;
    if (lane == 0) u = atomicAdd(p.ctrl + kCtrlTicket, 1u);
    u = __shfl_sync(0xffffffffu, u, 0);
    if ((long long)u >= p.num_units) break;
    const int pos = (int)(u / (uint32_t)p.units_per_region);
    const int sub = (int)(u - (uint32_t)pos * (uint32_t)p.units_per_region);
    const Region g = region_at(pos, p.mt_count, p.nt_count, p.band);
    const int region = g.mt * p.nt_count + g.nt;
    const int row_begin = g.mt * p.tile_rows + sub * p.unit_rows;
    if (row_begin >= p.M) continue;  // rows of a ragged last tile that do not exist
    if (!wait_region_flags(p, region, lane)) {
      if (lane == 0 && !ld_volatile_u32(p.ctrl + kCtrlAbort))
        record_error(p, kErrFlagTimeout, kWhereReducer, (uint32_t)region);
      break;
    }
    int row_end = row_begin + p.unit_rows;
    if (row_end > p.M) row_end = p.M;
    const int col = g.nt * kBN + lane * 8;
    if (col < p.N) {
      int row = row_begin;
#pragma unroll 1
      for (; row + 1 < row_end; row += 2) {
        const size_t off0 = (size_t)row * p.N + col;
        const size_t off1 = off0 + p.N;
        uint4 v0[kWorld], v1[kWorld];
#pragma unroll
        for (int r = 0; r < kWorld; ++r) {
          v0[r] = __ldcg(reinterpret_cast<const uint4*>(p.stage + r * plane + off0));
          v1[r] = __ldcg(reinterpret_cast<const uint4*>(p.stage + r * plane + off1));
        }
        *reinterpret_cast<uint4*>(p.out + off0) = reduce8(v0);
        *reinterpret_cast<uint4*>(p.out + off1) = reduce8(v1);
        if (p.staging_in_l2) {
          __syncwarp();  // every lane has consumed its loads (its stores depend on them)
          discard_row(p, plane, off0, lane);
          discard_row(p, plane, off1, lane);
        }
      }
      if (row < row_end) {
        const size_t off0 = (size_t)row * p.N + col;
        uint4 v0[kWorld];
#pragma unroll
        for (int r = 0; r < kWorld; ++r)
          v0[r] = __ldcg(reinterpret_cast<const uint4*>(p.stage + r * plane + off0));
        *reinterpret_cast<uint4*>(p.out + off0) = reduce8(v0);
        if (p.staging_in_l2) {
          __syncwarp();
          discard_row(p, plane, off0, lane);
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// The persistent GEMM kernel.  kFused = true adds flags and reducer warps;
// kPair = 2 shares each MMA between the two CTAs of a cluster.
template <bool kFused, int kPair>
__global__ void __launch_bounds__(32 * (kGemmWarps + (kFused ? kMaxReducerWarps : 0)), 1)
    gemm_rs_kernel(const __grid_constant__ GemmParams p) {
  using C = TileCfg<kPair>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t cta_rank = kPair == 2 ? cluster_ctarank() : 0u;
  const bool leader = cta_rank == 0;
  const long long first_tile = blockIdx.x / kPair;
  const long long tile_step = gridDim.x / kPair;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_full = sbase + C::kSmemBar;
  const uint32_t bar_empty = bar_full + 8 * C::kStages;
  const uint32_t bar_acc_full = bar_empty + 8 * C::kStages;
  const uint32_t bar_acc_empty = bar_acc_full + 16;
  const uint32_t bar_drain = bar_acc_empty + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kSmemMisc);
  volatile uint32_t* cta_abort = reinterpret_cast<volatile uint32_t*>(smem + C::kSmemMisc + 4);
  const uint64_t limit = p.timeout_ns;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar_full + 8 * s, 1);   // the leader's expect-tx arrival (+ bytes of the pair)
      mbar_init(bar_empty + 8 * s, 1);  // one MMA commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_acc_full + 8 * b, 1);
      mbar_init(bar_acc_empty + 8 * b, kEpiWarps * kPair);  // every epilogue warp of the pair
    }
    mbar_init(bar_drain, 1);
    *cta_abort = 0;
    fence_mbar_init();
    fence_proxy_async_shared();
    tma_prefetch_desc(&p.tmap_a);
    tma_prefetch_desc(&p.tmap_b);
    tma_prefetch_desc(&p.tmap_st);
  }
  if (warp == 1) {
    tmem_alloc<kPair>(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish<kPair>();
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (kPair == 2) cluster_sync();  // the peer's barriers exist before any remote use
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, issued_mask = 0, issued_par = 0;
      bool ok = true;
      for (long long idx = first_tile; ok && idx < p.num_tiles; idx += tile_step) {
        const TileCoord tc = tile_at(idx, p.mt_count, p.nt_count, p.band);
        const int m0 = tc.mt * C::kTileRows + (int)cta_rank * kBM;
        const int n0 = tc.nt * kBN + (int)cta_rank * C::kBCols;
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
          const uint32_t sb = sbase + C::kSmemB + stage * C::kBStage;
          if constexpr (kPair == 1) {
            mbar_arrive_expect_tx(fb, C::kStage);
            tma_load_3d(sa, &p.tmap_a, fb, kb * kBK, m0, tc.rank);
#pragma unroll
            for (int j = 0; j < C::kBBoxes; ++j)
              tma_load_3d(sb + j * C::kBBoxBytes, &p.tmap_b, fb, n0 + 64 * j, kb * kBK, tc.rank);
          } else {
            // both CTAs' bytes are counted on the leader's barrier
            if (leader) mbar_arrive_expect_tx(fb, kPair * C::kStage);
            const uint32_t fb_leader = mapa_shared(fb, 0);
            tma_load_3d_pair(sa, &p.tmap_a, fb_leader, kb * kBK, m0, tc.rank);
#pragma unroll
            for (int j = 0; j < C::kBBoxes; ++j)
              tma_load_3d_pair(sb + j * C::kBBoxBytes, &p.tmap_b, fb_leader, n0 + 64 * j,
                               kb * kBK, tc.rank);
          }
          issued_mask |= 1u << stage;
          issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Let every copy this thread started land before the CTA can exit (the
      // leader's barriers also count the peer's bytes).
      if (leader)
        for (int s = 0; s < C::kStages; ++s)
          if (issued_mask & (1u << s))
            bar_wait(bar_full + 8 * s, (issued_par >> s) & 1u, limit, cta_abort);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && leader) {
      constexpr uint32_t idesc = idesc_bf16_f32(C::kTileRows, kBN, /*b_mn_major=*/1);
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (long long idx = first_tile; ok && idx < p.num_tiles; idx += tile_step) {
        if (!bar_wait<kPair == 2>(bar_acc_empty + 8 * acc, acc_phase ^ 1u, limit, cta_abort)) {
          if (!*cta_abort) {
            record_error(p, kErrPipeTimeout, kWhereMma, (uint32_t)idx);
            *cta_abort = 1;
          }
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * kBN);
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
          const uint32_t sa = sbase + C::kSmemA + stage * C::kAStage;
          const uint32_t sb = sbase + C::kSmemB + stage * C::kBStage;
#pragma unroll
          for (int s = 0; s < kBK / 16; ++s) {
            // A: K-major rows of 128 bytes, 8-row groups 1024 bytes apart; a
            // 16-element K step moves 32 bytes inside the swizzled row.
            const uint64_t ad = smem_desc_sw128(sa + s * 32, 16, 1024);
            // B: N-major; 64-column boxes 8 KiB apart (leading), 8-k-row groups
            // 1024 bytes apart (stride); a 16-row K step moves 2 KiB.
            const uint64_t bd = smem_desc_sw128(sb + s * 2048, C::kBBoxBytes, 1024);
            mma_bf16<kPair>(d_tmem, ad, bd, idesc, (kb | s) != 0 ? 1u : 0u);
          }
          // frees the smem stage (in both CTAs) when these MMAs finish
          if constexpr (kPair == 1)
            mma_commit<1>(bar_empty + 8 * stage);
          else
            mma_commit_pair_multicast(bar_empty + 8 * stage, 0x3);
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        // accumulator ready for the epilogue warps (of both CTAs)
        if constexpr (kPair == 1)
          mma_commit<1>(bar_acc_full + 8 * acc);
        else
          mma_commit_pair_multicast(bar_acc_full + 8 * acc, 0x3);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      // All MMAs of this thread complete before TMEM can be released.
      mma_commit<kPair>(bar_drain);
      bar_wait(bar_drain, 0, limit, cta_abort);
    }
    __syncwarp();
  } else if (warp < kGemmWarps) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quadrant this warp can read
    const int ew = warp - 2;
    const uint32_t buf_s = sbase + C::kSmemEpi + ew * 2 * kEpiBufBytes;
    uint8_t* buf_p = smem + C::kSmemEpi + ew * 2 * kEpiBufBytes;
    const size_t regions = (size_t)p.mt_count * p.nt_count;
    const bool hint = kFused && p.staging_in_l2;
    const uint64_t keep_policy = hint ? policy_evict_last() : 0;
    int acc = 0, buf = 0;
    uint32_t acc_phase = 0;
    for (long long idx = first_tile; idx < p.num_tiles; idx += tile_step) {
      const TileCoord tc = tile_at(idx, p.mt_count, p.nt_count, p.band);
      int got = 0;
      if (lane == 0) got = bar_wait(bar_acc_full + 8 * acc, acc_phase, limit, cta_abort);
      got = __shfl_sync(0xffffffffu, got, 0);
      if (!got) {
        if (lane == 0 && !*cta_abort) {
          record_error(p, kErrPipeTimeout, kWhereEpi, (uint32_t)idx);
          *cta_abort = 1;
        }
        break;
      }
      tc_fence_after();
      const int row0 = tc.mt * C::kTileRows + (int)cta_rank * kBM + q * 32;
      const bool rows_in = row0 < p.M;
#pragma unroll 1
      for (int c = 0; c < kBN / 64; ++c) {
        uint32_t v0[32], v1[32];
        const uint32_t taddr =
            tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * kBN + c * 64);
        tmem_ld_32x32b_x32(taddr, v0);
        tmem_ld_32x32b_x32(taddr + 32, v1);
        tmem_ld_wait(v0);
        tmem_ld_wait(v1);
        if (c == kBN / 64 - 1) {
          // accumulator fully read: hand it back to the (leader's) MMA warp
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            if constexpr (kPair == 1)
              mbar_arrive(bar_acc_empty + 8 * acc);
            else
              mbar_arrive_cluster(mapa_shared(bar_acc_empty + 8 * acc, 0));
          }
        }
        const int col0 = tc.nt * kBN + c * 64;
        if (rows_in && col0 < p.N) {
          if (lane == 0) bulk_wait_read<1>();  // the store that used this buffer has read it
          __syncwarp();
          uint8_t* rowp = buf_p + buf * kEpiBufBytes + lane * 128;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint32_t* v = (j < 4) ? (v0 + 8 * j) : (v1 + 8 * (j - 4));
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(v[0]), __uint_as_float(v[1]));
            w.y = pack_bf16x2(__uint_as_float(v[2]), __uint_as_float(v[3]));
            w.z = pack_bf16x2(__uint_as_float(v[4]), __uint_as_float(v[5]));
            w.w = pack_bf16x2(__uint_as_float(v[6]), __uint_as_float(v[7]));
            // 128-byte swizzle: 16-byte chunk j of row t sits at chunk j ^ (t % 8)
            *reinterpret_cast<uint4*>(rowp + ((j ^ (lane & 7)) << 4)) = w;
          }
          fence_proxy_async_shared();
          __syncwarp();
          if (lane == 0) {
            if (hint)
              tma_store_3d_hint(&p.tmap_st, buf_s + buf * kEpiBufBytes, col0, row0, tc.rank,
                                keep_policy);
            else
              tma_store_3d(&p.tmap_st, buf_s + buf * kEpiBufBytes, col0, row0, tc.rank);
            bulk_commit();
          }
          buf ^= 1;
        }
      }
      if (kFused) {
        if (lane == 0) {
          bulk_wait_all<0>();          // this warp's part of the tile is in global memory
          fence_proxy_async_global();  // order the async-proxy writes before the release
          const bool skip = (p.debug_flags & 1u) && idx == 0 && ew == 0 && leader;
          if (!skip)
            red_release_gpu_add(p.flags + (size_t)tc.rank * regions +
                                    (size_t)tc.mt * p.nt_count + tc.nt,
                                1u);
        }
        __syncwarp();
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (lane == 0) bulk_wait_all<0>();
    __syncwarp();
    if (kFused) reducer_loop(p, lane);  // out of tiles: help with the reduction
  } else {
    // ------------------------------------------------------------ reducers
    if (kFused) reducer_loop(p, lane);
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (kPair == 2) cluster_sync();  // no MMA or remote arrive targets this CTA any more
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<kPair>(tmem_base, kTmemCols);
  }
  if (kFused && threadIdx.x == 0) {
    __threadfence();
    const uint32_t prev = atomicAdd(p.ctrl + kCtrlDone, 1u);
    if (prev == gridDim.x - 1) {  // last CTA: reset the per-run counters
      __threadfence();
      atomicExch(p.ctrl + kCtrlTicket, 0u);
      atomicExch(p.ctrl + kCtrlAbort, 0u);
      atomicExch(p.ctrl + kCtrlDone, 0u);
      __threadfence();
    }
  }
}

// ---------------------------------------------------------------------------
// Standalone reduce-scatter kernel of the unfused path: the same arithmetic
// (reduce8) over the whole output, one 16-byte vector per thread and step.
__global__ void __launch_bounds__(256) rs_reduce_kernel(const uint16_t* __restrict__ stage,
                                                        uint16_t* __restrict__ out,
                                                        long long mn) {
  const long long nvec = mn / 8;
  const long long stride = (long long)gridDim.x * blockDim.x;
  long long v = (long long)blockIdx.x * blockDim.x + threadIdx.x;
#pragma unroll 1
  for (; v + stride < nvec; v += 2 * stride) {
    uint4 a[kWorld], b[kWorld];
#pragma unroll
    for (int r = 0; r < kWorld; ++r) {
      a[r] = __ldcg(reinterpret_cast<const uint4*>(stage + r * mn) + v);
      b[r] = __ldcg(reinterpret_cast<const uint4*>(stage + r * mn) + v + stride);
    }
    reinterpret_cast<uint4*>(out)[v] = reduce8(a);
    reinterpret_cast<uint4*>(out)[v + stride] = reduce8(b);
  }
  if (v < nvec) {
    uint4 a[kWorld];
#pragma unroll
    for (int r = 0; r < kWorld; ++r)
      a[r] = __ldcg(reinterpret_cast<const uint4*>(stage + r * mn) + v);
    reinterpret_cast<uint4*>(out)[v] = reduce8(a);
  }
}

// Zero fill (empty contraction, K = 0): n16 16-byte vectors.
__global__ void __launch_bounds__(256) zero_fill_kernel(uint4* __restrict__ p, long long n16) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += stride)
    p[i] = make_uint4(0u, 0u, 0u, 0u);
}

}  // namespace grs
