// gemm_rs.cu -- host side of the C ABI declared in include/gemm_rs.h:
// argument checks, workspace layout, TMA tensor maps, launch configuration,
// the per-run epoch of the completion flags, and the device error word.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>

#include "../../include/gemm_rs.h"
#include "kernels.cuh"

using namespace grs;

namespace {

constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;  // 2 s
constexpr int kDefaultReducerWarps = 4;
// From K = 16384 on, the reduction is a small share of the work (T_rs / T_gemm
// ~ 9 P / (B K)): 2 reducer warps keep up and interfere less with the tiles'
// loads (interleaved A/B, fused: 8192 x 6144 x 16384 1110 -> 1024 us,
// 8192 x 8192 x 28672 2596 -> 2393 us; at K = 8192, 2 warps fall behind:
// o_proj 195 -> 227 us).
constexpr int kLargeKReducerWarps = 2;
constexpr int64_t kLargeK = 16384;
constexpr int kDefaultCopyWarps = 2;
// Up to K = 6144 the reduction is the larger share of the fused kernel's work
// and falls behind the tiles: 5 reducer warps, and 16-row items from M = 2048
// (fewer item operations), keep it closer (fused, loaders split: 2048 x 6144 x
// 6144 131 -> 121 us, 8192 x 6144 x 6144 504 -> 447 us; M = 512: 5 warps
// 53 -> 47 us; at K = 8192 no change on o_proj).
constexpr int kSmallKReducerWarps = 5;
constexpr int64_t kSmallK = 6144;
int default_reducer_warps(const gemm_rs_desc* d) {
  if (d->op == GEMM_RS_OP_AG) return kDefaultCopyWarps;
  if (d->K >= kLargeK) return kLargeKReducerWarps;
  return d->K <= kSmallK ? kSmallKReducerWarps : kDefaultReducerWarps;
}
// Reduce item size: small items leave less reduction in service when the
// last tiles finish, large ones cost fewer item operations where the
// reduction is a large share of the work.  8-row items, and 4-row items for
// the regions of the last 3 waves, were the best compromise measured (o_proj
// fused 211 -> 206 us, M = 512 78 -> 72 us against 16-row items and a
// 1-wave tail; 8192^3 at most 3% slower).
constexpr int kDefaultUnitRows = 8;
int default_unit_rows(const gemm_rs_desc* d) {
  return (d->K <= kSmallK && d->M >= 2048) ? 16 : kDefaultUnitRows;
}
constexpr int kDefaultTailWaves = 3;
constexpr int kDefaultMmaCtas = 2;
constexpr int kDefaultChunks = 4;
constexpr int kMaxChunks = 64;
constexpr long long kCopyChunk = 32768;  // elements per all-gather copy item (64 KiB)
constexpr int kMaxCopyStreams = 4;       // all-gather: side streams of copy-engine copies
constexpr int kDefaultCopyEngines = -1;  // all-gather: copy warps in the fused kernel

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct Layout {
  size_t staging_bytes, flags_off, flags_bytes, queue_off, ctrl_off, trace_off, total;
};

// blocks: 32-row blocks of the output (completion counts); items: reduce items
// of a run (debug stamp slots)
Layout layout_for(int64_t M, int64_t N, int64_t blocks, int64_t items) {
  Layout l;
  l.staging_bytes = (size_t)kWorld * (size_t)M * (size_t)N * 2;
  l.flags_off = align_up(l.staging_bytes, 256);
  l.flags_bytes = (size_t)blocks * kFlagStride * 4;
  l.queue_off = align_up(l.flags_off + l.flags_bytes, 256);
  l.ctrl_off = align_up(l.queue_off + (size_t)items * kQueueStride * 8, 256);
  l.trace_off = l.ctrl_off + (size_t)kCtrlWords * 4;
  l.total = l.trace_off + (size_t)kMaxTraceCtas * kTraceWords * 8;
  return l;
}

// All-gather + GEMM workspace: the 8 gather buffers [8][M][K], the 64
// per-(rank, shard) copy counts, the control words, the debug stamps.
Layout layout_ag(int64_t M, int64_t K) {
  Layout l;
  l.staging_bytes = (size_t)kWorld * (size_t)M * (size_t)K * 2;
  l.flags_off = align_up(l.staging_bytes, 256);
  l.flags_bytes = (size_t)kWorld * kWorld * kFlagStride * 4;
  l.queue_off = align_up(l.flags_off + l.flags_bytes, 256);
  l.ctrl_off = l.queue_off;
  l.trace_off = l.ctrl_off + (size_t)kCtrlWords * 4;
  l.total = l.trace_off + (size_t)kMaxTraceCtas * kTraceWords * 8;
  return l;
}

int check_desc(const gemm_rs_desc* d) {
  if (!d) return GEMM_RS_ERR_INVALID_ARG;
  if (d->world != GEMM_RS_WORLD) return GEMM_RS_ERR_INVALID_ARG;
  if (d->reducer_warps < 0 || d->reducer_warps > kMaxReducerWarps) return GEMM_RS_ERR_INVALID_ARG;
  if (d->grid < 0 || d->band_m < 0) return GEMM_RS_ERR_INVALID_ARG;
  if (d->unit_rows != 0 && d->unit_rows != 4 && d->unit_rows != 8 && d->unit_rows != 16 &&
      d->unit_rows != 32)
    return GEMM_RS_ERR_INVALID_ARG;
  if (d->mma_ctas < 0 || d->mma_ctas > 2) return GEMM_RS_ERR_INVALID_ARG;
  if (d->chunks < 0 || d->chunks > kMaxChunks) return GEMM_RS_ERR_INVALID_ARG;
  if (d->replicas != 0 && d->replicas != 1 && d->replicas != kWorld) return GEMM_RS_ERR_INVALID_ARG;
  if (d->op != GEMM_RS_OP_RS && d->op != GEMM_RS_OP_AG) return GEMM_RS_ERR_INVALID_ARG;
  if (d->adaptive != 0 && d->adaptive != 1) return GEMM_RS_ERR_INVALID_ARG;
  if (d->tail_waves < 0 || d->tail_waves > 64) return GEMM_RS_ERR_INVALID_ARG;
  if (d->half_regions < -1 || d->half_regions > 4096) return GEMM_RS_ERR_INVALID_ARG;
  if (d->copy_engines < -1 || d->copy_engines > kMaxCopyStreams) return GEMM_RS_ERR_INVALID_ARG;
  if (d->op == GEMM_RS_OP_AG && d->replicas > 1) return GEMM_RS_ERR_INVALID_ARG;
  if (d->M < 0 || d->N < 0 || d->K < 0) return GEMM_RS_ERR_UNSUPPORTED_SHAPE;
  if (d->M % 8 || d->N % 8 || d->K % 64) return GEMM_RS_ERR_UNSUPPORTED_SHAPE;
  // TMA coordinates and kernel indices are 32-bit.
  if (d->M > (1ll << 30) || d->N > (1ll << 30) || d->K / 8 > (1ll << 30))
    return GEMM_RS_ERR_UNSUPPORTED_SHAPE;
  if (d->op == GEMM_RS_OP_AG) {
    // out rows of N/8 elements must stay 16-byte aligned; K is every rank's
    if (d->N % 64) return GEMM_RS_ERR_UNSUPPORTED_SHAPE;
    if (d->K > (1ll << 30) || (d->M / 8) * d->K > (1ll << 40)) return GEMM_RS_ERR_UNSUPPORTED_SHAPE;
  }
  const int64_t cols = d->op == GEMM_RS_OP_AG ? d->N / kWorld : d->N;
  const int64_t mt = (d->M + kBM - 1) / kBM, nt = (cols + kBN - 1) / kBN;
  // tile order positions (half-width tiles count twice) stay below 2^31
  if (mt * nt * kWorld >= (1ll << 30)) return GEMM_RS_ERR_UNSUPPORTED_SHAPE;
  return GEMM_RS_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// Stream-ordered 32-bit write (the all-gather's copy-engine path publishes a
// copied shard's count with it, after the copy on the same stream).
PFN_cuStreamWriteValue32_v11070 write_value_fn() {
  static PFN_cuStreamWriteValue32_v11070 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuStreamWriteValue32", &ptr, 11070, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuStreamWriteValue32_v11070>(ptr);
  }
  return fn;
}

// 3-D bf16 tensor map, 128-byte swizzle, zero fill out of bounds.
bool make_map(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
              uint64_t s1_bytes, uint64_t s2_bytes, uint32_t b0, uint32_t b1) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {s1_bytes, s2_bytes};
  cuuint32_t box[3] = {b0, b1, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// W [8][rows][cols] as the 4-D map of GemmParams::tmap_w4: one box holds a
// CTA's columns of a 64-row stage (pair: 128 columns, one CTA: 256) as
// consecutive 8 KiB blocks of 64 columns, the layout the 3-D boxes gave.
// Leaves p->w4 = 0 (the kernel then copies 64 columns at a time) when the
// rows are not whole 64-column blocks.
bool make_map_w4(GemmParams* p, const void* w, uint64_t cols, uint64_t rows, int pair) {
  p->w4 = 0;
  if (cols % 64) return true;
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[4] = {64, rows, cols / 64, (cuuint64_t)kWorld};
  cuuint64_t strides[3] = {cols * 2, 128, cols * 2 * rows};
  cuuint32_t box[4] = {64, (cuuint32_t)kBK, (cuuint32_t)(kBN / pair / 64), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(&p->tmap_w4, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(w), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  p->w4 = 1;
  return true;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int mma_ctas_of(const gemm_rs_desc* d) { return d->mma_ctas > 0 ? d->mma_ctas : kDefaultMmaCtas; }
int replicas_of(const gemm_rs_desc* d) { return d->replicas > 1 ? d->replicas : 1; }

// First region completed by the last `waves` waves of tiles (tiles are
// claimed in order, `lanes` at a time; a region's 8 rank tiles are
// consecutive).
long long tail_region_of(long long tiles, long long lanes, long long regions, int waves) {
  long long first_last_wave_tile = tiles - lanes * waves;
  if (first_last_wave_tile < 0) first_last_wave_tile = 0;
  long long r = first_last_wave_tile / kWorld;
  return r < regions ? r : regions;
}

// Reduce items of a run: `splits` per 128-row block, 32 (4-row items) per
// block of a tail region.
long long items_of(long long blocks, int blocks_per_region, long long tail_region, int splits) {
  const long long tail_blocks = blocks - tail_region * blocks_per_region;
  return (blocks - tail_blocks) * splits + tail_blocks * (kBM / 4);
}

// kind: Kind (GEMM only, fused reduce-scatter, fused all-gather); ctas: CTAs
// of the cluster that share a tile (1 or 2).
template <int kKind>
const void* kernel_for(int ctas) {
  if (ctas == 2) return reinterpret_cast<const void*>(gemm_rs_kernel<kKind, 2>);
  return reinterpret_cast<const void*>(gemm_rs_kernel<kKind, 1>);
}
const void* gemm_kernel(int kind, int ctas) {
  if (kind == kKindRS) return kernel_for<kKindRS>(ctas);
  if (kind == kKindAG) return kernel_for<kKindAG>(ctas);
  return kernel_for<kKindGemm>(ctas);
}

template <int kKind>
int smem_for(int ctas) {
  return ctas == 2 ? TileCfg<kKind, 2>::kSmemAlloc : TileCfg<kKind, 1>::kSmemAlloc;
}
// Dynamic shared memory of the GEMM kernel of a Kind (stage counts differ).
int gemm_smem(int kind, int ctas) {
  if (kind == kKindRS) return smem_for<kKindRS>(ctas);
  if (kind == kKindAG) return smem_for<kKindAG>(ctas);
  return smem_for<kKindGemm>(ctas);
}
// The largest of them (what a plan needs from the device).
int gemm_smem_max(int ctas) {
  int m = gemm_smem(kKindGemm, ctas);
  for (int k = kKindRS; k <= kKindAG; ++k)
    if (gemm_smem(k, ctas) > m) m = gemm_smem(k, ctas);
  return m;
}

void fill_launch(cudaLaunchConfig_t* cfg, cudaLaunchAttribute* attr, int pair, int kind,
                 int grid, int threads, cudaStream_t st, bool overlap_previous = true) {
  memset(cfg, 0, sizeof(*cfg));
  cfg->gridDim = dim3((unsigned)grid);
  cfg->blockDim = dim3((unsigned)threads);
  cfg->dynamicSmemBytes = (size_t)gemm_smem(kind, pair);
  cfg->stream = st;
  // No co-residency is needed: GEMM tiles are claimed from an atomic ticket
  // by whichever CTAs run, and producers never wait for reducers.
  int n = 0;
  if (pair > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = (unsigned)pair;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  if (overlap_previous) {
    // programmatic dependent launch: the kernel's set-up may overlap the
    // previous kernel on the stream; it waits for that kernel (griddep_wait)
    // before its first access to global memory.  (The standalone reduce,
    // gather and zero kernels are launched plainly: a reduce launched this way
    // behind the GEMM made the unfused run 7 us slower on 2048 x 8192 x 8192.)
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg->attrs = attr;
  cfg->numAttrs = n;
}

// One launch of the persistent GEMM kernel of the given Kind.
int launch_gemm_kernel(int pair, int kind, int grid, int threads, const GemmParams& p,
                       cudaStream_t st) {
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[3];
  fill_launch(&cfg, attr, pair, kind, grid, threads, st);
  void* args[] = {const_cast<GemmParams*>(&p)};
  if (cudaLaunchKernelExC(&cfg, gemm_kernel(kind, pair), args) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_RS_ERR_CUDA;
  }
  return GEMM_RS_OK;
}

// Set the shared-memory limit of the GEMM kernels; persistent grid size
// (CTAs) for `pair` CTAs per MMA: one CTA per SM, whole clusters only.
int prepare_kernels(int dev, int num_sms, int pair, int requested, int threads_fused, int* grid) {
  for (int pr = 1; pr <= 2; ++pr)
    for (int kind = kKindGemm; kind <= kKindAG; ++kind)
      if (cudaFuncSetAttribute(gemm_kernel(kind, pr), cudaFuncAttributeMaxDynamicSharedMemorySize,
                               gemm_smem(kind, pr)) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_RS_ERR_CUDA;
      }
  (void)dev;
  int g = requested > 0 && requested < num_sms ? requested : num_sms;
  if (pair > 1) {
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[3];
    fill_launch(&cfg, attr, pair, kKindRS, pair * (num_sms / pair), threads_fused, 0, false);
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, gemm_kernel(kKindRS, pair), &cfg) != cudaSuccess) {
      cudaGetLastError();
      return GEMM_RS_ERR_CUDA;
    }
    if (clusters < 1) return GEMM_RS_ERR_UNSUPPORTED_DEVICE;
    int n_clusters = g / pair;
    if (n_clusters > clusters) n_clusters = clusters;
    if (n_clusters < 1) n_clusters = 1;
    g = pair * n_clusters;
  }
  *grid = g;
  return GEMM_RS_OK;
}

}  // namespace

struct gemm_rs_plan_s {
  gemm_rs_desc d;
  int device = 0, num_sms = 0;
  int pair = 2, tile_rows = 256;
  int grid = 0, reducer_warps = 0, band = 1, unit_rows = 16, splits = 8, blocks_per_region = 2;
  long long tail_region = 0, half_region = 0;
  int mt = 0, nt = 0, num_kb = 0;
  long long tiles = 0, items = 0;
  Layout lay;
  uint32_t epoch = 0;
  void* last_ws = nullptr;
  const void* map_A = nullptr;
  const void* map_W = nullptr;
  void* map_ws = nullptr;
  bool maps_valid = false;
  GemmParams params;
  // CHUNKED: row chunks, and the second stream and events (created on first use)
  int chunks = 0, chunk_rows = 0;
  cudaStream_t side = nullptr;
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
  cudaEvent_t ev_chunk[kMaxChunks] = {};
  // all-gather + GEMM (op == GEMM_RS_OP_AG)
  bool ag = false;
  int shard_rows = 0, ag_direct = 0, chunks_per_shard = 0, first_round = 0;
  long long copy_items = 0;
  // FUSED all-gather by copy engines: side streams and events (created on first use)
  int copy_engines = 0;
  cudaStream_t copy_st[kMaxCopyStreams] = {};
  cudaEvent_t copy_fork = nullptr;
  cudaEvent_t copy_join[kMaxCopyStreams] = {};
};

extern "C" {

const char* gemm_rs_strerror(int code) {
  switch (code) {
    case GEMM_RS_OK: return "ok";
    case GEMM_RS_ERR_INVALID_ARG: return "invalid argument";
    case GEMM_RS_ERR_UNSUPPORTED_SHAPE: return "unsupported shape (need M%8==0, N%8==0, K%64==0)";
    case GEMM_RS_ERR_UNSUPPORTED_DEVICE: return "no CUDA device, or not compute capability 10.3";
    case GEMM_RS_ERR_CUDA: return "CUDA call or kernel launch failed";
    case GEMM_RS_ERR_TIMEOUT: return "a device-side wait timed out; that run's output is incomplete";
    case GEMM_RS_ERR_MISALIGNED: return "buffer not 16-byte aligned";
    case GEMM_RS_ERR_WORKSPACE: return "workspace missing";
    case GEMM_RS_ERR_TOO_LARGE:
      return "problem larger than the static scratch of the no-allocation entry point";
    case GEMM_RS_ERR_INCOMPLETE:
      return "a fused run ended with output blocks whose 8 partials never all arrived";
    default: return "unknown status";
  }
}

int gemm_rs_schedule(const gemm_rs_desc* d, int64_t idx, int32_t* rank, int32_t* mt,
                     int32_t* nt, int32_t* half) {
  int rc = check_desc(d);
  if (rc) return rc;
  if (!rank || !mt || !nt) return GEMM_RS_ERR_INVALID_ARG;
  const int pair = mma_ctas_of(d);
  const int tile_rows = kBM * pair;
  const bool ag = d->op == GEMM_RS_OP_AG;
  const int64_t cols = ag ? d->N / kWorld : d->N;
  const int mtc = (int)((d->M + tile_rows - 1) / tile_rows), ntc = (int)((cols + kBN - 1) / kBN);
  const long long regions = (long long)mtc * ntc;
  const long long half_region = (!ag && pair == 2) ? half_region_of(regions, d->half_regions) : regions;
  const long long tiles = tiles_of(regions, half_region);
  if (idx < 0 || idx >= tiles) return GEMM_RS_ERR_INVALID_ARG;
  const int band =
      d->band_m > 0 ? (d->band_m < mtc ? d->band_m : mtc) : auto_band(d->M, d->K, tile_rows);
  const TileCoord t = ag ? ag_tile_at(idx, mtc, ntc, (int)(d->M / kWorld), tile_rows, band)
                         : tile_at(idx, mtc, ntc, band, half_region);
  *rank = t.rank;
  *mt = t.mt;
  *nt = t.nt;
  if (half) *half = t.half;
  return GEMM_RS_OK;
}

int gemm_rs_create(const gemm_rs_desc* d, gemm_rs_t* plan, size_t* workspace_bytes) {
  if (!plan) return GEMM_RS_ERR_INVALID_ARG;
  *plan = nullptr;
  int rc = check_desc(d);
  if (rc) return rc;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_RS_ERR_UNSUPPORTED_DEVICE;
  }
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_RS_ERR_UNSUPPORTED_DEVICE;
  }
  if (prop.major != 10 || prop.minor != 3) return GEMM_RS_ERR_UNSUPPORTED_DEVICE;
  const int pair = mma_ctas_of(d);
  if (prop.sharedMemPerBlockOptin < (size_t)gemm_smem_max(pair)) return GEMM_RS_ERR_UNSUPPORTED_DEVICE;
  // reducer warps (reduce-scatter) or copy warps (all-gather: 2 keep the
  // copies ahead of the tiles with the least interference)
  const int reducer_warps = d->reducer_warps > 0 ? d->reducer_warps : default_reducer_warps(d);
  int grid = 0;
  rc = prepare_kernels(dev, prop.multiProcessorCount, pair, d->grid,
                       32 * cta_warps(reducer_warps), &grid);
  if (rc) return rc;

  gemm_rs_plan_s* h = new (std::nothrow) gemm_rs_plan_s();
  if (!h) return GEMM_RS_ERR_CUDA;
  h->d = *d;
  h->device = dev;
  h->num_sms = prop.multiProcessorCount;
  h->pair = pair;
  h->tile_rows = kBM * pair;
  h->mt = (int)((d->M + h->tile_rows - 1) / h->tile_rows);
  h->nt = (int)((d->N + kBN - 1) / kBN);
  h->num_kb = (int)((d->K / kWorld + kBK - 1) / kBK);
  // the last regions in half-width tiles (CTA-pair tiles of the row-parallel layer)
  const long long regions = (long long)h->mt * h->nt;
  h->half_region = (d->op == GEMM_RS_OP_RS && pair == 2) ? half_region_of(regions, d->half_regions)
                                                        : regions;
  h->tiles = tiles_of(regions, h->half_region);
  h->grid = grid;
  h->reducer_warps = reducer_warps;
  h->band = d->band_m > 0 ? (d->band_m < h->mt ? d->band_m : h->mt)
                          : auto_band(d->M, d->K, h->tile_rows);
  if (h->band < 1) h->band = 1;
  h->unit_rows = d->unit_rows > 0 ? d->unit_rows : default_unit_rows(d);
  h->splits = kBM / h->unit_rows;
  h->blocks_per_region = h->tile_rows / kBM;
  const long long blocks = (long long)h->mt * h->nt * h->blocks_per_region;
  h->tail_region = tail_region_of(kWorld * regions, h->grid / pair, regions,
                                  d->tail_waves > 0 ? d->tail_waves : kDefaultTailWaves);
  h->items = items_of(blocks, h->blocks_per_region, h->tail_region, h->splits);
  h->lay = layout_for(d->M, d->N, blocks, h->items);
  {  // CHUNKED: whole tile rows per chunk
    const int want = d->chunks > 0 ? d->chunks : kDefaultChunks;
    const long long per = (d->M + want - 1) / want;
    long long rows = (per + h->tile_rows - 1) / h->tile_rows * h->tile_rows;
    if (rows < 8) rows = 8;
    h->chunk_rows = (int)rows;
    h->chunks = d->M > 0 ? (int)((d->M + rows - 1) / rows) : 0;
  }
  if (d->op == GEMM_RS_OP_AG) {
    h->ag = true;
    const int64_t cols = d->N / kWorld;  // each rank's column shard of W
    h->nt = (int)((cols + kBN - 1) / kBN);
    h->num_kb = (int)((d->K + kBK - 1) / kBK);
    h->tiles = (long long)kWorld * h->mt * h->nt;
    h->half_region = (long long)h->mt * h->nt;  // no half-width tiles
    // bands inside one rank's GEMM: A rows of that rank's gathered buffer
    h->band = d->band_m > 0 ? (d->band_m < h->mt ? d->band_m : h->mt)
                            : auto_band(d->M, d->K, h->tile_rows);
    if (h->band < 1) h->band = 1;
    h->shard_rows = (int)(d->M / kWorld);
    h->ag_direct = h->shard_rows > 0 && h->shard_rows % h->tile_rows == 0;
    const long long shard_elems = (long long)h->shard_rows * d->K;
    h->chunks_per_shard = (int)((shard_elems + kCopyChunk - 1) / kCopyChunk);
    h->first_round = h->ag_direct;
    h->copy_items = (long long)(kWorld - h->first_round) * kWorld * h->chunks_per_shard;
    h->copy_engines = d->copy_engines != 0 ? d->copy_engines : kDefaultCopyEngines;
    h->items = 0;
    h->tail_region = 0;
    h->chunks = 0;
    h->lay = layout_ag(d->M, d->K);
  }
  if (h->d.timeout_ns == 0) h->d.timeout_ns = kDefaultTimeoutNs;
  if (workspace_bytes) *workspace_bytes = h->lay.total;
  *plan = h;
  return GEMM_RS_OK;
}

int gemm_rs_get_info(gemm_rs_t h, gemm_rs_info* info) {
  if (!h || !info) return GEMM_RS_ERR_INVALID_ARG;
  memset(info, 0, sizeof(*info));
  info->num_sms = h->num_sms;
  info->grid = h->grid;
  info->threads_fused = 32 * cta_warps(h->reducer_warps);
  info->threads_gemm = 32 * cta_warps(0);
  info->smem_bytes = gemm_smem_max(h->pair);
  info->band_m = h->band;
  info->unit_rows = h->unit_rows;
  info->mt = h->mt;
  info->nt = h->nt;
  info->tiles = h->tiles;
  info->units = h->items;
  info->workspace_bytes = (int64_t)h->lay.total;
  info->staging_bytes = (int64_t)h->lay.staging_bytes;
  const bool empty = h->d.M == 0 || h->d.N == 0;
  info->launches[GEMM_RS_FUSED] = empty ? 0 : 1;
  info->launches[GEMM_RS_UNFUSED] = empty ? 0 : (h->d.K == 0 ? 1 : 2);
  info->launches[GEMM_RS_GEMM_ONLY] = empty ? 0 : 1;
  info->launches[GEMM_RS_RS_ONLY] = empty ? 0 : 1;
  info->launches[GEMM_RS_CHUNKED] = empty ? 0 : (h->d.K == 0 ? 1 : 2 * h->chunks);
  info->chunks = h->chunks;
  info->replicas = replicas_of(&h->d);
  info->op = h->d.op;
  info->queue_offset = (int64_t)h->lay.queue_off;
  if (h->ag) {
    info->launches[GEMM_RS_RS_ONLY] = empty || h->d.K == 0 ? 0 : 1;  // the gather kernel
    info->launches[GEMM_RS_CHUNKED] = 0;                           // not defined
    info->ag_direct = h->ag_direct;
    info->copy_items = h->copy_engines > 0 ? 0 : h->copy_items;
    info->copy_engines = h->copy_engines;
    if (h->copy_engines > 0) info->threads_fused = 32 * cta_warps(0);
  }
  info->mma_ctas = h->pair;
  info->tile_rows = h->tile_rows;
  info->trace_offset = (int64_t)h->lay.trace_off;
  info->half_region = h->half_region;
  return GEMM_RS_OK;
}

int gemm_rs_tune_candidates(const gemm_rs_desc* d, gemm_rs_desc* cands, int max, int* count,
                            size_t* workspace_bytes) {
  int rc = check_desc(d);
  if (rc) return rc;
  if (!count) return GEMM_RS_ERR_INVALID_ARG;
  const bool ag = d->op == GEMM_RS_OP_AG;
  // A candidate is d with some of these fields changed; zeros mean the defaults.
  struct Knobs {
    int ctas, warps, units, band, tail, half;
  };
  auto resolve = [&](Knobs k) {
    Knobs r;
    r.ctas = k.ctas > 0 ? k.ctas : kDefaultMmaCtas;
    r.warps = k.warps > 0 ? k.warps : default_reducer_warps(d);
    r.units = ag ? 0 : (k.units > 0 ? k.units : default_unit_rows(d));
    const int tile_rows = kBM * r.ctas;
    const int mtc = (int)((d->M + tile_rows - 1) / tile_rows);
    const int ab = auto_band(d->M, d->K, tile_rows);
    r.band = k.band > 0 ? (k.band < mtc ? k.band : (mtc > 0 ? mtc : 1)) : ab;
    r.tail = ag ? 0 : (k.tail > 0 ? k.tail : kDefaultTailWaves);
    r.half = (ag || r.ctas != 2 || k.half < 0) ? 0 : k.half;
    return r;
  };
  Knobs list[GEMM_RS_TUNE_MAX];
  int n = 0;
  auto add = [&](Knobs k) {
    const Knobs r = resolve(k);
    for (int i = 0; i < n; ++i) {
      const Knobs q = resolve(list[i]);
      if (q.ctas == r.ctas && q.warps == r.warps && q.units == r.units && q.band == r.band &&
          q.tail == r.tail && q.half == r.half)
        return;  // same plan as an earlier candidate
    }
    if (n < GEMM_RS_TUNE_MAX) list[n++] = k;
  };
  // the requested plan first, then tile shape x communication warps (x item rows)
  add({d->mma_ctas, d->reducer_warps, d->unit_rows, d->band_m, d->tail_waves, d->half_regions});
  static const int kCtas[2] = {2, 1};
  static const int kWarpsRs[3] = {2, 4, 5}, kWarpsAg[3] = {1, 2, 4};
  static const int kUnits[2] = {8, 16};
  for (int c = 0; c < 2; ++c)
    for (int w = 0; w < 3; ++w)
      for (int u = 0; u < (ag ? 1 : 2); ++u)
        add({kCtas[c], ag ? kWarpsAg[w] : kWarpsRs[w], ag ? 0 : kUnits[u], d->band_m, d->tail_waves,
             d->half_regions});
  // tile-order swizzle: narrower L2 bands than the automatic one (FLUX page,
  // TL;DR: tile coordinate swizzling), for the requested tile shape and warps
  {
    const Knobs r = resolve({d->mma_ctas, d->reducer_warps, d->unit_rows, d->band_m, d->tail_waves,
                             d->half_regions});
    const int ab = auto_band(d->M, d->K, kBM * r.ctas);
    for (int div = 2; div <= 4; div *= 2)
      if (ab / div >= 1)
        add({d->mma_ctas, d->reducer_warps, d->unit_rows, ab / div, d->tail_waves, d->half_regions});
    // how many final waves of regions are reduced in 4-row items
    if (!ag)
      for (int t : {1, 2, 6})
        add({d->mma_ctas, d->reducer_warps, d->unit_rows, d->band_m, t, d->half_regions});
    // final regions computed in half-width tiles (about one and two waves of
    // half tiles on 76 CTA pairs)
    if (!ag)
      for (int hr : {5, 10})
        add({d->mma_ctas, d->reducer_warps, d->unit_rows, d->band_m, d->tail_waves, hr});
  }
  size_t ws_max = 0;
  for (int i = 0; i < n; ++i) {
    gemm_rs_desc e = *d;
    e.mma_ctas = list[i].ctas;
    e.reducer_warps = list[i].warps;
    e.unit_rows = list[i].units;
    e.band_m = list[i].band;
    e.tail_waves = list[i].tail;
    e.half_regions = list[i].half;
    if (cands && i < max) cands[i] = e;
    // the workspace size depends only on the shape, the tile shape and the item count
    const int tile_rows = kBM * mma_ctas_of(&e);
    size_t bytes;
    if (ag) {
      bytes = layout_ag(e.M, e.K).total;
    } else {
      const int mt = (int)((e.M + tile_rows - 1) / tile_rows), nt = (int)((e.N + kBN - 1) / kBN);
      const long long blocks = (long long)mt * nt * (tile_rows / kBM);
      // the largest item count: every block in 4-row items
      bytes = layout_for(e.M, e.N, blocks, blocks * (kBM / 4)).total;
    }
    if (bytes > ws_max) ws_max = bytes;
  }
  *count = n;
  if (workspace_bytes) *workspace_bytes = ws_max;
  return GEMM_RS_OK;
}

int gemm_rs_tune(const gemm_rs_desc* d, int mode, const void* A, const void* W, void* out,
                 void* ws, size_t ws_bytes, int iters, int rounds, void* stream,
                 gemm_rs_desc* best, float* best_us, float* times_us) {
  gemm_rs_desc cands[GEMM_RS_TUNE_MAX];
  int n = 0;
  int rc = gemm_rs_tune_candidates(d, cands, GEMM_RS_TUNE_MAX, &n, nullptr);
  if (rc) return rc;
  if (!best || iters < 1 || rounds < 1 || !ws) return GEMM_RS_ERR_INVALID_ARG;
  if (n > GEMM_RS_TUNE_MAX) n = GEMM_RS_TUNE_MAX;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  gemm_rs_t plans[GEMM_RS_TUNE_MAX] = {};
  float per_round[GEMM_RS_TUNE_MAX][16];
  bool ok[GEMM_RS_TUNE_MAX];
  if (rounds > 16) rounds = 16;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) {
    cudaGetLastError();
    if (e0) cudaEventDestroy(e0);
    return GEMM_RS_ERR_CUDA;
  }
  // Plans share the caller's workspace: before a plan's launches, make it
  // clear the counters and restart its epoch (another plan advanced them).
  auto run_plan = [&](int i) {
    plans[i]->last_ws = nullptr;
    return gemm_rs_run(plans[i], mode, A, W, out, ws, stream);
  };
  for (int i = 0; i < n; ++i) {
    size_t need = 0;
    ok[i] = gemm_rs_create(&cands[i], &plans[i], &need) == GEMM_RS_OK && need <= ws_bytes;
    for (int w = 0; ok[i] && w < 3; ++w) ok[i] = run_plan(i) == GEMM_RS_OK;
    if (ok[i]) ok[i] = gemm_rs_status(plans[i], stream) == GEMM_RS_OK;
  }
  for (int r = 0; r < rounds; ++r)
    for (int i = 0; i < n; ++i) {
      if (!ok[i]) continue;
      plans[i]->last_ws = nullptr;
      if (gemm_rs_run(plans[i], mode, A, W, out, ws, stream) != GEMM_RS_OK) {  // clears, warms
        ok[i] = false;
        continue;
      }
      cudaEventRecord(e0, st);
      bool good = true;
      for (int k = 0; k < iters && good; ++k)
        good = gemm_rs_run(plans[i], mode, A, W, out, ws, stream) == GEMM_RS_OK;
      cudaEventRecord(e1, st);
      float ms = 0.f;
      if (!good || cudaEventSynchronize(e1) != cudaSuccess ||
          cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess ||
          gemm_rs_status(plans[i], stream) != GEMM_RS_OK) {
        cudaGetLastError();
        ok[i] = false;
        continue;
      }
      per_round[i][r] = ms * 1000.f / (float)iters;
    }
  int bi = -1;
  float bt = 0.f;
  float med[GEMM_RS_TUNE_MAX];
  for (int i = 0; i < n; ++i) {
    float t = -1.f;
    if (ok[i]) {  // median over rounds (insertion sort of a few values)
      float v[16];
      for (int r = 0; r < rounds; ++r) v[r] = per_round[i][r];
      for (int a = 1; a < rounds; ++a)
        for (int b = a; b > 0 && v[b] < v[b - 1]; --b) {
          const float x = v[b];
          v[b] = v[b - 1];
          v[b - 1] = x;
        }
      t = v[rounds / 2];
      if (bi < 0 || t < bt) {
        bi = i;
        bt = t;
      }
    }
    med[i] = t;
    if (times_us) times_us[i] = t;
    if (plans[i]) gemm_rs_destroy(plans[i]);
  }
  // Run-to-run noise is a few percent: keep the requested plan (candidate 0)
  // unless the fastest candidate beats it by more than 1%.
  if (bi > 0 && ok[0] && med[0] > 0.f && bt > 0.99f * med[0]) {
    bi = 0;
    bt = med[0];
  }
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  if (bi < 0) return GEMM_RS_ERR_CUDA;
  *best = cands[bi];
  if (best_us) *best_us = bt;
  return GEMM_RS_OK;
}

int gemm_rs_destroy(gemm_rs_t h) {
  if (!h) return GEMM_RS_OK;
  if (h->side) {
    cudaStreamDestroy(h->side);
    cudaEventDestroy(h->ev_fork);
    cudaEventDestroy(h->ev_join);
    for (int c = 0; c < kMaxChunks; ++c)
      if (h->ev_chunk[c]) cudaEventDestroy(h->ev_chunk[c]);
  }
  for (int e = 0; e < kMaxCopyStreams; ++e) {
    if (h->copy_st[e]) cudaStreamDestroy(h->copy_st[e]);
    if (h->copy_join[e]) cudaEventDestroy(h->copy_join[e]);
  }
  if (h->copy_fork) cudaEventDestroy(h->copy_fork);
  delete h;
  return GEMM_RS_OK;
}

static int launch_gemm(gemm_rs_t h, bool fused, cudaStream_t st) {
  return launch_gemm_kernel(h->pair, fused ? kKindRS : kKindGemm, h->grid,
                            32 * cta_warps(fused ? h->reducer_warps : 0), h->params, st);
}

// Reduce kernel over output rows [row0, row0 + rows).
static int launch_rs_rows(gemm_rs_t h, const void* ws, void* out, long long row0, long long rows,
                          cudaStream_t st) {
  const long long plane = (long long)h->d.M * h->d.N;  // between rank planes and output copies
  const long long elems = rows * h->d.N;
  long long blocks = (elems / 8 + 255) / 256;
  const long long cap = (long long)h->num_sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  rs_reduce_kernel<<<(unsigned)blocks, 256, 0, st>>>(
      static_cast<const uint16_t*>(ws) + row0 * h->d.N,
      static_cast<uint16_t*>(out) + row0 * h->d.N, elems, plane, replicas_of(&h->d), plane);
  return cudaGetLastError() == cudaSuccess ? GEMM_RS_OK : GEMM_RS_ERR_CUDA;
}

static int launch_rs(gemm_rs_t h, const void* ws, void* out, cudaStream_t st) {
  return launch_rs_rows(h, ws, out, 0, h->d.M, st);
}

// The prior stream-overlap method: GEMM of chunk c on `st`, reduce of chunk c
// on the plan's second stream once that GEMM is done, so the reduce of chunk c
// overlaps the GEMM of chunk c+1.  Same kernels and arithmetic as UNFUSED.
static int run_chunked(gemm_rs_t h, const void* A, void* out, void* ws, cudaStream_t st) {
  if (!h->side) {
    if (cudaStreamCreateWithFlags(&h->side, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&h->ev_fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&h->ev_join, cudaEventDisableTiming) != cudaSuccess) {
      cudaGetLastError();
      return GEMM_RS_ERR_CUDA;
    }
    for (int c = 0; c < h->chunks; ++c)
      if (cudaEventCreateWithFlags(&h->ev_chunk[c], cudaEventDisableTiming) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_RS_ERR_CUDA;
      }
  }
  const gemm_rs_desc& d = h->d;
  const uint64_t Kr = (uint64_t)(d.K / kWorld);
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  if (cudaEventRecord(h->ev_fork, st) != cudaSuccess ||
      cudaStreamWaitEvent(h->side, h->ev_fork, 0) != cudaSuccess)
    return GEMM_RS_ERR_CUDA;
  for (int c = 0; c < h->chunks; ++c) {
    const long long row0 = (long long)c * h->chunk_rows;
    long long rows = d.M - row0;
    if (rows > h->chunk_rows) rows = h->chunk_rows;
    GemmParams p = h->params;  // the whole problem's maps and settings, narrowed to the chunk
    if (!make_map(&p.tmap_a, static_cast<const uint8_t*>(A) + row0 * Kr * 2, Kr, (uint64_t)rows,
                  kWorld, Kr * 2, Kr * 2 * (uint64_t)d.M, kBK, kBM))
      return GEMM_RS_ERR_CUDA;
    p.stage = reinterpret_cast<uint16_t*>(wsb) + row0 * d.N;  // rank planes stay M * N apart
    if (!make_map(&p.tmap_s, p.stage, (uint64_t)d.N, (uint64_t)rows, kWorld, (uint64_t)d.N * 2,
                  (uint64_t)d.N * 2 * (uint64_t)d.M, 64, 32))
      return GEMM_RS_ERR_CUDA;
    p.M = (int)rows;
    p.mt_count = (int)((rows + h->tile_rows - 1) / h->tile_rows);
    const long long chunk_regions = (long long)p.mt_count * h->nt;
    p.half_region = (int)(h->pair == 2 ? half_region_of(chunk_regions, d.half_regions) : chunk_regions);
    p.num_tiles = tiles_of(chunk_regions, p.half_region);
    p.band = d.band_m > 0 ? (d.band_m < p.mt_count ? d.band_m : p.mt_count)
                          : auto_band(rows, d.K, h->tile_rows);
    if (p.band < 1) p.band = 1;
    p.staging_in_l2 = 0;
    p.trace = nullptr;
    int rc = launch_gemm_kernel(h->pair, kKindGemm, h->grid, 32 * cta_warps(0), p, st);
    if (rc != GEMM_RS_OK) return rc;
    if (cudaEventRecord(h->ev_chunk[c], st) != cudaSuccess ||
        cudaStreamWaitEvent(h->side, h->ev_chunk[c], 0) != cudaSuccess)
      return GEMM_RS_ERR_CUDA;
    rc = launch_rs_rows(h, wsb, out, row0, rows, h->side);
    if (rc != GEMM_RS_OK) return rc;
  }
  if (cudaEventRecord(h->ev_join, h->side) != cudaSuccess ||
      cudaStreamWaitEvent(st, h->ev_join, 0) != cudaSuccess)
    return GEMM_RS_ERR_CUDA;
  return GEMM_RS_OK;
}

static int launch_zero(gemm_rs_t h, void* p, size_t bytes, cudaStream_t st) {
  long long n16 = (long long)(bytes / 16);
  long long blocks = (n16 + 255) / 256;
  const long long cap = (long long)h->num_sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  zero_fill_kernel<<<(unsigned)blocks, 256, 0, st>>>(static_cast<uint4*>(p), n16);
  return cudaGetLastError() == cudaSuccess ? GEMM_RS_OK : GEMM_RS_ERR_CUDA;
}

// The all-gather + GEMM layer (op == GEMM_RS_OP_AG); see the header.
static int launch_gather(gemm_rs_t h, const void* A, void* gather, cudaStream_t st) {
  const long long rank_elems = h->d.M * h->d.K;
  long long blocks = ((long long)kWorld * rank_elems / 8 + 255) / 256;
  const long long cap = (long long)h->num_sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  ag_gather_kernel<<<(unsigned)blocks, 256, 0, st>>>(static_cast<const uint16_t*>(A),
                                                     static_cast<uint16_t*>(gather), rank_elems);
  return cudaGetLastError() == cudaSuccess ? GEMM_RS_OK : GEMM_RS_ERR_CUDA;
}

// FUSED all-gather by copy engines: fork the plan's side streams off st, then
// per rank (in the order the tiles take the ranks) and per shard (in the
// order the rank's tiles read them: its own shard + 1, + 2, ...) one
// device-to-device copy into the rank's gather buffer, followed on the same
// stream by a write of `target` to that (rank, shard)'s count.  The copies
// run on the copy engines, beside the kernel that holds the SMs.
static int issue_engine_copies(gemm_rs_t h, const void* A, uint8_t* wsb, uint32_t target,
                               cudaStream_t st) {
  const int E = h->copy_engines;
  if (!h->copy_fork) {  // all or nothing: a failed setup leaves no stream behind
    bool ok = cudaEventCreateWithFlags(&h->copy_fork, cudaEventDisableTiming) == cudaSuccess;
    for (int e = 0; ok && e < E; ++e)
      ok = cudaStreamCreateWithFlags(&h->copy_st[e], cudaStreamNonBlocking) == cudaSuccess &&
           cudaEventCreateWithFlags(&h->copy_join[e], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
      for (int e = 0; e < kMaxCopyStreams; ++e) {
        if (h->copy_st[e]) cudaStreamDestroy(h->copy_st[e]);
        if (h->copy_join[e]) cudaEventDestroy(h->copy_join[e]);
        h->copy_st[e] = nullptr;
        h->copy_join[e] = nullptr;
      }
      if (h->copy_fork) cudaEventDestroy(h->copy_fork);
      h->copy_fork = nullptr;
      cudaGetLastError();
      return GEMM_RS_ERR_CUDA;
    }
  }
  auto write_value = write_value_fn();
  if (!write_value) return GEMM_RS_ERR_CUDA;
  if (cudaEventRecord(h->copy_fork, st) != cudaSuccess) return GEMM_RS_ERR_CUDA;
  for (int e = 0; e < E; ++e)
    if (cudaStreamWaitEvent(h->copy_st[e], h->copy_fork, 0) != cudaSuccess) return GEMM_RS_ERR_CUDA;
  const size_t row_bytes = (size_t)h->d.K * 2;
  const size_t shard_bytes = (size_t)h->shard_rows * row_bytes;
  const uint8_t* src = static_cast<const uint8_t*>(A);
  uint32_t* counts = reinterpret_cast<uint32_t*>(wsb + h->lay.flags_off);
  int n = 0;
  for (int r = 0; r < kWorld; ++r)
    for (int k = h->first_round; k < kWorld; ++k) {
      const int s = (r + k) % kWorld;
      cudaStream_t cs = h->copy_st[n++ % E];
      uint8_t* dst = wsb + ((size_t)r * (size_t)h->d.M + (size_t)s * h->shard_rows) * row_bytes;
      if (cudaMemcpyAsync(dst, src + (size_t)s * shard_bytes, shard_bytes, cudaMemcpyDeviceToDevice,
                          cs) != cudaSuccess)
        return GEMM_RS_ERR_CUDA;
      // debug: the first (rank, shard) is copied but never published
      if ((h->d.debug_flags & GEMM_RS_DEBUG_SKIP_ONE_FLAG) && r == 0 && k == h->first_round) continue;
      const CUdeviceptr count = reinterpret_cast<CUdeviceptr>(counts + (size_t)(r * kWorld + s) * kFlagStride);
      if (write_value(reinterpret_cast<CUstream>(cs), count, target, CU_STREAM_WRITE_VALUE_DEFAULT) !=
          CUDA_SUCCESS)
        return GEMM_RS_ERR_CUDA;
    }
  return GEMM_RS_OK;
}

// st waits for the side streams' copies and count writes.
static int join_engine_copies(gemm_rs_t h, cudaStream_t st) {
  if (!h->copy_fork) return GEMM_RS_OK;  // never set up: nothing was queued on a side stream
  for (int e = 0; e < h->copy_engines; ++e)
    if (cudaEventRecord(h->copy_join[e], h->copy_st[e]) != cudaSuccess ||
        cudaStreamWaitEvent(st, h->copy_join[e], 0) != cudaSuccess)
      return GEMM_RS_ERR_CUDA;
  return GEMM_RS_OK;
}

static int run_ag(gemm_rs_t h, int mode, const void* A, const void* W, void* out, void* ws,
                  cudaStream_t st) {
  const gemm_rs_desc& d = h->d;
  if (mode == GEMM_RS_CHUNKED) return GEMM_RS_ERR_INVALID_ARG;
  if (d.M == 0 || d.N == 0) return GEMM_RS_OK;
  const bool needs_a = mode != GEMM_RS_GEMM_ONLY && d.K > 0;  // GEMM_ONLY reads the buffers
  const bool needs_w = mode != GEMM_RS_RS_ONLY && d.K > 0;
  const bool needs_out = mode != GEMM_RS_RS_ONLY;
  if (!ws) return GEMM_RS_ERR_WORKSPACE;
  if ((needs_a && !A) || (needs_w && !W) || (needs_out && !out)) return GEMM_RS_ERR_INVALID_ARG;
  if (!aligned16(ws) || (needs_a && !aligned16(A)) || (needs_w && !aligned16(W)) ||
      (needs_out && !aligned16(out)))
    return GEMM_RS_ERR_MISALIGNED;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess || cur != h->device) return GEMM_RS_ERR_INVALID_ARG;
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  if (ws != h->last_ws) {  // first use of this workspace: clear counts and control words
    if (cudaMemsetAsync(wsb + h->lay.flags_off, 0, h->lay.total - h->lay.flags_off, st) !=
        cudaSuccess)
      return GEMM_RS_ERR_CUDA;
    h->last_ws = ws;
    h->epoch = 0;
  }
  h->maps_valid = false;  // the reduce-scatter maps are not kept across ops
  if (d.K == 0) {  // empty contraction: C is zero, nothing to gather
    if (mode == GEMM_RS_RS_ONLY) return GEMM_RS_OK;
    return launch_zero(h, out, (size_t)d.M * d.N * 2, st);
  }
  if (mode == GEMM_RS_RS_ONLY) return launch_gather(h, A, wsb, st);

  const uint64_t M = (uint64_t)d.M, K = (uint64_t)d.K, cols = (uint64_t)(d.N / kWorld);
  const uint64_t shard = M / kWorld;
  GemmParams& p = h->params;
  memset(&p, 0, sizeof(p));
  const bool fused = mode == GEMM_RS_FUSED;
  // A: the input's row shards (fused: own rows) or the gather buffers
  bool ok = fused ? make_map(&p.tmap_a, A, K, shard, kWorld, K * 2, K * 2 * shard, kBK, kBM) &&
                        make_map(&p.tmap_g, wsb, K, M, kWorld, K * 2, K * 2 * M, kBK, kBM)
                  : make_map(&p.tmap_a, wsb, K, M, kWorld, K * 2, K * 2 * M, kBK, kBM);
  ok = ok && make_map(&p.tmap_b, W, cols, K, kWorld, cols * 2, cols * 2 * K, 64, kBK) &&
       make_map_w4(&p, W, cols, K, h->pair);
  // epilogue stores into the output [8][M][N/8]: 32 x 64 boxes
  ok = ok && make_map(&p.tmap_s, out, cols, M, kWorld, cols * 2, cols * 2 * M, 64, 32);
  if (!ok) return GEMM_RS_ERR_CUDA;
  p.stage = static_cast<uint16_t*>(out);  // the epilogue writes C_r = rank r's plane
  p.plane = (long long)(M * cols);
  p.out = static_cast<uint16_t*>(out);
  p.replicas = 1;
  p.out_stride = p.plane;
  p.ctrl = reinterpret_cast<uint32_t*>(wsb + h->lay.ctrl_off);
  p.flags = reinterpret_cast<uint32_t*>(wsb + h->lay.flags_off);
  p.M = (int)M;
  p.N = (int)cols;
  p.Kr = (int)K;
  p.mt_count = h->mt;
  p.nt_count = h->nt;
  p.band = h->band;
  p.num_kb = h->num_kb;
  p.unit_rows = h->unit_rows;
  p.splits = h->splits;
  p.blocks_per_region = h->blocks_per_region;
  p.tile_rows = h->tile_rows;
  p.num_tiles = h->tiles;
  p.half_region = (int)h->half_region;
  p.debug_flags = d.debug_flags;
  p.timeout_ns = d.timeout_ns;
  p.trace = (d.debug_flags & GEMM_RS_DEBUG_TRACE)
                ? reinterpret_cast<unsigned long long*>(wsb + h->lay.trace_off)
                : nullptr;
  p.ag_src = static_cast<const uint16_t*>(A);
  p.gather = reinterpret_cast<uint16_t*>(wsb);
  p.ag_flags = reinterpret_cast<uint32_t*>(wsb + h->lay.flags_off);
  p.shard_rows = h->shard_rows;
  p.ag_direct = h->ag_direct;
  p.chunks_per_shard = h->chunks_per_shard;
  p.first_round = h->first_round;
  p.ag_order = 1;
  p.copy_items = h->copy_items;
  p.copy_chunk = kCopyChunk;
  // pace the copies when one rank's tiles take at least two waves: then a
  // rank's gathered buffer written one rank ahead is still in L2 when read
  // (FLUX Figure 4 all-gather, M = 2048: 1597 -> 1521 us); shorter ranks
  // leave too little slack for it (QKV 2048 x 10240 x 8192: 251 -> 254 us)
  p.copy_paced = (long long)h->mt * h->nt >= 2LL * (h->grid / h->pair);
  if (fused) {
    h->epoch += 1;
    p.ag_target = (uint32_t)h->chunks_per_shard * h->epoch;  // every copied (rank, shard)
    if (h->copy_engines > 0) {  // copies by the copy engines; the kernel has no copy warps
      p.copy_items = 0;
      int rc = issue_engine_copies(h, A, wsb, p.ag_target, st);
      if (rc == GEMM_RS_OK)
        rc = launch_gemm_kernel(h->pair, kKindAG, h->grid, 32 * cta_warps(0), p, st);
      const int rj = join_engine_copies(h, st);  // also after a failed launch: st follows the copies
      return rc != GEMM_RS_OK ? rc : rj;
    }
    return launch_gemm_kernel(h->pair, kKindAG, h->grid, 32 * cta_warps(h->reducer_warps),
                              p, st);
  }
  if (mode == GEMM_RS_UNFUSED) {
    const int rc = launch_gather(h, A, wsb, st);
    if (rc != GEMM_RS_OK) return rc;
  }
  return launch_gemm_kernel(h->pair, kKindGemm, h->grid, 32 * cta_warps(0), p, st);
}

int gemm_rs_run(gemm_rs_t h, int mode, const void* A, const void* W, void* out, void* ws,
                void* stream) {
  if (!h) return GEMM_RS_ERR_INVALID_ARG;
  if (mode < GEMM_RS_FUSED || mode > GEMM_RS_CHUNKED) return GEMM_RS_ERR_INVALID_ARG;
  if (h->ag) {
    const int rc = run_ag(h, mode, A, W, out, ws, static_cast<cudaStream_t>(stream));
    if (rc != GEMM_RS_OK) cudaGetLastError();
    return rc;
  }
  const gemm_rs_desc& d = h->d;
  if (d.M == 0 || d.N == 0) return GEMM_RS_OK;  // nothing to read or write
  // A and W hold no element when K == 0: their pointers are not used then.
  const bool needs_ab = mode != GEMM_RS_RS_ONLY && d.K > 0;
  const bool needs_out = mode != GEMM_RS_GEMM_ONLY;
  if (!ws) return GEMM_RS_ERR_WORKSPACE;
  if ((needs_ab && (!A || !W)) || (needs_out && !out)) return GEMM_RS_ERR_INVALID_ARG;
  if (!aligned16(ws) || (needs_ab && (!aligned16(A) || !aligned16(W))) ||
      (needs_out && !aligned16(out)))
    return GEMM_RS_ERR_MISALIGNED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess || cur != h->device) return GEMM_RS_ERR_INVALID_ARG;

  uint8_t* wsb = static_cast<uint8_t*>(ws);
  if (ws != h->last_ws) {
    // first use of this workspace: clear flags and control words
    if (cudaMemsetAsync(wsb + h->lay.flags_off, 0, h->lay.total - h->lay.flags_off, st) !=
        cudaSuccess)
      return GEMM_RS_ERR_CUDA;
    h->last_ws = ws;
    h->epoch = 0;
  }

  if (d.K == 0) {  // empty contraction: every partial and the sum are zero
    if (mode == GEMM_RS_GEMM_ONLY) return launch_zero(h, wsb, h->lay.staging_bytes, st);
    if (mode == GEMM_RS_RS_ONLY) return launch_rs(h, wsb, out, st);
    return launch_zero(h, out, (size_t)replicas_of(&d) * d.M * d.N * 2, st);
  }

  if (!h->maps_valid || (needs_ab && (A != h->map_A || W != h->map_W)) || ws != h->map_ws) {
    GemmParams& p = h->params;
    memset(&p, 0, sizeof(p));
    const uint64_t Kr = (uint64_t)(d.K / kWorld);
    const void* a = needs_ab ? A : h->map_A;
    const void* w = needs_ab ? W : h->map_W;
    if (a && w) {
      if (!make_map(&p.tmap_a, a, Kr, (uint64_t)d.M, kWorld, Kr * 2, Kr * 2 * (uint64_t)d.M, kBK,
                    kBM) ||
          !make_map(&p.tmap_b, w, (uint64_t)d.N, Kr, kWorld, (uint64_t)d.N * 2,
                    (uint64_t)d.N * 2 * Kr, 64, kBK) ||
          !make_map_w4(&p, w, (uint64_t)d.N, Kr, h->pair))
        return GEMM_RS_ERR_CUDA;
    }
    // epilogue stores into the staging: 32 x 64 boxes
    if (!make_map(&p.tmap_s, wsb, (uint64_t)d.N, (uint64_t)d.M, kWorld, (uint64_t)d.N * 2,
                  (uint64_t)d.N * 2 * (uint64_t)d.M, 64, 32))
      return GEMM_RS_ERR_CUDA;
    p.stage = reinterpret_cast<uint16_t*>(wsb);
    p.plane = d.M * d.N;
    p.replicas = replicas_of(&d);
    p.out_stride = d.M * d.N;
    p.flags = reinterpret_cast<uint32_t*>(wsb + h->lay.flags_off);
    p.queue = reinterpret_cast<unsigned long long*>(wsb + h->lay.queue_off);
    p.ctrl = reinterpret_cast<uint32_t*>(wsb + h->lay.ctrl_off);
    p.M = (int)d.M;
    p.N = (int)d.N;
    p.Kr = (int)Kr;
    p.mt_count = h->mt;
    p.nt_count = h->nt;
    p.band = h->band;
    p.num_kb = h->num_kb;
    p.unit_rows = h->unit_rows;
    p.splits = h->splits;
    p.blocks_per_region = h->blocks_per_region;
    p.tail_region = (int)h->tail_region;
    p.half_region = (int)h->half_region;
    p.tile_rows = h->tile_rows;
    p.num_tiles = h->tiles;
    p.num_items = h->items;
    p.debug_flags = d.debug_flags;
    p.timeout_ns = d.timeout_ns;
    p.trace = (d.debug_flags & GEMM_RS_DEBUG_TRACE)
                  ? reinterpret_cast<unsigned long long*>(wsb + h->lay.trace_off)
                  : nullptr;
    p.adaptive = d.adaptive;
    p.reducer_warps = h->reducer_warps;
    h->map_A = a;
    h->map_W = w;
    h->map_ws = ws;
    h->maps_valid = a && w;
  }
  h->params.out = static_cast<uint16_t*>(out);

  int rc = GEMM_RS_OK;
  switch (mode) {
    case GEMM_RS_FUSED:
      // The reducers drop whole 128-byte staging lines from L2: only when every
      // line holds one reduce unit's columns (N % 64 == 0 and the staging base on
      // a 128-byte boundary); otherwise a dropped line could take unreduced
      // bytes of a neighbouring unit with it.
      h->params.staging_in_l2 = (d.N % 64 == 0) && (reinterpret_cast<uintptr_t>(wsb) & 127u) == 0 &&
                                !(d.debug_flags & GEMM_RS_DEBUG_NO_STAGING_L2);
      h->epoch += 1;
      h->params.epoch = h->epoch;
      rc = launch_gemm(h, true, st);
      break;
    case GEMM_RS_UNFUSED:
      h->params.staging_in_l2 = 0;
      rc = launch_gemm(h, false, st);
      if (rc == GEMM_RS_OK) rc = launch_rs(h, wsb, out, st);
      break;
    case GEMM_RS_GEMM_ONLY:
      h->params.staging_in_l2 = 0;
      rc = launch_gemm(h, false, st);
      break;
    case GEMM_RS_RS_ONLY:
      rc = launch_rs(h, wsb, out, st);
      break;
    case GEMM_RS_CHUNKED:
      rc = run_chunked(h, h->map_A, out, wsb, st);
      break;
  }
  if (rc != GEMM_RS_OK) cudaGetLastError();
  return rc;
}

int gemm_rs_status(gemm_rs_t h, void* stream) {
  if (!h) return GEMM_RS_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_RS_ERR_CUDA;
  }
  if (!h->last_ws) return GEMM_RS_OK;
  static thread_local uint32_t words[kCtrlWords];
  uint8_t* wsb = static_cast<uint8_t*>(h->last_ws);
  if (cudaMemcpyAsync(words, wsb + h->lay.ctrl_off, sizeof(words), cudaMemcpyDeviceToHost, st) !=
          cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_RS_ERR_CUDA;
  }
  const uint32_t err = words[kCtrlError * kCtrlStride];
  if (err == 0) return GEMM_RS_OK;
  // Start clean: zero flags and control words, restart the epoch.
  if (cudaMemsetAsync(wsb + h->lay.flags_off, 0, h->lay.total - h->lay.flags_off, st) !=
          cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_RS_ERR_CUDA;
  }
  h->epoch = 0;
  return (err & (kErrFlagTimeout | kErrPipeTimeout)) ? GEMM_RS_ERR_TIMEOUT
                                                                    : GEMM_RS_ERR_INCOMPLETE;
}

}  // extern "C"

extern "C" int gemm_rs_run_host(gemm_rs_t h, int mode, const void* A_host, const void* W_host,
                                void* out_host, void* A_dev, void* W_dev, void* out_dev,
                                void* ws, void* stream) {
  if (!h) return GEMM_RS_ERR_INVALID_ARG;
  if (mode < GEMM_RS_FUSED || mode > GEMM_RS_CHUNKED) return GEMM_RS_ERR_INVALID_ARG;
  // which buffers a mode reads and writes (all-gather: GEMM_ONLY reads only the
  // gather buffers and W, RS_ONLY is the gather: reads A, writes no output)
  const bool needs_a = h->ag ? mode != GEMM_RS_GEMM_ONLY : mode != GEMM_RS_RS_ONLY;
  const bool needs_w = mode != GEMM_RS_RS_ONLY;
  const bool needs_out = h->ag ? mode != GEMM_RS_RS_ONLY : mode != GEMM_RS_GEMM_ONLY;
  const gemm_rs_desc& d = h->d;
  const size_t a_bytes = (size_t)d.M * (size_t)d.K * 2;  // 8 shards of M x K/8
  const size_t w_bytes = (size_t)d.K * (size_t)d.N * 2;  // 8 shards of K/8 x N
  const size_t o_bytes = (size_t)replicas_of(&d) * (size_t)d.M * (size_t)d.N * 2;
  if ((needs_a && a_bytes && (!A_host || !A_dev)) || (needs_w && w_bytes && (!W_host || !W_dev)) ||
      (needs_out && o_bytes && (!out_host || !out_dev)))
    return GEMM_RS_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (needs_a && a_bytes &&
      cudaMemcpyAsync(A_dev, A_host, a_bytes, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return cudaGetLastError(), GEMM_RS_ERR_CUDA;
  if (needs_w && w_bytes &&
      cudaMemcpyAsync(W_dev, W_host, w_bytes, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return cudaGetLastError(), GEMM_RS_ERR_CUDA;
  int rc = gemm_rs_run(h, mode, A_dev, W_dev, out_dev, ws, stream);
  if (rc != GEMM_RS_OK) return rc;
  if (needs_out && o_bytes &&
      cudaMemcpyAsync(out_host, out_dev, o_bytes, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return cudaGetLastError(), GEMM_RS_ERR_CUDA;
  return GEMM_RS_OK;
}

// ---------------------------------------------------------------------------
// No-allocation entry point (gemm_rs_fused_noalloc).
//
// For callers that may not allocate device memory when they call in (a
// plug-in inside an application that owns the device-memory budget, a serving
// path that forbids cudaMalloc after start-up).  The fused kernel's scratch --
// bf16 staging, per-tile flags, control words -- lives in the file-scope array
// below instead of a caller workspace.  Host code never uses the array's name
// as an address (in host code it is only a stand-in for the device symbol):
// the first call on a device looks up the real device address with
// cudaGetSymbolAddress while that device is current and keeps it.
namespace {
constexpr size_t kNoallocStagingBytes = (size_t)32 << 20;  // 8*M*N*2 <= 32 MiB
constexpr size_t kNoallocFlagBytes = (size_t)4 << 20;      // completion counts + item stamps
constexpr size_t kNoallocCtrlBytes = (size_t)kCtrlWords * 4;
constexpr size_t kNoallocBytes = kNoallocStagingBytes + kNoallocFlagBytes + kNoallocCtrlBytes;
constexpr int kNoallocMaxDevices = 64;
}  // namespace

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoallocBytes];

namespace {
struct NoallocDevice {
  bool ready;
  uint8_t* scratch;  // device address of g_noalloc_scratch on this device
  int num_sms;
  int grid;
};
NoallocDevice g_noalloc_dev[kNoallocMaxDevices];
std::mutex g_noalloc_mu;

// Once per device, with that device current.
int noalloc_setup(int dev, const NoallocDevice** out) {
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoallocDevice& d = g_noalloc_dev[dev];
  if (!d.ready) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return GEMM_RS_ERR_UNSUPPORTED_DEVICE;
    }
    if (major != 10 || minor != 3) return GEMM_RS_ERR_UNSUPPORTED_DEVICE;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return GEMM_RS_ERR_CUDA;
    }
    int grid = 0;
    const int rc = prepare_kernels(dev, sms, kDefaultMmaCtas, 0,
                                   32 * cta_warps(kDefaultReducerWarps), &grid);
    if (rc != GEMM_RS_OK) return rc;
    d.scratch = static_cast<uint8_t*>(p);
    d.num_sms = sms;
    d.grid = grid;
    d.ready = true;
  }
  *out = &d;
  return GEMM_RS_OK;
}
}  // namespace

extern "C" int gemm_rs_fused_noalloc(const void* A, const void* W, void* out, int64_t M, int64_t N,
                                     int64_t K, void* error_word, void* stream) {
  if (M < 0 || N < 0 || K < 0 || M % 8 || N % 8 || K % 64) return GEMM_RS_ERR_UNSUPPORTED_SHAPE;
  if (M > (1ll << 30) || N > (1ll << 30)) return GEMM_RS_ERR_TOO_LARGE;
  const int tile_rows = kBM * kDefaultMmaCtas;
  const int64_t mt = (M + tile_rows - 1) / tile_rows, nt = (N + kBN - 1) / kBN;
  const size_t staging = (size_t)kWorld * (size_t)M * (size_t)N * 2;
  const int64_t blocks = mt * nt * (tile_rows / kBM);
  const int64_t items = blocks * (kBM / 4);  // at most 32 items per block
  const size_t count_bytes = (size_t)blocks * kFlagStride * 4;
  const size_t flag_bytes = align_up(count_bytes, 256) + (size_t)items * kQueueStride * 8;
  if (staging > kNoallocStagingBytes || flag_bytes > kNoallocFlagBytes) return GEMM_RS_ERR_TOO_LARGE;
  const bool empty = M == 0 || N == 0;
  if (!empty && (!out || (K > 0 && (!A || !W)))) return GEMM_RS_ERR_INVALID_ARG;
  if ((!empty && !aligned16(out)) || (!empty && K > 0 && (!aligned16(A) || !aligned16(W))) ||
      (error_word && (reinterpret_cast<uintptr_t>(error_word) & 3u)))
    return GEMM_RS_ERR_MISALIGNED;

  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoallocMaxDevices) {
    cudaGetLastError();
    return GEMM_RS_ERR_UNSUPPORTED_DEVICE;
  }
  const NoallocDevice* nd = nullptr;
  int rc = noalloc_setup(dev, &nd);
  if (rc != GEMM_RS_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* scratch = nd->scratch;
  uint32_t* flags = reinterpret_cast<uint32_t*>(scratch + kNoallocStagingBytes);
  uint32_t* ctrl = reinterpret_cast<uint32_t*>(scratch + kNoallocStagingBytes + kNoallocFlagBytes);

  // The array keeps the previous call's contents: the flags of this problem
  // and the control words must start at zero.
  if ((flag_bytes && cudaMemsetAsync(flags, 0, flag_bytes, st) != cudaSuccess) ||
      cudaMemsetAsync(ctrl, 0, kNoallocCtrlBytes, st) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_RS_ERR_CUDA;
  }

  if (!empty && K == 0) {  // empty contraction: the sum is zero
    const long long n16 = M * N * 2 / 16;
    long long blocks = (n16 + 255) / 256;
    if (blocks > (long long)nd->num_sms * 8) blocks = (long long)nd->num_sms * 8;
    zero_fill_kernel<<<(unsigned)blocks, 256, 0, st>>>(static_cast<uint4*>(out), n16);
    if (cudaGetLastError() != cudaSuccess) return GEMM_RS_ERR_CUDA;
  } else if (!empty) {
    GemmParams p;
    memset(&p, 0, sizeof(p));
    const uint64_t Kr = (uint64_t)(K / kWorld);
    if (!make_map(&p.tmap_a, A, Kr, (uint64_t)M, kWorld, Kr * 2, Kr * 2 * (uint64_t)M, kBK, kBM) ||
        !make_map(&p.tmap_b, W, (uint64_t)N, Kr, kWorld, (uint64_t)N * 2, (uint64_t)N * 2 * Kr, 64,
                  kBK) ||
        !make_map_w4(&p, W, (uint64_t)N, Kr, kDefaultMmaCtas))
      return GEMM_RS_ERR_CUDA;
    if (!make_map(&p.tmap_s, scratch, (uint64_t)N, (uint64_t)M, kWorld, (uint64_t)N * 2,
                  (uint64_t)N * 2 * (uint64_t)M, 64, 32))
      return GEMM_RS_ERR_CUDA;
    p.stage = reinterpret_cast<uint16_t*>(scratch);
    p.staging_in_l2 = (N % 64 == 0);  // as a default plan: the array is 256-byte aligned
    p.plane = M * N;
    p.replicas = 1;
    p.out_stride = M * N;
    p.out = static_cast<uint16_t*>(out);
    p.flags = flags;
    p.queue = reinterpret_cast<unsigned long long*>(reinterpret_cast<uint8_t*>(flags) +
                                                    align_up(count_bytes, 256));
    p.epoch = 1;  // first run on the counts just cleared
    p.ctrl = ctrl;
    p.M = (int)M;
    p.N = (int)N;
    p.Kr = (int)Kr;
    p.mt_count = (int)mt;
    p.nt_count = (int)nt;
    p.band = auto_band(M, K, tile_rows);
    p.num_kb = (int)((Kr + kBK - 1) / kBK);
    gemm_rs_desc dd;  // the default plan's reducer warps and item size for this shape
    memset(&dd, 0, sizeof(dd));
    dd.M = M;
    dd.N = N;
    dd.K = K;
    dd.op = GEMM_RS_OP_RS;
    const int reducers = default_reducer_warps(&dd);
    p.unit_rows = default_unit_rows(&dd);
    p.splits = kBM / p.unit_rows;
    p.blocks_per_region = tile_rows / kBM;
    p.tile_rows = tile_rows;
    p.half_region = (int)half_region_of(mt * nt, 0);
    p.num_tiles = tiles_of(mt * nt, p.half_region);
    const long long tail =
        tail_region_of(kWorld * mt * nt, nd->grid / kDefaultMmaCtas, mt * nt, kDefaultTailWaves);
    p.tail_region = (int)tail;
    p.num_items = items_of(blocks, p.blocks_per_region, tail, p.splits);
    p.timeout_ns = kDefaultTimeoutNs;
    p.reducer_warps = reducers;
    rc = launch_gemm_kernel(kDefaultMmaCtas, kKindRS, nd->grid, 32 * cta_warps(reducers), p, st);
    if (rc != GEMM_RS_OK) return rc;
  }
  if (error_word && cudaMemcpyAsync(error_word, ctrl + kCtrlError * kCtrlStride, sizeof(uint32_t),
                                    cudaMemcpyDeviceToDevice, st) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_RS_ERR_CUDA;
  }
  return GEMM_RS_OK;
}
