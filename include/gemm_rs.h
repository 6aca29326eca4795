/*
 * gemm_rs.h -- C ABI of the fused GEMM + reduce-scatter library (sm_103a).
 *
 * The operation (problem page "A fused GEMM + reduce-scatter kernel hiding
 * 90% of communication on 8 H100 GPUs", sections "What is asked" and "How it
 * gets verified"; FLUX page, abstract and Figure 2): a row-parallel linear
 * layer under tensor parallelism of degree 8.  Rank r holds the K-shard
 * A_r = A[:, r*K/8 : (r+1)*K/8] and W_r = W[r*K/8 : (r+1)*K/8, :], and
 * computes the partial product P_r = A_r W_r in bf16 with fp32 accumulation.
 * The partials are summed across the ranks (reduce) and rank s keeps rows
 * [s*M/8, (s+1)*M/8) of the sum (scatter).
 *
 * All-reduce variant (desc.replicas = 8; mKernel page, sections 3.1, 4 and
 * 5.2, GEMM+AllReduce: reduce within the node, then every rank holds the
 * whole sum): the same reduction, and the reducer of each output unit writes
 * the sum into all 8 ranks' copies of the output, i.e. the all-gather of the
 * reduced slices is fused into the reduction.
 *
 * On one GPU the 8 ranks are virtual.  Each rank's bf16 partial tiles are
 * written to a separate staging region in device memory (standing in for the
 * peer's receive buffer) and published with a per-tile completion flag.
 * Reducers add the 8 partials of an output tile in fp32, in rank order
 * 0..7, and round the total to bf16 (round to nearest even).
 *
 * Memory: the caller owns every device buffer and the CUDA stream.  The plan
 * owns host state only.  All pointers below are device pointers unless a
 * comment says "host".
 *
 * Errors: every entry point returns a gemm_rs_status code.  No C++ exception
 * and no abort crosses this boundary.  A plan serves one stream at a time.
 */
#ifndef GEMM_RS_H
#define GEMM_RS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GEMM_RS_WORLD 8

/* Status codes. */
enum gemm_rs_status {
  GEMM_RS_OK = 0,
  GEMM_RS_ERR_INVALID_ARG = -1,        /* null pointer, world != 8, bad mode or field */
  GEMM_RS_ERR_UNSUPPORTED_SHAPE = -2,  /* M%8, N%8 or K%64 != 0, negative or too large */
  GEMM_RS_ERR_UNSUPPORTED_DEVICE = -3, /* no CUDA device, or not compute capability 10.3 */
  GEMM_RS_ERR_CUDA = -4,               /* a CUDA runtime/driver call or launch failed */
  GEMM_RS_ERR_TIMEOUT = -5,            /* a device-side wait gave up (reported by status) */
  GEMM_RS_ERR_MISALIGNED = -6,         /* a buffer is not 16-byte aligned */
  GEMM_RS_ERR_WORKSPACE = -7,          /* workspace pointer missing for a mode that needs it */
  GEMM_RS_ERR_TOO_LARGE = -8,          /* beyond the fixed scratch of gemm_rs_fused_noalloc */
  GEMM_RS_ERR_INCOMPLETE = -9          /* a fused run ended with output blocks never reduced
                                          (some rank tile's completion never arrived) */
};

/* Execution modes of gemm_rs_run. */
enum gemm_rs_mode {
  GEMM_RS_FUSED = 0,     /* one persistent kernel: tile GEMM + flagged reduce-scatter */
  GEMM_RS_UNFUSED = 1,   /* GEMM kernel writes the staging, then a separate reduce kernel */
  GEMM_RS_GEMM_ONLY = 2, /* only the GEMM kernel (per-rank partials into staging) */
  GEMM_RS_RS_ONLY = 3,   /* only the reduce kernel (reads the staging as it is) */
  GEMM_RS_CHUNKED = 4    /* the prior stream-overlap method: the rows are cut into chunks;
                            the GEMM of chunk c runs on `stream` while the reduce kernel
                            of chunk c-1 runs on a second stream of the plan (FLUX page,
                            Figures 3 and 5); a comparison baseline, same result bits */
};

/* The layer a plan computes (gemm_rs_desc.op).
 *
 * GEMM_RS_OP_RS: the row-parallel layer above (GEMM, then reduce-scatter or
 *   all-reduce).
 * GEMM_RS_OP_AG: the column-parallel partner layer, all-gather then GEMM
 *   (FLUX page, abstract and Figure 1: all-gather fused into the GEMM's
 *   prologue; mKernel page, sections 3.1 and 4: the local shard first, then
 *   the other shards in the order they arrive).  Rank r holds the row shard
 *   A_r = A[r*M/8 : (r+1)*M/8, :] and the column shard W_r = W[:, r*N/8 :
 *   (r+1)*N/8]; it gathers all of A and computes C_r = A W_r (bf16, fp32
 *   accumulation, one rounding).  Layouts: A [8][M/8][K], W [8][K][N/8],
 *   out [8][M][N/8], all row-major bf16; N % 64 == 0.  The workspace holds
 *   the 8 gather buffers [8][M][K] (rank r's copy of every shard) instead of
 *   staging.  Modes: FUSED (copy warps gather while the tiles that need a
 *   shard wait for its completion counts), UNFUSED (a gather kernel, then the
 *   GEMM), GEMM_ONLY (the GEMM from the gather buffers as they are), RS_ONLY
 *   (the gather kernel alone); CHUNKED and replicas = 8 are not defined.
 */
#define GEMM_RS_OP_RS 0
#define GEMM_RS_OP_AG 1

/* Debug switches (gemm_rs_desc.debug_flags). */
#define GEMM_RS_DEBUG_SKIP_ONE_FLAG 0x1u /* FUSED: one producer warp never publishes its
                                            completion, so its block is never queued, the
                                            reducer waiting for it gives up after
                                            timeout_ns and the run reports
                                            GEMM_RS_ERR_TIMEOUT; tests the bounded wait
                                            (all-gather: the first copy item is never
                                            published, so the tiles that need that shard
                                            wait until timeout_ns) */
#define GEMM_RS_DEBUG_NO_STAGING_L2 0x2u /* FUSED: store staging tiles without the L2
                                            evict-last hint and keep them after reduction
                                            (by default reduced staging lines are dropped
                                            from L2 unwritten when N % 64 == 0 and the
                                            workspace is 128-byte aligned) */
#define GEMM_RS_DEBUG_TRACE 0x4u         /* GEMM kernels write, per CTA, four global-timer
                                            stamps (ns, u64): start, epilogue done with its
                                            tiles, MMA issue drained, all warps done; at
                                            workspace + gemm_rs_info.trace_offset (up to
                                            1024 CTAs).  The fused reduce-scatter also
                                            stamps every reduce item when its block became
                                            complete, when a reducer saw that and when it was
                                            done: u64 words 1..3 of a 32-byte slot per item
                                            (items in the order they are reduced) at workspace
                                            + gemm_rs_info.queue_offset (word 0 holds run << 32
                                            | item, item = 128-row block << 5 | part) */

/*
 * Problem description.  Shapes: A is [8][M][K/8] bf16 (row-major, K/8
 * contiguous: rank r's column block of A), W is [8][K/8][N] bf16 (row-major,
 * N contiguous: rank r's row block of W), out is [M][N] bf16 row-major, whose
 * rows [s*M/8, (s+1)*M/8) are the slice of virtual rank s.
 */
typedef struct gemm_rs_desc {
  int32_t world;          /* tensor-parallel degree; must be 8 */
  int64_t M, N, K;        /* M%8 == 0, N%8 == 0, K%64 == 0 (so K/8 is a multiple of 8); 0 allowed */
  int32_t reducer_warps;  /* FUSED: reducer warps per CTA (all-gather: copy warps), 1..5;
                             0 = default (4; 5 when K <= 6144, 2 when K >= 16384;
                             all-gather 2) */
  int32_t grid;           /* persistent CTAs; 0 = one per SM */
  int32_t band_m;         /* tile-order band height in 128-row tiles; 0 = automatic */
  int32_t unit_rows;      /* rows per reduce item in FUSED mode: 4, 8, 16 or 32; 0 = 8
                             (16 when K <= 6144 and M >= 2048) */
  uint64_t timeout_ns;    /* bound on every device-side wait; 0 = 2 s */
  uint32_t debug_flags;   /* GEMM_RS_DEBUG_* */
  int32_t mma_ctas;       /* CTAs of a cluster sharing one tile: 1 (128 x 256 tiles) or 2
                             (a 2-CTA MMA, 256 x 256 tiles); 0 = 2.  Every CTA loads its
                             own operand tiles (no load is multicast between CTAs) */
  int32_t chunks;         /* CHUNKED: row chunks, 1..64; 0 = 4 (each a whole number of tile
                             rows, the last one ragged) */
  int32_t replicas;       /* copies of the reduced output: 0 or 1 = reduce-scatter, out is
                             [M][N] (rank s's slice = rows [s*M/8, (s+1)*M/8)); 8 =
                             all-reduce, out is [8][M][N] and copy r is virtual rank r's
                             full sum (bitwise the reduce-scatter output) */
  int32_t op;             /* GEMM_RS_OP_RS (0) or GEMM_RS_OP_AG (1) */
  int32_t adaptive;       /* FUSED reduce-scatter: 1 = an on-GPU controller sets how many of
                             each CTA's reducer warps take items, from cycle and progress
                             counters (mKernel page, section 3.2); 0 = all of them */
  int32_t tail_waves;     /* FUSED reduce-scatter: regions completed by the last tail_waves
                             waves of tiles are reduced in 4-row items (fine grain where the
                             reduction is the critical path), the others in unit_rows-row
                             items; 0 = default (3), 1..64 */
  int32_t half_regions;   /* row-parallel layer, 2-CTA tiles: the last half_regions regions of
                             the tile order are computed in half-width tiles (256 rows x 128
                             columns), so the final wave is shorter; 0 or -1 = none (the
                             default), 1..4096 (clamped to the regions there are).  Every mode
                             uses the same tiles, and the results do not depend on it */
  int32_t copy_engines;   /* all-gather + GEMM, FUSED: what moves the 7 other ranks' row
                             shards into each rank's gather buffer while the tiles run.
                             -1 = copy warps inside the fused kernel (reducer_warps of them);
                             1..4 = the GPU's copy engines: one device-to-device copy per
                             (rank, shard) on that many side streams of the plan, each
                             followed on its stream by a write of that shard's count (the
                             value the tiles wait for), and no copy warps in the kernel; the
                             side streams start after the work already queued on the run's
                             stream, and that stream waits for them after the kernel.
                             0 = default (-1).  Ignored by the row-parallel layer */
} gemm_rs_desc;

typedef struct gemm_rs_plan_s* gemm_rs_t;

/* Facts about a plan (for tests and benchmarks). */
typedef struct gemm_rs_info {
  int32_t num_sms;        /* SMs on the device */
  int32_t grid;           /* CTAs of the GEMM / fused kernels */
  int32_t threads_fused;  /* threads per CTA of the fused kernel */
  int32_t threads_gemm;   /* threads per CTA of the unfused GEMM kernel */
  int32_t smem_bytes;     /* dynamic shared memory per CTA of the GEMM kernels (largest) */
  int32_t band_m;         /* tile-order band height in m-tiles */
  int32_t unit_rows;      /* rows per reduce unit (FUSED) */
  int32_t mt, nt;         /* tile rows (of tile_rows rows) and 256-column tiles of the output */
  int64_t tiles;          /* 8 * mt * nt rank tiles */
  int64_t units;          /* reduce items per FUSED run */
  int64_t workspace_bytes;
  int64_t staging_bytes;  /* 8 * M * N * 2 */
  int32_t launches[5];    /* kernels launched per gemm_rs_run, indexed by mode */
  int32_t mma_ctas;       /* CTAs of a cluster sharing one tile */
  int32_t tile_rows;      /* output rows of one rank tile: 128 * mma_ctas */
  int64_t trace_offset;   /* byte offset of the GEMM_RS_DEBUG_TRACE stamps in the workspace */
  int32_t chunks;         /* CHUNKED: chunks actually used */
  int32_t replicas;       /* 1 (reduce-scatter) or 8 (all-reduce) */
  int32_t op;             /* GEMM_RS_OP_RS or GEMM_RS_OP_AG */
  int32_t ag_direct;      /* AG: own shard read from the input, not copied */
  int64_t copy_items;     /* AG: copy items of a fused run */
  int64_t queue_offset;   /* byte offset of the reduce items' debug stamps in the workspace */
  int64_t half_region;    /* first region (in tile order) computed in half-width tiles; the
                             region count if none */
  int32_t copy_engines;   /* AG: side streams of copy-engine copies in FUSED runs; -1 = copy
                             warps; 0 for the row-parallel layer */
} gemm_rs_info;

/*
 * Validate d and build a plan for the current CUDA device.  On success
 * *plan is set and *workspace_bytes (may be NULL) receives the size of the
 * device workspace every gemm_rs_run call needs: the bf16 staging regions
 * (8*M*N*2 bytes), the per-block completion counts, the reduce items' stamps and
 * a few control words.  Arguments are
 * checked before any CUDA call, so INVALID_ARG / UNSUPPORTED_SHAPE come back
 * on a machine without a GPU too.
 */
int gemm_rs_create(const gemm_rs_desc* d, gemm_rs_t* plan, size_t* workspace_bytes);

/*
 * Enqueue one execution on `stream` (a cudaStream_t; NULL = legacy default).
 * A: [8][M][K/8] bf16, W: [8][K/8][N] bf16, out: [M][N] bf16 ([8][M][N] with
 * replicas = 8), workspace:
 * >= workspace_bytes, 16-byte aligned; at a 128-byte boundary (torch and
 * cudaMalloc allocations are) FUSED also keeps the staging in L2 and drops
 * each reduced line unwritten, which is faster; at other 16-byte offsets the
 * staging is written back as in the unfused path.
 * The caller may pass an uninitialised workspace: the first call that sees a
 * new workspace pointer clears its control words (a small memset on the
 * stream).  After GEMM_ONLY or UNFUSED the staging part holds the per-rank
 * partials of that GEMM; after FUSED it holds no defined values (reduced
 * staging lines are dropped from L2 without write-back, see above).
 * Returns after enqueueing; device-side failures (timeouts) are reported by
 * gemm_rs_status.  CHUNKED also uses a second stream and events that the plan
 * creates on its first CHUNKED call; that stream joins `stream` again before
 * the call returns (work after it on `stream` sees the whole output).  Modes
 * that do not read A/W (RS_ONLY) or write out (GEMM_ONLY) accept NULL for
 * them.  The GEMM kernels are launched with programmatic dependent launch:
 * their CTAs may start setting up shared memory and TMEM while the previous
 * kernel on `stream` finishes, but touch no global memory before that kernel
 * has completed, so stream order holds for every buffer; a kernel queued
 * after them that allows the same overlap may likewise start early and wait.
 */
int gemm_rs_run(gemm_rs_t plan, int mode, const void* A, const void* W,
                void* out, void* workspace, void* stream);

/*
 * Host-buffer variant of gemm_rs_run for callers whose A, W and out live in
 * host memory.  Enqueued on `stream`, in this order: copy A_host -> A_dev
 * (8*M*(K/8)*2 bytes) and W_host -> W_dev (8*(K/8)*N*2 bytes), run `mode`
 * exactly as gemm_rs_run would on the device buffers, copy out_dev -> out_host
 * (replicas*M*N*2 bytes).  All six buffers belong to the caller; host buffers
 * should be pinned (cudaHostAlloc / cudaHostRegister) for the copies to be
 * asynchronous, and must stay valid until the stream has passed the copies.
 * Two plans with their own device buffers, on two streams, let one call's
 * copies overlap the other's kernel.  RS_ONLY copies
 * nothing in, GEMM_ONLY copies nothing out.  Same return codes as gemm_rs_run,
 * plus GEMM_RS_ERR_CUDA if a copy cannot be enqueued.
 */
int gemm_rs_run_host(gemm_rs_t plan, int mode, const void* A_host, const void* W_host,
                     void* out_host, void* A_dev, void* W_dev, void* out_dev, void* workspace,
                     void* stream);

/*
 * Synchronise `stream` and report the device error word of the workspace the
 * plan used last: GEMM_RS_OK, GEMM_RS_ERR_TIMEOUT (a device wait gave up; the
 * output of that run is incomplete), GEMM_RS_ERR_INCOMPLETE (the run ended
 * with output blocks that never received all 8 partials) or GEMM_RS_ERR_CUDA.
 * A non-OK result also clears the workspace's control words and flags so the
 * next run starts clean.
 */
int gemm_rs_status(gemm_rs_t plan, void* stream);

/* Fill *info (host pointer).  */
int gemm_rs_get_info(gemm_rs_t plan, gemm_rs_info* info);

/*
 * Tile order used by the GEMM kernels, as a host-only computation (no CUDA
 * call): the idx-th rank tile (0 <= idx < the plan's tile count) is rank
 * *rank, tile row *mt (rows [mt*T, (mt+1)*T) with T = 128 * mma_ctas),
 * 256-column tile *nt, and *half (may be NULL) = -1 for the whole tile, 0 or
 * 1 for the left or right 128 columns of a half-width tile.  Row-parallel
 * order: 8 rank tiles per region (ranks 0..7), regions in L2 bands; the last
 * half_regions regions as 16 half-width tiles each (left halves of ranks
 * 0..7, then right halves).  Uses d->band_m or the automatic band.
 */
int gemm_rs_schedule(const gemm_rs_desc* d, int64_t idx, int32_t* rank, int32_t* mt, int32_t* nt,
                     int32_t* half);

/*
 * Fused run that allocates nothing.  The pages have no counterpart: this is a
 * convenience of this library for callers that cannot allocate device memory
 * when they call it -- a plug-in that runs inside a host application which
 * owns the whole device-memory budget, or a latency-bound serving path that
 * allows no cudaMalloc once it is up (a cudaMalloc may synchronise the device
 * and cost milliseconds).  Such a caller passes only its inputs and its
 * output; the staging regions, flags and control words live in one static
 * device array of this library (32 MiB of staging plus 4 MiB of completion
 * counts and reduce-item slots and 2 KiB of control words), which every GPU
 * that loads the library keeps until the process exits.
 *
 * Same operation, layouts and kernel as gemm_rs_run(..., GEMM_RS_FUSED, ...)
 * with the default plan settings.  Limits: 8*M*N*2 bytes of staging must fit
 * in 32 MiB (M*N <= 2,097,152), and the 128-byte completion count plus up
 * to 256 bytes of reduce-item slots per 32 x 256 output block in 4 MiB;
 * larger problems return GEMM_RS_ERR_TOO_LARGE before touching the GPU.
 * Shape rules and the other return codes are those of gemm_rs_create and
 * gemm_rs_run.
 *
 * error_word: optional device pointer to 4 bytes; after the run the stream
 * copies the device error bits of this call there (0 = ok, non-zero = a
 * device-side wait timed out and the output is incomplete).
 *
 * The first call on a device sets up that device (looks up the array's
 * device address, sets the kernel's shared-memory limit); make that first
 * call before any stream capture.  Every call clears the flags and control
 * words it uses on the stream, then reuses the array, which keeps the last
 * call's contents.  Calls share that one array: calls that can overlap on
 * the GPU (different streams, or several host threads) race and produce
 * garbage; order them on one stream.
 */
int gemm_rs_fused_noalloc(const void* A, const void* W, void* out, int64_t M, int64_t N,
                          int64_t K, void* error_word, void* stream);

/* Release the plan (host state only; device buffers stay the caller's). */
int gemm_rs_destroy(gemm_rs_t plan);

/*
 * Auto-tuning (FLUX page, TL;DR: tile swizzling and auto-tuning; mKernel page,
 * section 5.5: the best share of communication workers varies with the kernel
 * and the shape).  The candidates for d's problem are, without duplicates:
 *   d itself (first);
 *   d with mma_ctas in {2, 1} x reducer_warps in {2, 4, 5} x unit_rows in
 *     {8, 16} (all-gather: mma_ctas in {2, 1} x copy warps in {1, 2, 4});
 *   d with band_m (the tile-order swizzle band) at 1/2 and 1/4 of the
 *     automatic band;
 *   reduce-scatter: d with tail_waves in {1, 2, 6}, and half_regions in {5, 10};
 * every other field as in d (zeros stand for the defaults).  gemm_rs_tune_candidates
 * writes up to `max` of them to `cands` (may be NULL), sets *count, and
 * *workspace_bytes (may be NULL) to the largest workspace any of them needs.
 * Host only; checks d first.
 */
#define GEMM_RS_TUNE_MAX 32
int gemm_rs_tune_candidates(const gemm_rs_desc* d, gemm_rs_desc* cands, int max, int* count,
                            size_t* workspace_bytes);

/*
 * Time every candidate of gemm_rs_tune_candidates in `mode` on the caller's
 * buffers (as gemm_rs_run; ws of ws_bytes >= the candidates' largest
 * workspace) and return the fastest in *best with its time in *best_us; the
 * requested plan (candidate 0) is kept unless another beats it by over 1%.
 * Each candidate runs 3 warm-up launches, then `rounds` rounds in which every
 * candidate is timed over `iters` back-to-back runs with CUDA events on
 * `stream` (interleaved, so drifting clocks affect all alike); a candidate's
 * time is the median over rounds of its per-run mean.  times_us (may be NULL,
 * GEMM_RS_TUNE_MAX entries) receives every candidate's time, in candidate
 * order; a candidate that cannot be created or whose run fails gets -1 and is
 * skipped.  The output and workspace hold the last candidate's run afterwards.
 * Synchronises `stream`.
 */
int gemm_rs_tune(const gemm_rs_desc* d, int mode, const void* A, const void* W, void* out,
                 void* ws, size_t ws_bytes, int iters, int rounds, void* stream,
                 gemm_rs_desc* best, float* best_us, float* times_us);

/* Static text for a status code. */
const char* gemm_rs_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_RS_H */
