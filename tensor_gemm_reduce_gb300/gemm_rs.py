"""Python binding of the C ABI in include/gemm_rs.h (ctypes; marshalling only).

Every step of the operation runs in the CUDA library; this module checks
tensor shapes, dtypes and devices, passes raw pointers and the current CUDA
stream, and turns status codes into exceptions.  If the library is missing
the import of the binding fails loudly: there is no fallback path.

Layouts (problem page "A fused GEMM + reduce-scatter kernel hiding 90% of
communication on 8 H100 GPUs", "What is asked"; FLUX page, Figure 2):
  A   [8][M][K/8] bf16  rank r's column block of the activations
  W   [8][K/8][N] bf16  rank r's row block of the weight
  out [M][N]      bf16  rows [s*M/8, (s+1)*M/8) are virtual rank s's slice
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional

from . import build as _build

WORLD = 8

GEMM_RS_OK = 0
GEMM_RS_ERR_INVALID_ARG = -1
GEMM_RS_ERR_UNSUPPORTED_SHAPE = -2
GEMM_RS_ERR_UNSUPPORTED_DEVICE = -3
GEMM_RS_ERR_CUDA = -4
GEMM_RS_ERR_TIMEOUT = -5
GEMM_RS_ERR_MISALIGNED = -6
GEMM_RS_ERR_WORKSPACE = -7
GEMM_RS_ERR_TOO_LARGE = -8
GEMM_RS_ERR_INCOMPLETE = -9

# Fixed scratch of the no-allocation entry point (see gemm_rs_fused_noalloc).
NOALLOC_STAGING_BYTES = 32 << 20

FUSED, UNFUSED, GEMM_ONLY, RS_ONLY, CHUNKED = 0, 1, 2, 3, 4
# layers (gemm_rs_desc.op): GEMM then reduce-scatter / all-reduce, or all-gather then GEMM
OP_RS, OP_AG = 0, 1
MODES = {"fused": FUSED, "unfused": UNFUSED, "gemm_only": GEMM_ONLY, "rs_only": RS_ONLY,
         "chunked": CHUNKED}

DEBUG_SKIP_ONE_FLAG = 0x1
DEBUG_NO_STAGING_L2 = 0x2
DEBUG_TRACE = 0x4


class gemm_rs_desc(ctypes.Structure):
    _fields_ = [
        ("world", ctypes.c_int32),
        ("M", ctypes.c_int64),
        ("N", ctypes.c_int64),
        ("K", ctypes.c_int64),
        ("reducer_warps", ctypes.c_int32),
        ("grid", ctypes.c_int32),
        ("band_m", ctypes.c_int32),
        ("unit_rows", ctypes.c_int32),
        ("timeout_ns", ctypes.c_uint64),
        ("debug_flags", ctypes.c_uint32),
        ("mma_ctas", ctypes.c_int32),
        ("chunks", ctypes.c_int32),
        ("replicas", ctypes.c_int32),
        ("op", ctypes.c_int32),
        ("adaptive", ctypes.c_int32),
        ("tail_waves", ctypes.c_int32),
        ("half_regions", ctypes.c_int32),
        ("copy_engines", ctypes.c_int32),
    ]


class gemm_rs_info(ctypes.Structure):
    _fields_ = [
        ("num_sms", ctypes.c_int32),
        ("grid", ctypes.c_int32),
        ("threads_fused", ctypes.c_int32),
        ("threads_gemm", ctypes.c_int32),
        ("smem_bytes", ctypes.c_int32),
        ("band_m", ctypes.c_int32),
        ("unit_rows", ctypes.c_int32),
        ("mt", ctypes.c_int32),
        ("nt", ctypes.c_int32),
        ("tiles", ctypes.c_int64),
        ("units", ctypes.c_int64),
        ("workspace_bytes", ctypes.c_int64),
        ("staging_bytes", ctypes.c_int64),
        ("launches", ctypes.c_int32 * 5),
        ("mma_ctas", ctypes.c_int32),
        ("tile_rows", ctypes.c_int32),
        ("trace_offset", ctypes.c_int64),
        ("chunks", ctypes.c_int32),
        ("replicas", ctypes.c_int32),
        ("op", ctypes.c_int32),
        ("ag_direct", ctypes.c_int32),
        ("copy_items", ctypes.c_int64),
        ("queue_offset", ctypes.c_int64),
        ("half_region", ctypes.c_int64),
        ("copy_engines", ctypes.c_int32),
    ]

    def as_dict(self):
        d = {f: getattr(self, f) for f, _ in self._fields_ if f != "launches"}
        d["launches"] = list(self.launches)
        return d


class GemmRSError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        super().__init__(f"{what}: {strerror(code)} ({code})" if what else f"{strerror(code)} ({code})")


_LIB: Optional[ctypes.CDLL] = None

# Every entry point declared in include/gemm_rs.h with its ctypes signature.
_SIGS = {
    "gemm_rs_create": (ctypes.c_int, [ctypes.POINTER(gemm_rs_desc), ctypes.POINTER(ctypes.c_void_p),
                                      ctypes.POINTER(ctypes.c_size_t)]),
    "gemm_rs_run": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "gemm_rs_run_host": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int] + [ctypes.c_void_p] * 8),
    "gemm_rs_status": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p]),
    "gemm_rs_get_info": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(gemm_rs_info)]),
    "gemm_rs_schedule": (ctypes.c_int, [ctypes.POINTER(gemm_rs_desc), ctypes.c_int64,
                                        ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32),
                                        ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)]),
    "gemm_rs_fused_noalloc": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                             ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                             ctypes.c_void_p, ctypes.c_void_p]),
    "gemm_rs_destroy": (ctypes.c_int, [ctypes.c_void_p]),
    "gemm_rs_tune_candidates": (ctypes.c_int, [ctypes.POINTER(gemm_rs_desc), ctypes.POINTER(gemm_rs_desc),
                                               ctypes.c_int, ctypes.POINTER(ctypes.c_int),
                                               ctypes.POINTER(ctypes.c_size_t)]),
    "gemm_rs_tune": (ctypes.c_int, [ctypes.POINTER(gemm_rs_desc), ctypes.c_int, ctypes.c_void_p,
                                    ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                                    ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                    ctypes.POINTER(gemm_rs_desc), ctypes.POINTER(ctypes.c_float),
                                    ctypes.POINTER(ctypes.c_float)]),
    "gemm_rs_strerror": (ctypes.c_char_p, [ctypes.c_int]),
}


def library_path() -> str:
    return _build.LIB


def load_library(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libgemm_rs.so (building it first if asked and needed)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = _build.LIB
    if build_if_missing and (not os.path.exists(path)):
        _build.build_library()
    if not os.path.exists(path):
        raise ImportError(f"CUDA library not built: {path} (run tensor_gemm_reduce_gb300.build)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib


def header_symbols(header_path: Optional[str] = None):
    """Names of the functions declared in include/gemm_rs.h."""
    if header_path is None:
        header_path = os.path.join(_build.ROOT, "include", "gemm_rs.h")
    text = open(header_path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gemm_rs_[a-z_]+)\s*\(", text)))


def strerror(code: int) -> str:
    try:
        return load_library(build_if_missing=False).gemm_rs_strerror(code).decode()
    except Exception:
        return f"status {code}"


def _desc(M, N, K, reducer_warps=0, grid=0, band_m=0, unit_rows=0, timeout_ns=0, debug_flags=0,
          mma_ctas=0, chunks=0, replicas=0, op=OP_RS, adaptive=0, tail_waves=0, half_regions=0,
          copy_engines=0, world=WORLD):
    return gemm_rs_desc(world, M, N, K, reducer_warps, grid, band_m, unit_rows, timeout_ns,
                        debug_flags, mma_ctas, chunks, replicas, op, adaptive, tail_waves, half_regions,
                        copy_engines)


# ----------------------------------------------------------------------------
# thin wrappers with the C names
# ----------------------------------------------------------------------------


def gemm_rs_create(desc: gemm_rs_desc):
    """Returns (plan handle, workspace bytes); raises GemmRSError."""
    lib = load_library()
    h = ctypes.c_void_p()
    ws = ctypes.c_size_t()
    rc = lib.gemm_rs_create(ctypes.byref(desc), ctypes.byref(h), ctypes.byref(ws))
    if rc != GEMM_RS_OK:
        raise GemmRSError(rc, "gemm_rs_create")
    return h, ws.value


def gemm_rs_run(plan, mode: int, A_ptr: int, W_ptr: int, out_ptr: int, ws_ptr: int, stream_ptr: int) -> int:
    return load_library().gemm_rs_run(plan, mode, A_ptr, W_ptr, out_ptr, ws_ptr, stream_ptr)


def gemm_rs_run_host(plan, mode: int, A_host: int, W_host: int, out_host: int, A_dev: int, W_dev: int,
                     out_dev: int, ws_ptr: int, stream_ptr: int) -> int:
    return load_library().gemm_rs_run_host(plan, mode, A_host, W_host, out_host, A_dev, W_dev,
                                           out_dev, ws_ptr, stream_ptr)


def gemm_rs_status(plan, stream_ptr: int) -> int:
    return load_library().gemm_rs_status(plan, stream_ptr)


def gemm_rs_get_info(plan) -> gemm_rs_info:
    info = gemm_rs_info()
    rc = load_library().gemm_rs_get_info(plan, ctypes.byref(info))
    if rc != GEMM_RS_OK:
        raise GemmRSError(rc, "gemm_rs_get_info")
    return info


def gemm_rs_schedule(desc: gemm_rs_desc, idx: int):
    """(rank, tile row, 256-column tile, half) of the idx-th rank tile; half is
    -1 for a whole tile, 0 / 1 for the left / right half of a half-width one."""
    r, m, n, h = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    rc = load_library().gemm_rs_schedule(ctypes.byref(desc), idx, ctypes.byref(r), ctypes.byref(m),
                                         ctypes.byref(n), ctypes.byref(h))
    if rc != GEMM_RS_OK:
        raise GemmRSError(rc, "gemm_rs_schedule")
    return r.value, m.value, n.value, h.value


def gemm_rs_fused_noalloc(A_ptr: int, W_ptr: int, out_ptr: int, M: int, N: int, K: int,
                          error_word_ptr: int, stream_ptr: int) -> int:
    """Fused run with the library's static scratch instead of a workspace: for
    callers that may not allocate device memory at call time.  Returns the
    status code; the device error bits of the call land in *error_word_ptr
    (a 4-byte device buffer, or 0 for none)."""
    return load_library().gemm_rs_fused_noalloc(A_ptr, W_ptr, out_ptr, M, N, K, error_word_ptr,
                                                stream_ptr)


def gemm_rs_destroy(plan) -> int:
    return load_library().gemm_rs_destroy(plan)


def gemm_rs_strerror(code: int) -> str:
    return strerror(code)


# ----------------------------------------------------------------------------
# torch-facing plan object
# ----------------------------------------------------------------------------


class Plan:
    """A plan for one (M, N, K) on the current CUDA device."""

    def __init__(self, M: int, N: int, K: int, *, reducer_warps: int = 0, grid: int = 0,
                 band_m: int = 0, unit_rows: int = 0, timeout_ns: int = 0, debug_flags: int = 0,
                 mma_ctas: int = 0, chunks: int = 0, replicas: int = 0, op: int = OP_RS,
                 adaptive: int = 0, tail_waves: int = 0, half_regions: int = 0,
                 copy_engines: int = 0):
        self.M, self.N, self.K = int(M), int(N), int(K)
        self.replicas = max(1, int(replicas))
        self.op = int(op)
        self.desc = _desc(self.M, self.N, self.K, reducer_warps, grid, band_m, unit_rows,
                          timeout_ns, debug_flags, mma_ctas, chunks, replicas, op, adaptive,
                          tail_waves, half_regions, copy_engines)
        self._h, self.workspace_bytes = gemm_rs_create(self.desc)

    @property
    def a_shape(self):
        """[8][M][K/8] (row-parallel: K shards) or [8][M/8][K] (all-gather: row shards)."""
        if self.op == OP_AG:
            return (WORLD, self.M // WORLD, self.K)
        return (WORLD, self.M, self.K // WORLD)

    @property
    def w_shape(self):
        """[8][K/8][N] (row-parallel) or [8][K][N/8] (all-gather: column shards)."""
        if self.op == OP_AG:
            return (WORLD, self.K, self.N // WORLD)
        return (WORLD, self.K // WORLD, self.N)

    @property
    def out_shape(self):
        """[M][N] (reduce-scatter), [8][M][N] (all-reduce: one copy per rank) or
        [8][M][N/8] (all-gather + GEMM: rank r's column block)."""
        if self.op == OP_AG:
            return (WORLD, self.M, self.N // WORLD)
        return (self.M, self.N) if self.replicas == 1 else (self.replicas, self.M, self.N)

    @property
    def info(self) -> gemm_rs_info:
        return gemm_rs_get_info(self._h)

    def new_workspace(self, device=None):
        import torch
        dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
        return torch.empty(self.workspace_bytes, dtype=torch.uint8, device=dev)

    def _check(self, t, shape, name):
        import torch
        if t is None:
            return 0
        if t.dtype != torch.bfloat16:
            raise TypeError(f"{name} must be bfloat16, got {t.dtype}")
        if tuple(t.shape) != tuple(shape):
            raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
        return t.data_ptr()

    def run(self, A, W, out, workspace, mode: int = FUSED, stream=None) -> None:
        import torch
        a = self._check(A, self.a_shape, "A")
        w = self._check(W, self.w_shape, "W")
        o = self._check(out, self.out_shape, "out")
        if workspace is None or workspace.numel() * workspace.element_size() < self.workspace_bytes:
            raise ValueError("workspace missing or too small")
        s = stream if stream is not None else torch.cuda.current_stream()
        rc = gemm_rs_run(self._h, int(mode), a, w, o, workspace.data_ptr(), s.cuda_stream)
        if rc != GEMM_RS_OK:
            raise GemmRSError(rc, "gemm_rs_run")

    def run_host(self, A_host, W_host, out_host, A, W, out, workspace, mode: int = FUSED,
                 stream=None) -> None:
        """Host tensors in (pinned for asynchronous copies), host tensor out; the
        copies and the run are enqueued on one stream by the library."""
        import torch
        for t, shape, name in ((A_host, self.a_shape, "A_host"),
                               (W_host, self.w_shape, "W_host"),
                               (out_host, self.out_shape, "out_host")):
            if t.dtype != torch.bfloat16 or tuple(t.shape) != shape or t.is_cuda or not t.is_contiguous():
                raise ValueError(f"{name} must be a contiguous host bf16 tensor of shape {shape}")
        a = self._check(A, self.a_shape, "A")
        w = self._check(W, self.w_shape, "W")
        o = self._check(out, self.out_shape, "out")
        if workspace is None or workspace.numel() * workspace.element_size() < self.workspace_bytes:
            raise ValueError("workspace missing or too small")
        s = stream if stream is not None else torch.cuda.current_stream()
        rc = gemm_rs_run_host(self._h, int(mode), A_host.data_ptr(), W_host.data_ptr(),
                              out_host.data_ptr(), a, w, o, workspace.data_ptr(), s.cuda_stream)
        if rc != GEMM_RS_OK:
            raise GemmRSError(rc, "gemm_rs_run_host")

    def status(self, stream=None) -> int:
        import torch
        s = stream if stream is not None else torch.cuda.current_stream()
        return gemm_rs_status(self._h, s.cuda_stream)

    def trace(self, workspace):
        """GEMM_RS_DEBUG_TRACE stamps of the last run: int64 tensor [grid][4] (ns)."""
        import torch
        off = self.info.trace_offset
        n = self.info.grid * 4
        return workspace[off: off + 8 * n].view(torch.int64).view(-1, 4).cpu()

    def timeline(self, workspace) -> dict:
        """Timeline of the last FUSED reduce-scatter run of a plan made with
        debug_flags=DEBUG_TRACE, in microseconds from the earliest CTA start:
        per CTA (start, epilogue done, MMA drained, end) and per reduce item
        (item, queued, taken, done).  Plain lists, ready for json.dumps."""
        import torch
        info = self.info
        cta = self.trace(workspace).numpy()
        valid = cta[:, 0] > 0
        t0 = int(cta[valid, 0].min()) if valid.any() else 0
        us = lambda x: [round((int(v) - t0) / 1e3, 3) if v > 0 else None for v in x]
        q = workspace[info.queue_offset: info.queue_offset + 32 * info.units].view(torch.int64)
        q = q.view(-1, 4).cpu().numpy()
        items = [{"item": int(w0 & 0xFFFFFFFF), "queued": a, "taken": b, "done": c}
                 for w0, a, b, c in zip(q[:, 0], us(q[:, 1]), us(q[:, 2]), us(q[:, 3]))]
        return {"ctas": [{"start": a, "epilogue_done": b, "mma_drained": c, "end": d}
                         for a, b, c, d in zip(us(cta[:, 0]), us(cta[:, 1]), us(cta[:, 2]),
                                               us(cta[:, 3]))],
                "items": items}

    def close(self):
        if getattr(self, "_h", None):
            gemm_rs_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def gemm_rs(A, W, out=None, workspace=None, mode: int = FUSED, plan: Optional[Plan] = None,
            **plan_kw):
    """One call of a layer; the plan (made here from the tensors' shapes and
    plan_kw when not given) decides which.

    Row-parallel layer (default): A [8][M][K/8], W [8][K/8][N]; out[s*M/8:(s+1)*M/8]
    is rank s's slice (replicas=8: out[r] is rank r's copy of the whole sum).
    All-gather + GEMM (op=OP_AG): A [8][M/8][K], W [8][K][N/8]; out[r] = C_r.
    Returns (out, plan, workspace).
    """
    import torch
    if plan is None:
        if plan_kw.get("op", OP_RS) == OP_AG:
            R, h, K = A.shape
            plan = Plan(R * h, R * W.shape[2], K, **plan_kw)
        else:
            R, M, Kr = A.shape
            plan = Plan(M, W.shape[2], Kr * R, **plan_kw)
    if out is None:
        out = torch.empty(*plan.out_shape, dtype=torch.bfloat16, device=A.device)
    if workspace is None:
        workspace = plan.new_workspace(A.device)
    plan.run(A, W, out, workspace, mode)
    return out, plan, workspace


# ----------------------------------------------------------------------------
# auto-tuning
# ----------------------------------------------------------------------------

TUNE_MAX = 32
_DESC_KW = ("reducer_warps", "grid", "band_m", "unit_rows", "timeout_ns", "debug_flags",
            "mma_ctas", "chunks", "replicas", "op", "adaptive", "tail_waves", "half_regions",
            "copy_engines")


def tune_candidates(desc: gemm_rs_desc):
    """(list of candidate descs, workspace bytes that fits every one of them)."""
    lib = load_library()
    arr = (gemm_rs_desc * TUNE_MAX)()
    n = ctypes.c_int()
    ws = ctypes.c_size_t()
    rc = lib.gemm_rs_tune_candidates(ctypes.byref(desc), arr, TUNE_MAX, ctypes.byref(n),
                                     ctypes.byref(ws))
    if rc != GEMM_RS_OK:
        raise GemmRSError(rc, "gemm_rs_tune_candidates")
    return [arr[i] for i in range(min(n.value, TUNE_MAX))], ws.value


def desc_kwargs(desc: gemm_rs_desc) -> dict:
    """Plan(...) keyword arguments of a descriptor."""
    return {k: getattr(desc, k) for k in _DESC_KW}


def tune(M, N, K, A, W, out, mode: int = FUSED, iters: int = 10, rounds: int = 3, stream=None,
         workspace=None, **plan_kw):
    """Time the tuning candidates of (M, N, K, plan_kw) on these buffers.

    Returns (best Plan keyword arguments, best time in us, [(kwargs, us), ...]).
    """
    import torch
    desc = _desc(int(M), int(N), int(K), **plan_kw)
    cands, ws_bytes = tune_candidates(desc)
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=A.device)
    s = stream if stream is not None else torch.cuda.current_stream()
    best = gemm_rs_desc()
    best_us = ctypes.c_float()
    times = (ctypes.c_float * TUNE_MAX)()
    rc = load_library().gemm_rs_tune(ctypes.byref(desc), int(mode), A.data_ptr(), W.data_ptr(),
                                     out.data_ptr(), workspace.data_ptr(),
                                     workspace.numel() * workspace.element_size(), int(iters),
                                     int(rounds), s.cuda_stream, ctypes.byref(best),
                                     ctypes.byref(best_us), times)
    if rc != GEMM_RS_OK:
        raise GemmRSError(rc, "gemm_rs_tune")
    table = [(desc_kwargs(c), float(times[i])) for i, c in enumerate(cands)]
    return desc_kwargs(best), float(best_us.value), table
