#!/usr/bin/env python
"""Benchmark of the fused GEMM + reduce-scatter (row-parallel linear layer,
8 virtual tensor-parallel ranks on one GB300).

Metric (problem page "A fused GEMM + reduce-scatter kernel hiding 90% of
communication on 8 H100 GPUs", "How it gets verified"): throughput of the
fused kernel in TFLOP/s (2*M*N*K per step) and the overlap efficiency
(T_gemm + T_rs - T_fused) / T_rs, medians of 200 iterations after warm-up,
with T_gemm and T_rs the unfused path's GEMM and reduce-scatter kernels each
timed alone.

One step = one fused run over one batch of synthetic input: every rank tile of
the GEMM, its bf16 staging write, its completion flag and the rank-order fp32
reduction into the bf16 output.  Inputs stay resident in device memory for
`value`; `e2e` adds, every step, the host-to-device copy of A and W from
pinned memory and the device-to-host copy of the output, through the
library's host-buffer entry point.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs its own replica of the workload (the
emulated tensor-parallel group lives inside one GPU, so nothing is exchanged
between GPUs); rank 0 prints one JSON line.  --impl reference times the CPU
oracle instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import re
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused GEMM+reduce-scatter TFLOP/s and overlap efficiency vs unfused, 1 GB300"
DEFAULT_WORKLOAD = "llama3_70b_o_proj_m2048"
CLOCK_QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
               "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
KERNEL_SOURCES = ["tensor_gemm_reduce_gb300/csrc/kernels.cuh", "tensor_gemm_reduce_gb300/csrc/ptx.cuh",
                  "tensor_gemm_reduce_gb300/csrc/schedule.h", "tensor_gemm_reduce_gb300/csrc/gemm_rs.cu"]


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--overlap-iters", type=int, default=200)
    p.add_argument("--chunks", type=lambda s: [int(x) for x in s.split(",") if x], default=[2, 4, 8],
                   help="chunk counts of the stream-overlap comparison (empty: skip it)")
    p.add_argument("--sweep", default="",
                   help="comma-separated workloads ('all': every reduce-scatter shape, 'all_ag': every "
                        "all-gather shape) timed per shape instead of the benchmark line; for "
                        "all-gather shapes t_rs is the gather alone")
    p.add_argument("--sweep-rounds", type=int, default=3)
    p.add_argument("--tuned", action="store_true",
                   help="--sweep: also run the auto-tuner (gemm_rs_tune, FUSED) on each shape and time "
                        "its plan beside the default one")
    p.add_argument("--sweep-iters", type=int, default=0, help="timed launches per mode and round (0: auto)")
    p.add_argument("--ag-workload", default="llama3_70b_qkv_m2048",
                   help="all-gather + GEMM workload timed beside the main one ('' to skip)")
    p.add_argument("--no-allreduce", dest="allreduce", action="store_false",
                   help="skip the GEMM + all-reduce timing (8 output copies)")
    p.add_argument("--e2e-steps", type=int, default=50)
    p.add_argument("--cpu-seconds", type=float, default=10.0,
                   help="target CPU time of the oracle baseline sample")
    p.add_argument("--reference-seconds", type=float, default=120.0,
                   help="target length of the whole --impl reference run")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--profile", choices=["fused", "unfused", "gemm_only", "rs_only"], default=None,
                   help="only run --warmup + --steps launches of one mode of --workload (a target "
                        "for ncu; for an all-gather workload rs_only is the gather alone)")
    return p.parse_args(argv)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def source_sha256() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


def committed_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel sources (else None)."""
    sha = source_sha256()
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        text = open(path).read()
        m_k = re.search(r"^kernel:\s*(\S+)", text, re.M)
        m_w = re.search(r"^workload:\s*(\S+)", text, re.M)
        m_s = re.search(r"^source_sha256:\s*([0-9a-f]{64})", text, re.M)
        m_b = re.search(r"^dram_bytes_per_launch:\s*([0-9.eE+]+)", text, re.M)
        if m_k and m_w and m_s and m_b and m_k.group(1) == kernel and m_w.group(1) == workload:
            if m_s.group(1) == sha:
                return float(m_b.group(1))
    return None


class ClockSampler:
    """nvidia-smi samples every 100 ms while the timed region runs."""

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            import tempfile
            fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={CLOCK_QUERY}", "--format=csv",
                 "-lms", "100"], stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        from tensor_gemm_reduce_gb300 import metrics
        if not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        text = open(self.path).read()
        os.unlink(self.path)
        return metrics.summarize_clocks(text)


def time_batched(launch, iters: int, batches: int, stream) -> float:
    """Seconds per launch: the median of iters * batches per-launch times.
    Each batch is `iters` back-to-back launches with a CUDA event on `stream`
    between consecutive launches; a GPU-side sleep queued before each batch
    gives the host time to enqueue the whole batch, so host launch latency
    never shows in the device times."""
    import torch
    from tensor_gemm_reduce_gb300 import metrics
    per = []
    for _ in range(batches):
        torch.cuda._sleep(250_000 * iters)  # ~0.12 ms of host enqueue time per launch
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(iters + 1)]
        ev[0].record(stream)
        for i in range(iters):
            launch()
            ev[i + 1].record(stream)
        ev[-1].synchronize()
        per.extend(ev[i].elapsed_time(ev[i + 1]) * 1e-3 for i in range(iters))
    return metrics.median(per)


def device_info(index: int) -> dict:
    import torch
    prop = torch.cuda.get_device_properties(index)
    return {"name": prop.name, "sms": prop.multi_processor_count,
            "l2_mb": round(getattr(prop, "L2_cache_size", 0) / 2 ** 20, 1),
            "hbm_gib": round(prop.total_memory / 2 ** 30, 1), "cc": f"{prop.major}.{prop.minor}"}


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var):
            return int(os.environ[var])
    return len(os.sched_getaffinity(0))


def cpu_oracle_rate(A_bits, W_bits, N, K, target_s: float, max_rows: int):
    """Time the CPU oracle on a row sample of the workload: returns (TFLOP/s, rows, seconds)."""
    import numpy as np
    import oracle
    rows = 8
    while True:
        idx = np.arange(rows) % max_rows
        t0 = time.perf_counter()
        oracle.gemm_rs_rows(A_bits, W_bits, idx)
        dt = time.perf_counter() - t0
        if dt >= target_s or rows >= max_rows:
            break
        rows = int(min(max_rows, max(rows * 2, rows * target_s / max(dt, 1e-3) * 1.05)))
    return 2.0 * rows * N * K / dt / 1e12, rows, dt


# ---------------------------------------------------------------------------


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle as it stands, on host cores."""
    if rank != 0:
        return 0
    import numpy as np
    import oracle
    from tensor_gemm_reduce_gb300 import workloads
    w = workloads.WORKLOADS[args.workload]
    A_bits, W_bits = workloads.make_inputs(w)
    # size each step's row sample so the whole run stays near --reference-seconds
    t0 = time.perf_counter()
    oracle.gemm_rs_rows(A_bits, W_bits, np.arange(8))
    per_row = (time.perf_counter() - t0) / 8
    total_steps = args.warmup + args.steps
    rows = int(max(1, min(w.M, args.reference_seconds / total_steps / per_row)))
    cursor = 0

    def step():
        nonlocal cursor
        idx = (np.arange(rows) + cursor) % w.M
        cursor = (cursor + rows) % w.M
        oracle.gemm_rs_rows(A_bits, W_bits, idx)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    flops = 2.0 * rows * w.N * w.K * args.steps
    value = flops / dt / 1e12
    cores = blas_threads()
    sample = (f"{rows} of {w.M} output rows per step (all 8 ranks, full N={w.N}, K={w.K}); "
              f"float64 numpy oracle, {cores} BLAS threads")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "world": 8,
                   "sample_rows_per_step": rows},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args, rank, world, local):
    import numpy as np
    import torch
    import torch.distributed as dist

    from tensor_gemm_reduce_gb300 import gemm_rs as G
    from tensor_gemm_reduce_gb300 import metrics, workloads

    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    G.load_library(build_if_missing=True)
    w = workloads.WORKLOADS[args.workload]
    M, N, K = w.M, w.N, w.K
    A_bits, W_bits = workloads.make_inputs(w)
    # CPU baseline first (rank 0, one GPU): host work before the GPU gets busy
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, rows, dt = cpu_oracle_rate(A_bits, W_bits, N, K, args.cpu_seconds, M)
        cores = blas_threads()
        cpu = {"value": rate, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "sample": f"{rows} of {M} output rows of {w.name} (all 8 ranks, full N and K) in "
                         f"{dt:.1f} s; float64 numpy oracle"}

    A_host = torch.from_numpy(A_bits.view(np.int16)).view(torch.bfloat16).pin_memory()
    W_host = torch.from_numpy(W_bits.view(np.int16)).view(torch.bfloat16).pin_memory()
    A = A_host.cuda()
    W = W_host.cuda()
    out = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    out_host = torch.empty(M, N, dtype=torch.bfloat16).pin_memory()
    plan = G.Plan(M, N, K)
    info = plan.info
    ws = plan.new_workspace()
    stream = torch.cuda.current_stream()

    def check():
        rc = plan.status()
        if rc != G.GEMM_RS_OK:
            raise RuntimeError(f"device status: {G.strerror(rc)}")

    # sanity: fused and unfused agree bit for bit
    plan.run(A, W, out, ws, G.FUSED)
    check()
    f0 = out.clone()
    plan.run(A, W, out, ws, G.UNFUSED)
    check()
    if not torch.equal(f0.view(torch.int16), out.view(torch.int16)):
        raise RuntimeError("fused and unfused outputs differ")

    # overlap efficiency: per-iteration medians of each kernel alone
    def time_mode(mode, iters, warm, pl=None, w=None, o=None, a=None, b=None):
        pl = plan if pl is None else pl
        w = ws if w is None else w
        o = out if o is None else o
        a = A if a is None else a
        b = W if b is None else b
        for _ in range(warm):
            pl.run(a, b, o, w, mode)
        torch.cuda.synchronize()
        t = time_batched(lambda: pl.run(a, b, o, w, mode), 40, max(3, iters // 40), stream)
        rc = pl.status()
        if rc != G.GEMM_RS_OK:
            raise RuntimeError(f"device status: {G.strerror(rc)}")
        return t

    it = args.overlap_iters
    t_gemm = time_mode(G.GEMM_ONLY, it, 20)
    t_rs = time_mode(G.RS_ONLY, it, 20)
    t_fused = time_mode(G.FUSED, it, 20)
    t_unfused = time_mode(G.UNFUSED, it, 20)
    eff = metrics.overlap_efficiency(t_gemm, t_rs, t_fused)
    # The same fused run with the staging forced through HBM: staging stores
    # without the L2 evict-last hint and no discard after reduction, so the
    # partials are written back to DRAM as a peer write over a link would be
    # (the GEMM-alone run, T_gemm, writes its staging the same way).
    hplan = G.Plan(M, N, K, debug_flags=G.DEBUG_NO_STAGING_L2)
    ws_h = hplan.new_workspace()
    t_fused_hbm = time_mode(G.FUSED, it, 20, hplan, ws_h)
    hplan.close()
    del ws_h
    eff_hbm = metrics.overlap_efficiency(t_gemm, t_rs, t_fused_hbm)

    # the prior stream-overlap method (row chunks, reduce of chunk c beside the
    # GEMM of chunk c+1 on a second stream), on a workspace of its own
    ws_c = None
    t_chunked = {}
    for c in args.chunks:
        cplan = G.Plan(M, N, K, chunks=c)
        if ws_c is None:
            ws_c = cplan.new_workspace()
        cplan.run(A, W, out, ws_c, G.CHUNKED)
        torch.cuda.synchronize()
        if not torch.equal(f0.view(torch.int16), out.view(torch.int16)):
            raise RuntimeError(f"chunked ({c}) and fused outputs differ")
        t_chunked[str(cplan.info.chunks)] = time_mode(G.CHUNKED, it, 10, cplan, ws_c)
        cplan.close()
    del ws_c
    t_chunked_best = min(t_chunked.values()) if t_chunked else None

    # the column-parallel partner layer: all-gather + GEMM, fused and unfused
    ag = None
    if args.ag_workload:
        wa = workloads.WORKLOADS[args.ag_workload]
        Ab, Wb = workloads.make_inputs(wa)
        A_ag = torch.from_numpy(Ab.view(np.int16)).cuda().view(torch.bfloat16)
        W_ag = torch.from_numpy(Wb.view(np.int16)).cuda().view(torch.bfloat16)
        gplan = G.Plan(wa.M, wa.N, wa.K, op=G.OP_AG)
        ws_g = gplan.new_workspace()
        out_g = torch.empty(*gplan.out_shape, dtype=torch.bfloat16, device="cuda")
        gplan.run(A_ag, W_ag, out_g, ws_g, G.UNFUSED)
        torch.cuda.synchronize()
        ref_g = out_g.clone()
        gplan.run(A_ag, W_ag, out_g, ws_g, G.FUSED)
        torch.cuda.synchronize()
        if gplan.status() != G.GEMM_RS_OK or not torch.equal(ref_g.view(torch.int16), out_g.view(torch.int16)):
            raise RuntimeError("all-gather + GEMM: fused and unfused outputs differ")
        tg = {name: time_mode(mode, it, 10, gplan, ws_g, out_g, A_ag, W_ag)
              for mode, name in ((G.GEMM_ONLY, "gemm"), (G.RS_ONLY, "gather"),
                                 (G.FUSED, "fused"), (G.UNFUSED, "unfused"))}
        ag = {"workload": wa.name, "M": wa.M, "N": wa.N, "K": wa.K,
              "tflops_fused": metrics.gemm_flops(wa.M, wa.N, wa.K) / tg["fused"] / 1e12,
              "overlap_efficiency": metrics.overlap_efficiency(tg["gemm"], tg["gather"], tg["fused"]),
              "fused_speedup_vs_unfused": tg["unfused"] / tg["fused"],
              **{f"t_{k}_us": v * 1e6 for k, v in tg.items()}}
        gplan.close()
        del ws_g, out_g, A_ag, W_ag, ref_g

    # GEMM + all-reduce: the same reduction written to all 8 ranks' copies
    t_ar = {}
    if args.allreduce:
        aplan = G.Plan(M, N, K, replicas=8)
        ws_a = aplan.new_workspace()
        out_a = torch.empty(*aplan.out_shape, dtype=torch.bfloat16, device="cuda")
        for mode, name in ((G.FUSED, "fused"), (G.UNFUSED, "unfused")):
            aplan.run(A, W, out_a, ws_a, mode)
            torch.cuda.synchronize()
            if not all(torch.equal(out_a[r].view(torch.int16), f0.view(torch.int16)) for r in (0, 7)):
                raise RuntimeError(f"all-reduce ({name}) copies differ from the reduce-scatter output")
            t_ar[name] = time_mode(mode, it, 10, aplan, ws_a, out_a)
        aplan.close()
        del ws_a, out_a

    # the contract's timed region: K fused steps between events
    for _ in range(args.warmup):
        plan.run(A, W, out, ws, G.FUSED)
    check()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        # a GPU-side sleep before the start event lets the host enqueue all K
        # steps first, so the timed region holds the K launches back to back
        # and not the host's latency before the first one
        torch.cuda._sleep(int(2.0e9 * max(1e-3, 60e-6 * args.steps)))
        e0.record(stream)
        for _ in range(args.steps):
            plan.run(A, W, out, ws, G.FUSED)
        e1.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
    check()
    clocks = clk.summary()
    elapsed = e0.elapsed_time(e1) * 1e-3

    # end to end through the host-buffer entry point
    h2d = A_host.numel() * 2 + W_host.numel() * 2
    d2h = out_host.numel() * 2
    for _ in range(3):
        plan.run_host(A_host, W_host, out_host, A, W, out, ws, G.FUSED)
    check()
    ke = max(1, args.e2e_steps)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    e2 = torch.cuda.Event(enable_timing=True)
    e3 = torch.cuda.Event(enable_timing=True)
    e2.record(stream)
    for _ in range(ke):
        plan.run_host(A_host, W_host, out_host, A, W, out, ws, G.FUSED)
    e3.record(stream)
    torch.cuda.synchronize()
    check()
    e2e_serial = e2.elapsed_time(e3) * 1e-3
    if not torch.equal(out_host.view(torch.int16), f0.cpu().view(torch.int16)):
        raise RuntimeError("end-to-end output differs from the device-resident run")

    # The same calls double-buffered, as a serving or training loop issues
    # them: two plans, streams and device buffer sets, step s on set s % 2, so
    # step s + 1's input copies overlap step s's kernel and output copy (the
    # host-device link, ~200 GB/s each way here, bounds this path).
    plan2 = G.Plan(M, N, K)
    ws2 = plan2.new_workspace()
    A2, W2, out2 = torch.empty_like(A), torch.empty_like(W), torch.empty_like(out)
    out_host2 = torch.empty_like(out_host).pin_memory()
    s_a, s_b = torch.cuda.Stream(), torch.cuda.Stream()
    sets = [(plan, A, W, out, ws, out_host, s_a), (plan2, A2, W2, out2, ws2, out_host2, s_b)]
    for k in range(4):
        pk, ak, wk, ok_, wsk, ohk, sk = sets[k % 2]
        pk.run_host(A_host, W_host, ohk, ak, wk, ok_, wsk, G.FUSED, stream=sk)
    torch.cuda.synchronize()
    e4 = torch.cuda.Event(enable_timing=True)
    e5 = torch.cuda.Event(enable_timing=True)
    e4.record(stream)
    s_a.wait_stream(stream)
    s_b.wait_stream(stream)
    for k in range(ke):
        pk, ak, wk, ok_, wsk, ohk, sk = sets[k % 2]
        pk.run_host(A_host, W_host, ohk, ak, wk, ok_, wsk, G.FUSED, stream=sk)
    stream.wait_stream(s_a)
    stream.wait_stream(s_b)
    e5.record(stream)
    torch.cuda.synchronize()
    for pk in (plan, plan2):
        if pk.status() != G.GEMM_RS_OK:
            raise RuntimeError("pipelined end-to-end run: device status")
    for ohk in (out_host, out_host2):
        if not torch.equal(ohk.view(torch.int16), f0.cpu().view(torch.int16)):
            raise RuntimeError("pipelined end-to-end output differs from the device-resident run")
    e2e_elapsed = e4.elapsed_time(e5) * 1e-3
    plan2.close()
    del ws2, A2, W2, out2

    flops = metrics.gemm_flops(M, N, K)
    elapsed, e2e_elapsed, e2e_serial = metrics.max_over_ranks([elapsed, e2e_elapsed, e2e_serial],
                                                              device="cuda")
    agg = metrics.aggregate_ranks([flops * args.steps] * world, [elapsed])
    value = agg["rate"] / 1e12
    e2e_value = flops * ke * world / e2e_elapsed / 1e12
    e2e_serial_value = flops * ke * world / e2e_serial / 1e12

    peaks = load_peaks()
    per_launch = elapsed / args.steps
    # the sustained figure once the timed loop is long or ran into the power
    # cap (a loop of back-to-back launches, as the sustained peak was taken)
    long_region = elapsed > 1.0 or "sw_power_cap" in clocks.get("reasons", [])
    peak = peaks["bf16_tflops_sustained"] if long_region else peaks["bf16_tflops"]
    peak_kind = ("sustained" if long_region else "burst") + f" bf16, of {peaks['source']}"
    traffic = committed_traffic("gemm_rs_kernel_fused", w.name)
    roof = metrics.roofline("tensor", flops / per_launch / 1e12, peak, "TFLOP/s", traffic)
    roof["peak_kind"] = peak_kind
    roof["kernel"] = "gemm_rs_kernel<fused>"
    rs_gbs = metrics.rs_bytes(M, N) / t_rs / 1e9
    rs_roof = metrics.roofline("hbm", rs_gbs, peaks["hbm_gbs"], "GB/s",
                               committed_traffic("rs_reduce_kernel", w.name))
    rs_roof["kernel"] = "rs_reduce_kernel (unfused path, alone)"
    rs_roof["peak_kind"] = f"copy bandwidth, of {peaks['source']}"

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": elapsed / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": w.name, "M": M, "N": N, "K": K, "world": 8,
                   "parallelism": "8 virtual TP ranks per GPU" + (f", {world} replicas" if world > 1 else ""),
                   "l2": "no flush; inputs larger than L2 (A+W %.0f MB, staging %.0f MB written and read per step)"
                         % ((A.numel() + W.numel()) * 2 / 1e6, info.staging_bytes / 1e6),
                   "grid": info.grid, "threads_fused": info.threads_fused, "band_m": info.band_m,
                   "unit_rows": info.unit_rows,
                   "timing": "K launches back to back, queued behind a GPU sleep; CUDA events at "
                             "both ends (programmatic dependent launch overlaps each step's set-up "
                             "with the previous step's last CTAs)"},
        "overlap": {"efficiency": eff, "t_gemm_us": t_gemm * 1e6, "t_rs_us": t_rs * 1e6,
                    "t_fused_us": t_fused * 1e6, "t_unfused_us": t_unfused * 1e6,
                    "efficiency_staging_hbm": eff_hbm, "t_fused_staging_hbm_us": t_fused_hbm * 1e6,
                    "fused_speedup_vs_unfused": t_unfused / t_fused, "iters": it,
                    "t_chunked_us": {c: t * 1e6 for c, t in t_chunked.items()},
                    "fused_speedup_vs_best_chunked":
                        (t_chunked_best / t_fused) if t_chunked_best else None,
                    "allreduce_us": {k: v * 1e6 for k, v in t_ar.items()},
                    "statistic": "median of 200 per-launch CUDA-event times (5 batches of 40 "
                                 "back-to-back launches queued behind a GPU sleep), rank 0"},
        "device": device_info(local),
        "allgather_gemm": ag,
        "roofline": roof,
        "rs_roofline": rs_roof,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": ke,
                "how": "gemm_rs_run_host per step, double-buffered on 2 streams (step s+1's copies "
                       "overlap step s's kernel)",
                "serial_value": e2e_serial_value},
        "gpu_launches": args.steps * info.launches[G.FUSED],
        "clocks": clocks,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def run_profile_target(args, local):
    """Warm-up plus timed launches of one mode and nothing else, for ncu."""
    import numpy as np
    import torch
    from tensor_gemm_reduce_gb300 import gemm_rs as G
    from tensor_gemm_reduce_gb300 import workloads
    torch.cuda.set_device(local)
    w = workloads.WORKLOADS[args.workload]
    A_bits, W_bits = workloads.make_inputs(w)
    A = torch.from_numpy(A_bits.view(np.int16)).cuda().view(torch.bfloat16)
    W = torch.from_numpy(W_bits.view(np.int16)).cuda().view(torch.bfloat16)
    op = G.OP_AG if w.op == "ag" else G.OP_RS
    plan = G.Plan(w.M, w.N, w.K, op=op)
    out = torch.empty(*plan.out_shape, dtype=torch.bfloat16, device="cuda")
    ws = plan.new_workspace()
    mode = G.MODES[args.profile]
    if mode == G.RS_ONLY and op == G.OP_RS:
        plan.run(A, W, out, ws, G.GEMM_ONLY)  # partials in the staging for the reduce alone
    if mode == G.GEMM_ONLY and op == G.OP_AG:
        plan.run(A, W, out, ws, G.RS_ONLY)  # gathered buffers for the GEMM alone
    for _ in range(args.warmup + args.steps):
        plan.run(A, W, out, ws, mode)
    rc = plan.status()
    if rc != G.GEMM_RS_OK:
        raise RuntimeError(G.strerror(rc))
    print(json.dumps({"profile": args.profile, "workload": w.name, "launches": args.warmup + args.steps}))
    return 0


def run_sweep(args, local):
    """--sweep: per shape, medians of per-launch CUDA-event times of the GEMM
    alone, the reduce alone, FUSED and UNFUSED (interleaved rounds), one JSON
    line each.  Inputs: A ~ N(0,1), W ~ N(0,1/K) drawn on the device with a
    seeded torch generator (the large shapes would take minutes on the host),
    rounded to bf16 and sharded like the registered workloads; FUSED and
    UNFUSED must agree bit for bit."""
    import torch
    from tensor_gemm_reduce_gb300 import gemm_rs as G
    from tensor_gemm_reduce_gb300 import metrics, workloads
    torch.cuda.set_device(local)
    stream = torch.cuda.current_stream()
    if args.sweep == "all":
        names = [w.name for w in workloads.WORKLOADS.values() if w.op == "rs" and w.name != "tiny"]
    elif args.sweep == "all_ag":
        names = [w.name for w in workloads.WORKLOADS.values() if w.op == "ag" and w.name != "tiny_ag"]
    else:
        names = args.sweep.split(",")
    for name in names:
        w = workloads.WORKLOADS[name]
        g = torch.Generator(device="cuda")
        g.manual_seed(w.seed)
        A = torch.randn(w.M, w.K, device="cuda", generator=g).bfloat16()
        W = (torch.randn(w.K, w.N, device="cuda", generator=g) * w.K ** -0.5).bfloat16()
        if w.op == "ag":  # row shards of A, column shards of W (all-gather + GEMM)
            A = A.view(8, w.M // 8, w.K).contiguous()
            W = W.view(w.K, 8, w.N // 8).transpose(0, 1).contiguous()
        else:
            A = A.view(w.M, 8, w.K // 8).transpose(0, 1).contiguous()
            W = W.view(8, w.K // 8, w.N).contiguous()
        plan = G.Plan(w.M, w.N, w.K, op=G.OP_AG if w.op == "ag" else G.OP_RS)
        out = torch.empty(*plan.out_shape, dtype=torch.bfloat16, device="cuda")
        ws = plan.new_workspace()
        plan.run(A, W, out, ws, G.UNFUSED)
        ref = out.clone()
        plan.run(A, W, out, ws, G.FUSED)
        torch.cuda.synchronize()
        if plan.status() != G.GEMM_RS_OK or not torch.equal(ref.view(torch.int16), out.view(torch.int16)):
            raise RuntimeError(f"{name}: fused and unfused outputs differ")
        iters = args.sweep_iters or max(5, min(40, int(20e-3 / max(w.flops / 1.5e15, 1e-6))))
        times = {}
        for _ in range(args.sweep_rounds):  # rounds interleave the modes: drift affects all alike
            for mode, key in ((G.GEMM_ONLY, "gemm"), (G.RS_ONLY, "rs"), (G.FUSED, "fused"),
                              (G.UNFUSED, "unfused")):
                for _ in range(2):
                    plan.run(A, W, out, ws, mode)
                times.setdefault(key, []).append(
                    time_batched(lambda: plan.run(A, W, out, ws, mode), iters, 1, stream))
        if plan.status() != G.GEMM_RS_OK:
            raise RuntimeError(f"{name}: device status")
        t = {k: metrics.median(v) for k, v in times.items()}
        tuned = None
        if args.tuned:
            op = G.OP_AG if w.op == "ag" else G.OP_RS
            best, best_us, table = G.tune(w.M, w.N, w.K, A, W, out, mode=G.FUSED, iters=iters,
                                          rounds=args.sweep_rounds, op=op)
            tplan = G.Plan(w.M, w.N, w.K, **{k: v for k, v in best.items() if k != "timeout_ns"})
            tws = tplan.new_workspace()
            tplan.run(A, W, out, tws, G.FUSED)
            torch.cuda.synchronize()
            if tplan.status() != G.GEMM_RS_OK or not torch.equal(ref.view(torch.int16), out.view(torch.int16)):
                raise RuntimeError(f"{name}: the tuned plan's output differs")
            tt = []
            for _ in range(args.sweep_rounds):  # interleaved with the default plan again
                for pl, wsx, key in ((plan, ws, "default"), (tplan, tws, "tuned")):
                    for _ in range(2):
                        pl.run(A, W, out, wsx, G.FUSED)
                    tt.append((key, time_batched(lambda: pl.run(A, W, out, wsx, G.FUSED), iters, 1, stream)))
            t_def = metrics.median([v for k, v in tt if k == "default"])
            t_tun = metrics.median([v for k, v in tt if k == "tuned"])
            knobs = {k: best[k] for k in ("mma_ctas", "reducer_warps", "unit_rows", "band_m", "tail_waves",
                                          "half_regions", "copy_engines")}
            tuned = {"plan": knobs, "t_fused_tuned_us": t_tun * 1e6, "t_fused_default_us": t_def * 1e6,
                     "tuner_best_us": best_us, "candidates": len(table)}
            tplan.close()
            del tws
        print(json.dumps({
            "sweep": name, "layer": "all-gather + GEMM" if w.op == "ag" else "GEMM + reduce-scatter",
            "M": w.M, "N": w.N, "K": w.K,
            "tflops_fused": w.flops / t["fused"] / 1e12, "tflops_gemm": w.flops / t["gemm"] / 1e12,
            "overlap_efficiency": metrics.overlap_efficiency(t["gemm"], t["rs"], t["fused"]),
            "fused_speedup_vs_unfused": t["unfused"] / t["fused"],
            **{f"t_{k}_us": v * 1e6 for k, v in t.items()}, "iters": args.sweep_rounds * iters,
            "tuned": tuned}),
            flush=True)
        plan.close()
        del A, W, out, ws, ref
        torch.cuda.empty_cache()
    return 0


def main(argv=None):
    args = parse_args(argv)
    rank, world, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if args.profile:
        return run_profile_target(args, local)
    if args.sweep:
        return run_sweep(args, local)
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    try:
        return run_ours(args, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
