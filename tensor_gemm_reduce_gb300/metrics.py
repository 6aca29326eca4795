"""Measurement arithmetic (host only): overlap efficiency, throughput,
roofline fractions, clock-sample summaries and the multi-rank aggregate.

Overlap efficiency: the problem page "A fused GEMM + reduce-scatter kernel
hiding 90% of communication on 8 H100 GPUs" ("How it gets verified") asks for
the overlap efficiency of the fused kernel, as the median of 200 iterations
after warm-up, against the GEMM and the communication each timed alone; the
formula did not survive on the page and is taken as
    (T_gemm + T_rs - T_fused) / T_rs,
the share of the standalone reduce-scatter time that the fused kernel hides.
"""
from __future__ import annotations

import csv
import io
import statistics
from typing import Dict, Iterable, List, Optional


def overlap_efficiency(t_gemm: float, t_rs: float, t_fused: float) -> float:
    if t_rs <= 0:
        raise ValueError("t_rs must be positive")
    return (t_gemm + t_rs - t_fused) / t_rs


def tflops(flops: float, seconds: float) -> float:
    return flops / seconds / 1e12


def median(xs: Iterable[float]) -> float:
    return float(statistics.median(list(xs)))


def gemm_flops(M: int, N: int, K: int) -> int:
    """2*M*N*K: every rank's partial GEMM M x N x K/8, eight of them."""
    return 2 * M * N * K


def rs_bytes(M: int, N: int, world: int = 8) -> int:
    """Algorithmic bytes of the reduce-scatter: read 8 bf16 partials, write one bf16 output."""
    return (world + 1) * M * N * 2


def fused_bytes(M: int, N: int, K: int, world: int = 8) -> int:
    """Algorithmic DRAM bytes of one fused run: operands once, staging written
    and read once, output written once."""
    return 2 * (M * K + K * N) + 2 * world * M * N * 2 + 2 * M * N


def roofline(bound: str, achieved: float, peak: float, unit: str, traffic: Optional[float]) -> Dict:
    return {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
            "frac": achieved / peak if peak else None, "traffic": traffic}


_BAD_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


def summarize_clocks(csv_text: str) -> Dict:
    """Summarise `nvidia-smi --query-gpu=index,clocks.sm,clocks.max.sm,power.draw,
    clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,
    clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,
    clocks_event_reasons.sw_power_cap --format=csv` samples."""
    rows = [r for r in csv.reader(io.StringIO(csv_text)) if r and not r[0].startswith("index")]
    sm, smax, reasons = [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for r in rows:
        r = [x.strip() for x in r]
        if len(r) < 9:
            continue
        try:
            sm.append(float(r[1].split()[0]))
            smax.append(float(r[2].split()[0]))
        except ValueError:
            continue
        for name, val in zip(names, r[5:9]):
            if val.lower().startswith("active"):
                reasons.add(name)
    return {"sm_mhz": median(sm) if sm else None,
            "sm_max_mhz": max(smax) if smax else None,
            "reasons": sorted(reasons),
            "samples": len(sm),
            "rejected": bool(reasons & set(_BAD_REASONS))}


def aggregate_ranks(units_per_rank: List[float], seconds_per_rank: List[float]) -> Dict:
    """Whole-job throughput: all ranks' units over the slowest rank's time."""
    t = max(seconds_per_rank)
    return {"units": float(sum(units_per_rank)), "seconds": t, "rate": sum(units_per_rank) / t}


def max_over_ranks(values: List[float], device=None) -> List[float]:
    """Element-wise maximum of per-rank timings across the process group
    (identity when torch.distributed is not initialised)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.cpu()]


def timeline_tail(tl: Dict) -> Dict:
    """Where a traced fused run spends its end, from Plan.timeline() (times in
    microseconds from the earliest CTA start):
      mma_p50 / mma_max  when the median / last CTA's MMA issue drained (the
                         spread is the GEMM's own imbalance at the end);
      last_queued        when the last reduce item was queued (the final
                         tiles' epilogue and completion adds are done);
      last_done, end     the last item reduced, the last CTA finished;
      after_last_mma     items queued after the last MMA drained, and their
                         median time from taken to done (item_us_late);
      pickup_us, item_us medians over all items of queued -> taken and
                         taken -> done.
    Missing stamps (CTAs beyond the traced ones, items of other runs) are
    skipped."""
    ctas = [c for c in tl.get("ctas", []) if c.get("end") is not None]
    mma = sorted(c["mma_drained"] for c in ctas if c.get("mma_drained") is not None)
    items = [i for i in tl.get("items", [])
             if None not in (i.get("queued"), i.get("taken"), i.get("done"))]
    if not mma or not items:
        raise ValueError("timeline has no MMA stamps or no complete reduce items")
    mma_max = mma[-1]
    late = [i for i in items if i["queued"] > mma_max]
    return {
        "mma_p50": median(mma),
        "mma_max": mma_max,
        "last_queued": max(i["queued"] for i in items),
        "last_done": max(i["done"] for i in items),
        "end": max(c["end"] for c in ctas),
        "after_last_mma": len(late),
        "item_us_late": median(i["done"] - i["taken"] for i in late) if late else 0.0,
        "pickup_us": median(i["taken"] - i["queued"] for i in items),
        "item_us": median(i["done"] - i["taken"] for i in items),
        "items": len(items),
    }
