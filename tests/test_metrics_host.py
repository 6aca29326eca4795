"""Host logic of the measurement: overlap efficiency, clock summaries, the
multi-rank aggregate (gloo, world size 2, CPU) and the CPU reference arm."""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

from tensor_gemm_reduce_gb300 import metrics

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_overlap_efficiency():
    assert metrics.overlap_efficiency(100.0, 40.0, 100.0) == 1.0      # fully hidden
    assert metrics.overlap_efficiency(100.0, 40.0, 140.0) == 0.0      # nothing hidden
    assert metrics.overlap_efficiency(100.0, 40.0, 104.0) == pytest.approx(0.9)
    assert metrics.overlap_efficiency(100.0, 40.0, 96.0) == pytest.approx(1.1)
    with pytest.raises(ValueError):
        metrics.overlap_efficiency(1.0, 0.0, 1.0)


def test_work_figures():
    assert metrics.gemm_flops(2048, 8192, 8192) == 2 * 2048 * 8192 * 8192
    assert metrics.rs_bytes(2048, 8192) == 18 * 2048 * 8192
    assert metrics.fused_bytes(2, 3, 16) == 2 * (2 * 16 + 16 * 3) + 32 * 6 + 2 * 6
    r = metrics.roofline("tensor", 1500.0, 2000.0, "TFLOP/s", None)
    assert r["frac"] == 0.75 and r["traffic"] is None


def test_summarize_clocks():
    csv = (
        "index, clocks.current.sm [MHz], clocks.max.sm [MHz], power.draw [W], clocks_event_reasons.active, "
        "clocks_event_reasons.hw_slowdown, clocks_event_reasons.hw_thermal_slowdown, "
        "clocks_event_reasons.sw_thermal_slowdown, clocks_event_reasons.sw_power_cap\n"
        "0, 1965 MHz, 2070 MHz, 900.1 W, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n"
        "0, 1800 MHz, 2070 MHz, 1390.0 W, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n"
        "0, 1900 MHz, 2070 MHz, 1200.0 W, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n")
    s = metrics.summarize_clocks(csv)
    assert s["sm_mhz"] == 1900.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"] and not s["rejected"] and s["samples"] == 3
    s = metrics.summarize_clocks(csv.replace("Not Active, Not Active, Not Active, Active",
                                             "Active, Not Active, Not Active, Not Active"))
    assert s["rejected"]


def test_timeline_tail():
    tl = {"ctas": [{"start": 0.0, "epilogue_done": 9.0, "mma_drained": 8.0, "end": 12.0},
                   {"start": 0.1, "epilogue_done": 11.0, "mma_drained": 10.0, "end": 13.5},
                   {"start": 0.2, "epilogue_done": 7.0, "mma_drained": 6.0, "end": 12.5},
                   {"start": None, "epilogue_done": None, "mma_drained": None, "end": None}],
          "items": [{"item": 0, "queued": 2.0, "taken": 3.0, "done": 5.0},
                    {"item": 1, "queued": 10.5, "taken": 11.0, "done": 12.0},
                    {"item": 2, "queued": 11.0, "taken": 11.5, "done": 13.0},
                    {"item": 3, "queued": None, "taken": None, "done": None}]}
    t = metrics.timeline_tail(tl)
    assert t["mma_p50"] == 8.0 and t["mma_max"] == 10.0
    assert t["last_queued"] == 11.0 and t["last_done"] == 13.0 and t["end"] == 13.5
    assert t["after_last_mma"] == 2 and t["item_us_late"] == 1.25
    assert t["pickup_us"] == 0.5 and t["item_us"] == 1.5 and t["items"] == 3
    with pytest.raises(ValueError):
        metrics.timeline_tail({"ctas": [], "items": []})


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    elapsed = [1.0 + rank, 0.5 * (2 - rank)]  # rank 0: (1.0, 1.0); rank 1: (2.0, 0.5)
    mx = metrics.max_over_ranks(elapsed)
    agg = metrics.aggregate_ranks([10.0] * world, [mx[0]])
    q.put((rank, mx, agg))
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    ps = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    res = sorted(q.get(timeout=120) for _ in ps)
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, mx, agg in res:
        assert mx == [2.0, 1.0]
        assert agg == {"units": 20.0, "seconds": 2.0, "rate": 10.0}


def test_reference_arm_runs_on_cpu():
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
           "--warmup", "1", "--workload", "tiny", "--reference-seconds", "2"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
    # other ranks of a torchrun launch print nothing and exit 0
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0 and r.stdout.strip() == ""
