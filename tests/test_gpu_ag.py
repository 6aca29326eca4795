"""GPU parity of the all-gather + GEMM layer (op = OP_AG) against the oracle.

The column-parallel partner of the row-parallel layer (FLUX page, abstract
and Figure 1: all-gather fused into the GEMM; mKernel page, section 4: the
local shard first, then the others as they arrive).  Rank r holds rows
[r*M/8, (r+1)*M/8) of A and columns [r*N/8, (r+1)*N/8) of W and computes
C_r = A W_r after gathering A.  Checks: the output within the bf16 tolerance
of the oracle and each element within one bf16 step plus the fp32
accumulation bound; FUSED == UNFUSED == GEMM_ONLY bit for bit (same tiles);
after the unfused gather every rank's buffer holds all of A.  The gather
buffers are poisoned with NaN before fused runs, so a tile that read a shard
before its copy was published would show.
"""
import numpy as np
import pytest
import torch

import oracle
from tensor_gemm_reduce_gb300 import gemm_rs as G
from tensor_gemm_reduce_gb300 import workloads
from gpu_helpers import TOL, partial_ulp_check, to_dev, to_host_values

pytestmark = pytest.mark.gpu


class AGCase:
    def __init__(self, A_bits, W_bits, **plan_kw):
        self.A_bits, self.W_bits = A_bits, W_bits
        _, h, self.K = A_bits.shape
        self.M = 8 * h
        self.N = 8 * W_bits.shape[2]
        self.A = to_dev(A_bits)
        self.W = to_dev(W_bits)
        self.plan = G.Plan(self.M, self.N, self.K, op=G.OP_AG, **plan_kw)
        self.ws = self.plan.new_workspace()
        self.out = torch.empty(*self.plan.out_shape, dtype=torch.bfloat16, device="cuda")

    def run(self, mode=G.FUSED, poison=False):
        if poison:
            self.ws[: self.plan.info.staging_bytes].fill_(0xFF)  # NaN in every gather buffer
            self.out.view(torch.int16).fill_(-1)
        self.plan.run(self.A, self.W, self.out, self.ws, mode)
        rc = self.plan.status()
        assert rc == G.GEMM_RS_OK, G.strerror(rc)
        torch.cuda.synchronize()
        return self.out.clone()

    def gather_buffers(self):
        return self.ws[: 2 * 8 * self.M * self.K].view(torch.bfloat16).view(8, self.M, self.K)


def _abs_products(A_bits, W_bits):
    A = np.abs(np.concatenate(list(oracle.bf16_from_bits(A_bits)), axis=0))
    W = np.abs(oracle.bf16_from_bits(W_bits))
    return np.stack([A @ W[r] for r in range(8)])


def _check(A, W, **kw):
    c = AGCase(A, W, **kw)
    fused = c.run(G.FUSED, poison=True)
    C, ref = oracle.ag_gemm(A, W)
    fv = to_host_values(fused)
    e = oracle.err_vs_oracle(fv.reshape(-1, fv.shape[-1]), C.reshape(-1, C.shape[-1]))
    assert e <= TOL, f"max|err|/max|ref| = {e:.3e}"
    partial_ulp_check(fv, ref, _abs_products(A, W), c.K)
    unf = c.run(G.UNFUSED, poison=True)
    assert torch.equal(fused.view(torch.int16), unf.view(torch.int16)), "fused != unfused"
    g = c.gather_buffers()
    A_full = to_dev(np.concatenate(list(A), axis=0))
    for r in range(8):
        assert torch.equal(g[r].view(torch.int16), A_full.view(torch.int16)), r
    c.out.view(torch.int16).fill_(-1)
    only = c.run(G.GEMM_ONLY)
    assert torch.equal(only.view(torch.int16), unf.view(torch.int16))
    again = c.run(G.FUSED, poison=True)  # a second fused run on the same counts
    assert torch.equal(again.view(torch.int16), fused.view(torch.int16))
    return c


def test_tiny_workload():
    A, W = workloads.make_inputs(workloads.WORKLOADS["tiny_ag"])
    c = _check(A, W)
    assert not c.plan.info.ag_direct  # 16-row shards: own shard gathered too


@pytest.mark.parametrize("M,N,K,kw,direct", [
    (2048, 2560, 1024, {}, True),                  # 256-row shards = 2-CTA tile rows
    (1024, 1024, 512, dict(mma_ctas=1), True),     # 128-row shards = 1-CTA tile rows
    (1024, 1024, 512, {}, False),                  # 128-row shards inside 256-row tiles
    (392, 1536, 1600, {}, False),                  # ragged M and K; 49-row shards
    (8, 512, 64, {}, False),                       # one row per shard
    (2048, 2560, 1024, dict(reducer_warps=1, grid=6), True),  # one copy warp, few CTAs
    (2048, 2560, 1024, dict(reducer_warps=5), True),
    (2048, 4096, 512, dict(grid=8), True),   # 16 tiles per rank >= 2 waves of 4 clusters: paced copies
    (1024, 4096, 512, dict(grid=4, mma_ctas=1), True),  # paced, 1-CTA tiles
    # shards moved by the copy engines on 1..4 side streams, no copy warps
    (2048, 2560, 1024, dict(copy_engines=1), True),
    (2048, 2560, 1024, dict(copy_engines=4, grid=6), True),
    (1024, 1024, 512, dict(mma_ctas=1, copy_engines=2), True),
    (392, 1536, 1600, dict(copy_engines=3), False),       # own shard copied too
    (8, 512, 64, dict(copy_engines=2), False),
])
def test_shapes_and_plans(M, N, K, kw, direct):
    A, W = workloads.make_shape_inputs(M, N, K, seed=M + 2 * N + K, op="ag")
    c = _check(A, W, **kw)
    assert bool(c.plan.info.ag_direct) == direct
    n_rounds = 7 if direct else 8
    assert c.plan.info.copy_items % (8 * n_rounds) == 0
    engines = kw.get("copy_engines", 0)
    assert c.plan.info.copy_engines == (engines or -1)
    if engines > 0:  # the fused kernel runs without copy warps
        assert c.plan.info.copy_items == 0 and c.plan.info.threads_fused == c.plan.info.threads_gemm


def test_zero_k_and_host_copies():
    p = G.Plan(64, 512, 0, op=G.OP_AG)
    ws = p.new_workspace()
    out = torch.full(p.out_shape, 3.0, dtype=torch.bfloat16, device="cuda")
    p.run(torch.empty(8, 8, 0, dtype=torch.bfloat16, device="cuda"),
          torch.empty(8, 0, 64, dtype=torch.bfloat16, device="cuda"), out, ws, G.FUSED)
    assert p.status() == G.GEMM_RS_OK
    assert torch.count_nonzero(out).item() == 0
    A, W = workloads.make_shape_inputs(512, 2048, 1024, seed=71, op="ag")
    c = AGCase(A, W)
    ref = c.run(G.UNFUSED)
    A_h = torch.from_numpy(A.view(np.int16)).view(torch.bfloat16).pin_memory()
    W_h = torch.from_numpy(W.view(np.int16)).view(torch.bfloat16).pin_memory()
    out_h = torch.empty(*c.plan.out_shape, dtype=torch.bfloat16).pin_memory()
    c.plan.run_host(A_h, W_h, out_h, c.A, c.W, c.out, c.ws, G.FUSED)
    assert c.plan.status() == G.GEMM_RS_OK
    assert torch.equal(out_h.view(torch.int16), ref.view(torch.int16).cpu())


@pytest.mark.parametrize("engines", [0, 2])
def test_unpublished_copy_times_out_and_recovers(engines):
    """The first copy (a copy warp's item, or a copy engine's shard) is never
    published: the tiles that need its shard give up after 20 ms, the status
    says TIMEOUT, and the next run is clean."""
    A, W = workloads.make_shape_inputs(1024, 2048, 1024, seed=72, op="ag")
    bad = AGCase(A, W, timeout_ns=20_000_000, debug_flags=G.DEBUG_SKIP_ONE_FLAG, copy_engines=engines)
    bad.plan.run(bad.A, bad.W, bad.out, bad.ws, G.FUSED)
    assert bad.plan.status() == G.GEMM_RS_ERR_TIMEOUT
    good = AGCase(A, W, copy_engines=engines)
    C, _ = oracle.ag_gemm(A, W)
    out = to_host_values(good.run(G.FUSED, poison=True))
    assert oracle.err_vs_oracle(out.reshape(-1, out.shape[-1]), C.reshape(-1, C.shape[-1])) <= TOL
    bad.run(G.UNFUSED)  # the debug plan itself is usable again


@pytest.mark.parametrize("name", ["llama3_70b_qkv_m2048",
                                  pytest.param("flux_fig4_ag_m1024", marks=pytest.mark.slow)])
def test_workload_sampled(name):
    w = workloads.WORKLOADS[name]
    A, W = workloads.make_inputs(w)
    c = AGCase(A, W)
    fused = c.run(G.FUSED, poison=True)
    g = np.random.Generator(np.random.PCG64(w.seed))
    h = w.M // 8
    rows = sorted({0, w.M - 1, *(s * h for s in range(8)), *(s * h + h - 1 for s in range(8)),
                   *(int(x) for x in g.integers(0, w.M, size=24))})
    C, ref = oracle.ag_gemm_rows(A, W, rows)
    fv = to_host_values(fused[:, torch.as_tensor(rows, device="cuda")])
    e = oracle.err_vs_oracle(fv.reshape(-1, fv.shape[-1]), C.reshape(-1, C.shape[-1]))
    assert e <= TOL, e
    A_rows = np.abs(oracle.bf16_from_bits(np.concatenate(list(A), axis=0)[rows]))
    absAW = np.stack([A_rows @ np.abs(oracle.bf16_from_bits(W[r])) for r in range(8)])
    partial_ulp_check(fv, ref, absAW, w.K)
    unf = c.run(G.UNFUSED, poison=True)
    assert torch.equal(fused.view(torch.int16), unf.view(torch.int16))
    if name == "llama3_70b_qkv_m2048":  # the same run with the shards moved by the copy engines
        ce = AGCase(A, W, copy_engines=4)
        assert torch.equal(ce.run(G.FUSED, poison=True).view(torch.int16), unf.view(torch.int16))
