"""GPU parity at the full workload sizes, in the benchmark's launch
configuration (default plan): sampled output rows against the oracle, the
fused and unfused outputs bit for bit, the per-rank partials of the sampled
rows, and whole-output properties (finite, slice statistics).

Every registered row-parallel workload is covered: the Llama-3-70B and
Mixtral-8x22B projections, every shape of the full sweep (M in {512, 2048,
8192, 32768} x (N, K) in {(8192, 8192), (8192, 28672), (6144, 6144),
(6144, 16384)}) and the FLUX page's Figure 4 reduce-scatter shape
(n, k) = (12288, 49152), m = 1024..8192.

On two of them (o_proj and the largest-M 6144 x 6144 sweep shape) the
reduction is also checked exactly: the oracle's rank-order fp32 fold of the
GPU's own bf16 partials (read from the staging after the GEMM alone) must
equal the fused and the unfused outputs bit for bit, on every element.

Workloads: problem page "A fused GEMM + reduce-scatter kernel hiding 90% of
communication on 8 H100 GPUs", section "How it gets verified": token counts
M of 512 to 32768 and the output and inner dimensions of Llama-3-70B and
Mixtral-8x22B projection layers, 8-way tensor parallelism; FLUX page,
Figure 4 caption (the reduce-scatter GEMM shape).
"""
import numpy as np
import pytest
import torch

import oracle
from tensor_gemm_reduce_gb300 import gemm_rs as G
from tensor_gemm_reduce_gb300 import workloads
from gpu_helpers import Case, TOL, abs_partials, partial_ulp_check, to_host_bits, to_host_values

pytestmark = pytest.mark.gpu

# workloads whose fold is also checked bit for bit on every output element
EXACT_REDUCER = {"llama3_70b_o_proj_m2048", "sweep_m32768_n6144_k6144"}


def _sample_rows(M, seed, per_slice=3):
    g = np.random.Generator(np.random.PCG64(seed))
    h = M // 8
    rows = set()
    for s in range(8):
        rows.update({s * h, s * h + h - 1})
        rows.update(int(x) for x in g.integers(s * h, s * h + h, size=per_slice))
    rows.update(r for r in (127, 128, 255, 256, M - 1) if r < M)
    return np.array(sorted(rows))


def _exact_fold_check(c, fused, unf, block_rows=2048):
    """The GPU's own partials Q (staging after UNFUSED) folded by the oracle:
    bit for bit the fused and the unfused outputs, block of rows by block."""
    stage = c.staging()
    f_bits, u_bits = fused.view(torch.int16), unf.view(torch.int16)
    for r0 in range(0, c.M, block_rows):
        r1 = min(c.M, r0 + block_rows)
        Q = to_host_values(stage[:, r0:r1, :])
        out, _ = oracle.reduce_partials(Q, Q)
        exp = oracle.bf16_to_bits(out)
        got_f = f_bits[r0:r1].cpu().numpy().view(np.uint16)
        got_u = u_bits[r0:r1].cpu().numpy().view(np.uint16)
        bad = np.count_nonzero(got_f != exp)
        assert bad == 0, f"rows {r0}..{r1}: {bad} fused elements differ from the fold of the partials"
        assert np.array_equal(got_u, exp), f"rows {r0}..{r1}: unfused differs from the fold"


def _check_workload(w):
    A, W = workloads.make_inputs(w)
    c = Case(A, W)
    fused = c.run(G.FUSED, poison=True)
    rows = _sample_rows(w.M, w.seed)
    ridx = torch.as_tensor(rows, device="cuda")
    S = oracle.rank_partials(A[:, rows, :], W)
    out, ref = oracle.reduce_partials(S, oracle.partials_bf16(A[:, rows, :], W, S))
    fv = to_host_values(fused[ridx])
    e = oracle.err_vs_oracle(fv, out)
    assert e <= TOL, f"{w.name}: sampled err {e:.3e}"
    unf = c.run(G.UNFUSED, poison=True)  # leaves the GEMM's partials in the staging
    stage = to_host_values(c.staging()[:, ridx, :])
    partial_ulp_check(stage, S, abs_partials(A[:, rows, :], W), c.Kr)
    # the sampled rows: the oracle's fold of the GPU's own partials is the GPU's output
    fold, _ = oracle.reduce_partials(stage, stage)
    assert np.array_equal(oracle.bf16_to_bits(fold), to_host_bits(fused[ridx]))
    # whole output: finite, per-slice spread near the recipe's unit variance
    assert torch.isfinite(fused.float()).all()
    sl = fused.float().view(8, w.M // 8, w.N)
    std = sl.std(dim=(1, 2))
    assert torch.all((std > 0.7) & (std < (3.0 if w.outliers else 1.3))), std
    assert torch.equal(fused.view(torch.int16), unf.view(torch.int16))
    r_f = oracle.rel_vs_ref(fv, ref)
    r_u = oracle.rel_vs_ref(to_host_values(unf[ridx]), ref)
    assert r_f <= 1.1 * r_u + 1e-12
    if w.name in EXACT_REDUCER:
        _exact_fold_check(c, fused, unf)
    return e


def _rs_workloads():
    return [w for w in workloads.WORKLOADS.values() if w.op == "rs" and w.name != "tiny"]


def _is_large(w):
    # host-side input drawing dominates: mark the shapes with the most elements slow
    return w.M * w.K + w.K * w.N > 200_000_000


@pytest.mark.parametrize("name", [w.name for w in _rs_workloads() if not _is_large(w)])
def test_workload_sampled(name):
    _check_workload(workloads.WORKLOADS[name])


@pytest.mark.slow
@pytest.mark.parametrize("name", [w.name for w in _rs_workloads() if _is_large(w)])
def test_large_workload_sampled(name):
    _check_workload(workloads.WORKLOADS[name])


def test_every_config_shape_is_covered():
    """The benchmark's configurations, all in the registry checked above."""
    names = {w.name for w in _rs_workloads()}
    shapes = {(w.M, w.N, w.K) for w in _rs_workloads()}
    for n, k in ((8192, 8192), (8192, 28672), (6144, 6144), (6144, 16384)):
        for m in (512, 2048, 8192, 32768):
            assert (m, n, k) in shapes
    for m in (1024, 2048, 4096, 8192):
        assert (m, 12288, 49152) in shapes
    assert {"llama3_70b_o_proj_m2048", "llama3_70b_down_proj_m512", "llama3_70b_down_proj_m8192",
            "mixtral_8x22b_down_proj_m2048", "mixtral_8x22b_down_proj_m32768"} <= names
    assert EXACT_REDUCER <= names
