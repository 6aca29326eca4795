"""Shared helpers of the GPU tests: seeded inputs to device tensors, runs
through the C-ABI binding, comparisons against the oracle."""
import numpy as np
import torch

import oracle
from tensor_gemm_reduce_gb300 import gemm_rs as G
from tensor_gemm_reduce_gb300 import workloads

TOL = 1e-2  # max |X - oracle| / max |oracle|


def to_dev(bits: np.ndarray) -> torch.Tensor:
    """uint16 bf16 patterns -> contiguous bf16 CUDA tensor (same bits)."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.cuda().view(torch.bfloat16)


def to_host_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def to_host_values(t: torch.Tensor) -> np.ndarray:
    return oracle.bf16_from_bits(to_host_bits(t))


class Case:
    """Inputs on the device plus a plan and a workspace."""

    def __init__(self, A_bits, W_bits, **plan_kw):
        self.A_bits, self.W_bits = A_bits, W_bits
        _, self.M, self.Kr = A_bits.shape
        self.N = W_bits.shape[2]
        self.K = 8 * self.Kr
        self.A = to_dev(A_bits)
        self.W = to_dev(W_bits)
        self.plan = G.Plan(self.M, self.N, self.K, **plan_kw)
        self.ws = self.plan.new_workspace()
        self.out = torch.empty(*self.plan.out_shape, dtype=torch.bfloat16, device="cuda")

    def run(self, mode=G.FUSED, check_status=True, poison=False):
        if poison:
            self.ws[: self.plan.info.staging_bytes].fill_(0xFF)  # NaN bf16 everywhere
            self.out.view(torch.int16).fill_(-1)
        self.plan.run(self.A, self.W, self.out, self.ws, mode)
        if check_status:
            rc = self.plan.status()
            assert rc == G.GEMM_RS_OK, G.strerror(rc)
        torch.cuda.synchronize()
        return self.out.clone()

    def staging(self) -> torch.Tensor:
        n = 8 * self.M * self.N
        return self.ws[: 2 * n].view(torch.bfloat16).view(8, self.M, self.N)


def assert_parity(X_values: np.ndarray, out: np.ndarray, ref: np.ndarray):
    e = oracle.err_vs_oracle(X_values, out)
    assert e <= TOL, f"max|err|/max|ref| = {e:.3e} > {TOL}"
    return e


def partial_ulp_check(stage_vals: np.ndarray, S: np.ndarray, absAW: np.ndarray, Kr: int,
                      max_mismatch_frac=0.02):
    """GPU bf16 partials vs the exact partials rounded once to bf16.

    The GPU accumulates each partial in fp32 on the tensor cores, the oracle
    rounds the exact sum, so the two can differ by one bf16 step where the
    exact partial lies within the fp32 accumulation error of a rounding
    boundary.  Bound per element: one bf16 step of Q plus the fp32
    accumulation error 2 * Kr * 2**-24 * sum_k |a_k w_k| (absAW), taken
    with a margin of two for truncating adders.
    """
    Q = oracle.bf16_round(S)
    diff = np.abs(stage_vals - Q)
    _, e = np.frexp(np.maximum(np.maximum(np.abs(Q), np.abs(stage_vals)), 2.0 ** -126))
    step = np.ldexp(1.0, e - 8)
    bound = step + 2.0 * Kr * 2.0 ** -24 * absAW
    worst = float(np.max(diff / bound)) if diff.size else 0.0
    assert worst <= 1.0, f"partial error {worst:.2f} x the bound"
    frac = float(np.mean(diff > 0)) if diff.size else 0.0
    assert frac <= max_mismatch_frac, f"{frac:.4f} of partials differ from the rounded exact value"
    return frac


def abs_partials(A_bits, W_bits):
    """sum_k |a_k| |w_k| per rank, float64 [8][M][N]."""
    A = np.abs(oracle.bf16_from_bits(A_bits))
    W = np.abs(oracle.bf16_from_bits(W_bits))
    return np.stack([A[r] @ W[r] for r in range(A.shape[0])])
