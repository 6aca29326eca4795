"""CPU oracle for the row-parallel linear layer with a reduce-scatter (float64).

TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the benchmark's
CPU-baseline leg may import this module.  It shares no code with the CUDA
library (no kernels, headers, helpers or tables) and the library never calls
it.  It is deliberately plain and slow: every step is written out as the
definition states it, with library float64 matmuls as the only building block.

What is computed (problem page "A fused GEMM + reduce-scatter kernel hiding 90%
of communication on 8 H100 GPUs", sections "What is asked" and "How it gets
verified"; FLUX page, Figure 2):
  the tensor-parallel group has 8 ranks.  Rank r holds the K-shard A_r (columns
  [r*K/8, (r+1)*K/8) of A) and W_r (the same rows of W) and computes the
  partial product P_r = A_r W_r in BF16 with FP32 accumulation.  The partials
  are summed across ranks and each rank keeps one row slice of the total: rank
  s receives rows [s*M/8, (s+1)*M/8) (a reduce-scatter).

Readings of points the pages leave open:
  * each partial is rounded to bf16 once, round to nearest even, directly from
    its exact value (the bf16 tensor a real reduce-scatter would move): a
    float64 matmul, with the elements whose float64 error could change that
    rounding summed exactly (bf16_of_exact_product);
  * the sum over ranks is a left fold in FP32 (IEEE, round to nearest even),
    starting from the rank-0 partial and adding ranks 1..7 in order;
  * the FP32 total is rounded to bf16, round to nearest even;
  * the "FP32 reference" of the correctness rule is taken in float64: the
    unrounded sum of the exact partials.

The column-parallel partner layer, all-gather then GEMM (FLUX page, abstract
and Figure 1; mKernel page, section 4), is here too (ag_gemm): rank r holds
rows [r*M/8, (r+1)*M/8) of A and columns [r*N/8, (r+1)*N/8) of W, gathers all
rows of A (in rank order, which puts A back together) and computes
C_r = A W_r, rounded once to bf16 from its exact value (the GPU accumulates
in FP32, so parity there is a tolerance).

Pins that tie this module to something other than itself live in
tests/test_oracle_pins.py (exact rational brute force, also on arbitrary
wide-exponent inputs drawn by hypothesis, closed forms, invariants and
library routines).
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np

WORLD = 8

# ---------------------------------------------------------------------------
# bf16 helpers (own implementation: 8 significant bits, exponent range of fp32)
# ---------------------------------------------------------------------------


def bf16_round(x) -> np.ndarray:
    """Round to the nearest bf16 value, ties to even, straight from the input.

    The input is taken at its own precision (float64 or float32), so a float64
    value is rounded once, not through float32.  Returns float64 values that
    are exactly representable in bf16 (inf beyond the bf16 range, NaN kept).
    bf16 has an 8-bit significand, so a value with binary exponent e
    (x = m * 2**e, 0.5 <= |m| < 1) has quantum 2**(e-8); the quantum never
    goes below the smallest subnormal, 2**-133.
    """
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)
    qe = np.maximum(e - 8, -133)
    y = np.ldexp(np.rint(np.ldexp(x, -qe)), qe)  # rint rounds half to even
    y = np.where(np.abs(y) >= 2.0 ** 128, np.copysign(np.inf, x), y)
    return np.where(np.isfinite(x), y, x)


def bf16_round_fraction(x: Fraction) -> float:
    """Round an exact rational to the nearest bf16 value, ties to even
    (8 significant bits, quantum never below 2**-133, inf from 2**128 up)."""
    if x == 0:
        return 0.0
    sign = -1.0 if x < 0 else 1.0
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()  # 2**(e-1) < a < 2**(e+1)
    if a >= Fraction(2) ** e:
        e += 1                                                  # now 2**(e-1) <= a < 2**e
    qe = max(e - 8, -133)
    n = a / Fraction(2) ** qe
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    v = Fraction(fl) * Fraction(2) ** qe
    return sign * (float("inf") if v >= Fraction(2) ** 128 else float(v))


def bf16_of_exact_product(X, Y, S=None) -> np.ndarray:
    """bf16(X @ Y) rounded once from the exact value, for bf16 X [M][k] and
    Y [k][N] (values).

    S = X @ Y in float64 (computed here unless given): every product of two
    bf16 values is exact in float64 and only the k - 1 additions round, by at
    most k * 2**-53 * sum|x||y| whatever the summation order.  Where the
    interval S +- e (e = 4 times that bound, covering the interval's own
    rounding) rounds to one bf16 value, the exact value inside it rounds to
    the same value (rounding is monotone).  At the other elements the exact
    value could lie across a bf16 midpoint from S (products of very different
    magnitudes); those are summed exactly with fractions and rounded.
    """
    X = np.asarray(X, dtype=np.float64)
    Y = np.asarray(Y, dtype=np.float64)
    if S is None:
        S = X @ Y
    Q = bf16_round(S)
    k = X.shape[1]
    if k <= 1 or Q.size == 0:
        return Q  # one product (or none): S is exact
    e = 4.0 * k * 2.0 ** -53 * (np.abs(X) @ np.abs(Y))
    with np.errstate(invalid="ignore", over="ignore"):
        unsure = (bf16_round(S - e) != bf16_round(S + e)) & np.isfinite(S) & np.isfinite(e)
    for i, j in zip(*np.nonzero(unsure)):
        exact = sum((Fraction(float(X[i, t])) * Fraction(float(Y[t, j])) for t in range(k)),
                    Fraction(0))
        Q[i, j] = bf16_round_fraction(exact)
    return Q


def bf16_from_bits(bits) -> np.ndarray:
    """uint16 bf16 bit patterns -> float64 values (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def bf16_to_bits(values) -> np.ndarray:
    """bf16-representable float values -> uint16 bit patterns (exact)."""
    v = np.asarray(values, dtype=np.float64).astype(np.float32)
    return (v.view(np.uint32) >> 16).astype(np.uint16)


# ---------------------------------------------------------------------------
# The operation
# ---------------------------------------------------------------------------


def rank_partials(A_shards, W_shards) -> np.ndarray:
    """Per-rank partial products S_r = A_r @ W_r in float64.

    A_shards: [8][M][Kr] (bf16 bits or float values), W_shards: [8][Kr][N].
    Inputs are bf16, so every product is exact in float64 and the float64
    matmul only rounds its running sums (relative error ~ Kr * 2**-53); see
    partials_bf16 for the partials' exactly rounded bf16 values.
    """
    A = _as_values(A_shards)
    W = _as_values(W_shards)
    assert A.ndim == 3 and W.ndim == 3 and A.shape[0] == W.shape[0] == WORLD
    assert A.shape[2] == W.shape[1]
    return np.stack([A[r] @ W[r] for r in range(WORLD)])


def partials_bf16(A_shards, W_shards, S=None) -> np.ndarray:
    """Each rank's partial rounded once to bf16 from its exact value:
    Q_r = bf16(A_r @ W_r), [8][M][N].  S: rank_partials' result, if at hand."""
    A = _as_values(A_shards)
    W = _as_values(W_shards)
    if S is None:
        S = rank_partials(A, W)
    return np.stack([bf16_of_exact_product(A[r], W[r], S[r]) for r in range(WORLD)])


def reduce_partials(S: np.ndarray, Q=None):
    """Round each partial to bf16, fold in FP32 in rank order, round to bf16.

    S: the partials (exact values, or rank_partials' float64 values); Q: their
    bf16 roundings if already formed (partials_bf16), else bf16(S).
    Returns (out, ref): out [M][N] float64 values on the bf16 grid, ref [M][N]
    the unrounded float64 sum of the partials.
    """
    if Q is None:
        Q = [bf16_round(S[r]) for r in range(WORLD)]
    Q = [np.asarray(Q[r]).astype(np.float32) for r in range(WORLD)]  # exact casts
    T = Q[0].copy()
    for r in range(1, WORLD):
        T = (T + Q[r]).astype(np.float32)  # IEEE fp32 add, round to nearest even
    out = bf16_round(T)
    ref = np.zeros(S.shape[1:], dtype=np.float64)
    for r in range(WORLD):
        ref = ref + S[r]
    return out, ref


def gemm_rs(A_shards, W_shards):
    """Full output of the row-parallel linear layer.

    Returns (out, ref) as float64 arrays [M][N]; slice s of the reduce-scatter
    is rows [s*M/8, (s+1)*M/8) of out (see slices()).
    """
    S = rank_partials(A_shards, W_shards)
    return reduce_partials(S, partials_bf16(A_shards, W_shards, S))


def gemm_rs_rows(A_shards, W_shards, rows):
    """The same result evaluated only at the given output rows.

    Row i of every partial depends only on row i of each A_r, so this is the
    definition applied to a row subset (used to check sampled outputs of large
    workloads).  Returns (out[len(rows)][N], ref[len(rows)][N]).
    """
    rows = np.asarray(rows, dtype=np.int64)
    A = _as_values(A_shards)[:, rows, :]
    return gemm_rs(A, W_shards)


def gemm_allreduce(A_shards, W_shards):
    """GEMM + all-reduce of the same layer: every rank ends with the whole sum.

    mKernel page, sections 3.1, 4 and 5.2 (GEMM+AllReduce: a reduction within
    the node, after which every GPU holds the complete output).  The sum is the
    same rank-order fp32 fold of the bf16 partials as the reduce-scatter's;
    rank r's copy is all M rows of it.  Returns (out[8][M][N], ref[M][N]).
    """
    out, ref = gemm_rs(A_shards, W_shards)
    world = np.asarray(A_shards).shape[0]
    return np.stack([out.copy() for _ in range(world)]), ref


def ag_gemm(A_shards, W_shards):
    """All-gather + GEMM.  A_shards [8][M/8][K] (row shards), W_shards [8][K][N/8]
    (column shards).  The gather stacks the row shards in rank order; rank r's
    output is C_r = bf16(A W_r).  Returns (C[8][M][N/8], ref[8][M][N/8]), ref
    unrounded (float64)."""
    A = np.concatenate(list(_as_values(A_shards)), axis=0)
    Wv = _as_values(W_shards)
    ref = np.stack([A @ Wv[r] for r in range(Wv.shape[0])])
    return np.stack([bf16_of_exact_product(A, Wv[r], ref[r]) for r in range(Wv.shape[0])]), ref


def ag_gemm_rows(A_shards, W_shards, rows):
    """ag_gemm at the given rows of the gathered A only (row i of every C_r
    depends only on row i of A).  Returns (C[8][len(rows)][N/8], ref)."""
    A = np.concatenate(list(_as_values(A_shards)), axis=0)[np.asarray(rows, dtype=np.int64)]
    Wv = _as_values(W_shards)
    ref = np.stack([A @ Wv[r] for r in range(Wv.shape[0])])
    return np.stack([bf16_of_exact_product(A, Wv[r], ref[r]) for r in range(Wv.shape[0])]), ref


def slices(out: np.ndarray, world: int = WORLD):
    """Split the reduced output into the per-rank row slices of the scatter."""
    M = out.shape[0]
    assert M % world == 0
    h = M // world
    return [out[s * h:(s + 1) * h] for s in range(world)]


# ---------------------------------------------------------------------------
# The correctness rule (problem page, section "How it gets verified"): the
# output is accepted when it is within bf16 accuracy and its largest relative
# error against a high-precision reference is no more than 1.1 times the
# unfused path's
# ---------------------------------------------------------------------------


def err_vs_oracle(X, out) -> float:
    """max |X - out| / max |out| against the oracle's bf16 result."""
    X = np.asarray(X, dtype=np.float64)
    den = float(np.max(np.abs(out))) if out.size else 0.0
    num = float(np.max(np.abs(X - out))) if out.size else 0.0
    return num / den if den > 0 else num


def rel_vs_ref(X, ref) -> float:
    """max |X - ref| / max |ref| against the float64 (unrounded) reference."""
    X = np.asarray(X, dtype=np.float64)
    den = float(np.max(np.abs(ref))) if ref.size else 0.0
    num = float(np.max(np.abs(X - ref))) if ref.size else 0.0
    return num / den if den > 0 else num


def _as_values(x) -> np.ndarray:
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return bf16_from_bits(x)
    return x.astype(np.float64)
