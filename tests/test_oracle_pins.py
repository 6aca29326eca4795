"""Pins for the CPU oracle: it is checked against things other than itself.

  * exact rational brute force (fractions.Fraction) with an independent
    round-to-nearest-even for bf16 and fp32, on tiny random shapes and on
    arbitrary wide-exponent inputs drawn by hypothesis;
  * torch's float32 -> bfloat16 conversion (a library routine) for the bf16
    rounding of float32 inputs;
  * closed forms: integer inputs (everything exact), identity weights,
    a single non-zero rank, hand-derived rounding cases (tests/golden);
  * invariants: linearity and rank-permutation invariance in the exact range,
    the concatenated slices equal A @ W within the rounding bound of the
    definition, the output statistics of the N(0,1) x N(0,1/K) recipe.

Operation: problem page "A fused GEMM + reduce-scatter kernel hiding 90% of
communication on 8 H100 GPUs" (sections "What is asked", "How it gets
verified") and the FLUX page, Figure 2 (row-parallel partition).
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from tensor_gemm_reduce_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

# ---------------------------------------------------------------------------
# independent exact rounding (Fractions), used only by these pins
# ---------------------------------------------------------------------------


def _round_exact(x: Fraction, sig_bits: int, min_exp: int) -> Fraction:
    """Nearest value with sig_bits significant bits (quantum >= 2**min_exp), ties to even."""
    if x == 0:
        return Fraction(0)
    sign = 1 if x > 0 else -1
    a = abs(x)
    e = 0  # find e with 2**(e-1) <= a < 2**e
    while Fraction(2) ** e <= a:
        e += 1
    while Fraction(2) ** (e - 1) > a:
        e -= 1
    q = Fraction(2) ** max(e - sig_bits, min_exp)
    n = a / q
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return sign * fl * q


def rbf16(x: Fraction) -> Fraction:
    return _round_exact(x, 8, -133)


def rfp32(x: Fraction) -> Fraction:
    return _round_exact(x, 24, -149)


def brute_force(A_sh, W_sh):
    """Exact partials, exact bf16 rounding, exact fp32 fold emulation."""
    A = [[[Fraction(float(v)) for v in row] for row in oracle.bf16_from_bits(a)] for a in A_sh]
    W = [[[Fraction(float(v)) for v in row] for row in oracle.bf16_from_bits(w)] for w in W_sh]
    R, M, Kr = A_sh.shape
    N = W_sh.shape[2]
    out = np.zeros((M, N))
    for i in range(M):
        for j in range(N):
            t = None
            for r in range(R):
                s = sum((A[r][i][k] * W[r][k][j] for k in range(Kr)), Fraction(0))
                q = rbf16(s)
                t = q if t is None else rfp32(t + q)
            out[i, j] = float(rbf16(t))
    return out


def _bits_from_values(v):
    return oracle.bf16_to_bits(np.asarray(v, dtype=np.float64))


def _partials_to_shards(partials_per_rank):
    """Build shards whose exact partial at (0,0) is the given value per rank.

    A_r[0][0] = c_r with W_r[0][0] = 1 needs c_r to be a bf16 value; for
    general exact values the value is split over the K-shard as a sum of
    bf16 terms (each term times a weight of 1).
    """
    terms = []
    for c in partials_per_rank:
        c = Fraction(c)
        ts = []
        while c != 0:
            t = rbf16(c)
            if t == 0:
                break
            ts.append(t)
            c -= t
        assert c == 0
        terms.append(ts)
    Kr = max(1, max(len(t) for t in terms))
    Kr = ((Kr + 7) // 8) * 8
    A = np.zeros((8, 8, Kr))
    W = np.zeros((8, Kr, 8))
    for r, ts in enumerate(terms):
        for k, t in enumerate(ts):
            A[r, 0, k] = float(t)
            W[r, k, 0] = 1.0
    return _bits_from_values(A), _bits_from_values(W)


# ---------------------------------------------------------------------------
# bf16 rounding
# ---------------------------------------------------------------------------


def test_bf16_round_matches_torch_on_float32():
    g = np.random.Generator(np.random.PCG64(7))
    x = g.standard_normal(200000).astype(np.float32) * np.float32(3.0)
    x = np.concatenate([x,
                        (g.standard_normal(20000) * 1e-39).astype(np.float32),  # subnormals
                        (g.standard_normal(20000) * 3e38).astype(np.float32),   # near overflow
                        np.float32([0.0, -0.0, 1.00390625, -1.00390625, 1.01171875,
                                    3.3895314e38, 3.4e38, 1e-45, np.inf, -np.inf])])
    # exact ties: odd multiples of half a bf16 quantum
    m = g.integers(128, 256, size=5000)
    e = g.integers(-120, 120, size=5000)
    ties = np.ldexp(m * 2 + 1, e - 9).astype(np.float32)
    x = np.concatenate([x, ties, -ties])
    ours = oracle.bf16_to_bits(oracle.bf16_round(x))
    lib = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, lib)


def test_bf16_round_matches_exact_rounding_on_float64():
    g = np.random.Generator(np.random.PCG64(8))
    m = g.integers(2 ** 52, 2 ** 53, size=3000).astype(np.float64)
    e = g.integers(-140, 100, size=3000)
    x = np.ldexp(m, e - 52) * np.where(g.random(3000) < 0.5, -1, 1)
    # near-ties from float64: tie +/- a tiny amount
    base = np.ldexp(g.integers(256, 512, size=500).astype(np.float64) * 2 + 1, -9)
    x = np.concatenate([x, base, base + 2.0 ** -40, base - 2.0 ** -40])
    got = oracle.bf16_round(x)
    for xi, gi in zip(x, got):
        assert Fraction(float(gi)) == rbf16(Fraction(float(xi))), xi


def test_bf16_round_single_rounding_from_float64():
    x = 1.0 + 2.0 ** -8 + 2.0 ** -40  # above the tie; through float32 it would become the tie
    assert oracle.bf16_round(x) == 1.0 + 2.0 ** -7
    assert oracle.bf16_round(np.float32(x)) == 1.0  # the float32 value is the tie itself


def test_bf16_bits_roundtrip():
    bits = np.arange(0, 65536, dtype=np.uint32).astype(np.uint16)
    v = oracle.bf16_from_bits(bits)
    finite = np.isfinite(v)
    back = oracle.bf16_to_bits(v[finite])
    assert np.array_equal(back, bits[finite])
    assert np.array_equal(oracle.bf16_round(v[finite]), v[finite])


# ---------------------------------------------------------------------------
# the reduce step: hand-derived cases
# ---------------------------------------------------------------------------


def _golden_cases():
    with open(os.path.join(GOLDEN, "rounding_cases.json")) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["name"][:40])
def test_reduce_golden_cases(case):
    S = np.zeros((8, 1, 1))
    for r, (m, e) in enumerate(case["partials"]):
        S[r, 0, 0] = float(Fraction(m) * Fraction(2) ** e)
    out, _ = oracle.reduce_partials(S)
    exp = case["expected"]
    if exp == "inf":
        assert out[0, 0] == np.inf
    else:
        assert out[0, 0] == float(Fraction(exp[0]) * Fraction(2) ** exp[1])


@pytest.mark.parametrize("case", [c for c in _golden_cases() if c["expected"] != "inf"],
                         ids=lambda c: c["name"][:40])
def test_golden_cases_through_the_whole_pipeline(case):
    """The same cases built as GEMM inputs (exact partials) through gemm_rs and brute force."""
    vals = [Fraction(m) * Fraction(2) ** e for m, e in case["partials"]]
    A, W = _partials_to_shards(vals)
    out, _ = oracle.gemm_rs(A, W)
    exp = case["expected"]
    assert out[0, 0] == float(Fraction(exp[0]) * Fraction(2) ** exp[1])
    assert np.array_equal(out, brute_force(A, W))


# ---------------------------------------------------------------------------
# the whole pipeline against exact brute force
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("M,N,K,seed", [(16, 8, 16, 1), (8, 8, 40, 2), (24, 16, 64, 3)])
def test_pipeline_matches_brute_force(M, N, K, seed):
    A, W = workloads.make_shape_inputs(M, N, K, seed)
    out, ref = oracle.gemm_rs(A, W)
    assert np.array_equal(out, brute_force(A, W))


def test_pipeline_matches_brute_force_wide_exponents():
    """Inputs scaled by random powers of two so that the fp32 fold really rounds."""
    g = np.random.Generator(np.random.PCG64(11))
    M, N, K = 8, 8, 32
    A, W = workloads.make_shape_inputs(M, N, K, 5)
    Av = oracle.bf16_from_bits(A) * np.ldexp(1.0, g.integers(-30, 30, size=A.shape))
    Wv = oracle.bf16_from_bits(W) * np.ldexp(1.0, g.integers(-30, 30, size=W.shape))
    A2, W2 = _bits_from_values(Av), _bits_from_values(Wv)
    out, _ = oracle.gemm_rs(A2, W2)
    assert np.array_equal(out, brute_force(A2, W2))
    # and the fold really rounded somewhere: exact sum of bf16 partials differs
    S = oracle.rank_partials(A2, W2)
    Q = [oracle.bf16_round(S[r]) for r in range(8)]
    exact = [[sum(Fraction(float(q[i, j])) for q in Q) for j in range(N)] for i in range(M)]
    assert any(Fraction(float(rfp32(exact[i][j]))) != exact[i][j]
               for i in range(M) for j in range(N))


def test_partial_rounded_from_the_exact_value_not_the_float64_sum():
    """Products 1, 2^-8 and 2^-70: the exact sum 1 + 2^-8 + 2^-70 lies just
    above the bf16 midpoint 1 + 2^-8 and rounds up to 1 + 2^-7; the float64
    sum drops 2^-70, lands on the midpoint and would round to even (1)."""
    X = np.array([[1.0, 2.0 ** -4, 2.0 ** -35]])
    Y = np.array([[1.0], [2.0 ** -4], [2.0 ** -35]])
    assert oracle.bf16_round(X @ Y)[0, 0] == 1.0
    assert oracle.bf16_of_exact_product(X, Y)[0, 0] == 1.0 + 2.0 ** -7
    assert float(rbf16(Fraction(1) + Fraction(1, 2 ** 8) + Fraction(1, 2 ** 70))) == 1.0 + 2.0 ** -7
    # the same through the whole layer: one rank holds these products
    A = np.zeros((8, 8, 8)); W = np.zeros((8, 8, 8))
    A[5, 0, :3] = X[0]; W[5, :3, 0] = Y[:, 0]
    A_sh, W_sh = _bits_from_values(A), _bits_from_values(W)
    out, _ = oracle.gemm_rs(A_sh, W_sh)
    assert out[0, 0] == 1.0 + 2.0 ** -7
    assert np.array_equal(out, brute_force(A_sh, W_sh))
    C, _ = oracle.ag_gemm(_bits_from_values(np.tile(X, (8, 1)).reshape(8, 1, 3)),
                          _bits_from_values(np.tile(Y, (8, 1, 8))))
    assert np.all(C[:, :, 0] == 1.0 + 2.0 ** -7)


def test_bf16_round_fraction_matches_independent_rounding():
    g = np.random.Generator(np.random.PCG64(61))
    for _ in range(3000):
        num = int(g.integers(-2 ** 40, 2 ** 40))
        den = 2 ** int(g.integers(0, 200)) * int(g.integers(1, 2 ** 12))
        x = Fraction(num, den)
        assert oracle.bf16_round_fraction(x) == float(rbf16(x)), x
    for x in (Fraction(0), Fraction(2) ** 128, -Fraction(2) ** 130, Fraction(1, 2 ** 140),
              Fraction(3, 2 ** 134), Fraction(2) ** 127 * Fraction(511, 256)):
        r = rbf16(x)
        want = float(r) if abs(r) < Fraction(2) ** 128 else float("inf") * (1 if x > 0 else -1)
        assert oracle.bf16_round_fraction(x) == want, x


# ---------------------------------------------------------------------------
# closed forms and invariants
# ---------------------------------------------------------------------------


def _int_case(seed, M=16, N=24, K=128):
    g = np.random.Generator(np.random.PCG64(seed))
    A = g.integers(-1, 2, size=(M, K))
    W = g.integers(-1, 2, size=(K, N))
    return A, W


def test_exact_integer_case():
    A, W = _int_case(21)
    A_sh, W_sh = workloads.shard(_bits_from_values(A), _bits_from_values(W))
    out, ref = oracle.gemm_rs(A_sh, W_sh)
    exact = A.astype(np.int64) @ W.astype(np.int64)
    assert np.array_equal(out, exact.astype(np.float64))
    assert np.array_equal(ref, exact.astype(np.float64))


def test_linearity_in_exact_range():
    A, W1 = _int_case(22)
    _, W2 = _int_case(23)
    f = lambda a, w: oracle.gemm_rs(*workloads.shard(_bits_from_values(a), _bits_from_values(w)))[0]
    assert np.array_equal(f(A, W1 + W2), f(A, W1) + f(A, W2))
    assert np.array_equal(f(2 * A, W1), 2 * f(A, W1))


def test_rank_permutation_invariant_in_exact_range():
    A, W = _int_case(24)
    A_sh, W_sh = workloads.shard(_bits_from_values(A), _bits_from_values(W))
    perm = [3, 1, 7, 0, 5, 2, 6, 4]
    a, _ = oracle.gemm_rs(A_sh, W_sh)
    b, _ = oracle.gemm_rs(A_sh[perm], W_sh[perm])
    assert np.array_equal(a, b)


def test_identity_weights_return_A():
    M, K = 24, 64
    A, _ = workloads.draw_full(M, K, K, seed=31)
    W = _bits_from_values(np.eye(K))
    A_sh, W_sh = workloads.shard(A, W)
    out, _ = oracle.gemm_rs(A_sh, W_sh)
    assert np.array_equal(oracle.bf16_to_bits(out), A)


def test_single_nonzero_rank():
    M, N, K = 16, 32, 256
    A_sh, W_sh = workloads.make_shape_inputs(M, N, K, seed=41)
    q = 5
    A_sh = A_sh.copy()
    for r in range(8):
        if r != q:
            A_sh[r] = 0
    out, _ = oracle.gemm_rs(A_sh, W_sh)
    Aq = oracle.bf16_from_bits(A_sh[q])
    Wq = oracle.bf16_from_bits(W_sh[q])
    exact = np.array([[sum(Fraction(float(Aq[i, k])) * Fraction(float(Wq[k, j]))
                           for k in range(K // 8)) for j in range(N)] for i in range(M)])
    expected = np.array([[float(rbf16(v)) for v in row] for row in exact])
    assert np.array_equal(out, expected)


def test_slices_are_row_blocks():
    out = np.arange(16 * 3, dtype=np.float64).reshape(16, 3)
    sl = oracle.slices(out)
    assert len(sl) == 8
    for s in range(8):
        assert np.array_equal(sl[s], out[2 * s:2 * s + 2])
    assert np.array_equal(np.concatenate(sl), out)


def test_rows_subset_equals_full():
    A, W = workloads.make_shape_inputs(40, 24, 128, seed=51)
    out, ref = oracle.gemm_rs(A, W)
    rows = [0, 7, 8, 39, 20]
    o2, r2 = oracle.gemm_rs_rows(A, W, rows)
    assert np.array_equal(o2, out[rows])
    assert np.array_equal(r2, ref[rows])


def test_concatenated_slices_equal_full_gemm_within_bound():
    """out vs A @ W over the full K (one float64 matmul, not per shard)."""
    M, N, K = 64, 96, 512
    A_sh, W_sh = workloads.make_shape_inputs(M, N, K, seed=61)
    out, ref = oracle.gemm_rs(A_sh, W_sh)
    A = np.concatenate([oracle.bf16_from_bits(A_sh[r]) for r in range(8)], axis=1)
    W = np.concatenate([oracle.bf16_from_bits(W_sh[r]) for r in range(8)], axis=0)
    AW = A @ W
    absAW = np.abs(A) @ np.abs(W)
    ub, g7 = 2.0 ** -8, 7 * 2.0 ** -24
    bound = ub * np.abs(out) / (1 - ub) + (g7 * (1 + ub) + ub) * absAW + 1e-12 * absAW
    assert np.all(np.abs(out - AW) <= bound)
    assert np.max(np.abs(ref - AW)) <= 1e-12 * np.max(absAW)
    # a dropped rank, a sign error or a transposed shard must break the bound
    S = oracle.rank_partials(A_sh, W_sh)
    bad = S.copy(); bad[3] = 0
    assert not np.all(np.abs(oracle.reduce_partials(bad)[0] - AW) <= bound)
    bad = S.copy(); bad[6] = -bad[6]
    assert not np.all(np.abs(oracle.reduce_partials(bad)[0] - AW) <= bound)
    W_swapped = W_sh[[1, 0, 2, 3, 4, 5, 6, 7]]
    assert not np.all(np.abs(oracle.gemm_rs(A_sh, W_swapped)[0] - AW) <= bound)


def test_output_statistics_of_recipe():
    A_sh, W_sh = workloads.make_shape_inputs(256, 256, 1024, seed=71)
    out, _ = oracle.gemm_rs(A_sh, W_sh)
    assert abs(out.std() - 1.0) < 0.05
    assert abs(out.mean()) < 0.02


def test_error_metrics():
    out = np.array([[1.0, -2.0], [0.5, 4.0]])
    X = out.copy(); X[1, 1] = 4.03125
    assert oracle.err_vs_oracle(X, out) == pytest.approx(0.03125 / 4.0)
    ref = out + 0.01
    assert oracle.rel_vs_ref(out, ref) == pytest.approx(0.01 / 4.01)
    assert oracle.err_vs_oracle(np.zeros((0, 3)), np.zeros((0, 3))) == 0.0


@pytest.mark.parametrize("M,N,K,seed", [(16, 8, 16, 41), (24, 16, 64, 42)])
def test_allreduce_every_rank_holds_the_brute_force_sum(M, N, K, seed):
    """All-reduce (mKernel page, sections 3.1, 4, 5.2): each of the 8 copies is
    the exact rank-order sum of the rounded partials, all M rows of it."""
    A_sh, W_sh = workloads.make_shape_inputs(M, N, K, seed)
    out8, ref = oracle.gemm_allreduce(A_sh, W_sh)
    exact = brute_force(A_sh, W_sh)
    assert out8.shape == (8, M, N)
    for r in range(8):
        assert np.array_equal(out8[r], exact), r
    # rank s's slice of the reduce-scatter is rows [s*M/8, (s+1)*M/8) of every copy
    rs, _ = oracle.gemm_rs(A_sh, W_sh)
    for s_, sl in enumerate(oracle.slices(rs)):
        h = M // 8
        assert np.array_equal(out8[(s_ + 3) % 8][s_ * h:(s_ + 1) * h], sl)


# ---------------------------------------------------------------------------
# All-gather + GEMM (the column-parallel partner layer)

def _ag_brute_force(A_sh, W_sh):
    """Exact products of the gathered A with each column shard, rounded once."""
    A = [[Fraction(float(v)) for v in row] for a in A_sh for row in oracle.bf16_from_bits(a)]
    out = []
    for w in W_sh:
        Wv = [[Fraction(float(v)) for v in row] for row in oracle.bf16_from_bits(w)]
        K, n = len(Wv), len(Wv[0])
        out.append([[float(rbf16(sum((A[i][k] * Wv[k][j] for k in range(K)), Fraction(0))))
                     for j in range(n)] for i in range(len(A))])
    return np.array(out)


@pytest.mark.parametrize("M,N,K,seed", [(16, 16, 8, 51), (8, 64, 24, 52), (24, 8, 40, 53)])
def test_ag_gemm_matches_brute_force(M, N, K, seed):
    A_sh, W_sh = workloads.make_shape_inputs(M, N, K, seed, op="ag")
    C, ref = oracle.ag_gemm(A_sh, W_sh)
    assert C.shape == (8, M, N // 8)
    assert np.array_equal(C, _ag_brute_force(A_sh, W_sh))


def test_ag_gemm_column_blocks_form_one_product():
    """The ranks' column blocks side by side are the single rounding of the
    unsharded product A W (numpy's float64 matmul of the full matrices)."""
    M, N, K = 48, 128, 256
    A, W = workloads.draw_full(M, N, K, seed=54)
    A_sh, W_sh = workloads.shard_ag(A, W)
    C, _ = oracle.ag_gemm(A_sh, W_sh)
    full = oracle.bf16_round(oracle.bf16_from_bits(A) @ oracle.bf16_from_bits(W))
    assert np.array_equal(np.concatenate(list(C), axis=1), full)


def test_ag_gemm_identity_and_single_shard():
    M, K = 64, 64
    A, _ = workloads.draw_full(M, K, K, seed=55)
    A_sh, W_sh = workloads.shard_ag(A, oracle.bf16_to_bits(np.eye(K)))
    C, _ = oracle.ag_gemm(A_sh, W_sh)
    Av = oracle.bf16_from_bits(A)
    for r in range(8):
        assert np.array_equal(C[r], Av[:, r * K // 8:(r + 1) * K // 8])
    # only shard 3 non-zero: every rank's rows outside shard 3 are zero
    A2 = A_sh.copy()
    A2[[q for q in range(8) if q != 3]] = 0
    C2, _ = oracle.ag_gemm(A2, W_sh)
    h = M // 8
    assert np.count_nonzero(C2[:, :3 * h]) == 0 and np.count_nonzero(C2[:, 4 * h:]) == 0
    assert np.array_equal(C2[:, 3 * h:4 * h], C[:, 3 * h:4 * h])


def test_ag_gemm_rows_subset():
    A_sh, W_sh = workloads.make_shape_inputs(64, 128, 128, 56, op="ag")
    C, _ = oracle.ag_gemm(A_sh, W_sh)
    rows = [0, 7, 8, 33, 63]
    Cr, _ = oracle.ag_gemm_rows(A_sh, W_sh, rows)
    assert np.array_equal(Cr, C[:, rows])


# ---------------------------------------------------------------------------
# Property-based: arbitrary finite bf16 inputs over a wide exponent range
# (where the bf16 partial rounding and the fp32 fold both round), against the
# exact rational brute force.


def test_pipeline_matches_brute_force_on_arbitrary_bf16():
    hyp = pytest.importorskip("hypothesis")
    st = pytest.importorskip("hypothesis.strategies")

    def bf16_value(sign, exp, mant):
        return (-1) ** sign * (1 + mant / 128) * 2.0 ** exp

    value = st.builds(bf16_value, st.integers(0, 1), st.integers(-40, 40), st.integers(0, 127))
    entry = st.one_of(value, st.just(0.0))

    @hyp.settings(max_examples=40, deadline=None, derandomize=True,
                  phases=[hyp.Phase.explicit, hyp.Phase.generate])
    @hyp.given(st.integers(1, 3), st.integers(1, 3),
               st.lists(entry, min_size=8 * 8 * 3, max_size=8 * 8 * 3),
               st.lists(entry, min_size=8 * 3 * 3, max_size=8 * 3 * 3))
    def check(Kr, N, a_vals, w_vals):
        A = np.array(a_vals[:8 * 8 * Kr]).reshape(8, 8, Kr)
        W = np.array(w_vals[:8 * Kr * N]).reshape(8, Kr, N)
        A_sh, W_sh = _bits_from_values(A), _bits_from_values(W)
        out, _ = oracle.gemm_rs(A_sh, W_sh)
        assert np.array_equal(out, brute_force(A_sh, W_sh))

    check()


def test_fold_order_matters_on_powers_of_two():
    """Signed powers of two with K/8 = 1: every partial is one of ±1, ±2^13,
    ±2^26 and exact in bf16, so the fp32 fold alone decides the result.
    Next to 2^26 a 1 is absorbed (fp32 keeps 24 bits) and shows once the
    large terms cancel, so the rank order and the fp32 width both matter: a
    float64 fold or another order gives other results."""
    hyp = pytest.importorskip("hypothesis")
    st = pytest.importorskip("hypothesis.strategies")
    term = st.builds(lambda s, e: (-1) ** s * 2.0 ** e, st.integers(0, 1),
                     st.sampled_from([13, 0]))

    @hyp.settings(max_examples=100, deadline=None, derandomize=True,
                  phases=[hyp.Phase.explicit, hyp.Phase.generate])
    @hyp.given(st.lists(term, min_size=8 * 8, max_size=8 * 8),
               st.lists(term, min_size=8 * 4, max_size=8 * 4))
    def check(a_vals, w_vals):
        A = np.array(a_vals).reshape(8, 8, 1)
        W = np.array(w_vals).reshape(8, 1, 4)
        A_sh, W_sh = _bits_from_values(A), _bits_from_values(W)
        out, _ = oracle.gemm_rs(A_sh, W_sh)
        assert np.array_equal(out, brute_force(A_sh, W_sh))

    check()


def test_ag_gemm_matches_brute_force_on_arbitrary_bf16():
    """All-gather GEMM on arbitrary finite bf16 inputs over exponents -40..40:
    one rounding of the exact product, whatever the products' magnitudes."""
    hyp = pytest.importorskip("hypothesis")
    st = pytest.importorskip("hypothesis.strategies")
    value = st.builds(lambda s, e, m: (-1) ** s * (1 + m / 128) * 2.0 ** e,
                      st.integers(0, 1), st.integers(-40, 40), st.integers(0, 127))

    @hyp.settings(max_examples=40, deadline=None, derandomize=True,
                  phases=[hyp.Phase.explicit, hyp.Phase.generate])
    @hyp.given(st.integers(1, 4), st.lists(value, min_size=8 * 4, max_size=8 * 4),
               st.lists(value, min_size=8 * 4 * 2, max_size=8 * 4 * 2))
    def check(K, a_vals, w_vals):
        A = np.array(a_vals[:8 * K]).reshape(8, 1, K)      # one row per shard
        W = np.array(w_vals[:8 * K * 2]).reshape(8, K, 2)  # two columns per rank
        A_sh, W_sh = _bits_from_values(A), _bits_from_values(W)
        C, _ = oracle.ag_gemm(A_sh, W_sh)
        assert np.array_equal(C, _ag_brute_force(A_sh, W_sh))

    check()
