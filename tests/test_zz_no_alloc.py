"""The no-allocation entry point, gemm_rs_fused_noalloc.

It serves callers that may not allocate device memory when they call the
library (a plug-in inside an application that owns the device-memory budget,
a serving path that forbids cudaMalloc after start-up): they pass only their
inputs and output, and the fused kernel's staging, flags and control words
live in a fixed static device array of the library.  The pages have no
counterpart for this; it is checked here against the planned entry point
(gemm_rs_run in FUSED mode with a caller workspace).

This file is named to be collected last, so a run that stops at the first
failure has run every other test before it.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from tensor_gemm_reduce_gb300 import gemm_rs as G
from tensor_gemm_reduce_gb300 import workloads


def test_noalloc_rejects_oversize_before_any_cuda_call():
    """Size checks come first, so they also answer on a machine without a GPU."""
    lib = G.load_library()
    # 8 * 2048 * 8192 * 2 bytes of staging = 256 MiB > 32 MiB
    assert lib.gemm_rs_fused_noalloc(None, None, None, 2048, 8192, 8192, None, None) == G.GEMM_RS_ERR_TOO_LARGE
    # the staging limit is exact: 8 * 8 * 262144 * 2 bytes = 32 MiB fits (then the null
    # pointers are rejected), 8 more columns do not
    assert lib.gemm_rs_fused_noalloc(None, None, None, 8, 262152, 64, None, None) == G.GEMM_RS_ERR_TOO_LARGE
    assert lib.gemm_rs_fused_noalloc(None, None, None, 8, 262144, 64, None, None) == G.GEMM_RS_ERR_INVALID_ARG
    assert lib.gemm_rs_fused_noalloc(None, None, None, 100, 256, 64, None, None) == G.GEMM_RS_ERR_UNSUPPORTED_SHAPE
    assert lib.gemm_rs_fused_noalloc(None, None, None, 128, 256, 512, None, None) == G.GEMM_RS_ERR_INVALID_ARG


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


@pytest.mark.gpu
def test_noalloc_matches_planned_entry_point_on_two_calls():
    shapes = [(256, 1024, 2048, 101), (392, 776, 1600, 102)]  # the second one is ragged in M, N, K
    cases = []
    for M, N, K, seed in shapes:
        A_bits, W_bits = workloads.make_shape_inputs(M, N, K, seed)
        A, W = _dev(A_bits), _dev(W_bits)
        # the existing entry point, with a workspace from the caller
        plan = G.Plan(M, N, K)
        ws = plan.new_workspace()
        ref = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        plan.run(A, W, ref, ws, G.FUSED)
        assert plan.status() == G.GEMM_RS_OK
        out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        err = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
        cases.append((M, N, K, A, W, ref, out, err))
    torch.cuda.synchronize()

    stream = torch.cuda.current_stream().cuda_stream
    for M, N, K, A, W, ref, out, err in cases:  # two calls in a row on one stream
        rc = G.gemm_rs_fused_noalloc(A.data_ptr(), W.data_ptr(), out.data_ptr(), M, N, K,
                                     err.data_ptr(), stream)
        assert rc == G.GEMM_RS_OK, G.strerror(rc)
    torch.cuda.synchronize()

    for M, N, K, A, W, ref, out, err in cases:
        assert err.item() == 0
        got = oracle.bf16_from_bits(out.view(torch.int16).cpu().numpy().view(np.uint16))
        exp = oracle.bf16_from_bits(ref.view(torch.int16).cpu().numpy().view(np.uint16))
        assert np.all(np.isfinite(got))
        assert oracle.err_vs_oracle(got, exp) <= 1e-2
        # same kernel, same arithmetic: in practice the two agree bit for bit
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
