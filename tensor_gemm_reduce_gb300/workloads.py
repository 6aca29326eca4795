"""Workload registry and seeded synthetic inputs for the row-parallel linear layer.

This module is shared by the CUDA path (tests, bench) and the CPU oracle.  It
holds no arithmetic of the method itself: it only draws random numbers, rounds
them once to bf16 (through torch's float32 -> bfloat16 conversion, which rounds
to nearest even) and lays them out as per-rank shards.

Shapes follow the problem page "A fused GEMM + reduce-scatter kernel hiding 90%
of communication on 8 H100 GPUs" (section "How it gets verified": token counts
M of 512, 2048, 8192 and 32768, output and inner dimensions of Llama-3-70B and
Mixtral-8x22B projection layers, 8-way tensor parallelism).  Row-parallel sharding follows the FLUX page,
Figure 2 (N-way partition of the MLP forward, batch and sequence flattened
into the GEMM's M): rank r holds columns [r*K/8, (r+1)*K/8) of A and the
matching rows of W.

Recipe (identical bits on every machine):
  * A[M][K] ~ N(0, 1) drawn as float32 with numpy PCG64(seed);
  * W[K][N] ~ N(0, 1/K) drawn as float32 with PCG64(seed + 1), scaled by K**-0.5;
  * down_proj workloads: each entry of A independently (PCG64(seed + 2),
    probability 0.05) is multiplied by 8 (exact in bf16);
  * both rounded once to bf16 (round to nearest even);
  * A_shards = A reshaped to [8][M][K/8] (rank-major, K/8 contiguous),
    W_shards = W reshaped to [8][K/8][N] (rank-major, N contiguous).

All-gather + GEMM workloads (op "ag": the column-parallel partner layer,
FLUX page abstract and Figure 1, mKernel page section 4) draw A and W the
same way and shard them the other way round: rank r holds rows
[r*M/8, (r+1)*M/8) of A ([8][M/8][K]) and columns [r*N/8, (r+1)*N/8) of W
([8][K][N/8]).  Shapes: the Llama-3 70B attention QKV projection (N = 8192 +
2 * 1024) and the FLUX page's Figure 4 shapes, (n, k) = (49152, 12288) for
the all-gather and (12288, 49152) for the reduce-scatter, m from 1024 to 8192.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional

import numpy as np

WORLD = 8  # tensor-parallel degree of the emulated group


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    seed: int
    outliers: bool = False
    op: str = "rs"  # "rs": row-parallel (GEMM + reduce-scatter); "ag": all-gather + GEMM

    @property
    def Kr(self) -> int:
        return self.K // WORLD

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    def describe(self) -> str:
        o = ", 5% x8 outliers in A" if self.outliers else ""
        return f"{self.name}: M={self.M} N={self.N} K={self.K} (K/8={self.Kr}){o}"


def _registry() -> List[Workload]:
    w: List[Workload] = []
    # tiny row-parallel linear
    w.append(Workload("tiny", 128, 512, 1024, seed=0))
    # Llama-3-70B attention o_proj
    w.append(Workload("llama3_70b_o_proj_m2048", 2048, 8192, 8192, seed=1000))
    # Llama-3-70B MLP down_proj with activation outliers
    for i, m in enumerate((512, 8192)):
        w.append(Workload(f"llama3_70b_down_proj_m{m}", m, 8192, 28672,
                          seed=2000 + i, outliers=True))
    # Mixtral-8x22B expert down_proj
    for i, m in enumerate((2048, 32768)):
        w.append(Workload(f"mixtral_8x22b_down_proj_m{m}", m, 6144, 16384,
                          seed=3000 + i))
    # the FLUX page's Figure 4 reduce-scatter shape
    for i, m in enumerate((1024, 2048, 4096, 8192)):
        w.append(Workload(f"flux_fig4_rs_m{m}", m, 12288, 49152, seed=5200 + i))
    # all-gather + GEMM: tiny, Llama-3-70B QKV projection, FLUX Figure 4's shape
    w.append(Workload("tiny_ag", 128, 512, 1024, seed=100, op="ag"))
    w.append(Workload("llama3_70b_qkv_m2048", 2048, 10240, 8192, seed=5000, op="ag"))
    for i, m in enumerate((1024, 2048, 4096, 8192)):
        w.append(Workload(f"flux_fig4_ag_m{m}", m, 49152, 12288, seed=5100 + i, op="ag"))
    # the full sweep
    for j, (n, k) in enumerate(((8192, 8192), (8192, 28672), (6144, 6144), (6144, 16384))):
        for i, m in enumerate((512, 2048, 8192, 32768)):
            w.append(Workload(f"sweep_m{m}_n{n}_k{k}", m, n, k, seed=4000 + 10 * j + i))
    return w


WORKLOADS = {w.name: w for w in _registry()}
TINY = WORKLOADS["tiny"]
O_PROJ = WORKLOADS["llama3_70b_o_proj_m2048"]


def _to_bf16_bits(x32: np.ndarray) -> np.ndarray:
    """float32 array -> uint16 bf16 bit patterns, round to nearest even (torch)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def draw_full(M: int, N: int, K: int, seed: int, outliers: bool = False,
              w_scale: Optional[float] = None):
    """Return (A_bits[M][K], W_bits[K][N]) as uint16 bf16 patterns."""
    ga = np.random.Generator(np.random.PCG64(seed))
    a32 = ga.standard_normal((M, K), dtype=np.float32)
    if outliers:
        gm = np.random.Generator(np.random.PCG64(seed + 2))
        mask = gm.random((M, K), dtype=np.float32) < np.float32(0.05)
        a32[mask] *= np.float32(8.0)
    gw = np.random.Generator(np.random.PCG64(seed + 1))
    w32 = gw.standard_normal((K, N), dtype=np.float32)
    scale = np.float32(K ** -0.5 if w_scale is None else w_scale)
    w32 *= scale
    return _to_bf16_bits(a32), _to_bf16_bits(w32)


def shard(A_bits: np.ndarray, W_bits: np.ndarray, world: int = WORLD):
    """Split A[M][K] by columns and W[K][N] by rows into rank-major shards."""
    M, K = A_bits.shape
    K2, N = W_bits.shape
    assert K == K2 and K % world == 0
    Kr = K // world
    A_sh = np.ascontiguousarray(A_bits.reshape(M, world, Kr).transpose(1, 0, 2))
    W_sh = np.ascontiguousarray(W_bits.reshape(world, Kr, N))
    return A_sh, W_sh


def shard_ag(A_bits: np.ndarray, W_bits: np.ndarray, world: int = WORLD):
    """Split A[M][K] by rows and W[K][N] by columns: ([8][M/8][K], [8][K][N/8])."""
    M, K = A_bits.shape
    K2, N = W_bits.shape
    assert K == K2 and M % world == 0 and N % world == 0
    A_sh = np.ascontiguousarray(A_bits.reshape(world, M // world, K))
    W_sh = np.ascontiguousarray(W_bits.reshape(K, world, N // world).transpose(1, 0, 2))
    return A_sh, W_sh


def make_inputs(w: Workload):
    """Seeded shards for a registered workload (uint16 bf16 patterns): for "rs"
    (A_sh[8][M][K/8], W_sh[8][K/8][N]), for "ag" (A_sh[8][M/8][K], W_sh[8][K][N/8])."""
    A, W = draw_full(w.M, w.N, w.K, w.seed, w.outliers)
    return shard_ag(A, W) if w.op == "ag" else shard(A, W)


def make_shape_inputs(M: int, N: int, K: int, seed: int, outliers: bool = False, op: str = "rs"):
    """Seeded shards for an arbitrary shape (test cases)."""
    A, W = draw_full(M, N, K, seed, outliers)
    return shard_ag(A, W) if op == "ag" else shard(A, W)
