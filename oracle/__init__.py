"""CPU oracle (test infrastructure only; see gemm_rs_oracle)."""
from .gemm_rs_oracle import (WORLD, bf16_round, bf16_from_bits, bf16_to_bits,
                             rank_partials, reduce_partials, gemm_rs, gemm_rs_rows, gemm_allreduce,
                             ag_gemm, ag_gemm_rows,
                             slices, err_vs_oracle, rel_vs_ref)
