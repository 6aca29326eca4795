"""CPU oracle (test infrastructure only; see gemm_rs_oracle)."""
from .gemm_rs_oracle import (WORLD, bf16_round, bf16_round_fraction, bf16_from_bits, bf16_to_bits,
                             bf16_of_exact_product, rank_partials, partials_bf16, reduce_partials,
                             gemm_rs, gemm_rs_rows, gemm_allreduce, ag_gemm, ag_gemm_rows,
                             slices, err_vs_oracle, rel_vs_ref)
