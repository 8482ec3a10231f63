"""fp64 CPU oracle (test infrastructure; never imported by the product path)."""
from .flce_fp64 import (BadTarget, decode_bf16, flce_oracle, flce_oracle_f64, oracle_rows,
                          lse_all_rows, grad_weight_rows, rmsnorm_flce_oracle, rmsnorm_flce_oracle_f64)

__all__ = ["BadTarget", "decode_bf16", "flce_oracle", "flce_oracle_f64", "oracle_rows",
           "lse_all_rows", "grad_weight_rows", "rmsnorm_flce_oracle", "rmsnorm_flce_oracle_f64"]
