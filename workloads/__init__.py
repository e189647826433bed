"""Seeded synthetic workloads (inputs only; no attention arithmetic)."""
from .synth import (BF16, F32, CONFIG_NAMES, Problem, Structure, bf16_bits_to_f32,
                    chunk_queries, f32_to_bf16_bits, flatten_problem, make, make_chunked,
                    materialize, struct_grouped, struct_skewed, struct_two_level)

__all__ = ["BF16", "F32", "CONFIG_NAMES", "Problem", "Structure", "bf16_bits_to_f32",
           "chunk_queries", "f32_to_bf16_bits", "flatten_problem", "make", "make_chunked",
           "materialize", "struct_grouped",
           "struct_skewed", "struct_two_level"]
