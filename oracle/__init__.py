"""CPU oracle for C = alpha * A @ B + beta * C (test infrastructure only).

Only the tests, the smoke check and the benchmark's CPU-baseline leg use this package.
The product library never imports, links or calls it.
"""
from .oracle import (  # noqa: F401
    build,
    f16_bits_to_f32,
    f32_to_f16_bits,
    f64_to_f16_bits,
    gemm,
    gemm_f16out,
    gemm_at,
    num_threads,
    round_f16,
    set_num_threads,
)
