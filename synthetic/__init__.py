"""Seeded synthetic decode-attention inputs shared by the tests, the bench and smoke().

This package only draws random numbers and lays them out (q, a token-major K/V
cache with per-sequence offsets, and the per-head sampling offsets U).  It holds
none of the attention or sampling arithmetic: that lives in the CUDA library and,
independently, in the CPU oracle.
"""

from .workloads import (  # noqa: F401
    WORKLOADS,
    Inputs,
    Workload,
    bf16_bits_to_float32,
    float32_to_bf16_bits,
    generate,
    get_workload,
    max_length,
    to_torch,
)
