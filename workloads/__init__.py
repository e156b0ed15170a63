"""Seeded synthetic inputs for packed variable-length attention.

This package only draws random numbers and lays out document structure
(``cu_seqlens``) and mask specifications (the LTS/LTE/UTS/UTE column
intervals).  It performs none of the method's arithmetic, so both the CUDA
path and the float64 oracle may take their inputs from here.
"""

from .gen import (  # noqa: F401
    CONFIG_NAMES,
    Workload,
    bf16_bits_to_f32,
    bf16_bits_to_f64,
    f32_to_bf16_bits,
    make_workload,
)
