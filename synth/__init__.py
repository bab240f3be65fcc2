"""Seeded synthetic inputs for the W4A16 MoE grouped GEMM.

This package is shared by the CPU oracle's tests and by the CUDA path's tests
and benchmark. It only draws random inputs (activations, packed INT4 weights,
BF16 scales, routing); it contains none of the grouped GEMM's own arithmetic
(no unpacking, dequantisation, matmul, activation or combine).
"""

from .moe_inputs import *  # noqa: F401,F403
