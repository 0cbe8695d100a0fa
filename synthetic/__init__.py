"""Seeded synthetic inputs shared by the oracle tests, the CUDA parity tests and the bench.

This package only draws random tensors and names workload shapes.  It holds none of the
method's arithmetic (no Hadamard, no quantisation, no outlier detection), so both the oracle
and the CUDA path may use it without sharing any of the computation under test.
"""
from .gen import normal_bf16, bf16_bits, bits_to_f32, outlier_lines
from .workloads import WORKLOADS, Linear, Workload, tensor_recipes

__all__ = [
    "normal_bf16", "bf16_bits", "bits_to_f32", "outlier_lines",
    "WORKLOADS", "Linear", "Workload", "tensor_recipes",
]
