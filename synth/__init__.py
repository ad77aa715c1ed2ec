"""Seeded synthetic inputs for the quantized-KV decode path.

This package holds input generation only: random draws, bf16 rounding of the
draws, sequence lengths, block placement. It contains none of the method's
arithmetic (no quantizer, no attention), so that both the float64 oracle and
the CUDA path can consume the same bits without sharing any computation.
"""
from .workloads import (WORKLOADS, Workload, Inputs, make_inputs, f32_to_bf16_bits, bf16_bits_to_f32,
                        query_rows)

__all__ = ["WORKLOADS", "Workload", "Inputs", "make_inputs", "f32_to_bf16_bits", "bf16_bits_to_f32",
           "query_rows"]
