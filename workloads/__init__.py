"""Seeded synthetic decode workloads for the PrHS sparse-decode path.

This package only draws random inputs (KV caches, query sequences, paging
tables) and quantises them to the storage format; it holds none of the
method's arithmetic (no scores, softmax, selection, dilation or attention).
Both the CUDA path and the fp64 oracle consume the arrays it returns.
"""
from .generate import (Workload, make_workload, preset, PRESETS, bf16_bits_from_f32,
                       f32_from_bf16_bits)

__all__ = ["Workload", "make_workload", "preset", "PRESETS", "bf16_bits_from_f32",
           "f32_from_bf16_bits"]
