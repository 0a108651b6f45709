"""Seeded synthetic inputs for the NVFP4 MoE layer (shared by tests and bench).

This package draws random numbers and nothing else: no quantization, routing or
GEMM arithmetic lives here, so both the CUDA path and the CPU oracle can consume
the same buffers without sharing any of the method's code.
"""
from .workloads import CONFIGS, LayerConfig, make_inputs, expert_weights, gate_weights, zipf_bias  # noqa: F401
