"""Seeded synthetic workloads for the routed int4 MoE layer.

This package only draws inputs (activations, fp16 expert weights, fp32 router
weights, router bias) and names the five workload shapes. It contains none of
the layer's own arithmetic (no quantization, routing, GEMM or combine), so the
oracle and the CUDA path can both take their inputs from here without sharing
any step of the method.
"""
from .configs import CONFIGS, ZIPF_ALPHA, Workload, get  # noqa: F401
from . import gen  # noqa: F401
