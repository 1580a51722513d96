"""Seeded synthetic inputs for the fused MoE-LoRA expert layer.

This package only draws random numbers and lays them out in the shapes the
layer takes. It holds none of the layer's arithmetic (no routing, sorting,
matrix products or activations), so that both the fp64 CPU oracle and the CUDA
path can consume the very same inputs without sharing any computation.
"""
from .generators import (  # noqa: F401
    WORKLOADS,
    WORKLOAD_NAMES,
    EXTRA_WORKLOADS,
    ALL_WORKLOAD_NAMES,
    LayerInputs,
    workload_by_name,
    make_workload_inputs,
    make_workload_routing,
    make_layer_inputs,
)
