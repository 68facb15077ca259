"""Seeded synthetic inputs for the MoL LoRA hot path.

This package only draws inputs (routing, activations, adapter weights, the
initial MoE output). It holds none of the method's arithmetic: no remap, no
bucketing, no contraction, no rounding of results. Both the CPU oracle and the
CUDA path receive the arrays it produces.
"""

from .workloads import (  # noqa: F401
    Stage,
    Workload,
    WORKLOADS,
    WindowedWeights,
    LayerInputs,
    make_routing,
    make_layer,
    bf16_bits_from_f32,
)
