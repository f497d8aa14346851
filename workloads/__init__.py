"""Seeded synthetic inputs for the LRMoE backward-recalibration path.

This package only draws random numbers and arranges them into the tensors a
routed MoE layer hands to its backward pass (router logits, routed expert ids,
gate weights, output gradients, saved down-projection inputs, expert weights,
and for the FC1 side the expert inputs, saved FC1 outputs and FC1 weights).
It holds none of the recalibration arithmetic: no routing statistics, scores,
selection, compaction or gradients. Both the fp64 oracle (tests only) and the
CUDA path consume what it produces.
"""

from .generate import (  # noqa: F401
    WORKLOADS,
    Fc1Inputs,
    Workload,
    bf16_bits_to_f32,
    f32_to_bf16_bits,
    fc1_inputs,
    generate,
    get_workload,
)
