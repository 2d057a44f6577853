"""Seeded synthetic inputs for the routed-MoE expert computation.

This package only draws random bytes and ids in the checkpoint layouts the
pages describe; it holds none of the method's arithmetic (no decoding, no
quantisation, no GEMM).  Both the fp64 oracle and the CUDA path consume what
it produces, so that their results can be compared element by element.
"""
from .moe_inputs import (  # noqa: F401
    MoEConfig, CONFIGS, Checkpoint, make_checkpoint, make_routing, make_x, make_inputs,
    ep_mask_foreign, zipf_topk, uniform_topk, f32_to_bf16_bits,
    W13_UP_GATE, W13_GATE_UP, TIER_NVFP4, TIER_NF3,
)
