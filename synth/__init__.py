"""Seeded synthetic inputs for the weight-only NVFP4 MoE layer.

This package only *makes inputs*: router logits, BF16 activations and NVFP4
expert weights (FP32 weights drawn from a normal distribution and encoded to
E2M1 codes, E4M3 block scales and FP32 tensor scales).  It holds none of the
layer's arithmetic: no decoding of the formats, no routing, no matrix product.
Both the CPU oracle and the CUDA path consume what it returns.
"""
from .inputs import (  # noqa: F401
    CONFIGS,
    LayerConfig,
    LayerInputs,
    ExpertWeights,
    make_inputs,
    make_expert_weights,
    make_layer_weights,
    quantize_nvfp4,
    encode_e4m3_rne,
    encode_e2m1_rne,
    f32_to_bf16_bits,
    LINEAR_CONFIGS,
    LinearConfig,
    LinearInputs,
    make_linear_inputs,
    make_router_weight,
    make_input_scales,
)
