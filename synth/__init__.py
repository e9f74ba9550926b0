"""Seeded synthetic inputs for the quantized MoE expert layer.

This package is the one module shared by the CUDA path's tests/bench and by the
fp64 oracle.  It draws random numbers and encodes them into the canonical byte
formats (GGUF Q4_0 and OCP MXFP4 blocks).  It holds none of the layer's own
arithmetic: no block decode, no routing, no permutation, no FFN and no combine.
"""
from .gen import (  # noqa: F401
    CONFIGS,
    LayerInputs,
    QTYPE_BLOCK_BYTES,
    bf16_bits_to_f32,
    f32_to_bf16_bits,
    gen_gate_weights,
    gen_logits,
    gen_x_bf16,
    gen_expert_weights,
    make_layer,
    quantize_mxfp4,
    quantize_mxfp8,
    quantize_nvfp4,
    quantize_q4_0,
    stream_trace,
    zipf_bias,
)
