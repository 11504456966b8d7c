"""Seeded synthetic inputs for the top-2 sparse MoE feed-forward layer.

This package draws random tensors with the shapes and value distributions of the
Mixtral layer (d=4096, ffn=14336, 8 experts), of a tiny fp32 layer and of
the decoder block around the layer (norm gains, attention projections). It holds
none of the arithmetic: no router, no top-k, no expert, no norm or attention. Both the CUDA
path's tests/benchmark and the CPU oracle's tests take their inputs from here.
"""
from .gen import (  # noqa: F401
    CONFIGS,
    BLOCK_CONFIGS,
    make_block,
    make_block_config,
    Layer,
    make_config,
    make_layer,
    make_weights,
    make_tokens,
    make_token_stream,
    redraw_token_row,
    load_schedule,
    to_f64,
    normal_f32,
    skew_direction,
)
