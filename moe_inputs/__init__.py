"""Seeded synthetic inputs for the top-2 sparse MoE feed-forward layer.

This package draws random tensors with the shapes and value distributions of the
Mixtral layer (d=4096, ffn=14336, 8 experts) and of a tiny fp32 layer. It holds
none of the layer's arithmetic: no router, no top-k, no expert. Both the CUDA
path's tests/benchmark and the CPU oracle's tests take their inputs from here.
"""
from .gen import (  # noqa: F401
    CONFIGS,
    Layer,
    make_config,
    make_layer,
    make_weights,
    make_tokens,
    redraw_token_row,
    load_schedule,
    to_f64,
    normal_f32,
    skew_direction,
)
