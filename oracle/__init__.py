"""CPU fp64 oracle of the top-2 sparse MoE feed-forward layer (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may use this package. The CUDA library never imports it, and it
shares no code with the CUDA path.
"""
from .moe_oracle import (  # noqa: F401
    router_logits,
    top_k_gates,
    permute,
    silu,
    expert_forward,
    expert_ffn_slots,
    combine,
    layer_forward,
    layer_forward_tokens,
    aux_stats,
    mixtral_param_counts,
)
from .moe_backward import (  # noqa: F401
    silu_grad,
    topk_softmax_backward,
    aux_score_grad,
    layer_backward,
)
from .decoder_block import (  # noqa: F401
    rms_norm,
    rope,
    causal_gqa_attention,
    attention_sublayer,
    decoder_block,
    attention_one_query,
    decoder_block_decode,
)
