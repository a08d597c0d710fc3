"""CPU oracle of the MoE layer forward (test infrastructure; never used by the product path)."""
from .moe_oracle import *  # noqa: F401,F403
from .moe_oracle import capacity, route, router_logits, dispatch, dispatch_payload, expert_outputs, \
    swiglu_ffn, combine, moe_layer, moe_layer_tokens, near_tie_rows, ffn_flops, dispatch_bytes, \
    expert_choice, expert_choice_layer, sinkhorn_scaling, route_sinkhorn, route_selbias  # noqa: F401
