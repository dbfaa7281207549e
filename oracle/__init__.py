"""CPU oracle of the fused MoE layer: test infrastructure, not product code.

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.
"""
from .moe_oracle import (  # noqa: F401
    align, align_capacity, experts_dense_bruteforce, experts_loop, moe_layer,
    near_tie_tokens, route, router_logits, routing_weights, select_topk,
    silu_and_mul, softmax_over_experts, widen_bf16,
)
