"""Float64 CPU oracle for the fused MoE layer (test infrastructure only).

Imported by the test suite, the package smoke check and the benchmark's CPU-baseline
leg; never by the product path. See ``oracle.moe_oracle`` for the definitions.
"""
from .moe_oracle import *  # noqa: F401,F403
from .moe_oracle import (add_shared_experts, apply_expert_map, bf16_bits_to_f64,
                         dequant_blockwise, dequant_w13, dispatch_masked, e4m3_to_f64, masked_forward, brute_align, brute_topk, expert_ffn,  # noqa: F401
                         max_padded_rows, moe_align, moe_dense, moe_forward, moe_loop,
                         route, route_sigmoid_grouped, route_softmax,
                         route_topk_then_softmax, router_logits, selection_margins,
                         sigmoid, silu, softmax, topk_desc)
