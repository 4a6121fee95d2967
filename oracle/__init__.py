"""CPU oracle of the blockwise-FP8 routed-MoE layer.

TEST INFRASTRUCTURE ONLY: imported by tests/, __graft_entry__.smoke() and
bench.py's CPU-baseline and reference legs.  The CUDA library and its Python
binding never import it.
"""
from .moe_oracle import (E4M3_TABLE, bf16_to_f64, combine, dequantize, e4m3_value,  # noqa: F401
                         expert_ffn, moe_forward, permutation, round_to_bf16, router_logits,
                         select_topk, silu, topk_weights)
