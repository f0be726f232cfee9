"""CPU oracle of the FP4 routed-MoE layer: test infrastructure only.

Only the tests, the smoke check and the benchmark's CPU-baseline leg use
this package; the library's compute path never imports it.
"""
from .moe_oracle import (E2M1_MAGNITUDE, MX_BLOCK, bf16_bits_to_f64, bf16_round, dequantize_rows,
                         e2m1_decode, e8m0_decode, expert_ffn, expert_sort, fnv1a64, forward,
                         forward_tokens, route, route_hash, silu)

from .router import forward_gated, router_logits, router_logits_f32

__all__ = ["forward_gated", "router_logits", "router_logits_f32", "E2M1_MAGNITUDE", "MX_BLOCK", "bf16_bits_to_f64", "bf16_round", "dequantize_rows",
           "e2m1_decode", "e8m0_decode", "expert_ffn", "expert_sort", "fnv1a64", "forward",
           "forward_tokens", "route", "route_hash", "silu"]
