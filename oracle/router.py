"""CPU oracle of the router GEMM ahead of top-k (test infrastructure).

This file is test infrastructure only, under the same rules as moe_oracle:
tests, the smoke check and the benchmark's CPU-baseline leg may call it; the
product path never does.  Plain numpy in fp64; no code shared with the CUDA
path.

The routing step of the layer starts from router logits; the step before it
is the router (gate) projection of the token's hidden state, logits =
x . Wg^T.  The MI250 correctness blog puts this projection among the paths
that may take low-precision inputs with FP32 accumulation (section 4.1: the
gate network's layers in the "low precision allowed" class) and requires the
top-k comparison itself in FP32 (section 4.1 table, "MoE routing top-k: FP32
comparison + fixed tie-break").  Readings used here, where the pages say
nothing:

* Wg is bf16 [E, d], row e the gate vector of expert e; x is the layer's bf16
  input [T, d].
* logits[t, e] = sum_K x[t, K] * Wg[e, K]: the products of two bf16 values are
  exact, the sum is the exact real sum (fp64 here; the accumulation precision
  required of an implementation is fp32).
* The top-k decision is taken in fp32: on the exact logits rounded to the
  nearest fp32 value, with the routing rules of moe_oracle.route.
"""
from __future__ import annotations

import numpy as np

from .moe_oracle import bf16_bits_to_f64, forward


def router_logits(x_bf16: np.ndarray, w_gate_bf16: np.ndarray) -> np.ndarray:
    """logits fp64 [T, E] = x [T, d] . Wg [E, d]^T, both given as bf16 bit patterns."""
    x = bf16_bits_to_f64(x_bf16)
    wg = bf16_bits_to_f64(w_gate_bf16)
    if x.shape[1] != wg.shape[1]:
        raise ValueError("x and Wg must share the hidden size d")
    return x @ wg.T


def router_logits_f32(x_bf16: np.ndarray, w_gate_bf16: np.ndarray) -> np.ndarray:
    """The exact logits rounded to the nearest fp32 value (the values the top-k compares)."""
    return router_logits(x_bf16, w_gate_bf16).astype(np.float32)


def forward_gated(x_bf16: np.ndarray, w_gate_bf16: np.ndarray, w13: np.ndarray, w13_scale: np.ndarray,
                  w2: np.ndarray, w2_scale: np.ndarray, k: int):
    """The layer starting from x and the router weights: the router projection,
    then moe_oracle.forward on its fp32 logits.  Returns forward's dict plus
    "logits" (fp64, exact)."""
    logits = router_logits(x_bf16, w_gate_bf16)
    r = forward(x_bf16, logits.astype(np.float32), w13, w13_scale, w2, w2_scale, k)
    r["logits"] = logits
    return r
