"""Seeded generators for the five MoE layer workloads and for small parity shapes.

Recipe (one numpy PCG64 stream per layer, seeded with ``seed``; the draws
happen in this order):

1. ``x``: fp32 standard normal [T, d], rounded to bf16 (round to nearest
   even on the fp32 bit pattern) and kept as its uint16 bit pattern.
2. ``router_logits``: fp32 standard normal [T, E].  For the skewed
   workload a per-expert bias ``2.0 * log(1 / rank)`` with ``rank = e + 1``
   (natural log) is added in fp32, which gives a Zipf-like load where high
   indices are rarely picked.
3. ``w13``: uint8 [E, 2I, d/2], the little-endian bytes of raw 64-bit
   PCG64 outputs (``bit_generator.random_raw``), each uniform on 0..255, so every 4-bit E2M1 code (both nibbles) is
   uniform over the 16 codes.
4. ``w13_scale``: uint8 [E, 2I, d/32], E8M0 bytes ``127 + u`` with the
   unbiased exponent ``u`` uniform on ``[exp_lo, exp_hi]``.
5. ``w2``: uint8 [E, d, I/2], raw generator bytes as for ``w13``.
6. ``w2_scale``: uint8 [E, d, I/32], E8M0 bytes as for ``w13_scale``.

Router weights (for the router projection ahead of top-k) come from a
stream of their own, ``make_gate_weights(E, d, seed)``: a PCG64 generator
seeded with ``[seed, 1]`` draws fp32 standard normal [E, d], divided by
sqrt(d) (so that logits of N(0, 1) tokens are about N(0, 1), like the
workloads' router logits) and rounded to bf16.

The five named workloads are the ones the FP4 routed-MoE layer is measured
on: a tiny layer, a decode-shaped layer (T=32), a prefill-shaped layer
(T=4608, the paper's 4,604-token prompt rounded up to 36 x 128), a skewed
routing layer and a large layer with d=7168.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

CONFIGS = {
    "tiny": dict(T=16, d=256, I=128, E=8, k=2, exp_lo=-7, exp_hi=-5, skew=False, seed=0),
    "decode": dict(T=32, d=4096, I=2048, E=256, k=8, exp_lo=-7, exp_hi=-5, skew=False, seed=0),
    "prefill": dict(T=4608, d=4096, I=2048, E=256, k=8, exp_lo=-7, exp_hi=-5, skew=False, seed=0),
    "skewed": dict(T=2048, d=4096, I=2048, E=256, k=8, exp_lo=-7, exp_hi=-5, skew=True, seed=0),
    "large": dict(T=16384, d=7168, I=2048, E=256, k=8, exp_lo=-8, exp_hi=-6, skew=False, seed=0),
}


@dataclasses.dataclass
class LayerInputs:
    """Host arrays of one MoE layer problem (all C-contiguous numpy)."""

    T: int
    d: int
    I: int
    E: int
    k: int
    x_bf16: np.ndarray        # uint16 [T, d], bf16 bit patterns
    router_logits: np.ndarray  # float32 [T, E]
    w13: np.ndarray           # uint8 [E, 2I, d/2]
    w13_scale: np.ndarray     # uint8 [E, 2I, d/32]
    w2: np.ndarray            # uint8 [E, d, I/2]
    w2_scale: np.ndarray      # uint8 [E, d, I/32]

    @property
    def dims(self):
        return dict(T=self.T, d=self.d, I=self.I, E=self.E, k=self.k)


def _f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even) and return bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return r.astype(np.uint16)


def _uniform_bytes(rng: np.random.Generator, shape) -> np.ndarray:
    n = int(np.prod(shape))
    words = rng.bit_generator.random_raw((n + 7) // 8).astype("<u8", copy=False)
    return words.view(np.uint8)[:n].reshape(shape)


def _scale_bytes(rng: np.random.Generator, shape, exp_lo: int, exp_hi: int) -> np.ndarray:
    return rng.integers(127 + exp_lo, 127 + exp_hi + 1, size=shape, dtype=np.uint8)


def make_layer(T: int, d: int, I: int, E: int, k: int, exp_lo: int = -7, exp_hi: int = -5,
               skew: bool = False, seed: int = 0) -> LayerInputs:
    """Draw one layer problem following the recipe in the module docstring."""
    if d % 32 or I % 32:
        raise ValueError("d and I must be multiples of 32 (E8M0 block size)")
    rng = np.random.default_rng(seed)
    x = _f32_to_bf16_bits(rng.standard_normal((T, d), dtype=np.float32))
    logits = rng.standard_normal((T, E), dtype=np.float32)
    if skew:
        bias = np.array([2.0 * math.log(1.0 / (e + 1)) for e in range(E)], dtype=np.float32)
        logits = (logits + bias[None, :]).astype(np.float32)
    w13 = _uniform_bytes(rng, (E, 2 * I, d // 2))
    w13_scale = _scale_bytes(rng, (E, 2 * I, d // 32), exp_lo, exp_hi)
    w2 = _uniform_bytes(rng, (E, d, I // 2))
    w2_scale = _scale_bytes(rng, (E, d, I // 32), exp_lo, exp_hi)
    return LayerInputs(T, d, I, E, k, x, np.ascontiguousarray(logits), w13, w13_scale, w2, w2_scale)


def make_gate_weights(E: int, d: int, seed: int = 0) -> np.ndarray:
    """Router weights Wg as bf16 bit patterns [E, d] (see the module docstring)."""
    rng = np.random.default_rng([seed, 1])
    w = rng.standard_normal((E, d), dtype=np.float32) / np.float32(math.sqrt(d))
    return _f32_to_bf16_bits(w.astype(np.float32))


def make_config(name: str, seed: int | None = None) -> LayerInputs:
    """Draw one of the named workloads (``CONFIGS``)."""
    c = dict(CONFIGS[name])
    if seed is not None:
        c["seed"] = seed
    return make_layer(**c)


def routing_sample_tokens(T: int, n: int, seed: int = 1) -> np.ndarray:
    """A fixed, sorted sample of token indices (always includes the first and last token)."""
    if n >= T:
        return np.arange(T)
    rng = np.random.default_rng(seed)
    pick = rng.choice(np.arange(1, T - 1), size=max(n - 2, 0), replace=False)
    return np.unique(np.concatenate([[0, T - 1], pick])).astype(np.int64)
