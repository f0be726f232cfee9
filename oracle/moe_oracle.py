"""CPU oracle of the FP4 routed mixture-of-experts layer (test infrastructure).

This file is test infrastructure only. Tests, the smoke check and the
benchmark's CPU-baseline leg may call it; the product path never does.
It is plain numpy in fp64 and shares no code with the CUDA path.

What it computes follows "DeepSeek-V4-Flash on AMD gfx90a: Correctness
Recovery and Inference Performance Engineering" (abstract: FP4 routed MoE,
expert sorting, the routed-expert W2 layout, fixed-token and hash checks),
the MXFP4 MoE path of the vLLM MI300X write-up ("MXFP4 MoE"), and the
top-k rules of the MI250 correctness blog (section 4.1 table, "MoE routing
top-k: FP32 comparison + fixed tie-break"; section 4.2, ties broken by
expert_id rather than memory address).  Where the pages are silent the
readings used are:

* MXFP4 element: E2M1 code (sign, 2 exponent bits, 1 mantissa bit), two
  codes per byte along K, the low nibble holding the even K element; E8M0
  scale byte s meaning 2**(s - 127), one per 32 consecutive K elements.
* W13 rows [0, I) are the gate projection, rows [I, 2I) the up projection;
  W2 row n is output feature n, packed along I.
* Routing: experts ordered by (logit descending, expert index ascending),
  the first k kept in that order; weights are the softmax over the k kept
  logits (no routed scaling, no shared expert, no expert groups).
* Expert sort: stable counting sort of the flat slots f = t*k + j by expert.
* Activation: SwiGLU, h = silu(g) * u with silu(z) = z / (1 + exp(-z)); h
  is rounded to bf16 (nearest, ties to even) before the down projection.
* out[t] = sum over the token's slots j, in slot order, of w[t, j] * y[slot].

Arithmetic is fp64 throughout except the one rounding point the layer
fixes (h to bf16).  Every function states the passage or reading it follows.
"""
from __future__ import annotations

import numpy as np

# E2M1 magnitudes indexed by the 3 low bits of a code (exponent bits e1 e0,
# mantissa bit m): e = 0 is the subnormal row (0, 0.5), otherwise
# 2**(e - 1) * (1 + m / 2).  OCP Microscaling (MX) v1.0, FP4 E2M1 element.
E2M1_MAGNITUDE = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)

MX_BLOCK = 32  # K elements per E8M0 scale (MXFP4)


# ----------------------------------------------------------------------------
# Formats
# ----------------------------------------------------------------------------
def e2m1_decode(codes: np.ndarray) -> np.ndarray:
    """Value of 4-bit E2M1 codes: bit 3 is the sign, bits 0..2 index the magnitude."""
    codes = np.asarray(codes).astype(np.int64)
    mag = E2M1_MAGNITUDE[codes & 7]
    return np.where((codes >> 3) & 1, -mag, mag)


def e8m0_decode(s: np.ndarray) -> np.ndarray:
    """Value of E8M0 scale bytes: 2**(s - 127); the byte 0xFF is NaN."""
    s = np.asarray(s).astype(np.int64)
    v = np.ldexp(1.0, s - 127)
    return np.where(s == 255, np.nan, v)


# (low-nibble value, high-nibble value) for every byte: byte b holds the even
# K element in its low nibble and the odd one in its high nibble.
_BYTE_PAIR = np.stack([e2m1_decode(np.arange(256) & 15), e2m1_decode(np.arange(256) >> 4)], axis=1)


def dequantize_rows(packed: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Dequantise MXFP4 rows: packed uint8 [R, K/2] and E8M0 uint8 [R, K/32] -> fp64 [R, K].

    Element K of row r is e2m1(code) * 2**(s - 127) with
    code = packed[r, K // 2] & 15 for even K, packed[r, K // 2] >> 4 for odd K,
    and s = scales[r, K // 32].
    """
    packed = np.asarray(packed, dtype=np.uint8)
    R, half = packed.shape
    K = 2 * half
    if scales.shape != (R, K // MX_BLOCK):
        raise ValueError(f"scales shape {scales.shape} does not match rows {R} x K {K}")
    vals = _BYTE_PAIR[packed].reshape(R, K)
    return vals * np.repeat(e8m0_decode(scales), MX_BLOCK, axis=1)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Decode bf16 bit patterns (uint16): the top half of an IEEE binary32."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):
        return b.view(np.float32).astype(np.float64)


def bf16_round(v: np.ndarray) -> np.ndarray:
    """Round real values to bf16 (8 significant bits, exponent range of binary32),
    nearest with ties to even; returns the rounded values as fp64.

    Written from the format's definition: the spacing of bf16 numbers in
    [2**e, 2**(e+1)) is 2**(e - 7) for e >= -126, and 2**-133 below (subnormals);
    values at or beyond the overflow threshold go to +-inf.
    """
    v = np.asarray(v, dtype=np.float64)
    out = np.zeros_like(v)
    nz = (v != 0) & np.isfinite(v)
    a = np.abs(v[nz])
    _, ex = np.frexp(a)             # a = m * 2**ex with m in [0.5, 1)
    e = ex - 1                      # a in [2**e, 2**(e+1))
    e = np.maximum(e, -126)
    ulp = np.ldexp(1.0, e - 7)
    q = np.rint(a / ulp) * ulp      # np.rint rounds halves to even
    q = np.where(q >= np.ldexp(1.0, 128), np.inf, q)  # past the largest bf16, (2 - 2**-7) * 2**127
    out[nz] = np.copysign(q, v[nz])
    out[~np.isfinite(v)] = v[~np.isfinite(v)]
    out[v == 0] = v[v == 0]
    return out


# ----------------------------------------------------------------------------
# Routing (top-k with fixed tie-break, softmax over the selected logits)
# ----------------------------------------------------------------------------
def route(router_logits: np.ndarray, k: int):
    """Top-k expert selection per token.

    Experts are ordered by (logit descending, index ascending) and the first
    k kept in that order (MI250 blog, section 4.1 table and section 4.2:
    FP32 comparison, ties to the lower expert id).  The weights are the
    softmax over the k kept logits, computed with the slot-0 logit as the
    shift: w_j = exp(l_j - l_0) / sum_j' exp(l_j' - l_0), sums in slot order.
    +0 and -0 compare equal and fall to the index rule.

    Returns topk_ids int32 [T, k] and topk_w fp64 [T, k].
    """
    logits = np.asarray(router_logits, dtype=np.float32)
    T, E = logits.shape
    if not 1 <= k <= E:
        raise ValueError("need 1 <= k <= E")
    idx = np.broadcast_to(np.arange(E), (T, E))
    # lexsort: the last key is primary.  -logits as float64 keeps -0 == +0.
    order = np.lexsort((idx, -logits.astype(np.float64)), axis=1)
    ids = order[:, :k].astype(np.int32)
    sel = np.take_along_axis(logits, ids.astype(np.int64), axis=1).astype(np.float64)
    ex = np.exp(sel - sel[:, :1])
    tot = np.zeros(T)
    for j in range(k):
        tot = tot + ex[:, j]
    return ids, ex / tot[:, None]


def expert_sort(topk_ids: np.ndarray, E: int):
    """Stable counting sort of the S = T*k slots by expert ("retuned expert sorting").

    expert_offsets[e] = number of slots routed to experts < e (E+1 entries);
    sorted_slot[r] = flat slot index t*k + j of sorted position r, increasing
    within each expert; slot_pos is the inverse permutation.
    """
    flat = np.asarray(topk_ids, dtype=np.int64).ravel()
    counts = np.bincount(flat, minlength=E)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    sorted_slot = np.argsort(flat, kind="stable").astype(np.int32)
    slot_pos = np.empty_like(sorted_slot)
    slot_pos[sorted_slot] = np.arange(flat.size, dtype=np.int32)
    return offsets, sorted_slot, slot_pos


def route_hash(topk_ids: np.ndarray, sorted_slot: np.ndarray, expert_offsets: np.ndarray) -> int:
    """FNV-1a 64-bit hash over the little-endian int32 bytes of topk_ids, then
    sorted_slot, then expert_offsets (the paper's hash-based routing check).
    FNV-1a: h = 0xcbf29ce484222325; per byte h = (h xor byte) * 0x100000001b3 mod 2**64.
    """
    data = b"".join(np.ascontiguousarray(a, dtype="<i4").tobytes()
                    for a in (topk_ids, sorted_slot, expert_offsets))
    return fnv1a64(data)


def fnv1a64(data: bytes) -> int:
    h = 0xCBF29CE484222325
    for byte in data:
        h ^= byte
        h = (h * 0x100000001B3) & 0xFFFFFFFFFFFFFFFF
    return h


# ----------------------------------------------------------------------------
# Expert FFN and the full layer
# ----------------------------------------------------------------------------
def silu(z: np.ndarray) -> np.ndarray:
    return z / (1.0 + np.exp(-z))


def expert_ffn(x_rows: np.ndarray, w13_e: np.ndarray, w13s_e: np.ndarray,
               w2_e: np.ndarray, w2s_e: np.ndarray):
    """One expert on m token rows: x_rows fp64 [m, d] -> (h fp64 [m, I] (bf16 values), y fp64 [m, d]).

    g = x W_gate^T, u = x W_up^T (W13 rows [0, I) and [I, 2I)), h = bf16(silu(g) * u),
    y = h W2^T.  Weights are dequantised once per call.
    """
    W13 = dequantize_rows(w13_e, w13s_e)          # [2I, d]
    I = W13.shape[0] // 2
    g = x_rows @ W13[:I].T
    u = x_rows @ W13[I:].T
    h = bf16_round(silu(g) * u)
    W2 = dequantize_rows(w2_e, w2s_e)              # [d, I]
    y = h @ W2.T
    return h, y


def forward(x_bf16: np.ndarray, router_logits: np.ndarray, w13: np.ndarray, w13_scale: np.ndarray,
            w2: np.ndarray, w2_scale: np.ndarray, k: int):
    """The whole layer: route, sort, per-expert FFN over the sorted rows, combine.

    Returns a dict with topk_ids, topk_w, expert_offsets, sorted_slot,
    slot_pos, h (fp64 [S, I], sorted order, bf16 values) and out (fp64 [T, d]).
    """
    x = bf16_bits_to_f64(x_bf16)
    T, d = x.shape
    E = w13.shape[0]
    I = w13.shape[1] // 2
    ids, w = route(router_logits, k)
    offsets, sorted_slot, slot_pos = expert_sort(ids, E)
    S = T * k
    h = np.zeros((S, I))
    y = np.zeros((S, d))
    for e in range(E):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r0 == r1:
            continue
        tokens = sorted_slot[r0:r1] // k
        h[r0:r1], y[r0:r1] = expert_ffn(x[tokens], w13[e], w13_scale[e], w2[e], w2_scale[e])
    out = np.zeros((T, d))
    for j in range(k):
        out += w[:, j:j + 1] * y[slot_pos.reshape(T, k)[:, j]]
    return dict(topk_ids=ids, topk_w=w, expert_offsets=offsets, sorted_slot=sorted_slot,
                slot_pos=slot_pos, h=h, out=out)


def forward_tokens(x_bf16: np.ndarray, router_logits: np.ndarray, w13: np.ndarray, w13_scale: np.ndarray,
                   w2: np.ndarray, w2_scale: np.ndarray, k: int, tokens: np.ndarray):
    """out rows for a subset of tokens only (each token's output depends only on
    its own x row and logits).  Returns (topk_ids, topk_w, out fp64 [len(tokens), d])."""
    tokens = np.asarray(tokens, dtype=np.int64)
    x = bf16_bits_to_f64(x_bf16[tokens])
    ids, w = route(router_logits[tokens], k)
    y = np.zeros((len(tokens), k, x.shape[1]))
    for e in np.unique(ids):
        rows, slots = np.nonzero(ids == e)
        _, y[rows, slots] = expert_ffn(x[rows], w13[e], w13_scale[e], w2[e], w2_scale[e])
    out = np.zeros((len(tokens), x.shape[1]))
    for j in range(k):
        out += w[:, j:j + 1] * y[:, j]
    return ids, w, out
