"""CPU oracle of the layer with block-scaled (MXFP8) activations (test infrastructure).

This file is test infrastructure only, under the same rules as moe_oracle:
tests, the smoke check and the benchmark's CPU-baseline leg may call it; the
product path never does.  Plain numpy in fp64; no code shared with the CUDA
path.

The paper's decode path quantises its activations ("DeepSeek-V4-Flash on AMD
gfx90a: Correctness Recovery and Inference Performance Engineering", abstract:
INT8 activation quantisation on the decode path), and the MI250 blog that
reads it names block-wise FP8 quantisation as the next gain (its closing
outlook).  A tensor core that consumes MX operands directly takes the
activations in the MX form of the weights: one E8M0 scale per 32 K elements.
The readings used here, where the pages say nothing:

* Element: E4M3 of the OCP 8-bit floating-point formats (the "FN" variant):
  sign bit, 4 exponent bits with bias 7, 3 mantissa bits; exponent field 0
  holds the subnormals m/8 * 2**-6; S.1111.111 is NaN; there are no
  infinities; the largest finite magnitude is 448 = 1.75 * 2**8.
* Block: 32 consecutive elements along the reduction dimension (d for x
  before W13, I for h before W2), aligned like the weights' scale blocks.
* Scale (OCP Microscaling v1.0 conversion): X = 2**(floor(log2(amax)) - 8),
  8 being the largest E4M3 exponent, the exponent clamped to [-127, 127] and
  stored as the E8M0 byte exponent + 127.  A block of zeros gets the byte 0.
* Elements: v / X (exact: X is a power of two) rounded to the nearest E4M3
  value, ties to the even mantissa; magnitudes beyond 448 saturate to 448
  (amax / X lies in [256, 512), so only the top binade can exceed it).  The
  sign of zero is kept: -0 gives the code 0x80.
* Non-finite input: a block holding an infinity or a NaN has no finite
  power-of-two scale, and E8M0 has no infinity, so its scale is the NaN byte
  0xFF (OCP Microscaling v1.0: a NaN scale makes the whole block NaN) and its
  elements are the E4M3 NaN code 0x7F.
* Where: x (bf16) per token row before W13; h after its bf16 rounding, per
  slot row, before W2.  Routing, the sort, SwiGLU, the bf16 rounding of h and
  the combine are those of moe_oracle.forward.
"""
from __future__ import annotations

import numpy as np

from .moe_oracle import MX_BLOCK, bf16_bits_to_f64, bf16_round, dequantize_rows, expert_sort, route, silu

E4M3_MAX = 448.0
E4M3_EMAX = 8      # exponent of the largest binade
E4M3_EMIN = -6     # exponent of the smallest normal binade
E4M3_MANT = 3      # mantissa bits


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """Value of E4M3 codes (uint8): (-1)**s * 2**(e-7) * (1 + m/8) for e >= 1,
    (-1)**s * 2**-6 * m/8 for e = 0; the codes 0x7F and 0xFF are NaN."""
    c = np.asarray(codes).astype(np.int64)
    s, e, m = (c >> 7) & 1, (c >> 3) & 15, c & 7
    mag = np.where(e == 0, np.ldexp(m / 8.0, E4M3_EMIN), np.ldexp(1.0 + m / 8.0, e - 7))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(s == 1, -mag, mag)


def e4m3_round(v: np.ndarray) -> np.ndarray:
    """Round real values to E4M3 values: nearest, ties to even mantissa,
    saturating at +-448, sign kept (also for zero).  Returns fp64 values.

    Spacing of E4M3 values in [2**e, 2**(e+1)) is 2**(e-3) for e >= -6, and
    2**-9 below 2**-6 (subnormals)."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    out = np.zeros_like(a)
    nz = a > 0
    _, ex = np.frexp(a[nz])                 # a = f * 2**ex, f in [0.5, 1)
    e = np.maximum(ex - 1, E4M3_EMIN)
    ulp = np.ldexp(1.0, e - E4M3_MANT)
    out[nz] = np.minimum(np.rint(a[nz] / ulp) * ulp, E4M3_MAX)   # np.rint: halves to even
    return np.copysign(out, v)


def e4m3_encode(q: np.ndarray) -> np.ndarray:
    """Codes of E4M3-representable values q (finite, |q| <= 448), sign of zero kept."""
    q = np.asarray(q, dtype=np.float64)
    a = np.abs(q)
    if np.any(~np.isfinite(a)) or np.any(a > E4M3_MAX):
        raise ValueError("value outside the finite E4M3 range")
    sign = np.signbit(q).astype(np.int64)
    normal = a >= np.ldexp(1.0, E4M3_EMIN)
    _, ex = np.frexp(np.where(normal, a, 1.0))
    e = ex - 1
    m_norm = (np.ldexp(np.where(normal, a, 1.0), -e) - 1.0) * 8.0
    m_sub = np.ldexp(a, 9)
    m = np.where(normal, m_norm, m_sub)
    ebits = np.where(normal, e + 7, 0)
    if np.any(m != np.rint(m)) or np.any((m < 0) | (m > 7)):
        raise ValueError("value not representable in E4M3")
    return ((sign << 7) | (ebits << 3) | m.astype(np.int64)).astype(np.uint8)


def mxfp8_quantize(rows: np.ndarray):
    """MXFP8 (E4M3 elements, E8M0 scales) of real rows [R, K], K a multiple of 32.

    Returns codes uint8 [R, K] and scale bytes uint8 [R, K/32]; element j of
    block b is e4m3_round(rows[r, 32 b + j] / X_b) with X_b = 2**(floor(log2(amax_b)) - 8)."""
    rows = np.asarray(rows, dtype=np.float64)
    R, K = rows.shape
    if K % MX_BLOCK:
        raise ValueError("K must be a multiple of 32")
    blocks = rows.reshape(R, K // MX_BLOCK, MX_BLOCK)
    bad = ~np.all(np.isfinite(blocks), axis=2)          # blocks holding an infinity or a NaN
    blocks = np.where(bad[:, :, None], 0.0, blocks)
    amax = np.abs(blocks).max(axis=2)
    _, ex = np.frexp(np.where(amax > 0, amax, 1.0))
    shared = np.where(amax > 0, ex - 1 - E4M3_EMAX, -127)
    shared = np.clip(shared, -127, 127)
    q = e4m3_round(blocks / np.ldexp(1.0, shared)[:, :, None])
    codes = np.where(bad[:, :, None], np.uint8(0x7F), e4m3_encode(q))
    scales = np.where(bad, np.uint8(0xFF), (shared + 127).astype(np.uint8))
    return codes.reshape(R, K).astype(np.uint8), scales.astype(np.uint8)


def mxfp8_dequantize(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Values of MXFP8 rows: e4m3(code) * 2**(s - 127) -> fp64 [R, K]; the
    scale byte 0xFF is NaN."""
    codes = np.asarray(codes, dtype=np.uint8)
    R, K = codes.shape
    s = np.asarray(scales).astype(np.int64)
    X = np.where(s == 255, np.nan, np.ldexp(1.0, s - 127))
    return e4m3_decode(codes) * np.repeat(X, MX_BLOCK, axis=1)


def mx_round_trip(rows: np.ndarray) -> np.ndarray:
    """rows as the block-scaled operand sees them: dequantise(quantise(rows))."""
    return mxfp8_dequantize(*mxfp8_quantize(rows))


def expert_ffn_mx(x_rows_q: np.ndarray, w13_e: np.ndarray, w13s_e: np.ndarray,
                  w2_e: np.ndarray, w2s_e: np.ndarray):
    """One expert on m token rows already in MXFP8 form (fp64 values):
    g, u from x_rows_q; h = bf16(silu(g) * u); h_q = MXFP8 round trip of h; y = h_q W2^T.
    Returns (h, h_q, y)."""
    W13 = dequantize_rows(w13_e, w13s_e)
    I = W13.shape[0] // 2
    g = x_rows_q @ W13[:I].T
    u = x_rows_q @ W13[I:].T
    h = bf16_round(silu(g) * u)
    h_q = mx_round_trip(h)
    y = h_q @ dequantize_rows(w2_e, w2s_e).T
    return h, h_q, y


def forward_mx(x_bf16: np.ndarray, router_logits: np.ndarray, w13: np.ndarray, w13_scale: np.ndarray,
               w2: np.ndarray, w2_scale: np.ndarray, k: int):
    """The layer with MXFP8 activations into both projections.

    Returns the keys of moe_oracle.forward (h: bf16 values before the
    quantisation, sorted order) plus x_codes / x_scales (MXFP8 of x, per token)
    and h_q (the W2 operand, sorted order)."""
    x = bf16_bits_to_f64(x_bf16)
    T, d = x.shape
    E = w13.shape[0]
    I = w13.shape[1] // 2
    x_codes, x_scales = mxfp8_quantize(x)
    x_q = mxfp8_dequantize(x_codes, x_scales)
    ids, w = route(router_logits, k)
    offsets, sorted_slot, slot_pos = expert_sort(ids, E)
    S = T * k
    h = np.zeros((S, I))
    h_q = np.zeros((S, I))
    y = np.zeros((S, d))
    for e in range(E):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r0 == r1:
            continue
        tokens = sorted_slot[r0:r1] // k
        h[r0:r1], h_q[r0:r1], y[r0:r1] = expert_ffn_mx(x_q[tokens], w13[e], w13_scale[e], w2[e], w2_scale[e])
    out = np.zeros((T, d))
    for j in range(k):
        out += w[:, j:j + 1] * y[slot_pos.reshape(T, k)[:, j]]
    return dict(topk_ids=ids, topk_w=w, expert_offsets=offsets, sorted_slot=sorted_slot, slot_pos=slot_pos,
                x_codes=x_codes, x_scales=x_scales, h=h, h_q=h_q, out=out)
