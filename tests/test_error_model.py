"""The h error model of the parity tests, checked on the CPU.

h on the GPU is bf16(silu(g) u) with g and u summed in fp32; the parity tests
accept any bf16 value in the interval _layer_util.h_interval derives from the
exact g and u.  Here an fp32 emulation of that arithmetic (products exact,
recursive fp32 sums in several random orders, fp32 SiLU) must always land in
the interval, and the interval must stay narrow (one bf16 value for most
elements), so that it cannot hide a real error.
"""
import numpy as np

import oracle
from moe_inputs import make_layer

from _layer_util import h_interval


def emulate_h_fp32(x_rows, W, rng):
    """h with fp32 recursive sums over K in a random order, SiLU in fp32."""
    I = W.shape[0] // 2
    K = W.shape[1]
    order = rng.permutation(K)
    prod_g = (x_rows[:, None, order] * W[None, :I, order]).astype(np.float32)  # exact products, rounded to fp32
    prod_u = (x_rows[:, None, order] * W[None, I:, order]).astype(np.float32)
    g = np.zeros(prod_g.shape[:2], dtype=np.float32)
    u = np.zeros(prod_u.shape[:2], dtype=np.float32)
    for j in range(K):
        g = g + prod_g[:, :, j]
        u = u + prod_u[:, :, j]
    with np.errstate(over="ignore"):
        v = (g / (np.float32(1) + np.exp(-g))) * u
    return oracle.bf16_round(v.astype(np.float64))


def test_fp32_emulation_lands_in_the_interval():
    L = make_layer(T=24, d=512, I=64, E=1, k=1, seed=71)
    x = oracle.bf16_bits_to_f64(L.x_bf16)
    W = oracle.dequantize_rows(L.w13[0], L.w13_scale[0])
    lo, hi = h_interval(x, L.w13[0], L.w13_scale[0])
    rng = np.random.default_rng(72)
    h_exact = oracle.expert_ffn(x, L.w13[0], L.w13_scale[0], L.w2[0], L.w2_scale[0])[0]
    n_diff = 0
    for _ in range(4):
        h = emulate_h_fp32(x, W, rng)
        assert np.all((h >= lo) & (h <= hi))
        n_diff += int((h != h_exact).sum())
    # the emulation does differ from the exact h somewhere, and the interval is
    # a single bf16 value for most elements
    assert n_diff > 0
    assert np.mean(lo == hi) > 0.9


def test_interval_rejects_a_one_percent_error():
    L = make_layer(T=16, d=256, I=64, E=1, k=1, seed=73)
    x = oracle.bf16_bits_to_f64(L.x_bf16)
    lo, hi = h_interval(x, L.w13[0], L.w13_scale[0])
    h = oracle.expert_ffn(x, L.w13[0], L.w13_scale[0], L.w2[0], L.w2_scale[0])[0]
    bad = oracle.bf16_round(h * 1.01)
    big = np.abs(h) > 1e-3 * np.abs(h).max()
    assert np.mean((bad[big] < lo[big]) | (bad[big] > hi[big])) > 0.9
