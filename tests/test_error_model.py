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


def test_interval_reaches_zero_where_fp32_silu_underflows():
    # g far below -88: exp(-g) overflows fp32 and the fast SiLU gives 0, while
    # the exact h is a tiny nonzero value; 0 must lie in the interval
    L = make_layer(T=4, d=64, I=32, E=1, k=1, seed=74)
    x = oracle.bf16_bits_to_f64(L.x_bf16)
    W = oracle.dequantize_rows(L.w13[0], L.w13_scale[0])
    W[:32] *= 200.0 / np.abs(x @ W[:32].T).max()   # |g| up to 200
    from _layer_util import h_interval_w
    lo, hi = h_interval_w(x, W)
    g = x @ W[:32].T
    deep = g < -100
    assert deep.any()
    assert np.all((lo[deep] <= 0) & (hi[deep] >= 0))


def test_out_slack_covers_a_flip_and_nothing_more():
    # an h element one bf16 ulp off (inside its interval) moves out by at most
    # the slack; an error in W2 (a weight doubled) is not covered
    from _layer_util import MAX_ABS, assert_out_within, h_interval_w
    L = make_layer(T=6, d=128, I=64, E=2, k=1, seed=75)
    ref = oracle.forward(L.x_bf16, L.router_logits, L.w13, L.w13_scale, L.w2, L.w2_scale, L.k)
    assert_out_within(ref["out"], ref["out"], L)
    wrong = ref["out"].copy()
    wrong[2, 5] += 50 * MAX_ABS
    import pytest
    with pytest.raises(AssertionError):
        assert_out_within(wrong, ref["out"], L)
