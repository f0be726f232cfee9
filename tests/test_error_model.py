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


# ---- the MXFP8 layer: h's interval passed through the block quantiser ----
def _bf16_neighbours(v):
    """the bf16 values one ulp below and above v (bf16 values, fp64)"""
    b = (np.asarray(v, dtype=np.float32).view(np.uint32) >> 16).astype(np.int64)
    up = np.where(v >= 0, b + 1, b - 1)
    dn = np.where(v > 0, b - 1, np.where(v == 0, 0x8001, b + 1))
    f = lambda bits: ((bits.astype(np.uint32) & 0xFFFF) << 16).view(np.float32).astype(np.float64)
    return np.minimum(f(dn), f(up)), np.maximum(f(dn), f(up))


def test_mx_hq_bound_covers_every_choice_inside_the_interval():
    """brute force: for blocks with up to three elements whose h may be either
    bf16 neighbour (one of them the block's largest, next to a power of two,
    so that the scale can move), every choice quantises within the bound"""
    import itertools

    from oracle import mx_activations as mxa

    from _layer_util import mx_hq_bound
    rng = np.random.default_rng(91)
    for case in range(40):
        h = oracle.bf16_round(rng.standard_normal((1, 32)) * np.exp2(rng.integers(-8, 8)))
        if case % 2 == 0:   # the largest element right at a power of two: the scale exponent may step
            j = int(np.argmax(np.abs(h)))
            h[0, j] = np.copysign(np.exp2(np.floor(np.log2(np.abs(h[0, j]))) + 1), h[0, j])
        idx = rng.choice(32, size=3, replace=False)
        if case % 2 == 0:
            idx[0] = int(np.argmax(np.abs(h)))
        lo, hi = h.copy(), h.copy()
        a, b = _bf16_neighbours(h[0, idx])
        lo[0, idx], hi[0, idx] = a, b
        hq = mxa.mx_round_trip(h)
        bound = mx_hq_bound(lo, hi, hq)
        for choice in itertools.product(range(3), repeat=3):
            hp = h.copy()
            for c, i in zip(choice, idx):
                hp[0, i] = (lo[0, i], h[0, i], hi[0, i])[c]
            d = np.abs(mxa.mx_round_trip(hp) - hq)
            assert np.all(d <= bound), (case, choice)
        # not vacuous: nothing moves by more than a few top-binade E4M3 ulps
        top = np.exp2(np.floor(np.log2(np.abs(hi).max())) - 3)
        assert bound.max() <= 4 * top


def test_mx_hq_bound_is_zero_for_single_point_intervals():
    from oracle import mx_activations as mxa

    from _layer_util import mx_hq_bound
    rng = np.random.default_rng(92)
    h = oracle.bf16_round(rng.standard_normal((5, 64)))
    assert not mx_hq_bound(h, h, mxa.mx_round_trip(h)).any()


def test_mx_out_slack_rejects_a_real_error():
    import pytest

    from oracle import mx_activations as mxa

    from _layer_util import MAX_ABS, assert_out_within_mx
    L = make_layer(T=6, d=128, I=64, E=2, k=1, seed=93)
    ref = mxa.forward_mx(L.x_bf16, L.router_logits, L.w13, L.w13_scale, L.w2, L.w2_scale, L.k)
    assert_out_within_mx(ref["out"], ref["out"], L)
    wrong = ref["out"].copy()
    wrong[3, 7] += 50 * MAX_ABS
    with pytest.raises(AssertionError):
        assert_out_within_mx(wrong, ref["out"], L)
