"""The seeded input recipe: shapes, value ranges and determinism."""
import numpy as np

from moe_inputs import CONFIGS, make_config, make_layer, routing_sample_tokens


def test_tiny_config_recipe():
    L = make_config("tiny")
    assert (L.T, L.d, L.I, L.E, L.k) == (16, 256, 128, 8, 2)
    assert L.x_bf16.dtype == np.uint16 and L.x_bf16.shape == (16, 256)
    assert L.router_logits.dtype == np.float32 and L.router_logits.shape == (16, 8)
    assert L.w13.shape == (8, 256, 128) and L.w13_scale.shape == (8, 256, 8)
    assert L.w2.shape == (8, 256, 64) and L.w2_scale.shape == (8, 256, 4)
    assert L.w13_scale.min() >= 120 and L.w13_scale.max() <= 122
    assert set(np.unique(L.w2_scale)) == {120, 121, 122}


def test_determinism_and_seed():
    a, b, c = make_layer(8, 64, 32, 4, 2, seed=5), make_layer(8, 64, 32, 4, 2, seed=5), make_layer(8, 64, 32, 4, 2, seed=6)
    for f in ("x_bf16", "router_logits", "w13", "w13_scale", "w2", "w2_scale"):
        assert np.array_equal(getattr(a, f), getattr(b, f))
        assert not np.array_equal(getattr(a, f), getattr(c, f))


def test_codes_uniform_and_skew_bias():
    L = make_layer(T=64, d=512, I=256, E=16, k=4, seed=1, skew=True)
    lo = np.bincount((L.w13 & 15).ravel(), minlength=16)
    hi = np.bincount((L.w13 >> 4).ravel(), minlength=16)
    n = L.w13.size / 16
    assert np.all(np.abs(lo - n) < 6 * np.sqrt(n)) and np.all(np.abs(hi - n) < 6 * np.sqrt(n))
    # the per-expert bias 2 log(1/(e+1)) shifts column means down with the rank
    m = L.router_logits.mean(0)
    assert m[0] > m[3] > m[15]


def test_named_configs_and_sampling():
    assert CONFIGS["prefill"]["T"] == 4608 and CONFIGS["large"]["d"] == 7168
    s = routing_sample_tokens(100, 10)
    assert s[0] == 0 and s[-1] == 99 and len(s) == 10 and (np.diff(s) > 0).all()
