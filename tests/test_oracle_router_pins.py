"""Pins of the router-projection oracle (oracle/router.py) to what the
definition fixes: a hand-worked example, the orientation of Wg (one-hot gate
rows select one hidden element), relabelling experts, exact power-of-two
scaling, and the fp32 rounding of the compared values; planted mistakes in
the oracle must make a pin fail."""
import os

import numpy as np
import pytest

import oracle
from oracle import router as orr
from moe_inputs import make_gate_weights, make_layer

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16(v):
    b = np.asarray(v, dtype=np.float32).view(np.uint32)
    assert not np.any(b & 0xFFFF)
    return (b >> 16).astype(np.uint16)


def golden_inputs():
    x = np.zeros((2, 32))
    x[0, :16], x[0, 16:], x[1] = 1.0, 0.5, -2.0
    wg = np.zeros((3, 32))
    wg[0] = 0.25
    wg[1] = np.where(np.arange(32) % 2 == 0, 1.0, -1.0)
    wg[2, 31] = 3.0
    return bf16(x), bf16(wg)


def read_golden():
    vals = {}
    for ln in open(os.path.join(GOLDEN, "router_logits.txt")):
        ln = ln.strip()
        if ln and not ln.startswith("#") and not ln.startswith("key"):
            key, *rest = ln.split()
            vals[key] = [float(v) for v in rest]
    return vals


def test_router_hand_worked_example():
    x, wg = golden_inputs()
    g = read_golden()
    logits = orr.router_logits(x, wg)
    for t in range(2):
        for e in range(3):
            assert logits[t, e] == g[f"logit_{t}_{e}"][0]
    ids, _ = oracle.route(orr.router_logits_f32(x, wg), 2)
    assert ids[0].tolist() == g["ids_0"] and ids[1].tolist() == g["ids_1"]


def test_one_hot_gate_rows_select_hidden_elements():
    L = make_layer(T=7, d=64, I=32, E=5, k=2, seed=81)
    picks = [3, 17, 40, 63, 0]
    wg = np.zeros((5, 64))
    for e, K in enumerate(picks):
        wg[e, K] = 1.0
    logits = orr.router_logits(L.x_bf16, bf16(wg))
    x = oracle.bf16_bits_to_f64(L.x_bf16)
    for e, K in enumerate(picks):
        assert np.array_equal(logits[:, e], x[:, K])


def test_relabelling_experts_permutes_columns_and_scaling_is_exact():
    L = make_layer(T=9, d=128, I=32, E=6, k=2, seed=82)
    wg = make_gate_weights(6, 128, seed=82)
    base = orr.router_logits(L.x_bf16, wg)
    perm = np.array([4, 0, 5, 2, 1, 3])
    assert np.array_equal(orr.router_logits(L.x_bf16, wg[perm]), base[:, perm])
    w2x = bf16(oracle.bf16_bits_to_f64(wg) * 2.0)
    assert np.array_equal(orr.router_logits(L.x_bf16, w2x), 2.0 * base)


def test_compared_values_are_the_exact_logits_rounded_to_fp32():
    L = make_layer(T=5, d=256, I=32, E=4, k=2, seed=83)
    wg = make_gate_weights(4, 256, seed=83)
    exact = orr.router_logits(L.x_bf16, wg)
    f32 = orr.router_logits_f32(L.x_bf16, wg)
    assert f32.dtype == np.float32
    spacing = np.spacing(np.abs(f32).astype(np.float32)).astype(np.float64)
    assert np.all(np.abs(f32.astype(np.float64) - exact) <= spacing / 2)


def test_gate_weights_recipe_gives_unit_scale_logits():
    L = make_layer(T=64, d=4096, I=32, E=64, k=2, seed=84)
    logits = orr.router_logits(L.x_bf16, make_gate_weights(64, 4096, seed=84))
    assert 0.8 < logits.std() < 1.2


def test_forward_gated_routes_on_the_fp32_logits():
    L = make_layer(T=12, d=128, I=64, E=6, k=2, seed=85)
    wg = make_gate_weights(6, 128, seed=85)
    r = orr.forward_gated(L.x_bf16, wg, L.w13, L.w13_scale, L.w2, L.w2_scale, L.k)
    ref = oracle.forward(L.x_bf16, orr.router_logits_f32(L.x_bf16, wg), L.w13, L.w13_scale, L.w2, L.w2_scale, L.k)
    assert np.array_equal(r["topk_ids"], ref["topk_ids"]) and np.array_equal(r["out"], ref["out"])


def _fails(fn):
    try:
        fn()
    except AssertionError:
        return True
    return False


def test_planted_transposed_gate_is_caught(monkeypatch):
    def bad(x_bf16, w_gate_bf16):
        x = oracle.bf16_bits_to_f64(x_bf16)
        wg = oracle.bf16_bits_to_f64(w_gate_bf16)
        return x @ wg.reshape(wg.shape[1], wg.shape[0])   # rows read as columns
    monkeypatch.setattr(orr, "router_logits", bad)
    assert _fails(test_one_hot_gate_rows_select_hidden_elements)


def test_planted_dropped_last_element_is_caught(monkeypatch):
    def bad(x_bf16, w_gate_bf16):
        x = oracle.bf16_bits_to_f64(x_bf16)
        wg = oracle.bf16_bits_to_f64(w_gate_bf16)
        return x[:, :-1] @ wg[:, :-1].T
    monkeypatch.setattr(orr, "router_logits", bad)
    assert _fails(test_router_hand_worked_example)


def test_planted_truncated_fp32_is_caught(monkeypatch):
    def bad(x_bf16, w_gate_bf16):
        v = orr.router_logits(x_bf16, w_gate_bf16)
        return (v.astype(np.float32).view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32)  # bf16 truncation
    monkeypatch.setattr(orr, "router_logits_f32", bad)
    assert _fails(test_compared_values_are_the_exact_logits_rounded_to_fp32)
