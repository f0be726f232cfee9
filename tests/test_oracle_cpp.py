"""The second CPU oracle (plain C++ loops, oracle/moe_oracle_ref.cpp) against
the hand-worked layer and against the numpy oracle: two independent programs
of the layer's definition."""
import numpy as np
import pytest

import oracle
from moe_inputs import make_layer
from oracle import cpp_ref
from test_oracle_pins import _golden_values, _hand_layer


@pytest.fixture(scope="module", autouse=True)
def _built():
    cpp_ref.build()


def test_cpp_oracle_hand_worked_layer():
    g = _golden_values()
    x, logits, w13, w13s, w2, w2s, k = _hand_layer()
    r = cpp_ref.forward(x, logits, w13, w13s, w2, w2s, k)
    assert r["topk_ids"].tolist() == [[0, 1], [0, 1]]
    assert r["sorted_slot"].tolist() == [0, 2, 1, 3]
    h = r["h"]
    assert (h[0] == g["h_t0_e0"]).all() and (h[1] == g["h_t1_e0"]).all()
    assert (h[2] == g["h_t0_e1"]).all() and (h[3] == g["h_t1_e1"]).all()
    w0 = 1.0 / (1.0 + np.exp(-1.0))
    np.testing.assert_allclose(r["out"][0], w0 * g["y_t0_e0"] + (1.0 - w0) * g["y_t0_e1"], rtol=1e-15)
    np.testing.assert_allclose(r["out"][1], 0.5 * g["y_t1_e0"] + 0.5 * g["y_t1_e1"], rtol=1e-15)


@pytest.mark.parametrize("shape", [dict(T=16, d=256, I=128, E=8, k=2, seed=0),
                                   dict(T=23, d=64, I=96, E=13, k=4, seed=3),
                                   dict(T=40, d=128, I=64, E=64, k=6, seed=4),
                                   dict(T=7, d=32, I=32, E=3, k=3, seed=5)])
def test_cpp_oracle_matches_numpy_oracle(shape):
    L = make_layer(**shape)
    a = oracle.forward(L.x_bf16, L.router_logits, L.w13, L.w13_scale, L.w2, L.w2_scale, L.k)
    b = cpp_ref.forward(L.x_bf16, L.router_logits, L.w13, L.w13_scale, L.w2, L.w2_scale, L.k)
    for key in ("topk_ids", "expert_offsets", "sorted_slot"):
        np.testing.assert_array_equal(a[key], b[key])
    np.testing.assert_allclose(a["topk_w"], b["topk_w"], rtol=1e-15, atol=0)
    # h: both programs sum exact fp64 products (in different orders) and round
    # to bf16 once; the roundings agree unless a sum lies within fp64 error of a
    # bf16 boundary, which these inputs never do
    np.testing.assert_array_equal(a["h"], b["h"])
    scale = np.abs(a["out"]).max()
    np.testing.assert_allclose(b["out"], a["out"], rtol=1e-12, atol=1e-13 * scale)


def test_cpp_oracle_ties_and_signed_zero():
    # equal logits and +-0 fall to the lower expert index, as in the numpy oracle
    logits = np.array([[0.0, -0.0, 1.0, 1.0, -1.0, 0.0],
                       [2.0, 2.0, 2.0, 2.0, 2.0, 2.0],
                       [-0.0, 0.0, -0.0, 0.0, -3.0, 5.0]], dtype=np.float32)
    for k in (1, 3, 6):
        ids_a, w_a = oracle.route(logits, k)
        ids_b, w_b = cpp_ref.route(logits, k)
        np.testing.assert_array_equal(ids_a, ids_b)
        np.testing.assert_allclose(w_a, w_b, rtol=1e-15, atol=0)
        assert np.allclose(w_b.sum(axis=1), 1.0, rtol=1e-15)


def test_cpp_oracle_sort_is_stable_counting_sort():
    ids = np.array([[3, 0], [0, 3], [2, 0], [3, 1]], dtype=np.int32)
    off, ss, sp = cpp_ref.expert_sort(ids, 5)
    assert off.tolist() == [0, 3, 4, 5, 8, 8]
    assert ss.tolist() == [1, 2, 5, 7, 4, 0, 3, 6]
    assert (ss[sp] == np.arange(8)).all()


def test_cpp_oracle_does_not_depend_on_thread_count():
    L = make_layer(T=24, d=128, I=64, E=9, k=3, seed=6)
    args = (L.x_bf16, L.router_logits, L.w13, L.w13_scale, L.w2, L.w2_scale, L.k)
    a = cpp_ref.forward(*args, threads=1)
    b = cpp_ref.forward(*args, threads=5)
    for key in a:
        np.testing.assert_array_equal(a[key], b[key])
