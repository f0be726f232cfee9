"""Pins of the CPU oracle to facts fixed outside the oracle itself.

Each test checks the oracle against a published table or test vector, a
closed form worked by hand, a library routine, a brute-force evaluation or
an invariant of the layer, so that a plausible mistake in the oracle (nibble
order, gate/up split, W2 orientation, tie-break, softmax support, sort
stability, rounding) fails at least one of them.  The mutation tests at the
end plant such mistakes in the oracle and check that the pins catch them.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import moe_oracle as om
from moe_inputs import make_layer

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------
# helpers that are independent of the oracle's code
# ----------------------------------------------------------------------------
def e2m1_closed_form(code: int) -> float:
    """E2M1 from its bit fields: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0."""
    s, e, m = (code >> 3) & 1, (code >> 1) & 3, code & 1
    mag = 0.5 * m if e == 0 else 2.0 ** (e - 1) * (1.0 + 0.5 * m)
    return -mag if s else mag


def dequant_by_loops(packed: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Element-by-element dequantisation with the closed-form E2M1 decoder."""
    R, half = packed.shape
    out = np.zeros((R, 2 * half))
    for r in range(R):
        for K in range(2 * half):
            byte = int(packed[r, K // 2])
            code = byte & 15 if K % 2 == 0 else byte >> 4
            out[r, K] = e2m1_closed_form(code) * math.ldexp(1.0, int(scales[r, K // 32]) - 127)
    return out


def bf16_torch(v: np.ndarray) -> np.ndarray:
    """fp64 -> fp32 -> bf16 through torch (the values used here are fp32-exact or far from ties)."""
    return torch.from_numpy(np.asarray(v, dtype=np.float64)).to(torch.float32).to(torch.bfloat16).to(torch.float64).numpy()


def dense_layer_torch(L, ids_w=None):
    """The layer as sum_e g_te * FFN_e(x_t) over ALL experts (g_te = 0 unless selected),
    with no sort, permutation or combine step; torch fp64 matmuls and F.silu."""
    x = torch.from_numpy(oracle.bf16_bits_to_f64(L.x_bf16))
    ids, w = ids_w if ids_w is not None else oracle.route(L.router_logits, L.k)
    gate = np.zeros((L.T, L.E))
    for t in range(L.T):
        for j in range(L.k):
            gate[t, ids[t, j]] += w[t, j]
    out = torch.zeros(L.T, L.d, dtype=torch.float64)
    for e in range(L.E):
        W13 = torch.from_numpy(dequant_by_loops(L.w13[e], L.w13_scale[e]))
        W2 = torch.from_numpy(dequant_by_loops(L.w2[e], L.w2_scale[e]))
        g = x @ W13[:L.I].T
        u = x @ W13[L.I:].T
        h = torch.from_numpy(bf16_torch((torch.nn.functional.silu(g) * u).numpy()))
        out += torch.from_numpy(gate[:, e:e + 1]) * (h @ W2.T)
    return out.numpy()


def small_layer(seed=0, T=12, d=64, I=64, E=6, k=3, **kw):
    return make_layer(T=T, d=d, I=I, E=E, k=k, seed=seed, **kw)


def run(L):
    return oracle.forward(L.x_bf16, L.router_logits, L.w13, L.w13_scale, L.w2, L.w2_scale, L.k)


# ----------------------------------------------------------------------------
# formats
# ----------------------------------------------------------------------------
def test_e2m1_matches_published_table():
    rows = [ln.split() for ln in open(os.path.join(GOLDEN, "e2m1_codes.txt")) if ln.strip() and not ln.startswith("#")]
    assert len(rows) == 16
    for code_hex, sign, exp, man, value in rows:
        code = int(code_hex, 16)
        got = oracle.e2m1_decode(np.array([code]))[0]
        assert got == float(value) and math.copysign(1.0, got) == math.copysign(1.0, float(value)), code_hex
        assert got == e2m1_closed_form(code)
        assert (code >> 3) == int(sign) and ((code >> 1) & 3) == int(exp, 2) and (code & 1) == int(man)


def test_e8m0_is_power_of_two_with_bias_127():
    for s in [0, 1, 2, 119, 120, 121, 122, 126, 127, 128, 200, 254]:
        assert oracle.e8m0_decode(np.array([s]))[0] == math.ldexp(1.0, s - 127)
    assert np.isnan(oracle.e8m0_decode(np.array([255]))[0])


def test_dequant_matches_element_loops_and_nibble_order():
    rng = np.random.default_rng(3)
    packed = rng.integers(0, 256, (5, 48), dtype=np.uint8)
    scales = rng.integers(110, 140, (5, 3), dtype=np.uint8)
    np.testing.assert_array_equal(oracle.dequantize_rows(packed, scales), dequant_by_loops(packed, scales))
    # byte 0x7A: low nibble 0xA (-1.0) is element K=0, high nibble 0x7 (6.0) is K=1
    p = np.zeros((1, 16), np.uint8)
    p[0, 0] = 0x7A
    v = oracle.dequantize_rows(p, np.full((1, 1), 127, np.uint8))
    assert v[0, 0] == -1.0 and v[0, 1] == 6.0 and not v[0, 2:].any()
    # scale block j covers K in [32j, 32j+32)
    p = np.full((1, 32), 0x22, np.uint8)
    v = oracle.dequantize_rows(p, np.array([[127, 130]], np.uint8))
    assert (v[0, :32] == 1.0).all() and (v[0, 32:] == 8.0).all()


def test_bf16_decode_matches_torch():
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.bf16_bits_to_f64(bits)
    fin = np.isfinite(ref)
    np.testing.assert_array_equal(got[fin], ref[fin])
    assert np.array_equal(np.isnan(got), np.isnan(ref))


def test_bf16_round_matches_torch_on_fp32_values():
    rng = np.random.default_rng(0)
    # random fp32 bit patterns across the whole range, plus every tie and
    # near-tie pattern around a few exponents, subnormals and the overflow edge
    pats = [rng.integers(0, 1 << 32, 200_000, dtype=np.uint64).astype(np.uint32)]
    for hi in [0x3F80, 0x3F81, 0x4000, 0x0001, 0x0080, 0x7F7F, 0xBF80, 0x8001, 0x0000]:
        base = np.uint32(hi) << np.uint32(16)
        low = np.array([0x0000, 0x0001, 0x7FFF, 0x8000, 0x8001, 0xFFFF], dtype=np.uint32)
        pats.append(base + low)
    bits = np.concatenate(pats)
    f = bits.view(np.float32)
    f = f[np.isfinite(f)]
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.bf16_round(f.astype(np.float64))
    np.testing.assert_array_equal(got, ref)
    assert oracle.bf16_round(np.array([3.397e38]))[0] == np.inf    # at or above (2 - 2^-8) * 2^127
    assert oracle.bf16_round(np.array([3.395e38]))[0] == 255 * 2.0 ** 120  # largest bf16


# ----------------------------------------------------------------------------
# routing
# ----------------------------------------------------------------------------
def test_route_matches_brute_force_sort():
    rng = np.random.default_rng(1)
    for E, k in [(8, 2), (16, 5), (33, 33), (64, 8)]:
        logits = rng.standard_normal((20, E)).astype(np.float32)
        logits[3, :] = 0.0                       # all tied
        logits[4, ::2] = 1.25                    # half tied at the top
        logits[5, 1] = -0.0                      # -0 vs +0 tie
        logits[5, 0] = 0.0
        logits[5, 2:] = -1.0
        ids, w = oracle.route(logits, k)
        for t in range(logits.shape[0]):
            order = sorted(range(E), key=lambda e: (-float(logits[t, e]), e))[:k]
            assert list(ids[t]) == order
            sel = [float(logits[t, e]) for e in order]
            ex = [math.exp(v - sel[0]) for v in sel]
            np.testing.assert_allclose(w[t], [v / sum(ex) for v in ex], rtol=1e-14)
        np.testing.assert_allclose(w.sum(1), 1.0, rtol=1e-14)
    assert list(oracle.route(np.zeros((1, 5), np.float32), 3)[0][0]) == [0, 1, 2]
    assert list(oracle.route(np.array([[0.0, -0.0, 0.0]], np.float32), 3)[0][0]) == [0, 1, 2]


def test_route_top2_closed_form_and_top1_weight_one():
    rng = np.random.default_rng(2)
    logits = rng.standard_normal((50, 7)).astype(np.float32)
    ids, w = oracle.route(logits, 2)
    l0 = np.take_along_axis(logits, ids[:, :1].astype(np.int64), 1)[:, 0].astype(np.float64)
    l1 = np.take_along_axis(logits, ids[:, 1:].astype(np.int64), 1)[:, 0].astype(np.float64)
    np.testing.assert_allclose(w[:, 0], 1.0 / (1.0 + np.exp(l1 - l0)), rtol=1e-14)
    ids1, w1 = oracle.route(logits, 1)
    assert (w1 == 1.0).all()
    np.testing.assert_array_equal(ids1[:, 0], np.argmax(logits, axis=1))  # numpy argmax: first max


def test_route_softmax_equals_renormalised_full_softmax():
    rng = np.random.default_rng(4)
    logits = rng.standard_normal((30, 16)).astype(np.float32)
    ids, w = oracle.route(logits, 4)
    full = torch.softmax(torch.from_numpy(logits.astype(np.float64)), dim=1).numpy()
    sel = np.take_along_axis(full, ids.astype(np.int64), 1)
    np.testing.assert_allclose(w, sel / sel.sum(1, keepdims=True), rtol=1e-13)


# ----------------------------------------------------------------------------
# expert sort and hash
# ----------------------------------------------------------------------------
def test_expert_sort_properties_and_hand_example():
    ids = np.array([[2, 0], [0, 1], [2, 1], [3, 2]], np.int32)   # T=4, k=2, E=5
    off, ss, pos = oracle.expert_sort(ids, 5)
    # by hand: expert 0 <- flat 1, 2; expert 1 <- 3, 5; expert 2 <- 0, 4, 7; expert 3 <- 6; expert 4 empty
    assert list(off) == [0, 2, 4, 7, 8, 8]
    assert list(ss) == [1, 2, 3, 5, 0, 4, 7, 6]
    assert list(pos) == [4, 0, 1, 2, 5, 3, 7, 6]
    rng = np.random.default_rng(5)
    for E, k, T in [(8, 2, 40), (256, 8, 100), (3, 3, 7)]:
        ids, _ = oracle.route(rng.standard_normal((T, E)).astype(np.float32), k)
        off, ss, pos = oracle.expert_sort(ids, E)
        flat = ids.ravel()
        assert off[0] == 0 and off[-1] == T * k and (np.diff(off) >= 0).all()
        np.testing.assert_array_equal(np.diff(off), np.bincount(flat, minlength=E))
        assert sorted(ss) == list(range(T * k))
        np.testing.assert_array_equal(pos[ss], np.arange(T * k))
        for e in range(E):
            seg = ss[off[e]:off[e + 1]]
            assert (flat[seg] == e).all() and (np.diff(seg) > 0).all()


def test_fnv1a64_published_vectors_and_route_hash_bytes():
    for ln in open(os.path.join(GOLDEN, "fnv1a64_vectors.txt")):
        if ln.startswith("#") or not ln.strip():
            continue
        text, hx = ln.split()
        assert oracle.fnv1a64(text.strip('"').encode()) == int(hx, 16)
    a, b, c = np.array([1], np.int32), np.array([2, 3], np.int32), np.array([0, 256], np.int32)
    raw = bytes([1, 0, 0, 0, 2, 0, 0, 0, 3, 0, 0, 0, 0, 0, 0, 0, 0, 1, 0, 0])
    assert oracle.route_hash(a, b, c) == oracle.fnv1a64(raw)


# ----------------------------------------------------------------------------
# the whole layer
# ----------------------------------------------------------------------------
def _hand_layer():
    T, d, I, E, k = 2, 32, 32, 2, 2
    x = np.zeros((T, d), np.uint16)
    x[0] = 0x3F00
    x[1] = 0xBF80
    logits = np.array([[1.0, 0.0], [0.0, 0.0]], np.float32)
    w13 = np.zeros((E, 2 * I, d // 2), np.uint8)
    w13s = np.full((E, 2 * I, d // 32), 127, np.uint8)
    w2 = np.zeros((E, d, I // 2), np.uint8)
    w2s = np.full((E, d, I // 32), 127, np.uint8)
    w13[0] = 0x22
    w2[0] = 0x11
    w2s[0] = 126
    w13[1, :I] = 0x99
    w13[1, I:] = 0x22
    w2[1] = 0x33
    return x, logits, w13, w13s, w2, w2s, k


def _golden_values():
    vals = {}
    for ln in open(os.path.join(GOLDEN, "hand_worked_layer.txt")):
        if ln.startswith("#") or not ln.strip():
            continue
        key, v = ln.split()
        if "*2^" in v:
            m, p = v.split("*2^")
            vals[key] = float(m) * 2.0 ** int(p)
        else:
            vals[key] = float(v)
    return vals


def test_hand_worked_layer():
    g = _golden_values()
    r = oracle.forward(*_hand_layer())
    assert r["topk_ids"].tolist() == [[0, 1], [0, 1]]
    # sorted rows: expert 0 <- slots 0 (t0), 2 (t1); expert 1 <- slots 1 (t0), 3 (t1)
    assert r["sorted_slot"].tolist() == [0, 2, 1, 3]
    h = r["h"]
    assert (h[0] == g["h_t0_e0"]).all() and (h[1] == g["h_t1_e0"]).all()
    assert (h[2] == g["h_t0_e1"]).all() and (h[3] == g["h_t1_e1"]).all()
    w0 = 1.0 / (1.0 + math.exp(-1.0))
    out0 = w0 * g["y_t0_e0"] + (1.0 - w0) * g["y_t0_e1"]
    out1 = 0.5 * g["y_t1_e0"] + 0.5 * g["y_t1_e1"]
    np.testing.assert_allclose(r["out"][0], out0, rtol=1e-15)
    np.testing.assert_allclose(r["out"][1], out1, rtol=1e-15)


def test_forward_equals_dense_brute_force():
    L = make_layer(T=10, d=64, I=32, E=5, k=2, seed=7)
    got = run(L)["out"]
    ref = dense_layer_torch(L)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_top1_reduces_to_dense_swiglu_mlp():
    L = make_layer(T=9, d=64, I=64, E=4, k=1, seed=8)
    got = run(L)["out"]
    e_star = np.argmax(L.router_logits, axis=1)
    x = torch.from_numpy(oracle.bf16_bits_to_f64(L.x_bf16))
    for t in range(L.T):
        e = int(e_star[t])
        W13 = torch.from_numpy(dequant_by_loops(L.w13[e], L.w13_scale[e]))
        W2 = torch.from_numpy(dequant_by_loops(L.w2[e], L.w2_scale[e]))
        gu = torch.nn.functional.linear(x[t], W13)
        h = bf16_torch((torch.nn.functional.silu(gu[:L.I]) * gu[L.I:]).numpy())
        ref = torch.nn.functional.linear(torch.from_numpy(h), W2).numpy()
        np.testing.assert_allclose(got[t], ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_single_expert_layer():
    L = make_layer(T=5, d=32, I=32, E=1, k=1, seed=9)
    r = run(L)
    assert (r["topk_ids"] == 0).all() and (r["topk_w"] == 1.0).all()
    assert r["expert_offsets"].tolist() == [0, 5]


def test_token_permutation_invariance():
    L = small_layer(seed=10)
    perm = np.random.default_rng(0).permutation(L.T)
    a = run(L)
    L2 = small_layer(seed=10)
    L2.x_bf16 = L.x_bf16[perm].copy()
    L2.router_logits = L.router_logits[perm].copy()
    b = run(L2)
    np.testing.assert_allclose(b["out"], a["out"][perm], rtol=1e-13, atol=1e-13)
    np.testing.assert_array_equal(b["topk_ids"], a["topk_ids"][perm])


def test_expert_relabelling_invariance():
    L = small_layer(seed=11)
    sigma = np.random.default_rng(1).permutation(L.E)     # new label of expert e is sigma[e]
    L2 = small_layer(seed=11)
    inv = np.argsort(sigma)
    L2.router_logits = L.router_logits[:, inv].copy()
    L2.w13, L2.w13_scale = L.w13[inv].copy(), L.w13_scale[inv].copy()
    L2.w2, L2.w2_scale = L.w2[inv].copy(), L.w2_scale[inv].copy()
    a, b = run(L), run(L2)
    # logits are distinct here, so the relabelled ids are sigma of the old ones, in the same slot order
    np.testing.assert_array_equal(b["topk_ids"], sigma[a["topk_ids"]])
    np.testing.assert_allclose(b["out"], a["out"], rtol=1e-13, atol=1e-13)


def test_w2_layout_probe():
    """One nonzero W2 code at (e*, n0, m0): the output is nonzero only in column n0,
    for tokens routed to e*, and equals w * h[m0] * value there."""
    L = small_layer(seed=12, T=16, d=64, I=64, E=4, k=2)
    e_star, n0, m0 = 2, 37, 21                   # m0 odd: high nibble of byte m0 // 2
    L.w2[:] = 0
    L.w2[e_star, n0, m0 // 2] = 0x50             # code 5 (3.0) in the high nibble
    L.w2_scale[:] = 128                          # x2
    r = run(L)
    out = r["out"]
    cols = np.nonzero(np.abs(out).sum(0))[0]
    assert set(cols.tolist()) <= {n0} and len(cols) == 1
    for t in range(L.T):
        j = np.nonzero(r["topk_ids"][t] == e_star)[0]
        if len(j) == 0:
            assert out[t, n0] == 0.0
            continue
        row = r["slot_pos"][t * L.k + j[0]]
        assert out[t, n0] == r["topk_w"][t, j[0]] * (r["h"][row, m0] * 6.0)


def test_w13_probes_nibble_order_and_gate_up_split():
    """One nonzero W13 code: in the gate half it makes g nonzero with u = 0 (h = 0);
    in the up half u is nonzero with g = 0 (silu(0) = 0, h = 0); a gate+up pair
    gives h = bf16(silu(a x_K) * b x_K) at the probe column, with K even or odd."""
    d, I = 64, 32
    L = make_layer(T=6, d=d, I=I, E=1, k=1, seed=13)
    xs = oracle.bf16_bits_to_f64(L.x_bf16)
    for K in (10, 11):
        for i0 in (0, 5):
            L.w13[:] = 0
            L.w13_scale[:] = 127
            sh = 0 if K % 2 == 0 else 4
            L.w13[0, i0, K // 2] = 0x4 << sh          # gate: 2.0 at K
            L.w13[0, I + i0, K // 2] = 0xB << sh      # up: -1.5 at K
            r = run(L)
            h = r["h"]
            assert not np.delete(h, i0, axis=1).any()
            for row in range(L.T):
                t = r["sorted_slot"][row]
                g, u = 2.0 * xs[t, K], -1.5 * xs[t, K]
                assert h[row, i0] == bf16_torch(np.array([g / (1 + math.exp(-g)) * u]))[0]
            # gate alone: h = 0; up alone: h = 0
            L.w13[0, I + i0, K // 2] = 0
            assert not run(L)["h"].any()
            L.w13[0, i0, K // 2] = 0
            L.w13[0, I + i0, K // 2] = 0xB << sh
            assert not run(L)["h"].any()


def test_exact_scaling_laws_and_zero_codes():
    L = small_layer(seed=14)
    base = run(L)["out"]
    L2 = small_layer(seed=14)
    L2.w2_scale = (L.w2_scale + 1).astype(np.uint8)
    np.testing.assert_array_equal(run(L2)["out"], 2.0 * base)
    L3 = small_layer(seed=14)
    L3.w13_scale = L.w13_scale.copy()
    L3.w13_scale[:, L.I:] += 1                   # up half doubled: u -> 2u, bf16(2v) = 2 bf16(v)
    np.testing.assert_array_equal(run(L3)["out"], 2.0 * base)
    L4 = small_layer(seed=14)
    L4.w13[:] = 0x88                             # -0 codes
    assert not run(L4)["out"].any()


def test_forward_tokens_matches_forward():
    L = small_layer(seed=15, T=20)
    r = run(L)
    toks = np.array([0, 3, 19])
    ids, w, out = oracle.forward_tokens(L.x_bf16, L.router_logits, L.w13, L.w13_scale, L.w2, L.w2_scale, L.k, toks)
    np.testing.assert_array_equal(ids, r["topk_ids"][toks])
    np.testing.assert_allclose(out, r["out"][toks], rtol=1e-13, atol=1e-13)


# ----------------------------------------------------------------------------
# planted mistakes: each must make at least one pin above fail
# ----------------------------------------------------------------------------
def _fails(test_fn):
    try:
        test_fn()
    except AssertionError:
        return True
    return False


def test_planted_nibble_swap_is_caught(monkeypatch):
    swapped = np.stack([om.e2m1_decode(np.arange(256) >> 4), om.e2m1_decode(np.arange(256) & 15)], axis=1)
    monkeypatch.setattr(om, "_BYTE_PAIR", swapped)
    assert _fails(test_dequant_matches_element_loops_and_nibble_order)
    assert _fails(test_w13_probes_nibble_order_and_gate_up_split)


def test_planted_gate_up_swap_is_caught(monkeypatch):
    real = om.dequantize_rows

    def ffn(x_rows, w13_e, w13s_e, w2_e, w2s_e):
        W13 = real(w13_e, w13s_e)
        I = W13.shape[0] // 2
        # wrong: rows [0, I) used as the up projection and [I, 2I) as the gate
        h = om.bf16_round(om.silu(x_rows @ W13[I:].T) * (x_rows @ W13[:I].T))
        return h, h @ real(w2_e, w2s_e).T
    monkeypatch.setattr(om, "expert_ffn", ffn)
    assert _fails(test_hand_worked_layer)


def test_planted_w2_transpose_is_caught(monkeypatch):
    real = om.dequantize_rows

    def ffn(x_rows, w13_e, w13s_e, w2_e, w2s_e):
        W13 = real(w13_e, w13s_e)
        I = W13.shape[0] // 2
        h = om.bf16_round(om.silu(x_rows @ W13[:I].T) * (x_rows @ W13[I:].T))
        W2 = real(w2_e, w2s_e)
        d = W2.shape[0]
        # wrong: read W2 as if stored [I, d] and reshape
        W2 = W2.reshape(-1).reshape(I, d).T
        return h, h @ W2.T
    monkeypatch.setattr(om, "expert_ffn", ffn)
    assert _fails(test_w2_layout_probe)


def test_planted_tie_to_higher_index_is_caught(monkeypatch):
    real = om.route

    def route_hi(logits, k):
        E = logits.shape[1]
        ids, w = real(logits[:, ::-1].copy(), k)
        return (E - 1 - ids).astype(np.int32), w
    monkeypatch.setattr(om, "route", route_hi)
    monkeypatch.setattr(oracle, "route", route_hi)
    assert _fails(test_route_matches_brute_force_sort)
    assert _fails(test_hand_worked_layer)


def test_planted_full_softmax_is_caught(monkeypatch):
    real = om.route

    def route_full(logits, k):
        ids, _ = real(logits, k)
        full = np.exp(logits.astype(np.float64) - logits.max(1, keepdims=True))
        full /= full.sum(1, keepdims=True)
        return ids, np.take_along_axis(full, ids.astype(np.int64), 1)
    monkeypatch.setattr(om, "route", route_full)
    monkeypatch.setattr(oracle, "route", route_full)
    assert _fails(test_route_matches_brute_force_sort)


def test_planted_unstable_sort_is_caught(monkeypatch):
    real = om.expert_sort

    def unstable(ids, E):
        off, ss, pos = real(ids, E)
        ss = ss.copy()
        for e in range(E):
            ss[off[e]:off[e + 1]] = ss[off[e]:off[e + 1]][::-1]
        pos = np.empty_like(ss)
        pos[ss] = np.arange(ss.size, dtype=np.int32)
        return off, ss, pos
    monkeypatch.setattr(om, "expert_sort", unstable)
    monkeypatch.setattr(oracle, "expert_sort", unstable)
    assert _fails(test_expert_sort_properties_and_hand_example)


def test_planted_missing_h_rounding_is_caught(monkeypatch):
    monkeypatch.setattr(om, "bf16_round", lambda v: np.asarray(v, dtype=np.float64))
    assert _fails(test_hand_worked_layer)


def test_planted_e8m0_bias_off_by_one_is_caught(monkeypatch):
    """The format-dialect bug class: an E8M0 bias of 126 instead of 127 doubles every weight."""
    def e8m0_bias126(s):
        s = np.asarray(s).astype(np.int64)
        return np.where(s == 255, np.nan, np.ldexp(1.0, s - 126))
    monkeypatch.setattr(om, "e8m0_decode", e8m0_bias126)
    monkeypatch.setattr(oracle, "e8m0_decode", e8m0_bias126)
    assert _fails(test_e8m0_is_power_of_two_with_bias_127)
    assert _fails(test_dequant_matches_element_loops_and_nibble_order)
    assert _fails(test_hand_worked_layer)


def test_planted_silu_sign_is_caught(monkeypatch):
    monkeypatch.setattr(om, "silu", lambda z: z / (1.0 + np.exp(z)))
    assert _fails(test_top1_reduces_to_dense_swiglu_mlp)
    assert _fails(test_forward_equals_dense_brute_force)


def _forward_with(token_of_slot, combine_rows):
    """oracle.forward with two of its index choices replaced (for planting mistakes)."""
    def forward(x_bf16, router_logits, w13, w13_scale, w2, w2_scale, k):
        x = om.bf16_bits_to_f64(x_bf16)
        T, d = x.shape
        E, I = w13.shape[0], w13.shape[1] // 2
        ids, w = om.route(router_logits, k)
        offsets, sorted_slot, slot_pos = om.expert_sort(ids, E)
        h, y = np.zeros((T * k, I)), np.zeros((T * k, d))
        for e in range(E):
            r0, r1 = int(offsets[e]), int(offsets[e + 1])
            if r0 < r1:
                tokens = token_of_slot(sorted_slot[r0:r1], k)
                h[r0:r1], y[r0:r1] = om.expert_ffn(x[tokens], w13[e], w13_scale[e], w2[e], w2_scale[e])
        out = np.zeros((T, d))
        rows = combine_rows(sorted_slot, slot_pos).reshape(T, k)
        for j in range(k):
            out += w[:, j:j + 1] * y[rows[:, j]]
        return dict(topk_ids=ids, topk_w=w, expert_offsets=offsets, sorted_slot=sorted_slot, slot_pos=slot_pos,
                    h=h, out=out)
    return forward


def test_planted_forward_rewrite_is_faithful(monkeypatch):
    """the helper above with the right choices reproduces the oracle (so the plants below test one change each)"""
    f = _forward_with(lambda ss, k: ss // k, lambda ss, pos: pos)
    L = make_layer(T=10, d=64, I=32, E=5, k=2, seed=7)
    a = f(L.x_bf16, L.router_logits, L.w13, L.w13_scale, L.w2, L.w2_scale, L.k)["out"]
    assert np.array_equal(a, run(L)["out"])


def test_planted_wrong_token_of_slot_is_caught(monkeypatch):
    f = _forward_with(lambda ss, k: ss % k, lambda ss, pos: pos)
    monkeypatch.setattr(om, "forward", f)
    monkeypatch.setattr(oracle, "forward", f)
    assert _fails(test_forward_equals_dense_brute_force)


def test_planted_combine_through_the_wrong_permutation_is_caught(monkeypatch):
    f = _forward_with(lambda ss, k: ss // k, lambda ss, pos: ss)
    monkeypatch.setattr(om, "forward", f)
    monkeypatch.setattr(oracle, "forward", f)
    assert _fails(test_forward_equals_dense_brute_force)


def test_planted_bf16_round_half_away_is_caught(monkeypatch):
    def away(v):
        v = np.asarray(v, dtype=np.float64)
        out = np.zeros_like(v)
        nz = (v != 0) & np.isfinite(v)
        a = np.abs(v[nz])
        _, ex = np.frexp(a)
        ulp = np.ldexp(1.0, np.maximum(ex - 1, -126) - 7)
        out[nz] = np.copysign(np.floor(a / ulp + 0.5) * ulp, v[nz])
        return out
    monkeypatch.setattr(om, "bf16_round", away)
    monkeypatch.setattr(oracle, "bf16_round", away)
    assert _fails(test_bf16_round_matches_torch_on_fp32_values)
