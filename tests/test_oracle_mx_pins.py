"""Pins of the MXFP8-activation oracle (oracle/mx_activations.py) to facts
fixed outside it.

The E4M3 decoder is checked against torch's float8_e4m3fn on all 256 codes,
the rounding against torch's float -> float8_e4m3fn conversion, and the MX
block quantiser against an exhaustive nearest-value search over the decoded
code table with a scale found by brute force over powers of two.  The layer
is checked against a dense evaluation over all experts (no sort, no
permutation, no combine step), an exact scaling law and a bounded distance
from the unquantised layer.  Planted mistakes at the end must be caught.
"""
import numpy as np
import pytest
import torch

from oracle import mx_activations as mx
from oracle import moe_oracle as om
from moe_inputs import make_layer


# ----------------------------------------------------------------------------
# helpers independent of the oracle's code
# ----------------------------------------------------------------------------
def torch_e4m3_table() -> np.ndarray:
    """Values of all 256 E4M3 codes, decoded by torch."""
    return torch.from_numpy(np.arange(256, dtype=np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def torch_e4m3_round(v: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.asarray(v, np.float64)).to(torch.float32).to(torch.float8_e4m3fn).to(
        torch.float64).numpy()


def scale_exponent_by_search(amax: float) -> int:
    """The integer s with 2**(s + 8) <= amax < 2**(s + 9), by stepping through powers of two."""
    s = -200
    while 2.0 ** (s + 9) <= amax:
        s += 1
    return s


def nearest_code(v: float, table: np.ndarray) -> int:
    """Code of the finite E4M3 value nearest to v; on a tie the even code (mantissa LSB 0)."""
    fin = np.nonzero(np.isfinite(table))[0]
    dist = np.abs(table[fin] - v)
    best = fin[dist == dist.min()]
    if len(best) > 1:
        # equal values (+0 and -0) or a true tie between neighbours
        vals = table[best]
        if np.all(vals == vals[0]):
            return int(best[0])
        best = best[(best & 1) == 0]
    return int(best[0])


def bf16_exact(rng, shape, lo_exp, hi_exp):
    """Random values exactly representable in bf16 with magnitudes in [2**lo_exp, 2**hi_exp)."""
    mant = rng.integers(128, 256, size=shape)        # 8 significant bits
    e = rng.integers(lo_exp, hi_exp, size=shape)
    sign = rng.choice([-1.0, 1.0], size=shape)
    return sign * np.ldexp(mant / 128.0, e)


# ----------------------------------------------------------------------------
# the element format
# ----------------------------------------------------------------------------
def test_e4m3_decode_matches_torch_on_all_codes():
    got = mx.e4m3_decode(np.arange(256))
    ref = torch_e4m3_table()
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(ref[ok]))   # 0x80 is -0
    assert np.nanmax(ref) == mx.E4M3_MAX


def test_e4m3_round_matches_torch_conversion():
    rng = np.random.default_rng(0)
    table = torch_e4m3_table()
    fin = np.sort(np.unique(table[np.isfinite(table)]))
    mids = (fin[1:] + fin[:-1]) / 2.0                # exact ties between neighbours
    rnd = np.concatenate([bf16_exact(rng, 4000, -12, 9), rng.uniform(-448, 448, 4000)])
    v = np.concatenate([mids, -mids, fin, rnd])
    v = v[np.abs(v) <= mx.E4M3_MAX]                  # torch gives NaN instead of saturating beyond 464
    v = v.astype(np.float32).astype(np.float64)      # inputs torch sees exactly
    got, ref = mx.e4m3_round(v), torch_e4m3_round(v)
    assert np.array_equal(got, ref)


def test_e4m3_round_saturates_and_keeps_the_sign_of_zero():
    got = mx.e4m3_round(np.array([448.0, 463.9, 464.0, 500.0, 511.9, -480.0, 0.0, -0.0]))
    assert list(got[:6]) == [448.0, 448.0, 448.0, 448.0, 448.0, -448.0]
    assert got[6] == 0 and not np.signbit(got[6]) and np.signbit(got[7])


def test_e4m3_encode_inverts_decode():
    table = torch_e4m3_table()
    codes = np.array([c for c in range(256) if np.isfinite(table[c])], dtype=np.uint8)
    assert np.array_equal(mx.e4m3_encode(table[codes]), codes)


# ----------------------------------------------------------------------------
# the MX block quantiser
# ----------------------------------------------------------------------------
def test_mx_quantize_matches_exhaustive_nearest_search():
    rng = np.random.default_rng(1)
    table = torch_e4m3_table()
    rows = []
    # the fourth range puts every block maximum below 2**-119: the scale clamps at 2**-127
    for lo, hi in [(-3, 3), (-20, -10), (5, 30), (-126, -120), (100, 120)]:
        rows.append(bf16_exact(rng, (2, 64), lo, hi))
    mixed = bf16_exact(rng, (2, 64), -10, 3)
    mixed[0, :32] *= 0.0                              # an all-zero block
    mixed[1, 5] = 2.0 ** 40                           # one large element in a small block
    rows.append(mixed)
    rows = np.concatenate(rows)
    codes, scales = mx.mxfp8_quantize(rows)
    for r in range(rows.shape[0]):
        for b in range(rows.shape[1] // 32):
            blk = rows[r, 32 * b:32 * b + 32]
            amax = np.abs(blk).max()
            s = -127 if amax == 0 else min(max(scale_exponent_by_search(amax), -127), 127)
            assert scales[r, b] == s + 127
            for j in range(32):
                want = nearest_code(blk[j] / 2.0 ** s, table)
                got = int(codes[r, 32 * b + j])
                assert table[got] == table[want], (r, b, j, blk[j], got, want)


def test_mx_round_trip_is_exact_for_representable_blocks():
    rng = np.random.default_rng(2)
    table = torch_e4m3_table()
    fin = np.nonzero(np.isfinite(table) & (table != 0))[0]
    top = np.nonzero(np.isfinite(table) & (np.abs(table) >= 256))[0]   # the top binade: 256..448
    for trial in range(50):
        c = rng.choice(fin, size=32)
        c[rng.integers(32)] = rng.choice(top)          # the block maximum sits in [256, 448]
        s = int(rng.integers(-100, 100))
        blk = table[c] * 2.0 ** s
        codes, scales = mx.mxfp8_quantize(blk[None, :])
        assert scales[0, 0] == s + 127
        assert np.array_equal(codes[0], c.astype(np.uint8))
        assert np.array_equal(mx.mxfp8_dequantize(codes, scales)[0], blk)


def test_mx_zero_block_and_negative_zero():
    rows = np.zeros((1, 64))
    rows[0, 3] = -0.0
    rows[0, 40] = 1.0
    rows[0, 41] = -0.0
    codes, scales = mx.mxfp8_quantize(rows)
    assert scales[0, 0] == 0 and scales[0, 1] == 127 - 8
    assert codes[0, 3] == 0x80 and codes[0, 41] == 0x80 and codes[0, 0] == 0
    assert mx.e4m3_decode(codes[0, 40]) * 2.0 ** (int(scales[0, 1]) - 127) == 1.0


def test_mx_non_finite_block_gets_the_nan_scale_and_leaves_its_neighbours_alone():
    # an infinity or a NaN has no finite power-of-two scale and E8M0 has no
    # infinity: the block's scale is the NaN byte, which makes every element
    # of that block NaN, while the other blocks of the row quantise exactly as
    # they would alone
    rng = np.random.default_rng(31)
    rows = rng.standard_normal((3, 128))
    rows[0, 5] = np.inf
    rows[1, 70] = -np.inf
    rows[2, 100] = np.nan
    codes, scales = mx.mxfp8_quantize(rows)
    bad = {(0, 0), (1, 2), (2, 3)}
    for r in range(3):
        for b in range(4):
            blk = rows[r, 32 * b:32 * b + 32]
            if (r, b) in bad:
                assert scales[r, b] == 0xFF and np.all(codes[r, 32 * b:32 * b + 32] == 0x7F)
                assert np.all(np.isnan(mx.mxfp8_dequantize(codes[r:r + 1, 32 * b:32 * b + 32],
                                                           scales[r:r + 1, b:b + 1])))
            else:
                c1, s1 = mx.mxfp8_quantize(blk[None, :])
                assert scales[r, b] == s1[0, 0] and np.array_equal(codes[r, 32 * b:32 * b + 32], c1[0])


# ----------------------------------------------------------------------------
# the layer
# ----------------------------------------------------------------------------
def dense_mx_layer(L):
    """sum_e g_te * FFN_e(x_t) over ALL experts with the MXFP8 round trips of x and h,
    token by token, through torch (no sort, permutation or combine step)."""
    x = om.bf16_bits_to_f64(L.x_bf16)
    ids, w = om.route(L.router_logits, L.k)
    gate = np.zeros((L.T, L.E))
    for t in range(L.T):
        for j in range(L.k):
            gate[t, ids[t, j]] += w[t, j]
    out = np.zeros((L.T, L.d))
    for t in range(L.T):
        xq = torch.from_numpy(mx.mx_round_trip(x[t:t + 1]))
        for e in range(L.E):
            if gate[t, e] == 0:
                continue
            W13 = torch.from_numpy(om.dequantize_rows(L.w13[e], L.w13_scale[e]))
            W2 = torch.from_numpy(om.dequantize_rows(L.w2[e], L.w2_scale[e]))
            gu = torch.nn.functional.linear(xq, W13)
            h = (torch.nn.functional.silu(gu[:, :L.I]) * gu[:, L.I:]).to(torch.float32).to(torch.bfloat16)
            hq = torch.from_numpy(mx.mx_round_trip(h.to(torch.float64).numpy()))
            out[t] += gate[t, e] * torch.nn.functional.linear(hq, W2)[0].numpy()
    return out


def run_mx(L):
    return mx.forward_mx(L.x_bf16, L.router_logits, L.w13, L.w13_scale, L.w2, L.w2_scale, L.k)


def test_forward_mx_equals_dense_brute_force():
    L = make_layer(T=10, d=64, I=64, E=5, k=2, seed=21)
    got = run_mx(L)["out"]
    ref = dense_mx_layer(L)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_forward_mx_w2_scale_law():
    L = make_layer(T=12, d=64, I=64, E=4, k=2, seed=22)
    a = run_mx(L)["out"]
    L.w2_scale = (L.w2_scale.astype(np.int64) + 1).astype(np.uint8)
    b = run_mx(L)["out"]
    assert np.array_equal(b, 2.0 * a)


def test_forward_mx_stays_near_the_unquantised_layer():
    """E4M3 keeps 4 significant bits: per element a relative error of at most
    2**-4, so the output moves by a few percent at most, and not by nothing."""
    L = make_layer(T=16, d=256, I=128, E=6, k=3, seed=23)
    a = run_mx(L)["out"]
    b = om.forward(L.x_bf16, L.router_logits, L.w13, L.w13_scale, L.w2, L.w2_scale, L.k)["out"]
    rel = np.linalg.norm(a - b) / np.linalg.norm(b)
    assert 1e-3 < rel < 5e-2, rel


def test_forward_mx_operands_are_the_quantised_values():
    L = make_layer(T=8, d=64, I=64, E=3, k=2, seed=24)
    r = run_mx(L)
    x = om.bf16_bits_to_f64(L.x_bf16)
    np.testing.assert_array_equal(mx.mxfp8_dequantize(r["x_codes"], r["x_scales"]), mx.mx_round_trip(x))
    np.testing.assert_array_equal(r["h_q"], mx.mx_round_trip(r["h"]))
    assert np.array_equal(r["h"], om.bf16_round(r["h"]))


# ----------------------------------------------------------------------------
# planted mistakes: each must make at least one pin above fail
# ----------------------------------------------------------------------------
def _fails(test_fn):
    try:
        test_fn()
    except AssertionError:
        return True
    return False


def test_planted_scale_off_by_one_is_caught(monkeypatch):
    monkeypatch.setattr(mx, "E4M3_EMAX", 7)
    assert _fails(test_mx_quantize_matches_exhaustive_nearest_search)
    assert _fails(test_mx_round_trip_is_exact_for_representable_blocks)


def test_planted_round_half_away_is_caught(monkeypatch):
    real = mx.e4m3_round

    def away(v):
        v = np.asarray(v, dtype=np.float64)
        a = np.abs(v)
        out = np.zeros_like(a)
        nz = a > 0
        _, ex = np.frexp(a[nz])
        ulp = np.ldexp(1.0, np.maximum(ex - 1, mx.E4M3_EMIN) - mx.E4M3_MANT)
        out[nz] = np.minimum(np.floor(a[nz] / ulp + 0.5) * ulp, mx.E4M3_MAX)
        return np.copysign(out, v)
    monkeypatch.setattr(mx, "e4m3_round", away)
    assert _fails(test_e4m3_round_matches_torch_conversion)
    monkeypatch.setattr(mx, "e4m3_round", real)


def test_planted_missing_h_quantisation_is_caught(monkeypatch):
    def ffn(x_rows_q, w13_e, w13s_e, w2_e, w2s_e):
        W13 = om.dequantize_rows(w13_e, w13s_e)
        I = W13.shape[0] // 2
        h = om.bf16_round(om.silu(x_rows_q @ W13[:I].T) * (x_rows_q @ W13[I:].T))
        return h, h, h @ om.dequantize_rows(w2_e, w2s_e).T     # wrong: W2 reads h unquantised
    monkeypatch.setattr(mx, "expert_ffn_mx", ffn)
    assert _fails(test_forward_mx_equals_dense_brute_force)


def test_planted_row_wide_scale_is_caught(monkeypatch):
    """one scale per row instead of one per 32-element block"""
    def per_row(rows):
        rows = np.asarray(rows, dtype=np.float64)
        R, K = rows.shape
        amax = np.abs(rows).max(axis=1, keepdims=True)
        _, ex = np.frexp(np.where(amax > 0, amax, 1.0))
        shared = np.clip(np.where(amax > 0, ex - 1 - mx.E4M3_EMAX, -127), -127, 127)
        q = mx.e4m3_round(rows / np.ldexp(1.0, shared))
        return mx.e4m3_encode(q), np.repeat(shared + 127, K // 32, axis=1).astype(np.uint8)
    monkeypatch.setattr(mx, "mxfp8_quantize", per_row)
    assert _fails(test_mx_quantize_matches_exhaustive_nearest_search)
