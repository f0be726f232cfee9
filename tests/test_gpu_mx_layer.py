"""Parity of the block-scaled (MXFP8-activation) layer with its oracle.

moe_fp4_forward_mx runs both projections on kind::mxf8f6f4 tensor cores: the
E2M1 weights and E8M0 scales as stored, x and h quantised to MXFP8 (E4M3,
one E8M0 scale per 32 elements).  The oracle is oracle.mx_activations
(fp64, the same quantisation readings).  Compared here:
* x's MXFP8 codes and scales (sorted-row order): bit-exact;
* h (bf16): equal to the oracle's, or inside the fp32 error model's interval
  (the products are exact on both sides, as in the exact layer);
* h's MXFP8 codes and scales: bit-exact in every block whose 32 h values
  equal the oracle's; elsewhere within the bound that h's interval implies;
* out: relative L2 <= 5e-3, cosine >= 0.9999, max abs <= 2e-2 plus the slack
  of legitimate h rounding decisions passed through the quantiser.
"""
import numpy as np
import pytest

import oracle
from moe_inputs import make_config, make_layer, routing_sample_tokens
from oracle import mx_activations as mxa

from _layer_util import (assert_h_within, assert_out_within_mx, bf16_bits, h_interval_w, mx_hq_bound,
                         to_device)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import fp4_mixture_experts_gb300 as m
    m.load_library()
    return m


def run_mx(moe, L):
    D = to_device(L)
    r = moe.forward_mx(D["x"], D["logits"], D["w13"], D["w13_scale"], D["w2"], D["w2_scale"], L.k,
                       return_operands=True)
    torch.cuda.synchronize()
    return {k: v.cpu() for k, v in r.items()}


def h_bounds_mx(L, ref, experts=None):
    """h_interval of every sorted row (or those of `experts`), from x's MXFP8 values."""
    xq = mxa.mxfp8_dequantize(ref["x_codes"], ref["x_scales"])
    S = L.T * L.k
    lo = np.full((S, L.I), np.nan)
    hi = np.full((S, L.I), np.nan)
    off, ss = ref["expert_offsets"], ref["sorted_slot"]
    for e in range(L.E) if experts is None else experts:
        r0, r1 = int(off[e]), int(off[e + 1])
        if r0 == r1:
            continue
        W13 = oracle.dequantize_rows(L.w13[e], L.w13_scale[e])
        lo[r0:r1], hi[r0:r1] = h_interval_w(xq[ss[r0:r1] // L.k], W13)
    return lo, hi


def check_layer(moe, L, rows=None, what=""):
    """Whole-layer comparison (rows: sorted-row ranges of h to compare, default all)."""
    ref = mxa.forward_mx(L.x_bf16, L.router_logits, L.w13, L.w13_scale, L.w2, L.w2_scale, L.k)
    r = run_mx(moe, L)
    ss = ref["sorted_slot"]
    # x's MXFP8 form, per sorted row: bit-exact
    np.testing.assert_array_equal(r["x_codes"].numpy(), ref["x_codes"][ss // L.k])
    np.testing.assert_array_equal(r["x_scales"].numpy(), ref["x_scales"][ss // L.k])
    lo, hi = h_bounds_mx(L, ref)
    got_h = bf16_bits(r["h"])
    sel = np.arange(L.T * L.k) if rows is None else np.concatenate([np.arange(a, b) for a, b in rows])
    n_diff = assert_h_within(got_h[sel], ref["h"][sel], lo[sel], hi[sel], what)
    check_hq(r, ref, lo, hi, sel, what)
    m, excess = assert_out_within_mx(r["out"].numpy(), ref["out"], L, what=what)
    print(what, m, "h elements rounded the other way:", n_diff, "largest excess over max abs:", excess)
    return m


def check_hq(r, ref, lo, hi, sel, what):
    """h's MXFP8 form: bit-exact where the block's h equals the oracle's,
    else within the bound of h's interval."""
    got_h = oracle.bf16_bits_to_f64(bf16_bits(r["h"])[sel])
    want_h = ref["h"][sel]
    codes, scales = mxa.mxfp8_quantize(want_h)
    R, I = want_h.shape
    same = np.all((got_h == want_h).reshape(R, I // 32, 32), axis=2)
    gc = r["h_codes"].numpy()[sel].reshape(R, I // 32, 32)
    gs = r["h_scales"].numpy()[sel]
    np.testing.assert_array_equal(gc[same], codes.reshape(R, I // 32, 32)[same], err_msg=f"{what}: h codes")
    np.testing.assert_array_equal(gs[same], scales[same], err_msg=f"{what}: h scales")
    if not same.all():
        got_q = mxa.mxfp8_dequantize(r["h_codes"].numpy()[sel], gs)
        want_q = mxa.mxfp8_dequantize(codes, scales)
        bound = mx_hq_bound(lo[sel], hi[sel], want_q)
        assert np.all(np.abs(got_q - want_q) <= bound), f"{what}: h_q beyond its interval's bound"


# ----------------------------------------------------------------------------
def test_mx_tiny(moe):
    check_layer(moe, make_config("tiny"), what="tiny")


@pytest.mark.parametrize("T,d,I,E,k,skew", [
    (700, 512, 256, 8, 2, False),     # ~175 rows an expert: one ragged tile each
    (1500, 384, 384, 6, 2, True),     # skewed: several tiles for the hot experts; d % 256 = 128 (half W2 block)
    (64, 1024, 640, 16, 4, False),    # few rows an expert, I not a multiple of 256
])
def test_mx_ragged_shapes(moe, T, d, I, E, k, skew):
    L = make_layer(T, d, I, E, k, skew=skew, seed=5)
    check_layer(moe, L, what=f"T={T} d={d} I={I} E={E} k={k}")


def test_mx_wide_dynamic_range(moe):
    """E8M0 weight exponents over 24 binades, token rows scaled by powers of
    two from 2^-16 to 2^16 and one all-zero token (all-zero blocks: scale
    byte 0, codes 0): the block scales carry the range, so each token's
    output keeps the usual relative accuracy whatever its magnitude"""
    L = make_layer(T=48, d=1024, I=512, E=6, k=2, exp_lo=-20, exp_hi=3, seed=41)
    rng = np.random.default_rng(41)
    shift = rng.integers(-16, 17, size=L.T)
    x32 = (L.x_bf16.astype(np.uint32) << 16).view(np.float32) * np.ldexp(1.0, shift)[:, None].astype(np.float32)
    x32[5] = 0.0
    L.x_bf16 = (x32.view(np.uint32) >> 16).astype(np.uint16)  # exact: power-of-two scaling of bf16 values
    ref = mxa.forward_mx(L.x_bf16, L.router_logits, L.w13, L.w13_scale, L.w2, L.w2_scale, L.k)
    r = run_mx(moe, L)
    ss = ref["sorted_slot"]
    np.testing.assert_array_equal(r["x_codes"].numpy(), ref["x_codes"][ss // L.k])
    np.testing.assert_array_equal(r["x_scales"].numpy(), ref["x_scales"][ss // L.k])
    lo, hi = h_bounds_mx(L, ref)
    assert_h_within(bf16_bits(r["h"]), ref["h"], lo, hi, "wide range")
    check_hq(r, ref, lo, hi, np.arange(L.T * L.k), "wide range")
    got = r["out"].numpy().astype(np.float64)
    want = ref["out"]
    assert not got[5].any() and not want[5].any()
    for t in range(L.T):
        if t == 5:
            continue
        rel = np.linalg.norm(got[t] - want[t]) / np.linalg.norm(want[t])
        assert rel <= 5e-3, f"token {t} (x scaled by 2^{shift[t]}): relative L2 {rel}"


def test_mx_nonfinite_block_poisons_its_rows(moe):
    """a NaN in one 32-element block of x: that block's scale is 0xFF and its
    codes NaN; the token's rows (h and out) come out NaN, the others match"""
    L = make_layer(40, 256, 128, 4, 2, seed=11)
    L.x_bf16[3, 70] = 0x7FC0
    ref = mxa.forward_mx(L.x_bf16, L.router_logits, L.w13, L.w13_scale, L.w2, L.w2_scale, L.k)
    r = run_mx(moe, L)
    ss = ref["sorted_slot"]
    np.testing.assert_array_equal(r["x_codes"].numpy(), ref["x_codes"][ss // L.k])
    np.testing.assert_array_equal(r["x_scales"].numpy(), ref["x_scales"][ss // L.k])
    assert (r["x_scales"].numpy()[ss // L.k == 3][:, 2] == 0xFF).all()
    out = r["out"].numpy()
    assert np.isnan(out[3]).all()
    keep = np.arange(L.T) != 3
    assert np.isfinite(out[keep]).all()
    m, _ = assert_out_within_mx(out[keep], ref["out"][keep], L, toks=np.nonzero(keep)[0], what="nan block")


def test_mx_prefill_full_size(moe):
    """the prefill workload (T=4608, d=4096, I=2048, E=256, k=8) at full size:
    x's MXFP8 form for all 36,864 rows bit-exact; h and h's MXFP8 form for
    the most and the least loaded expert whole; out for 192 sampled tokens
    (the oracle on those tokens alone: routing is per token)"""
    L = make_config("prefill")
    r = run_mx(moe, L)
    ids, w = oracle.route(L.router_logits, L.k)
    off, ss, _ = oracle.expert_sort(ids, L.E)
    xc, xs = mxa.mxfp8_quantize(oracle.bf16_bits_to_f64(L.x_bf16))
    np.testing.assert_array_equal(r["x_codes"].numpy(), xc[ss // L.k])
    np.testing.assert_array_equal(r["x_scales"].numpy(), xs[ss // L.k])
    counts = np.diff(off)
    xq = mxa.mxfp8_dequantize(xc, xs)
    for e in (int(np.argmax(counts)), int(np.argmin(np.where(counts > 0, counts, 1 << 30)))):
        r0, r1 = int(off[e]), int(off[e + 1])
        xr = xq[ss[r0:r1] // L.k]
        h, hq, _ = mxa.expert_ffn_mx(xr, L.w13[e], L.w13_scale[e], L.w2[e], L.w2_scale[e])
        lo, hi = h_interval_w(xr, oracle.dequantize_rows(L.w13[e], L.w13_scale[e]))
        rr = {"h": r["h"][r0:r1], "h_codes": r["h_codes"][r0:r1], "h_scales": r["h_scales"][r0:r1]}
        assert_h_within(bf16_bits(rr["h"]), h, lo, hi, f"expert {e}")
        check_hq(rr, {"h": h}, lo, hi, np.arange(r1 - r0), f"expert {e}")
    toks = routing_sample_tokens(L.T, 192)
    sub = mxa.forward_mx(L.x_bf16[toks], L.router_logits[toks], L.w13, L.w13_scale, L.w2, L.w2_scale, L.k)
    m, excess = assert_out_within_mx(r["out"].numpy()[toks], sub["out"], L, toks, "prefill")
    print("prefill mx", m, "largest excess over max abs:", excess)


def test_mx_decode_shape(moe):
    """the decode workload's sizes (T=32, d=4096, I=2048, E=256, k=8): about one
    row per expert, so every token tile is the smallest (N = 16) and the
    ragged-tile paths of the block-scaled kernel run on every item"""
    check_layer(moe, make_config("decode"), what="decode shape")


def test_mx_graph_capture_replays_bit_identical(moe):
    """the MXFP8-activation layer allocates nothing and never waits on the
    host, so one call can be captured in a CUDA graph; replays give the eager
    call's output bit for bit"""
    L = make_layer(T=300, d=1024, I=512, E=16, k=4, seed=21)
    D = to_device(L)
    args = (D["x"], D["logits"], D["w13"], D["w13_scale"], D["w2"], D["w2_scale"], L.k)
    ws = torch.empty(moe.mx_workspace_bytes(L.T, L.d, L.I, L.E, L.k), dtype=torch.uint8, device="cuda")
    out = torch.empty(L.T, L.d, dtype=torch.float32, device="cuda")
    eager = moe.forward_mx(*args, workspace=ws).clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        moe.forward_mx(*args, out=out, workspace=ws)
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        moe.forward_mx(*args, out=out, workspace=ws)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eager)
    moe.check(ws)
