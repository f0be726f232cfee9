"""Shared helpers of the parity tests: upload inputs, compare with the oracle."""
import numpy as np

import oracle

# tolerances of the layer output against the fp64 oracle (fp32 accumulation,
# h rounded to bf16 on both sides)
REL_L2 = 5e-3
COSINE = 0.9999
MAX_ABS = 2e-2

# Error model of h on the GPU.  The products x_K * w_K are exact on both
# sides; the GPU adds them in fp32, whose rounding errors (at most half an ulp
# of each partial sum, of random sign) add up like a random walk: for
# recursive summation of K terms the standard deviation is about
# 0.2 * 2^-23 * sqrt(K) * ||x o w||_2, and blocked (MMA) summation is
# smaller.  The model allows H_SUM_ERR * 2^-24 * sqrt(K) * ||x o w||_2 for
# each of g and u, about ten standard deviations.  The fp32 evaluation of
# silu(g) * u with the fast exponential and division (a few ulp each) adds
# at most H_EVAL_ERR of |silu(g) u|.  First-order propagation through
# v = silu(g) u gives the interval of v, and h may be the bf16 rounding of
# any value in it: an element whose exact v lies within that distance of a
# bf16 rounding boundary may come out one bf16 ulp away from the oracle's h,
# and where g or u cancel the interval widens accordingly.  At the bottom of
# the fp32 range the fast SiLU loses its result: for g below about -88,
# exp(-g) overflows and silu(g) evaluates to 0 although its exact value,
# about g e^g, is still a (tiny) fp32 number, and products below the smallest
# normal fp32 are flushed to zero; where |silu(g)| < 2^-119 or |v| < 2^-125
# the interval reaches 0.
H_SUM_ERR = 4.0
H_EVAL_ERR = 2.0 ** -20
SILU_UNDERFLOW = 2.0 ** -119
V_UNDERFLOW = 2.0 ** -125


def to_device(L, dev="cuda:0"):
    import torch
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    return dict(x=t(L.x_bf16.view(np.int16)).view(torch.bfloat16), logits=t(L.router_logits), w13=t(L.w13),
                w13_scale=t(L.w13_scale), w2=t(L.w2), w2_scale=t(L.w2_scale))


def out_metrics(got, want):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    diff = got - want
    nw = np.linalg.norm(want)
    rel = np.linalg.norm(diff) / nw if nw > 0 else np.linalg.norm(diff)
    cos = float(np.dot(got.ravel(), want.ravel()) / (np.linalg.norm(got) * nw)) if nw > 0 else 1.0
    return dict(rel_l2=float(rel), cosine=cos, max_abs=float(np.abs(diff).max()) if diff.size else 0.0)


def assert_out_close(got, want, what=""):
    m = out_metrics(got, want)
    assert m["rel_l2"] <= REL_L2 and m["cosine"] >= COSINE and m["max_abs"] <= MAX_ABS, f"{what}: {m}"
    return m


def bf16_bits(t):
    """torch bf16 tensor -> numpy uint16 bit patterns"""
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def h_interval(x_rows, w13_e, w13s_e):
    """For token rows x_rows (fp64 [m, d]) of one expert: the range of bf16 values
    an fp32 evaluation of h = bf16(silu(g) u) may produce, from the exact g and
    u and the error model above.  Returns (lo, hi), fp64 [m, I]."""
    return h_interval_w(x_rows, oracle.dequantize_rows(w13_e, w13s_e))


def h_interval_w(x_rows, W):
    """h_interval with the expert's dequantised W13 rows W (fp64 [2I, d])."""
    I = W.shape[0] // 2
    K = W.shape[1]
    g = x_rows @ W[:I].T
    u = x_rows @ W[I:].T
    x2 = x_rows * x_rows
    ng = np.sqrt(x2 @ (W[:I] * W[:I]).T)
    nu = np.sqrt(x2 @ (W[I:] * W[I:]).T)
    eg = H_SUM_ERR * 2.0 ** -24 * np.sqrt(K) * ng
    eu = H_SUM_ERR * 2.0 ** -24 * np.sqrt(K) * nu
    with np.errstate(over="ignore", invalid="ignore"):
        sig = 1.0 / (1.0 + np.exp(-g))
        silu = g * sig
        dsilu = sig * (1.0 + g * (1.0 - sig))
        v = silu * u
        dv = np.abs(dsilu * u) * eg + np.abs(silu) * eu + H_EVAL_ERR * np.abs(v)
    dv = np.nan_to_num(dv, nan=np.inf)
    under = (np.abs(silu) < SILU_UNDERFLOW) | (np.abs(v) < V_UNDERFLOW)
    dv = np.where(under, np.maximum(dv, np.abs(v)), dv)
    return oracle.bf16_round(v - dv), oracle.bf16_round(v + dv)


def h_bounds_sorted(L, ref, rows=None):
    """h_interval for the sorted rows of a layer (all rows, or the sorted-row
    ranges [r0, r1) listed in `rows`), expert by expert."""
    x = oracle.bf16_bits_to_f64(L.x_bf16)
    S = L.T * L.k
    lo = np.full((S, L.I), np.nan)
    hi = np.full((S, L.I), np.nan)
    off, ss = ref["expert_offsets"], ref["sorted_slot"]
    for e in range(L.E):
        r0, r1 = int(off[e]), int(off[e + 1])
        if r0 == r1 or (rows is not None and not any(a <= r0 and r1 <= b for a, b in rows)):
            continue
        lo[r0:r1], hi[r0:r1] = h_interval(x[ss[r0:r1] // L.k], L.w13[e], L.w13_scale[e])
    return lo, hi


def assert_h_within(got_bits, want, lo, hi, what=""):
    """h from the GPU (bf16 bits) against the oracle's h: equal, or (where the
    fp32 sums lie near a bf16 rounding boundary, or g or u cancel) a bf16
    value inside the error model's interval [lo, hi].  Returns the number of
    elements that differ from the oracle."""
    got = oracle.bf16_bits_to_f64(got_bits)
    mism = got != want
    if mism.any():
        ok = (got[mism] >= lo[mism]) & (got[mism] <= hi[mism])
        assert ok.all(), (f"{what}: h outside the error model at {np.argwhere(mism)[~ok][:4].tolist()}: "
                          f"got {got[mism][~ok][:4]}, want {want[mism][~ok][:4]}, "
                          f"interval {lo[mism][~ok][:4]} .. {hi[mism][~ok][:4]}")
    return int(mism.sum())


def assert_out_within(got, want, L, toks=None, what=""):
    """out from the GPU against the oracle's out (rows `toks` of the layer, or
    all): relative L2 and cosine over the whole array, and every element
    within MAX_ABS plus the slack that legitimate h rounding decisions imply.

    Where an exact h value lies within fp32 error of a bf16 rounding boundary
    the kernel may round it the other way (h_interval); one bf16 ulp of a large
    h (ulp 1 at |h| >= 128) times a W2 weight (up to 6 * 2^-5) times the
    routing weight moves out by several 1e-2.  For every token with an element
    beyond MAX_ABS the slack is sum_j w_tj sum_i dh_i |W2_e[n, i]|, with dh the
    distance from the oracle's h to the far end of its interval: computed from
    the oracle's own values only.  Returns the metrics and the largest excess
    over MAX_ABS that the slack had to cover."""
    m = out_metrics(got, want)
    assert m["rel_l2"] <= REL_L2 and m["cosine"] >= COSINE, f"{what}: {m}"
    got = np.asarray(got, dtype=np.float64)
    toks = np.arange(L.T) if toks is None else np.asarray(toks)
    diff = np.abs(got - want)
    bad = np.nonzero((diff > MAX_ABS).any(axis=1))[0]
    if bad.size == 0:
        return m, 0.0
    x = oracle.bf16_bits_to_f64(L.x_bf16)
    ids, w = oracle.route(L.router_logits[toks[bad]], L.k)
    slack = np.zeros((bad.size, L.d))
    for e in np.unique(ids):
        rows, slots = np.nonzero(ids == e)
        xr = x[toks[bad][rows]]
        W13 = oracle.dequantize_rows(L.w13[e], L.w13_scale[e])
        lo, hi = h_interval_w(xr, W13)
        h, _ = oracle.expert_ffn(xr, L.w13[e], L.w13_scale[e], L.w2[e], L.w2_scale[e])
        dh = np.maximum(hi - h, h - lo)
        W2 = np.abs(oracle.dequantize_rows(L.w2[e], L.w2_scale[e]))
        slack[rows] += w[rows, slots][:, None] * (dh @ W2.T)
    excess = diff[bad] - MAX_ABS
    ok = excess <= slack * (1 + 1e-6)
    assert ok.all(), (f"{what}: out beyond MAX_ABS + h-rounding slack at token {toks[bad][np.nonzero(~ok)[0][:4]]}: "
                      f"excess {excess[~ok][:4]}, slack {slack[~ok][:4]}")
    m["tokens_beyond_max_abs"] = int(bad.size)
    return m, float(excess.max())


def mx_hq_bound(lo, hi, hq):
    """Per element, the largest distance between the oracle's MXFP8 h_q (fp64
    values [R, I]) and the MXFP8 form of any h' with lo <= h' <= hi (the bf16
    values the error model allows for h, h_interval).

    A block whose 32 intervals are single points has one MXFP8 form: 0.  Else
    the block's scale exponent floor(log2 amax') - 8 ranges over the binades
    of amax' in [amax_min, amax_max], and for each scale X the rounding
    RN(h'/X) X is monotone in h', so its extremes are those of lo and hi; if
    every interval holds 0 the block may also be all zero (any scale), and
    |q(h')| <= 2 |h'| covers every scale."""
    from oracle.mx_activations import E4M3_EMAX, e4m3_round
    R, I = lo.shape
    nb = I // 32
    lo3, hi3, hq3 = (np.asarray(a, dtype=np.float64).reshape(R, nb, 32) for a in (lo, hi, hq))
    out = np.zeros((R, nb, 32))
    wide = np.any(lo3 != hi3, axis=2)
    if not wide.any():
        return out.reshape(R, I)
    L, H, Q = lo3[wide], hi3[wide], hq3[wide]
    mag_min = np.where((L <= 0) & (H >= 0), 0.0, np.minimum(np.abs(L), np.abs(H)))
    mag_max = np.maximum(np.abs(L), np.abs(H))
    amin, amax = mag_min.max(axis=1), mag_max.max(axis=1)
    ex = lambda a: np.frexp(np.where(a > 0, a, 1.0))[1] - 1
    e_hi = ex(amax)
    e_lo = np.where(amin > 0, ex(amin), e_hi)
    dev = np.zeros_like(L)
    for o in range(int((e_hi - e_lo).max()) + 1):
        e = np.minimum(e_lo + o, e_hi)
        X = np.ldexp(1.0, np.clip(e - E4M3_EMAX, -127, 127))[:, None]
        qlo = e4m3_round(L / X) * X
        qhi = e4m3_round(H / X) * X
        dev = np.maximum(dev, np.maximum(np.abs(qlo - Q), np.abs(qhi - Q)))
    zero_ok = (amin == 0)[:, None]
    dev = np.where(zero_ok, np.maximum(dev, np.abs(Q) + 2.0 * mag_max.max(axis=1, keepdims=True)), dev)
    out[wide] = dev
    return out.reshape(R, I)


def assert_out_within_mx(got, want, L, toks=None, what=""):
    """out of the MXFP8 layer against the oracle's (oracle.mx_activations):
    relative L2 and cosine over the whole array; every element within MAX_ABS
    plus the slack of legitimate h rounding decisions, which here reach the
    W2 operand through its MXFP8 form: sum_j w_tj sum_i dq_i |W2_e[n, i]| with
    dq = mx_hq_bound of h's interval (computed from the oracle's values
    only).  Returns the metrics and the largest excess over MAX_ABS."""
    from oracle import mx_activations as mxa
    m = out_metrics(got, want)
    assert m["rel_l2"] <= REL_L2 and m["cosine"] >= COSINE, f"{what}: {m}"
    got = np.asarray(got, dtype=np.float64)
    toks = np.arange(L.T) if toks is None else np.asarray(toks)
    diff = np.abs(got - want)
    bad = np.nonzero((diff > MAX_ABS).any(axis=1))[0]
    if bad.size == 0:
        return m, 0.0
    xq = mxa.mx_round_trip(oracle.bf16_bits_to_f64(L.x_bf16[toks[bad]]))
    ids, w = oracle.route(L.router_logits[toks[bad]], L.k)
    slack = np.zeros((bad.size, L.d))
    for e in np.unique(ids):
        rows, slots = np.nonzero(ids == e)
        W13 = oracle.dequantize_rows(L.w13[e], L.w13_scale[e])
        lo, hi = h_interval_w(xq[rows], W13)
        _, hq, _ = mxa.expert_ffn_mx(xq[rows], L.w13[e], L.w13_scale[e], L.w2[e], L.w2_scale[e])
        dq = mx_hq_bound(lo, hi, hq)
        W2 = np.abs(oracle.dequantize_rows(L.w2[e], L.w2_scale[e]))
        slack[rows] += w[rows, slots][:, None] * (dq @ W2.T)
    excess = diff[bad] - MAX_ABS
    ok = excess <= slack * (1 + 1e-6)
    assert ok.all(), (f"{what}: out beyond MAX_ABS + h-rounding slack at token {toks[bad][np.nonzero(~ok)[0][:4]]}: "
                      f"excess {excess[~ok][:4]}, slack {slack[~ok][:4]}")
    m["tokens_beyond_max_abs"] = int(bad.size)
    return m, float(excess.max())
