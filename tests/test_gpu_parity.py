"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Routing ids, the expert permutation, the offsets and their FNV-1a hash must
be bit-exact; routing weights agree to fp32 rounding; h agrees up to rare
one-ulp bf16 flips (fp32 vs fp64 sums before the rounding); out must reach
relative L2 <= 5e-3, cosine >= 0.9999 and max abs <= 2e-2.
"""
import numpy as np
import pytest

import oracle
from moe_inputs import make_config, make_layer, routing_sample_tokens

from _layer_util import (assert_h_within, assert_out_close, assert_out_within, bf16_bits, h_bounds_sorted,
                         h_interval, out_metrics, to_device)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

GEMV = 0x1
TC = 0x2
PERSIST = 0x4
PAIRS = TC | 0x8
DET = 0x10  # the combine in slot order: bitwise reproducible


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import fp4_mixture_experts_gb300 as m
    m.load_library()
    return m


def run_gpu(moe, L, flags=0, return_h=True):
    D = to_device(L)
    r = moe.forward(D["x"], D["logits"], D["w13"], D["w13_scale"], D["w2"], D["w2_scale"], L.k, flags=flags,
                    return_routing=True, return_h=return_h)
    torch.cuda.synchronize()
    return {k: v for k, v in r.items()}


def check_routing(r, ref):
    ids = r["topk_ids"].cpu().numpy()
    ss = r["sorted_slot"].cpu().numpy()
    off = r["expert_offsets"].cpu().numpy()
    np.testing.assert_array_equal(ids, ref["topk_ids"])
    np.testing.assert_array_equal(off, ref["expert_offsets"])
    np.testing.assert_array_equal(ss, ref["sorted_slot"])
    assert oracle.route_hash(ids, ss, off) == oracle.route_hash(ref["topk_ids"], ref["sorted_slot"],
                                                                ref["expert_offsets"])
    np.testing.assert_allclose(r["topk_weights"].cpu().numpy(), ref["topk_w"], rtol=2e-6, atol=1e-7)


def check_h(r, ref, L, rows=None):
    """h equal to the oracle's, or a bf16 value the fp32 error model allows
    (see _layer_util.h_interval); `rows`: only these sorted-row ranges."""
    lo, hi = h_bounds_sorted(L, ref, rows)
    got = bf16_bits(r["h"])
    want = ref["h"]
    if rows is not None:
        sel = np.concatenate([np.arange(a, b) for a, b in rows])
        got, want, lo, hi = got[sel], want[sel], lo[sel], hi[sel]
    return assert_h_within(got, want, lo, hi)


def full_check(moe, L, flags=0):
    ref = oracle.forward(L.x_bf16, L.router_logits, L.w13, L.w13_scale, L.w2, L.w2_scale, L.k)
    r = run_gpu(moe, L, flags)
    check_routing(r, ref)
    check_h(r, ref, L)
    return assert_out_close(r["out"].cpu().numpy(), ref["out"], f"flags={flags}")


# ----------------------------------------------------------------------------
def test_tiny_config(moe):
    full_check(moe, make_config("tiny"))


@pytest.mark.parametrize("flags", [GEMV, TC, GEMV | PERSIST, PAIRS])
def test_several_tiles_ragged(moe, flags):
    # 300 tokens x 4 slots over 16 experts: ~75 rows per expert, ragged chunk and tile tails
    L = make_layer(T=300, d=1024, I=1024, E=16, k=4, seed=3)
    full_check(moe, L, flags)


@pytest.mark.parametrize("flags", [0, TC, PAIRS])
def test_non_1024_multiples(moe, flags):
    L = make_layer(T=37, d=384, I=640, E=12, k=3, seed=4)
    full_check(moe, L, flags)


@pytest.mark.parametrize("flags", [GEMV, TC])
def test_single_token(moe, flags):
    full_check(moe, make_layer(T=1, d=1024, I=1024, E=8, k=2, seed=5), flags)


@pytest.mark.parametrize("flags", [GEMV, TC, GEMV | DET, TC | DET])
def test_against_the_cpp_oracle(moe, flags):
    """The same checks against the second CPU oracle (plain C++ loops)"""
    from oracle import cpp_ref
    L = make_layer(T=24, d=1024, I=1024, E=12, k=3, seed=36)
    ref = cpp_ref.forward(L.x_bf16, L.router_logits, L.w13, L.w13_scale, L.w2, L.w2_scale, L.k)
    ref["slot_pos"] = np.argsort(ref["sorted_slot"]).astype(np.int32)
    r = run_gpu(moe, L, flags)
    check_routing(r, ref)
    check_h(r, ref, L)
    assert_out_within(r["out"].cpu().numpy(), ref["out"], L, what=f"C++ oracle, flags={flags}")


@pytest.mark.parametrize("flags", [GEMV, TC])
def test_top1_and_single_expert(moe, flags):
    full_check(moe, make_layer(T=20, d=1024, I=1024, E=6, k=1, seed=6), flags)
    full_check(moe, make_layer(T=20, d=1024, I=1024, E=1, k=1, seed=7), flags)


@pytest.mark.parametrize("flags", [GEMV, TC])
def test_all_tokens_one_expert_and_empty_experts(moe, flags):
    L = make_layer(T=70, d=1024, I=1024, E=32, k=2, seed=8)
    L.router_logits[:, 5] += 50.0     # expert 5 first for every token
    L.router_logits[:, 9] += 40.0     # expert 9 second
    full_check(moe, L, flags)


def test_ties_and_signed_zero(moe):
    L = make_layer(T=40, d=1024, I=1024, E=16, k=4, seed=9)
    L.router_logits[:10] = 0.0
    L.router_logits[10:20, ::2] = 1.5
    L.router_logits[20:30] = np.where(np.arange(16) % 2, -0.0, 0.0).astype(np.float32)
    full_check(moe, L)


def test_k_equals_E(moe):
    full_check(moe, make_layer(T=9, d=1024, I=1024, E=5, k=5, seed=10), GEMV)
    full_check(moe, make_layer(T=9, d=256, I=256, E=5, k=5, seed=10), TC)


@pytest.mark.parametrize("flags", [GEMV, TC, PAIRS])
def test_w2_layout_probe(moe, flags):
    """A single nonzero W2 code must land on its own output column only."""
    L = make_layer(T=24, d=1024, I=1024, E=4, k=2, seed=11)
    e_star, n0, m0 = 1, 517, 301
    L.w2[:] = 0
    L.w2[e_star, n0, m0 // 2] = 0x50
    r = run_gpu(moe, L, flags)
    ref = oracle.forward(L.x_bf16, L.router_logits, L.w13, L.w13_scale, L.w2, L.w2_scale, L.k)
    out = r["out"].cpu().numpy()
    assert set(np.nonzero(np.abs(out).sum(0))[0].tolist()) <= {n0}
    assert_out_close(out, ref["out"], "w2 probe")


@pytest.mark.parametrize("flags", [GEMV, TC, PAIRS])
def test_w13_nibble_and_gate_up_probe(moe, flags):
    L = make_layer(T=12, d=1024, I=1024, E=2, k=1, seed=12)
    L.w13[:] = 0
    L.w13[:, 7, 100] = 0x04        # gate row 7, K=200 (low nibble): 2.0
    L.w13[:, 1024 + 7, 100] = 0xB0  # up row 7, K=201 (high nibble): -1.5
    L.w13[:, 1024 + 9, 33] = 0x22   # up row 9 only: h must stay 0 (silu(0) = 0)
    r = run_gpu(moe, L, flags)
    ref = oracle.forward(L.x_bf16, L.router_logits, L.w13, L.w13_scale, L.w2, L.w2_scale, L.k)
    check_h(r, ref, L)
    h = oracle.bf16_bits_to_f64(bf16_bits(r["h"]))
    assert not np.delete(h, 7, axis=1).any()


def test_zero_codes_give_zero(moe):
    L = make_layer(T=16, d=1024, I=1024, E=4, k=2, seed=13)
    L.w2[:] = 0x88
    for flags in (GEMV, TC):
        r = run_gpu(moe, L, flags)
        assert not r["out"].cpu().numpy().any()


def test_run_twice_bit_identical(moe):
    L = make_layer(T=200, d=1024, I=1024, E=16, k=4, seed=14)
    for flags in (GEMV | DET, TC | DET, PAIRS):
        a = run_gpu(moe, L, flags)["out"].cpu().numpy()
        b = run_gpu(moe, L, flags)["out"].cpu().numpy()
        assert np.array_equal(a, b)


@pytest.mark.parametrize("shape", [dict(T=200, d=1024, I=1024, E=16, k=4, seed=14),
                                   dict(T=32, d=4096, I=2048, E=256, k=8, seed=0),
                                   dict(T=77, d=384, I=640, E=12, k=3, seed=35)])
def test_epilogue_combine_matches_slot_order_combine(moe, shape):
    """The default combine (atomic adds in the W2 epilogue, in no fixed order)
    against the slot-order pass: the same k fp32 terms per element summed in
    another order, so equal up to fp32 rounding of the partial sums; h and the
    routing are bitwise the same."""
    L = make_layer(**shape)
    for flags in (GEMV, TC, GEMV | PERSIST):
        if flags & GEMV and (L.d % 1024 or L.I % 1024):
            continue
        a = run_gpu(moe, L, flags)
        b = run_gpu(moe, L, flags | DET)
        assert torch.equal(a["h"], b["h"]) and torch.equal(a["sorted_slot"], b["sorted_slot"])
        x, y = a["out"].cpu().numpy().astype(np.float64), b["out"].cpu().numpy().astype(np.float64)
        # the epilogue adds up to 2k fp32 terms per element (the streaming
        # kernel's two K halves of each slot separately), each rounded at 2^-24
        # like every partial sum: bound the difference by 4 k 2^-24 times the
        # terms' magnitude, taken as k max|out| of the token
        scale = np.abs(y).max(axis=1, keepdims=True) + 1e-30
        assert (np.abs(x - y) <= 4 * L.k * L.k * 2.0 ** -24 * scale).all(), f"flags {flags}"
        assert np.linalg.norm(x - y) <= 1e-6 * np.linalg.norm(y), f"flags {flags}"


def test_route_entry_point(moe):
    L = make_layer(T=333, d=128, I=128, E=64, k=6, seed=15)
    ids, w, off, ss = moe.route(torch.from_numpy(L.router_logits).cuda(), L.k)
    torch.cuda.synchronize()
    ref_ids, ref_w = oracle.route(L.router_logits, L.k)
    ref_off, ref_ss, _ = oracle.expert_sort(ref_ids, L.E)
    np.testing.assert_array_equal(ids.cpu().numpy(), ref_ids)
    np.testing.assert_array_equal(off.cpu().numpy(), ref_off)
    np.testing.assert_array_equal(ss.cpu().numpy(), ref_ss)
    np.testing.assert_allclose(w.cpu().numpy(), ref_w, rtol=2e-6, atol=1e-7)


@pytest.mark.parametrize("T,E,k", [(32, 1024, 32), (17, 300, 7), (1, 1000, 3), (32, 257, 8), (5, 8, 8),
                                   (100, 1024, 32), (77, 8, 3), (70, 1000, 5), (64, 512, 8)])
def test_route_wide_expert_counts(moe, T, E, k):
    """both routing paths (T <= 32: one cluster; T > 32: three kernels) over
    expert counts and k beyond the layer configs, with ties on every third token"""
    L = make_layer(T=T, d=32, I=32, E=E, k=k, seed=T * 7 + E + k)
    logits = L.router_logits.copy()
    logits[::3] = np.round(logits[::3] * 2.0) / 2.0
    ids, w, off, ss = moe.route(torch.from_numpy(logits).cuda(), k)
    torch.cuda.synchronize()
    ref_ids, ref_w = oracle.route(logits, k)
    ref_off, ref_ss, _ = oracle.expert_sort(ref_ids, E)
    np.testing.assert_array_equal(ids.cpu().numpy(), ref_ids)
    np.testing.assert_array_equal(off.cpu().numpy(), ref_off)
    np.testing.assert_array_equal(ss.cpu().numpy(), ref_ss)
    np.testing.assert_allclose(w.cpu().numpy(), ref_w, rtol=2e-6, atol=1e-7)


@pytest.mark.parametrize("flags", [GEMV, TC])
def test_small_batch_many_experts_forward(moe, flags):
    """T <= 32 routing with E > 256 (work lists for many sparse experts)"""
    full_check(moe, make_layer(T=32, d=1024, I=1024, E=300, k=2, seed=51), flags)


def test_forward_host_matches_forward(moe):
    L = make_layer(T=40, d=1024, I=1024, E=16, k=4, seed=16)
    D = to_device(L)
    dev_out = moe.forward(D["x"], D["logits"], D["w13"], D["w13_scale"], D["w2"], D["w2_scale"], L.k, flags=DET)
    xh = torch.from_numpy(L.x_bf16.view(np.int16)).view(torch.bfloat16).pin_memory()
    lh = torch.from_numpy(L.router_logits).pin_memory()
    host_out = moe.forward_host(xh, lh, D["w13"], D["w13_scale"], D["w2"], D["w2_scale"], L.k, flags=DET)
    torch.cuda.synchronize()
    assert np.array_equal(host_out.numpy(), dev_out.cpu().numpy())
    # pinned logits and out are used in place, pageable ones go through device staging: the
    # same result either way, and for each mix of the two
    xp = torch.from_numpy(L.x_bf16.view(np.int16).copy()).view(torch.bfloat16)
    lp = torch.from_numpy(L.router_logits.copy())
    for x_, l_, pinned_out in ((xp, lp, False), (xh, lp, True), (xp, lh, False), (xh, lh, True)):
        o_ = torch.full((L.T, L.d), float("nan"), dtype=torch.float32)
        if pinned_out:
            o_ = o_.pin_memory()
        moe.forward_host(x_, l_, D["w13"], D["w13_scale"], D["w2"], D["w2_scale"], L.k, out_host=o_, flags=DET)
        assert np.array_equal(o_.numpy(), dev_out.cpu().numpy())
        # the default combine: pinned out is written by the slot-order pass
        # (bitwise the same), pageable out through the epilogue combine
        o_.fill_(float("nan"))
        moe.forward_host(x_, l_, D["w13"], D["w13_scale"], D["w2"], D["w2_scale"], L.k, out_host=o_)
        if pinned_out:
            assert np.array_equal(o_.numpy(), dev_out.cpu().numpy())
        else:
            x_o, y_o = o_.numpy().astype(np.float64), dev_out.cpu().numpy().astype(np.float64)
            scale = np.abs(y_o).max(axis=1, keepdims=True)
            assert (np.abs(x_o - y_o) <= 4 * L.k * L.k * 2.0 ** -24 * scale).all()


def test_check_reports_clean_workspace(moe):
    L = make_layer(T=16, d=1024, I=1024, E=4, k=2, seed=17)
    D = to_device(L)
    ws = torch.empty(moe.workspace_bytes(L.T, L.d, L.I, L.E, L.k), dtype=torch.uint8, device="cuda")
    moe.forward(D["x"], D["logits"], D["w13"], D["w13_scale"], D["w2"], D["w2_scale"], L.k, workspace=ws)
    moe.check(ws)


# ----------------------------------------------------------------------------
# the five named workloads at full size
# ----------------------------------------------------------------------------
def test_decode_config_full(moe):
    L = make_config("decode")
    m = full_check(moe, L)
    print("decode", m)


@pytest.mark.parametrize("shape", [dict(T=32, d=4096, I=2048, E=256, k=8, seed=0),
                                   dict(T=3, d=7168, I=2048, E=16, k=2, seed=33),
                                   dict(T=29, d=1024, I=3072, E=64, k=6, seed=34)])
def test_persistent_decode_is_bit_identical_to_two_launches(moe, shape):
    """the single-launch decode layer (W13, grid-wide arrival counter, W2)
    runs the same arithmetic in the same order as the two launches"""
    L = make_layer(**shape)
    a = run_gpu(moe, L, GEMV | DET)
    b = run_gpu(moe, L, GEMV | PERSIST | DET)
    assert torch.equal(a["h"], b["h"]) and torch.equal(a["out"], b["out"])


@pytest.mark.parametrize("name,flags", [("prefill", 0), ("skewed", 0), ("skewed", PAIRS)])
def test_full_size_every_token(moe, name, flags):
    """the prefill and skewed workloads, whole: routing bit-exact, every h
    element and every out element against the oracle (the default path, the
    tensor-core kernels, with the launch configuration the benchmark times)"""
    L = make_config(name)
    r = run_gpu(moe, L, flags)
    ref = oracle.forward(L.x_bf16, L.router_logits, L.w13, L.w13_scale, L.w2, L.w2_scale, L.k)
    check_routing(r, ref)
    n_diff = check_h(r, ref, L)
    m, excess = assert_out_within(r["out"].cpu().numpy(), ref["out"], L, what=name)
    print(name, m, "h elements rounded the other way:", n_diff, "largest excess over max abs:", excess)


def large_picks(counts):
    """experts of the large workload to compare whole: the most and the least
    loaded, and ones whose row counts leave ragged tiles (token tiles of up to
    192 rows, split evenly and padded to 16; 64-row token boxes)"""
    nz = np.nonzero(counts)[0]
    picks = [int(nz[np.argmax(counts[nz])]), int(nz[np.argmin(counts[nz])])]
    for cond in (lambda c: c % 16 != 0, lambda c: c % 64 not in (0, 16, 32, 48) or c % 192 > 128,
                 lambda c: c % 192 != 0 and c % 192 < 16):
        for e in nz:
            if cond(int(counts[e])) and int(e) not in picks:
                picks.append(int(e))
                break
    return picks


def test_large_config_whole_experts_and_their_tokens(moe):
    """the large workload (d = 7168, 131,072 slots): routing bit-exact; every
    h row of a handful of whole experts; out for every token routed to those
    experts plus 256 more tokens, against the oracle token by token"""
    L = make_config("large")
    r = run_gpu(moe, L)
    ids, w = oracle.route(L.router_logits, L.k)
    off, ss, _ = oracle.expert_sort(ids, L.E)
    check_routing(r, dict(topk_ids=ids, topk_w=w, expert_offsets=off, sorted_slot=ss))
    picks = large_picks(np.diff(off))
    x = oracle.bf16_bits_to_f64(L.x_bf16)
    got_h = bf16_bits(r["h"])
    toks = set()
    for e in picks:
        r0, r1 = int(off[e]), int(off[e + 1])
        tok = ss[r0:r1] // L.k
        toks.update(tok.tolist())
        h_ref, _ = oracle.expert_ffn(x[tok], L.w13[e], L.w13_scale[e], L.w2[e], L.w2_scale[e])
        lo, hi = h_interval(x[tok], L.w13[e], L.w13_scale[e])
        assert_h_within(got_h[r0:r1], h_ref, lo, hi, f"expert {e} ({r1 - r0} rows)")
    toks.update(routing_sample_tokens(L.T, 256).tolist())
    toks = np.array(sorted(toks), dtype=np.int64)
    _, _, want = oracle.forward_tokens(L.x_bf16, L.router_logits, L.w13, L.w13_scale, L.w2, L.w2_scale, L.k, toks)
    got = r["out"][torch.from_numpy(toks).cuda()].cpu().numpy()
    m, excess = assert_out_within(got, want, L, toks, "large")
    print("large", picks, len(toks), "tokens", m, "largest excess over max abs:", excess)


def test_d7168_streaming_path(moe):
    """the decode (streaming) path at the large layer's d = 7168 (3-deep ring)"""
    full_check(moe, make_layer(T=12, d=7168, I=2048, E=12, k=2, exp_lo=-8, exp_hi=-6, seed=31), GEMV)


@pytest.mark.parametrize("d,I", [(8192, 1024), (1024, 9216)])
def test_streaming_path_beyond_7168(moe, d, I):
    """d or I above 7168 on the streaming path: the activations of 8 tokens no
    longer fit next to the weight ring, so the CUDA-core row kernels
    (w13_swiglu_rows, w2_rows) run instead; they must match the oracle too"""
    full_check(moe, make_layer(T=8, d=d, I=I, E=8, k=2, seed=d + I), GEMV)


def test_routing_block_boundary(moe):
    """T = 32 runs the one-cluster routing kernel, T = 33 the three-kernel one"""
    for T in (32, 33):
        full_check(moe, make_layer(T=T, d=1024, I=1024, E=64, k=8, seed=32 + T))


@pytest.mark.parametrize("flags", [GEMV, TC, PAIRS])
def test_wide_dynamic_range(moe, flags):
    # E8M0 exponents spread over 24 binades inside every weight row, token rows
    # scaled by powers of two from 2^-16 to 2^16 and one all-zero token: every
    # power-of-two rescaling on the path (weight rows against their largest
    # block scale, x rows, h rows) must stay exact, so each token's output keeps
    # the usual relative accuracy whatever its magnitude
    L = make_layer(T=48, d=1024, I=1024, E=6, k=2, exp_lo=-20, exp_hi=3, seed=41)
    rng = np.random.default_rng(41)
    shift = rng.integers(-16, 17, size=L.T)
    x32 = (L.x_bf16.astype(np.uint32) << 16).view(np.float32) * np.ldexp(1.0, shift)[:, None].astype(np.float32)
    x32[5] = 0.0
    L.x_bf16 = (x32.view(np.uint32) >> 16).astype(np.uint16)  # exact: power-of-two scaling of bf16 values
    ref = oracle.forward(L.x_bf16, L.router_logits, L.w13, L.w13_scale, L.w2, L.w2_scale, L.k)
    r = run_gpu(moe, L, flags)
    check_routing(r, ref)
    # blocks 2^23 apart in scale cancel more in the fp32 sums than the usual
    # workloads do: the error model's interval, computed from each element's
    # own g, u and magnitude sums, covers it
    check_h(r, ref, L)
    got = r["out"].cpu().numpy().astype(np.float64)
    want = ref["out"]
    assert not got[5].any() and not want[5].any()
    for t in range(L.T):
        if t == 5:
            continue
        rel = np.linalg.norm(got[t] - want[t]) / np.linalg.norm(want[t])
        assert rel <= 5e-3, f"token {t} (x scaled by 2^{shift[t]}): relative L2 {rel}"


@pytest.mark.parametrize("flags", [GEMV | DET, TC | DET, GEMV | PERSIST | DET, PAIRS, GEMV, TC])
def test_cuda_graph_capture_replays_bit_identical(moe, flags):
    # the layer call allocates nothing and never waits on the host, so it can
    # be captured in a CUDA graph; replays recompute everything from the inputs
    L = make_layer(T=40, d=1024, I=1024, E=16, k=4, seed=42)
    D = to_device(L)
    ws = torch.empty(moe.workspace_bytes(L.T, L.d, L.I, L.E, L.k), dtype=torch.uint8, device="cuda")
    out = torch.empty(L.T, L.d, dtype=torch.float32, device="cuda")
    args = (D["x"], D["logits"], D["w13"], D["w13_scale"], D["w2"], D["w2_scale"], L.k)
    moe.forward(*args, out=out, workspace=ws, flags=flags)
    torch.cuda.synchronize()
    eager = out.clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        moe.forward(*args, out=out, workspace=ws, flags=flags)
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        moe.forward(*args, out=out, workspace=ws, flags=flags)
    out.fill_(float("nan"))
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    moe.check(ws)
    if flags & DET or flags == PAIRS:
        assert torch.equal(out, eager)
    else:
        # the epilogue combine zeroes out inside the graph and adds the k terms
        # in no fixed order: each replay gives the layer once, up to fp32 rounding
        x, y = out.cpu().numpy().astype(np.float64), eager.cpu().numpy().astype(np.float64)
        scale = np.abs(y).max(axis=1, keepdims=True)
        assert (np.abs(x - y) <= 4 * L.k * L.k * 2.0 ** -24 * scale).all()
