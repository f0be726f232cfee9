"""Parity of the router projection (moe_fp4_router, moe_fp4_forward_gated,
through the C ABI) with the oracle (oracle/router.py).

The logits are fp32 sums of exact bf16 x bf16 products: each must lie within
the fp32 accumulation bound 4 * 2^-24 * sqrt(d) * ||x o w||_2 of the exact
logit (the random-walk model of the h checks).  The top-k is an integer
decision taken on fp32 values: where a token's exact logits leave no near-tie
(every gap in its top k + 1 larger than both values' uncertainty), the GPU
must pick the oracle's experts in the oracle's order; elsewhere its choice
must be a valid one for logits within that uncertainty.  The layer output of
the gated forward is then compared token by token where the routing agrees.
"""
import numpy as np
import pytest

import oracle
from oracle import router as orr
from moe_inputs import make_config, make_gate_weights, make_layer

from _layer_util import assert_out_within, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ERR = 4.0


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import fp4_mixture_experts_gb300 as m
    m.load_library()
    return m


def logit_bound(x_bf16, wg_bf16):
    x = oracle.bf16_bits_to_f64(x_bf16)
    w = oracle.bf16_bits_to_f64(wg_bf16)
    return ERR * 2.0 ** -24 * np.sqrt(x.shape[1]) * np.sqrt((x * x) @ (w * w).T)


def dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def check_logits(got, x_bf16, wg_bf16):
    exact = orr.router_logits(x_bf16, wg_bf16)
    b = logit_bound(x_bf16, wg_bf16)
    err = np.abs(got.astype(np.float64) - exact)
    assert np.all(err <= b), f"logits beyond the fp32 bound: worst {np.max(err / np.maximum(b, 1e-300))}x"
    return exact, b


def routing_verdicts(gpu_ids, exact, b, k):
    """per token: True where the decision is robust (then it must equal the
    oracle's), and checks that every GPU choice is valid for logits within the
    uncertainty u = b + one fp32 ulp."""
    u = b + np.spacing(np.abs(exact).astype(np.float32)).astype(np.float64)
    ref_ids, _ = oracle.route(exact.astype(np.float32), k)
    robust = np.ones(len(exact), dtype=bool)
    for t in range(len(exact)):
        order = list(ref_ids[t])
        rest = [e for e in np.argsort(-exact[t], kind="stable") if e not in order]
        chain = order + rest[:1]
        for a, c in zip(chain, chain[1:]):
            if exact[t, a] - exact[t, c] <= u[t, a] + u[t, c]:
                robust[t] = False
        if robust[t]:
            assert list(gpu_ids[t]) == order, f"token {t}: {list(gpu_ids[t])} vs {order}"
        else:
            chosen = []
            for c in gpu_ids[t]:
                others = [e for e in range(exact.shape[1]) if e not in chosen and e != c]
                assert all(exact[t, e] - u[t, e] <= exact[t, c] + u[t, c] for e in others), \
                    f"token {t}: expert {c} cannot come next"
                chosen.append(int(c))
    return robust, ref_ids


@pytest.mark.parametrize("T,d,E", [(1, 128, 8), (7, 256, 64), (32, 4096, 256), (33, 1024, 300), (300, 4096, 256),
                                   (4608, 4096, 256), (100, 7168, 256), (64, 2048, 1024)])
def test_router_logits(moe, T, d, E):
    L = make_layer(T=T, d=d, I=32, E=1, k=1, seed=T + d + E)
    wg = make_gate_weights(E, d, seed=T + E)
    got = moe.router(dev_bf16(L.x_bf16), dev_bf16(wg))
    again = moe.router(dev_bf16(L.x_bf16), dev_bf16(wg))
    torch.cuda.synchronize()
    check_logits(got.cpu().numpy(), L.x_bf16, wg)
    assert torch.equal(got, again), "router logits differ between two calls"


@pytest.mark.parametrize("name,flags", [("decode", 0), ("tiny", 0)])
def test_forward_gated(moe, name, flags):
    L = make_config(name)
    wg = make_gate_weights(L.E, L.d, seed=7)
    D = to_device(L)
    r = moe.forward_gated(D["x"], dev_bf16(wg), D["w13"], D["w13_scale"], D["w2"], D["w2_scale"], L.k,
                          flags=flags, return_routing=True)
    torch.cuda.synchronize()
    exact, b = check_logits(r["router_logits"].cpu().numpy(), L.x_bf16, wg)
    gpu_ids = r["topk_ids"].cpu().numpy()
    robust, ref_ids = routing_verdicts(gpu_ids, exact, b, L.k)
    same = np.all(gpu_ids == ref_ids, axis=1)
    assert same.mean() >= 0.99
    ref = orr.forward_gated(L.x_bf16, wg, L.w13, L.w13_scale, L.w2, L.w2_scale, L.k)
    if same.all():
        np.testing.assert_array_equal(r["sorted_slot"].cpu().numpy(), ref["sorted_slot"])
        np.testing.assert_array_equal(r["expert_offsets"].cpu().numpy(), ref["expert_offsets"])
    toks = np.nonzero(same)[0]
    assert_out_within(r["out"].cpu().numpy()[toks], ref["out"][toks], L, toks, f"gated {name}")


def test_prefill_size_routing_from_the_router(moe):
    """the router at the prefill workload's size (T = 4608): logits element by
    element, every robust token's experts exactly, the rest valid"""
    L = make_config("prefill")
    wg = make_gate_weights(L.E, L.d, seed=11)
    logits = moe.router(dev_bf16(L.x_bf16), dev_bf16(wg))
    ids, w, off, ss = moe.route(logits, L.k)
    torch.cuda.synchronize()
    exact, b = check_logits(logits.cpu().numpy(), L.x_bf16, wg)
    robust, _ = routing_verdicts(ids.cpu().numpy(), exact, b, L.k)
    assert robust.mean() > 0.99
    print("robust tokens", robust.sum(), "of", L.T)
