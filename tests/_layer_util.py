"""Shared helpers of the parity tests: upload inputs, compare with the oracle."""
import numpy as np

# tolerances of the layer output against the fp64 oracle (fp32 accumulation,
# h rounded to bf16 on both sides)
REL_L2 = 5e-3
COSINE = 0.9999
MAX_ABS = 2e-2


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
