"""Failure handling on the GPU without a GPU fault.

Every pipeline wait in the expert kernels is bounded.  A host-chosen fault
(moe_fp4_set_fault_injection: the first CTA never loads its first tile or
stage, so a wait on it can never complete) with a short wait limit makes one
wait run out; the call must return, moe_fp4_check must report
MOE_FP4_ERR_DEVICE with the timed-out bit, and the next ordinary call must be
correct (tensor memory was freed and every copy in flight had landed).
"""
import time

import numpy as np
import pytest

import oracle
from moe_inputs import make_layer

from _layer_util import assert_out_close, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

GEMV, TC = 0x1, 0x2


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import fp4_mixture_experts_gb300 as m
    m.load_library()
    return m


@pytest.mark.parametrize("site,flags", [(1, TC), (1, TC | 0x8), (2, GEMV), (2, GEMV | 0x4)])
def test_timed_out_wait_is_reported_and_the_next_call_is_correct(moe, site, flags):
    L = make_layer(T=48, d=1024, I=1024, E=8, k=2, seed=61)
    D = to_device(L)
    args = (D["x"], D["logits"], D["w13"], D["w13_scale"], D["w2"], D["w2_scale"], L.k)
    ws = torch.empty(moe.workspace_bytes(L.T, L.d, L.I, L.E, L.k), dtype=torch.uint8, device="cuda")
    moe.set_fault_injection(site, 20000)  # waits give up after 20 ms
    try:
        t0 = time.perf_counter()
        moe.forward(*args, workspace=ws, flags=flags)
        with pytest.raises(moe.MoeFp4Error) as ei:
            moe.check(ws)
        elapsed = time.perf_counter() - t0
    finally:
        moe.set_fault_injection(moe.FAULT_NONE)
    assert ei.value.status == -5
    assert elapsed < 30.0
    moe.check(ws)  # the error word was cleared
    out = moe.forward(*args, workspace=ws, flags=flags)
    moe.check(ws)
    ref = oracle.forward(L.x_bf16, L.router_logits, L.w13, L.w13_scale, L.w2, L.w2_scale, L.k)
    assert_out_close(out.cpu().numpy(), ref["out"], f"after fault site {site}")


def test_timed_out_wait_in_the_block_scaled_kernel(moe):
    """the MXFP8-activation layer: its W13 kernel's first stage withheld"""
    from oracle import mx_activations as mxa

    from _layer_util import assert_out_within_mx
    L = make_layer(T=48, d=1024, I=1024, E=8, k=2, seed=62)
    D = to_device(L)
    args = (D["x"], D["logits"], D["w13"], D["w13_scale"], D["w2"], D["w2_scale"], L.k)
    ws = torch.empty(moe.mx_workspace_bytes(L.T, L.d, L.I, L.E, L.k), dtype=torch.uint8, device="cuda")
    moe.set_fault_injection(moe.FAULT_TC_TOKEN_TILE, 20000)
    try:
        t0 = time.perf_counter()
        moe.forward_mx(*args, workspace=ws)
        with pytest.raises(moe.MoeFp4Error) as ei:
            moe.check(ws)
        elapsed = time.perf_counter() - t0
    finally:
        moe.set_fault_injection(moe.FAULT_NONE)
    assert ei.value.status == -5
    assert elapsed < 30.0
    moe.check(ws)
    out = moe.forward_mx(*args, workspace=ws)
    moe.check(ws)
    ref = mxa.forward_mx(L.x_bf16, L.router_logits, L.w13, L.w13_scale, L.w2, L.w2_scale, L.k)
    assert_out_within_mx(out.cpu().numpy(), ref["out"], L, what="after the block-scaled fault")


def test_fault_injection_arguments(moe):
    with pytest.raises(moe.MoeFp4Error):
        moe.set_fault_injection(7, 1000)
    with pytest.raises(moe.MoeFp4Error):
        moe.set_fault_injection(moe.FAULT_TC_TOKEN_TILE, 0)
    moe.set_fault_injection(moe.FAULT_NONE)
