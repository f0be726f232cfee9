"""The allocation-free entry point (collected late on purpose).

moe_fp4_forward_noalloc serves callers that cannot allocate device memory:
it takes only inputs and outputs and runs on the library's fixed device
scratch.  Both run the same deterministic kernels as moe_fp4_forward, so the
results must be bit-identical; checked through the C ABI on two calls in a
row (the second with other inputs, so that leftovers of the first call in the
shared scratch would show), on the streaming and the tensor-core path, at the
largest problem the scratch holds, and for the size limit.
"""
import ctypes

import numpy as np
import pytest

from moe_inputs import make_layer

from _layer_util import to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

GEMV, TC, DET = 0x1, 0x2, 0x10
SCRATCH = 16 * 1024 * 1024


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import fp4_mixture_experts_gb300 as m
    m.load_library()
    return m


def _noalloc_raw(moe, L, D, out, flags=0):
    lib = moe.load_library()
    dims = moe.Dims(L.T, L.d, L.I, L.E, L.k)
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.moe_fp4_forward_noalloc(ctypes.byref(dims), P(D["x"]), P(D["logits"]), P(D["w13"]),
                                       P(D["w13_scale"]), P(D["w2"]), P(D["w2_scale"]), P(out), flags, stream)


def _check_raw(moe):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return moe.load_library().moe_fp4_noalloc_check(stream)


def _compare(moe, L, flags, what):
    D = to_device(L)
    ref = moe.forward(D["x"], D["logits"], D["w13"], D["w13_scale"], D["w2"], D["w2_scale"], L.k, flags=flags)
    out = torch.full((L.T, L.d), float("nan"), dtype=torch.float32, device="cuda")
    assert _noalloc_raw(moe, L, D, out, flags) == 0
    assert _check_raw(moe) == 0
    torch.cuda.synchronize()
    assert torch.equal(out, ref), f"{what}: noalloc differs from forward"


@pytest.mark.parametrize("flags", [GEMV | DET, TC | DET])
def test_noalloc_matches_forward_twice(moe, flags):
    for seed in (21, 22):
        _compare(moe, make_layer(T=32, d=1024, I=1024, E=32, k=4, seed=seed), flags, f"flags {flags} seed {seed}")


def test_noalloc_tensor_core_call_after_streaming_call(moe):
    # the tensor-core path reads regions of the shared scratch (64-row token
    # boxes, the f16 copy of h) that a streaming call before it left dirty
    _compare(moe, make_layer(T=40, d=1024, I=1024, E=16, k=4, seed=23), GEMV | DET, "streaming")
    _compare(moe, make_layer(T=96, d=1024, I=1024, E=4, k=2, seed=24), TC | DET, "tensor-core after streaming")


def _largest_T(moe, d, I, E, k):
    T = 1
    while moe.workspace_bytes(T + 1, d, I, E, k) <= SCRATCH:
        T += 1
    return T


def test_noalloc_largest_problem_and_one_token_more(moe):
    d, I, E, k = 1024, 1024, 16, 4
    T = _largest_T(moe, d, I, E, k)
    _compare(moe, make_layer(T=T, d=d, I=I, E=E, k=k, seed=25), DET, f"largest T={T}")
    L = make_layer(T=T + 1, d=d, I=I, E=E, k=k, seed=26)
    D = to_device(L)
    out = torch.empty(L.T, L.d, dtype=torch.float32, device="cuda")
    assert _noalloc_raw(moe, L, D, out) == -3


def test_noalloc_rejects_problems_beyond_its_scratch(moe):
    # T=4096 tokens at d=4096 need far more than the fixed scratch; the
    # decode-shaped limits stated in the header hold
    lib = moe.load_library()
    dims = moe.Dims(4096, 4096, 2048, 256, 8)
    assert moe.workspace_bytes(4096, 4096, 2048, 256, 8) > SCRATCH
    assert _largest_T(moe, 4096, 2048, 256, 8) == 72
    assert _largest_T(moe, 7168, 2048, 256, 8) == 44
    fake = ctypes.c_void_p(0x100000)  # never dereferenced: the size check comes first
    rc = lib.moe_fp4_forward_noalloc(ctypes.byref(dims), fake, fake, fake, fake, fake, fake, fake, 0, None)
    assert rc == -3


def test_noalloc_check_reports_a_timed_out_wait(moe):
    # a host-planted fault (a token tile that never arrives) makes a pipeline
    # wait run out; the error word in the internal scratch reports it once
    L = make_layer(T=64, d=1024, I=1024, E=4, k=2, seed=27)
    D = to_device(L)
    out = torch.empty(L.T, L.d, dtype=torch.float32, device="cuda")
    moe.set_fault_injection(moe.FAULT_TC_TOKEN_TILE, 20000)
    try:
        assert _noalloc_raw(moe, L, D, out, TC) == 0
        assert _check_raw(moe) == -5
    finally:
        moe.set_fault_injection(moe.FAULT_NONE)
    assert _check_raw(moe) == 0
    _compare(moe, L, TC | DET, "after the fault")
