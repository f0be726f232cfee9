"""The allocation-free entry point (collected last on purpose).

moe_fp4_forward_noalloc serves callers that cannot allocate device memory:
it takes only inputs and outputs and runs on the library's fixed device
scratch.  Checked through the C ABI against moe_fp4_forward on two calls in
a row (the second with other inputs, so that leftovers of the first call in
the shared scratch would show), and for the size limit.
"""
import ctypes

import numpy as np
import pytest

from moe_inputs import make_layer

from _layer_util import assert_out_close, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import fp4_mixture_experts_gb300 as m
    m.load_library()
    return m


def _noalloc_raw(moe, L, D, out):
    lib = moe.load_library()
    dims = moe.Dims(L.T, L.d, L.I, L.E, L.k)
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.moe_fp4_forward_noalloc(ctypes.byref(dims), P(D["x"]), P(D["logits"]), P(D["w13"]),
                                       P(D["w13_scale"]), P(D["w2"]), P(D["w2_scale"]), P(out), 0, stream)


def test_noalloc_matches_forward_twice(moe):
    for seed in (21, 22):
        L = make_layer(T=32, d=1024, I=1024, E=32, k=4, seed=seed)
        D = to_device(L)
        ref = moe.forward(D["x"], D["logits"], D["w13"], D["w13_scale"], D["w2"], D["w2_scale"], L.k)
        out = torch.full((L.T, L.d), float("nan"), dtype=torch.float32, device="cuda")
        assert _noalloc_raw(moe, L, D, out) == 0
        torch.cuda.synchronize()
        assert_out_close(out.cpu().numpy(), ref.cpu().numpy(), f"noalloc seed {seed}")


def test_noalloc_rejects_problems_beyond_its_scratch(moe):
    # T=4096 tokens at d=4096 need far more than the fixed scratch
    lib = moe.load_library()
    dims = moe.Dims(4096, 4096, 2048, 256, 8)
    assert moe.workspace_bytes(4096, 4096, 2048, 256, 8) > 16 * 1024 * 1024
    fake = ctypes.c_void_p(0x100000)  # never dereferenced: the size check comes first
    rc = lib.moe_fp4_forward_noalloc(ctypes.byref(dims), fake, fake, fake, fake, fake, fake, fake, 0, None)
    assert rc == -3
