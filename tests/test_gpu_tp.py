"""The tensor-parallel split of I with the CUDA kernels: every rank's share of
the layer (its weight shard through moe_fp4_forward) run one after another on
one GPU, summed in rank order as the all-reduce would, must match the oracle's
unsplit layer (the cross-GPU all-reduce itself is torch.distributed, covered
by the gloo test on the host)."""
import numpy as np
import pytest

import oracle
from moe_inputs import make_layer

from _layer_util import assert_out_within, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import fp4_mixture_experts_gb300 as m
    m.load_library()
    return m


@pytest.mark.parametrize("world,flags", [(2, 0x1), (4, 0x2), (2, 0x2)])
def test_shards_sum_to_the_layer(moe, world, flags):
    from fp4_mixture_experts_gb300 import tp
    # shards must suit the path: multiples of 1024 for the streaming path, of 128 for the tensor cores
    I = world * (1024 if flags & 0x1 else 256)
    L = make_layer(T=64, d=1024, I=I, E=16, k=4, seed=95 + world)
    D = to_device(L)
    total = torch.zeros(L.T, L.d, dtype=torch.float32, device="cuda")
    for rank in range(world):
        shard = tp.shard_weights(D["w13"], D["w13_scale"], D["w2"], D["w2_scale"], rank, world)
        total += moe.forward(D["x"], D["logits"], *shard, L.k, flags=flags)
    torch.cuda.synchronize()
    ref = oracle.forward(L.x_bf16, L.router_logits, L.w13, L.w13_scale, L.w2, L.w2_scale, L.k)
    assert_out_within(total.cpu().numpy(), ref["out"], L, what=f"TP{world}")
