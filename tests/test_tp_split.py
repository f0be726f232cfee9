"""The tensor-parallel split of I on the host: two gloo ranks each take their
shard of the weights (shard_weights), compute their partial layer output with
the CPU oracle, and sum it with the library's all-reduce; the result must be
the oracle's unsplit output (up to fp64 rounding), because SwiGLU acts on
each i separately and W2 is linear in h."""
import os

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from fp4_mixture_experts_gb300 import tp


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        from moe_inputs import make_layer
        L = make_layer(T=10, d=256, I=512, E=4, k=2, seed=91)
        shard = tp.shard_weights(*(torch.from_numpy(a) for a in (L.w13, L.w13_scale, L.w2, L.w2_scale)), rank, world)
        part = oracle.forward(L.x_bf16, L.router_logits, *(s.numpy() for s in shard), L.k)
        out = torch.from_numpy(part["out"].copy())
        tp.all_reduce_out(out)
        full = oracle.forward(L.x_bf16, L.router_logits, L.w13, L.w13_scale, L.w2, L.w2_scale, L.k)
        q.put((rank, float(np.abs(out.numpy() - full["out"]).max()), float(np.abs(full["out"]).max())))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_sum_to_the_unsplit_layer():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29700 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, err, scale in res:
        assert err <= 1e-12 * scale, (rank, err, scale)


def test_shard_layout_and_bounds():
    I, d, E = 512, 256, 3
    w13 = torch.arange(E * 2 * I * (d // 2), dtype=torch.int64).reshape(E, 2 * I, d // 2)
    w2 = torch.arange(E * d * (I // 2), dtype=torch.int64).reshape(E, d, I // 2)
    s13 = torch.zeros(E, 2 * I, d // 32, dtype=torch.uint8)
    s2 = torch.zeros(E, d, I // 32, dtype=torch.uint8)
    a, _, b, _ = tp.shard_weights(w13, s13, w2, s2, 1, 4)     # i in [128, 256)
    assert torch.equal(a[:, :128], w13[:, 128:256]) and torch.equal(a[:, 128:], w13[:, I + 128:I + 256])
    assert torch.equal(b, w2[:, :, 64:128])
    for bad in [(I, 0, 3), (I, 0, 8), (I, 2, 2), (384, 0, 2)]:
        with pytest.raises(ValueError):
            tp.shard_bounds(*bad)
