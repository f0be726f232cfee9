"""The multi-rank bench logic on CPU: two gloo ranks, barrier and max over ranks."""
import os

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    bench.barrier(dist, device="cpu")
    v = bench.max_over_ranks(dist, 1.5 + rank, device="cpu")
    tot = bench.sum_over_ranks(dist, 10 * (rank + 1), device="cpu")
    q.put((rank, v, tot))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert out == [(0, 2.5, 30.0), (1, 2.5, 30.0)]


def test_cpu_baseline_reports_parity_of_a_given_result():
    """The CPU-baseline leg compares its oracle sample with the CUDA path's result it is given."""
    import numpy as np

    import bench
    import oracle
    from moe_inputs import make_config
    L = make_config("tiny")
    ref = oracle.forward(L.x_bf16, L.router_logits, L.w13, L.w13_scale, L.w2, L.w2_scale, L.k)
    good = {"out": ref["out"].astype(np.float32), "topk_ids": ref["topk_ids"]}
    r = bench.cpu_baseline_sample("tiny", 0.0, good)
    p = r["parity"]
    assert p["tokens"] >= 1 and p["topk_ids_equal"] and p["rel_l2"] < 1e-6 and r["kind"] == "oracle"
    bad_out = good["out"].copy()
    bad_out[0] *= 1.1
    bad_ids = good["topk_ids"].copy()
    bad_ids[0] = bad_ids[0][::-1]
    p = bench.cpu_baseline_sample("tiny", 0.0, {"out": bad_out, "topk_ids": bad_ids})["parity"]
    assert not p["topk_ids_equal"] and p["rel_l2"] > 0.05
