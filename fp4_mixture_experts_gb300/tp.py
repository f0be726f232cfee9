"""Tensor-parallel split of the expert intermediate size I.

The DeepSeek-V4-Flash-on-gfx90a paper serves the model with tensor
parallelism over four devices (TP4/EP1, abstract) and an all-reduce of the
layer output.  For the routed-expert layer the natural split is I: rank r of
N holds, for every expert, the gate and up rows [i0, i1) of W13 (i0 = r I/N)
and the matching K range [i0, i1) of W2.  SwiGLU acts on each i separately
and W2 is linear in h, so

    out = sum_r out_r,   out_r[t] = sum_j w_tj * sum_{i in [i0, i1)} h_i W2[:, i]

and every rank computes out_r with the ordinary layer call on its shard
(routing is replicated: every rank routes the same logits).  The only
exchange is one sum all-reduce of out [T, d] fp32 over torch.distributed.
I / N must be a multiple of 128 (the kernels' granularity).

shard_weights only slices tensors (once, when the weights are loaded); every
step of the layer still runs in the library's kernels.
"""
from __future__ import annotations


def shard_bounds(I: int, rank: int, world: int):
    """[i0, i1) of rank `rank` out of `world`; raises unless I / world is a multiple of 128."""
    if world < 1 or not 0 <= rank < world or I % world or (I // world) % 128:
        raise ValueError(f"I={I} does not split into {world} shards of a multiple of 128")
    n = I // world
    return rank * n, (rank + 1) * n


def shard_weights(w13, w13_scale, w2, w2_scale, rank: int, world: int):
    """The rank's shard of the expert weights (torch tensors, any device):
    w13 [E, 2I, d/2] -> [E, 2n, d/2] (gate rows i0..i1, then up rows I+i0..I+i1),
    w13_scale likewise, w2 [E, d, I/2] -> [E, d, n/2], w2_scale [E, d, I/32] -> [E, d, n/32]."""
    import torch
    I = w13.shape[1] // 2
    i0, i1 = shard_bounds(I, rank, world)
    w13_r = torch.cat([w13[:, i0:i1], w13[:, I + i0:I + i1]], dim=1).contiguous()
    w13s_r = torch.cat([w13_scale[:, i0:i1], w13_scale[:, I + i0:I + i1]], dim=1).contiguous()
    w2_r = w2[:, :, i0 // 2:i1 // 2].contiguous()
    w2s_r = w2_scale[:, :, i0 // 32:i1 // 32].contiguous()
    return w13_r, w13s_r, w2_r, w2s_r


def all_reduce_out(out, group=None):
    """Sum the ranks' partial outputs in place (torch.distributed, the
    process group's backend: NCCL between GPUs, gloo on the host)."""
    import torch.distributed as dist
    dist.all_reduce(out, op=dist.ReduceOp.SUM, group=group)
    return out


def forward_tp(x_bf16, router_logits, shard, k: int, group=None, flags: int = 0, workspace=None, stream=None):
    """This rank's share of the layer on its weight shard (from shard_weights),
    followed by the all-reduce: every rank returns the whole layer output."""
    from ._binding import forward
    w13_r, w13s_r, w2_r, w2s_r = shard
    out = forward(x_bf16, router_logits, w13_r, w13s_r, w2_r, w2s_r, k, flags=flags, workspace=workspace,
                  stream=stream)
    return all_reduce_out(out, group)
