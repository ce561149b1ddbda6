"""The multi-device half of the fixed-order shard gradient sum.

"MojoLearn 162M" model card, table "Training": 64 logical shards, each a mean
over 4 x 2,048 tokens, their gradients summed in a fixed order. Profile v1
reads the order as left to right over the global shard index. A collective's
own reduction (all-reduce, reduce-scatter) adds in an order of its own, so it
is never used: the ranks all-gather their shard gradients unreduced (bytes
only, no arithmetic), in global shard order, and every rank then runs the
same ordered sum (detshardsum_f32) over the gathered stack. Every rank ends
with the same bits, and they equal a single device's sum of all shards.

Rank r holds the contiguous block of shards r*k .. r*k + k - 1, one per row.
"""
from __future__ import annotations


def gather_shards(local, group=None):
    """All-gather the ranks' k x n blocks of shard gradients unreduced; returns
    the (world * k) x n stack in global shard order."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group)
    local = local.contiguous()
    blocks = [torch.empty_like(local) for _ in range(world)]
    dist.all_gather(blocks, local, group=group)
    return torch.cat(blocks, dim=0)


def ordered_shard_mean(local, group=None, sum_fn=None):
    """The mean of all ranks' shard gradients: gather, then the left-to-right
    sum scaled by 1 / (number of shards). sum_fn(stack, scale) defaults to
    the library's detshardsum_f32 on the stack's device."""
    stack = gather_shards(local, group)
    if sum_fn is None:
        from bitwise_reproducible_fp32_gb300 import detlib
        sum_fn = lambda g, scale: detlib.detshardsum_f32(g, scale=scale)  # noqa: E731
    return sum_fn(stack, 1.0 / stack.shape[0])
