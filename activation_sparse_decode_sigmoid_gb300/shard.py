"""Decode step over a neuron-sharded layer stack: one sum over the devices
per layer.

Multi-GPU support is listed as future work on the PowerInfer pages
(de.news.hada.io summary, "Jüngste Updates und Pläne").  Splitting every
layer's neurons round-robin over G devices (``pi_load_layer_shard``) leaves
each device a 1/G share of the predictor's output rows and of the FFN rows;
W1 is replicated, so every device computes the whole hidden layer.  Each
device computes its part u_g of the layer's update of the residual stream
(``pi_layer_partial``); the update is sum_g u_g -- one all-reduce of B x
d_model floats per layer -- which every device adds into its own copy of x
(``pi_residual_add``), so the copies stay identical.  The pages' hybrid
merges the CPU's and the GPU's partial results the same way (blog.csdn.net
QbitAI/IPADS article, "CPU/GPU混合推理设计").

The collective is torch.distributed's (NCCL between GPUs, gloo on CPUs);
this module only sequences the library calls around it.
"""
from __future__ import annotations


def stack_layers(ctx) -> list[int]:
    """The loaded slots 0..L-1 of a context (a ``pi.Context`` or any object
    with the same ``descs`` mapping)."""
    L = 0
    while L in ctx.descs:
        L += 1
    return list(range(L))


def decode_step_sharded(ctx, x, group=None, u=None):
    """One decode step in place on x (this device's copy of the fp32
    residual, [B][d]) over the context's shard of every layer: per layer the
    shard's update, an all-reduce (sum) over `group`, then the add into x.
    Every rank of the group calls it with the same x and the same stack
    split into its own shards."""
    import torch
    import torch.distributed as dist

    if u is None:
        u = torch.empty_like(x)
    for l in stack_layers(ctx):
        ctx.layer_partial(l, x, u)
        dist.all_reduce(u, op=dist.ReduceOp.SUM, group=group)
        ctx.residual_add(x, u)
    return x
