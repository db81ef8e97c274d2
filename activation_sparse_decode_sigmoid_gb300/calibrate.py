"""Offline placement: profile a layer's predictor on calibration inputs and
reload it with its neurons in descending activation-count order.

PowerInfer profiles, offline, how often each neuron activates and places the
frequently activated ("hot") neurons where they are cheapest to reach
(blog.csdn.net QbitAI/IPADS article, "CPU/GPU混合推理设计" and
"PowerInfer的整体架构").  On one GB300 everything is resident, so placement
becomes a permutation: hot neurons first, contiguous.  The counting runs in
the library (pi_layer_counts), the ordering in pi_perm_from_counts, the
permuted copy in pi_load_layer.
"""
from __future__ import annotations

import numpy as np

from . import pi
from . import workload as W


def calibrate_and_load(ctx: "pi.Context", slot: int, layer: dict, cal_xhat, hot_batch: int = 0) -> np.ndarray:
    """Load `layer` into `slot` in hot-first order; returns the permutation
    (perm[i] = original id of physical neuron i).  With hot_batch > 0 the
    layer also gets the always-active prefix at which computing a neuron
    costs no more bytes than predicting it, for batches of hot_batch tokens
    (pi_choose_hot_prefix on the calibration counts)."""
    ctx.load_layer(slot, layer)
    counts = ctx.layer_counts(slot, cal_xhat).cpu().numpy()
    perm = pi.pi_perm_from_counts(counts)
    ctx.load_layer(slot, layer, perm)
    if hot_batch > 0:
        ctx.set_hot_prefix(slot, ctx.choose_hot_prefix(slot, counts[perm], cal_xhat.shape[0], hot_batch))
    return perm


def load_synthetic_stack(cfg: W.LayerConfig, L: int, seed: int, device: int, max_batch: int,
                         keep_host=(), cal_tokens: int = 256, hot_batch: int = 0):
    """Draw an L-layer synthetic stack on the GPU, calibrate and load it
    (with hot_batch > 0, each layer with its crossover hot prefix).

    Returns (ctx, host) where host[l] = (host copy of layer l, perm) for the
    layers in `keep_host` (for checking against a CPU reference)."""
    import torch

    # calibration runs 64 tokens per launch; decode calls use their own batch
    ctx = pi.Context(device, max_layers=L, max_batch=max(max_batch, 64))
    host = {}
    dev = torch.device("cuda", device)
    for l in range(L):
        lw = W.make_layer_device(cfg, l, seed, dev)
        cal = torch.from_numpy(W.calibration_inputs(cfg, l, seed, T=cal_tokens).view(np.int16)).to(dev)
        perm = calibrate_and_load(ctx, l, lw, cal, hot_batch)
        if l in keep_host:
            host[l] = (W.layer_to_host(lw), perm)
        del lw, cal
    torch.cuda.synchronize(dev)
    ctx.check()
    return ctx, host
