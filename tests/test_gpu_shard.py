"""Neuron-sharded layers through the C ABI on one GPU: two contexts, each
holding one of two round-robin shards of the same calibrated layer
(pi_load_layer_shard), compute their parts of the layer's update
(pi_layer_partial); the parts, summed, must match the oracle's unsplit layer:
the union of the shards' lists (local ids mapped back to the layer's
neurons) equals the oracle's list bit for bit, and the summed update is
within the tolerance of the other parity tests.  One token runs in the
persistent kernel, 3 and 8 tokens layer by layer (CUDA-core and tensor-core
FFN).  A whole layer's pi_layer_partial + pi_residual_add is the decode step,
bit for bit."""
from __future__ import annotations

import numpy as np
import pytest

import oracle as O
from activation_sparse_decode_sigmoid_gb300 import pi
from activation_sparse_decode_sigmoid_gb300 import workload as W
from tests import _gpu as G
from tests._helpers import max_rel_err

pytestmark = pytest.mark.gpu

CFGS = {
    "relu_f16": W.LayerConfig("sh_relu_f16", 256, 1000, 64, 2, W.RELU, W.F16, W.F16, alpha=0.8, cfg_id=601),
    "reglu_bf16": W.LayerConfig("sh_reglu_bf16", 264, 777, 32, 2, W.REGLU, W.BF16, W.BF16, alpha=0.7, cfg_id=602),
    "relu_q4": W.LayerConfig("sh_relu_q4", 512, 640, 64, 2, W.RELU, W.Q4_0, W.F16, alpha=0.9, cfg_id=603),
}


def _calibrated(cfg, l):
    """A layer and its calibrated permutation (counted on a whole-layer context)."""
    lw = W.make_layer(cfg, l, 0, random_b1=True, random_bdown=True)
    c = G.ctx(max_layers=1, max_batch=64)
    c.load_layer(0, lw)
    perm = pi.pi_perm_from_counts(c.layer_counts(0, G.dev16(W.calibration_inputs(cfg, l, 0, T=64))).cpu().numpy())
    c.close()
    return lw, perm


@pytest.mark.parametrize("name", list(CFGS))
@pytest.mark.parametrize("B", [1, 3, 8])
def test_two_shards_sum_to_the_unsplit_layer(name, B):
    t = G.torch()
    cfg = CFGS[name]
    lw, perm = _calibrated(cfg, 0)
    world = 2
    ctxs, traces = [], []
    for r in range(world):
        c = G.ctx(max_layers=1, max_batch=8)
        c.load_layer_shard(0, lw, r, world, perm)
        assert pi.pi_layer_shard(c.handle, 0) == (r, world)
        nl = (cfg.n - r + world - 1) // world
        tr = (t.zeros((1, B, cfg.d), dtype=t.float32, device="cuda"),
              t.zeros((1, B, cfg.d), dtype=t.int16, device="cuda"),
              t.full((1, nl), -1, dtype=t.int32, device="cuda"), t.zeros(1, dtype=t.int32, device="cuda"))
        c.set_trace(*tr)
        ctxs.append(c)
        traces.append(tr)
    x0 = W.decode_inputs(cfg, B, 9)
    x = t.from_numpy(x0.copy()).cuda()
    parts = [c.layer_partial(0, x) for c in ctxs]
    for c in ctxs:
        c.check()
    assert t.equal(x, t.from_numpy(x0).cuda())  # x is only read
    xh = G.host16(traces[0][1])[0]
    assert np.array_equal(xh, G.host16(traces[1][1])[0])  # both shards normalise the same x
    want_xh = O.rmsnorm(x0, cfg.act_dtype)
    assert np.abs(xh.astype(np.int32) - want_xh.astype(np.int32)).max() <= 1
    sel = []
    for r, tr in enumerate(traces):
        m = int(tr[3][0].item())
        local = tr[2][0, :m].cpu().numpy()
        assert np.all(np.diff(local) > 0)
        sel.append(perm[r + world * local])  # local -> physical -> original ids
    sel = np.sort(np.concatenate(sel))
    assert np.array_equal(sel, O.union(O.layer_predict(lw, xh)["mask"]))
    u = (parts[0] + parts[1]).cpu().numpy().astype(np.float64)
    assert max_rel_err(u, O.masked_ffn(lw, xh, sel)) <= G.tol(lw)
    for c in ctxs:
        c.close()


@pytest.mark.parametrize("B", [1, 8])
def test_layer_partial_plus_residual_add_is_the_decode_step(B):
    t = G.torch()
    cfg = CFGS["relu_f16"]
    c = G.ctx(max_layers=1, max_batch=8)
    c.load_layer(0, W.make_layer(cfg, 0, 0, random_b1=True, random_bdown=True))
    x0 = t.from_numpy(W.decode_inputs(cfg, B, 10)).cuda()
    ref = x0.clone()
    c.decode_step(ref)
    x = x0.clone()
    u = c.layer_partial(0, x)
    c.residual_add(x, u)
    c.check()
    assert t.equal(x, ref)
    c.close()


def test_sharded_stack_decode_matches_the_whole_stack():
    """Two layers, each split into two shards held by two contexts: per layer
    both compute their part, the parts are summed (standing in for the
    all-reduce between devices) and both add the sum into their copy of x.
    The result equals the whole-layer decode step within the tolerance (the
    split changes only the order of the fp32 sums)."""
    t = G.torch()
    cfg = CFGS["reglu_bf16"]
    B, L, world = 3, 2, 2
    layers = [_calibrated(cfg, l) for l in range(L)]
    whole = G.ctx(max_layers=L, max_batch=8)
    shards = [G.ctx(max_layers=L, max_batch=8) for _ in range(world)]
    for l, (lw, perm) in enumerate(layers):
        whole.load_layer(l, lw, perm)
        for r, c in enumerate(shards):
            c.load_layer_shard(l, lw, r, world, perm)
    x0 = W.decode_inputs(cfg, B, 11)
    ref = t.from_numpy(x0.copy()).cuda()
    whole.decode_step(ref)
    whole.check()
    xs = [t.from_numpy(x0.copy()).cuda() for _ in range(world)]
    for l in range(L):
        parts = [c.layer_partial(l, x) for c, x in zip(shards, xs)]
        total = parts[0] + parts[1]
        for c, x in zip(shards, xs):
            c.residual_add(x, total)
    for c in shards:
        c.check()
    assert t.equal(xs[0], xs[1])
    upd = (xs[0] - t.from_numpy(x0).cuda()).cpu().numpy().astype(np.float64)
    want = (ref - t.from_numpy(x0).cuda()).cpu().numpy().astype(np.float64)
    assert max_rel_err(upd, want) <= 1e-2
    for c in [whole] + shards:
        c.close()
