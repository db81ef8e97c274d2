"""The sharded decode loop (shard.decode_step_sharded) on two gloo ranks on
CPU, with an oracle-backed stand-in for the library context: each rank holds
the round-robin neuron shard of every layer of a three-layer stack, computes
its part of each layer's update, the ranks sum the parts with one all-reduce
per layer, and both add it.  The final residual must equal the unsplit stack
decoded by the oracle (fp64, up to summation order), and both ranks must end
with identical copies of x.  The library side of the same sequence runs on
one GPU in tests/test_gpu_shard.py."""
from __future__ import annotations

import os
import socket
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class OracleShard:
    """Stand-in for pi.Context holding shard `rank` of `world` of every layer:
    layer_partial / residual_add follow the library's contract, computed by
    the oracle in fp64."""

    def __init__(self, layers, rank, world, act_dtype):
        from tests.test_oracle_shard import shard
        self.parts = [shard(lw, rank, world)[0] for lw in layers]
        self.descs = {l: None for l in range(len(layers))}
        self.dt = act_dtype

    def layer_partial(self, l, x, u):
        import oracle as O
        import torch
        xh = O.rmsnorm(x.numpy().astype(np.float32), self.dt)
        part = self.parts[l]
        idx = O.union(O.layer_predict(part, xh)["mask"])
        u.copy_(torch.from_numpy(O.masked_ffn(part, xh, idx)))

    def residual_add(self, x, u):
        x.add_(u)


def _unsplit(layers, x, dt):
    import oracle as O
    x = x.copy()
    for lw in layers:
        xh = O.rmsnorm(x.astype(np.float32), dt)
        x = x + O.masked_ffn(lw, xh, O.union(O.layer_predict(lw, xh)["mask"]))
    return x


def _rank_main(rank, world, port, name, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist

    from activation_sparse_decode_sigmoid_gb300 import shard as SH
    from activation_sparse_decode_sigmoid_gb300 import workload as W

    dist.init_process_group("gloo", rank=rank, world_size=world)
    cfg = W.LayerConfig(name, 128, 300, 32, 3, W.REGLU if name == "reglu" else W.RELU, W.F16, W.F16,
                        alpha=0.8, cfg_id=503)
    layers = [W.make_layer(cfg, l, 0, random_b1=True, random_bdown=True) for l in range(3)]
    x0 = W.decode_inputs(cfg, 2, 5).astype(np.float64)
    ctx = OracleShard(layers, rank, world, cfg.act_dtype)
    x = torch.from_numpy(x0.copy())
    SH.decode_step_sharded(ctx, x)
    got = [None] * world
    dist.all_gather_object(got, x.numpy().tolist())
    dist.destroy_process_group()
    if rank == 0:
        want = _unsplit(layers, x0, cfg.act_dtype)
        a = np.asarray(got[0])
        out.put((np.array_equal(a, np.asarray(got[1])), float(np.max(np.abs(a - want))), float(np.max(np.abs(want)))))


@pytest.mark.parametrize("name", ["relu", "reglu"])
def test_sharded_decode_loop_equals_unsplit_stack(name):
    pytest.importorskip("torch")
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, name, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
    assert [p.exitcode for p in procs] == [0, 0]
    same, err, scale = out.get(timeout=5)
    assert same, "the ranks' residual copies differ"
    # the residual feeds the next layer's RMSNorm and predictor: equal lists
    # need the same x_hat bytes, so the split must not move x beyond rounding
    assert err <= 1e-9 * max(1.0, scale), err
