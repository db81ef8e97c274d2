"""The neuron-sharded decomposition of one layer, emulated with the oracle on
two CPU ranks (gloo, world size 2).

Sharding a layer over G devices gives neuron j to rank j mod G (round-robin,
so the hot neurons at the front of the calibrated order spread over all
ranks).  W1 is replicated, so every rank computes the whole hidden layer h;
each rank evaluates the predictor rows of its own neurons and the FFN of its
own predicted neurons, and one sum over the ranks merges the partial outputs
(b_down added once).  The pages' worked example merges the partial results
of two executors the same way ("CPU/GPU混合推理设计", CSDN page).  These
tests check that decomposition against the unsplit layer: the union of the
ranks' lists is the layer's list (bit for bit), and the reduced output
equals the unsplit masked FFN up to fp64 rounding of the summation order.
No multi-device path is built; this pins the arithmetic it would follow."""
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


def shard(layer: dict, rank: int, world: int) -> tuple[dict, np.ndarray]:
    """Rank `rank`'s part of a layer dict: its neurons' W2 rows, b2, W_up /
    W_gate rows, biases and W_down columns; b_down on rank 0 only."""
    ids = np.arange(rank, layer["n"], world, dtype=np.int32)
    part = dict(layer)
    part["n"] = ids.size
    for k in ("p_w2", "p_b2", "w_up", "w_gate", "b"):
        if part.get(k) is not None:
            part[k] = np.ascontiguousarray(layer[k][ids])
    part["w_down"] = np.ascontiguousarray(layer["w_down"][:, ids])
    if rank != 0:
        part["b_down"] = None
    return part, ids


def _rank_main(rank: int, world: int, port: int, name: str, out) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist

    import oracle as O
    from activation_sparse_decode_sigmoid_gb300 import workload as W

    dist.init_process_group("gloo", rank=rank, world_size=world)
    cfg = W.LayerConfig(name, 128, 300, 32, 1, W.REGLU if name == "reglu" else W.RELU, W.F16, W.F16,
                        alpha=0.8, cfg_id=501)
    layer = W.make_layer(cfg, 0, 0, random_b1=True, random_bdown=True)
    x = W.xhat_inputs(cfg, 3, 4)
    part, ids = shard(layer, rank, world)
    mask = O.layer_predict(part, x)["mask"]
    mine = ids[O.union(mask)]  # this rank's predicted neurons, as layer ids
    y = O.masked_ffn(part, x, O.union(mask))  # its partial output (+ b_down on rank 0)
    yt = torch.from_numpy(y)
    dist.all_reduce(yt, op=dist.ReduceOp.SUM)
    lists = [None] * world
    dist.all_gather_object(lists, mine.tolist())
    dist.destroy_process_group()
    if rank == 0:
        whole = O.union(O.layer_predict(layer, x)["mask"])
        want = O.masked_ffn(layer, x, whole)
        merged = np.sort(np.concatenate([np.asarray(l, np.int32) for l in lists]))
        out.put((merged.tolist() == whole.tolist(), float(np.max(np.abs(yt.numpy() - want))),
                 float(np.max(np.abs(want)))))


@pytest.mark.parametrize("name", ["relu", "reglu"])
def test_round_robin_shards_reduce_to_the_unsplit_layer(name):
    pytest.importorskip("torch")
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, name, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    codes = [p.exitcode for p in procs]
    assert codes == [0, 0], codes
    same_list, err, scale = out.get(timeout=5)
    assert same_list
    assert err <= 1e-12 * max(1.0, scale)


def test_shards_cover_every_neuron_once():
    sys.path.insert(0, ROOT)
    from activation_sparse_decode_sigmoid_gb300 import workload as W
    cfg = W.LayerConfig("s", 64, 101, 16, 1, W.RELU, W.F16, W.F16, alpha=0.8, cfg_id=502)
    layer = W.make_layer(cfg, 0, 0)
    parts = [shard(layer, r, 3) for r in range(3)]
    ids = np.sort(np.concatenate([p[1] for p in parts]))
    assert np.array_equal(ids, np.arange(cfg.n))
    for r, (part, own) in enumerate(parts):
        assert np.array_equal(part["p_w2"], layer["p_w2"][own])
        assert np.array_equal(part["w_down"], layer["w_down"][:, own])
        assert (part["b_down"] is None) == (r != 0) or layer["b_down"] is None
