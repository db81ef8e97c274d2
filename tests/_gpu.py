"""Helpers for the GPU parity tests: contexts, device copies, oracle checks."""
from __future__ import annotations

import numpy as np

import oracle as O
from activation_sparse_decode_sigmoid_gb300 import pi
from activation_sparse_decode_sigmoid_gb300 import workload as W
from tests._helpers import max_rel_err

TOL = {W.F16: 1e-2, W.BF16: 1e-2, W.Q4_0: 2e-2}


def torch():
    import torch as t
    return t


def ensure_built():
    from activation_sparse_decode_sigmoid_gb300 import build
    build.build()


def dev16(a: np.ndarray):
    """uint16 bit patterns -> int16 CUDA tensor (same bytes)."""
    t = torch()
    return t.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def host16(t) -> np.ndarray:
    return t.detach().cpu().numpy().view(np.uint16)


def y_to_f64(y, dt) -> np.ndarray:
    t = torch()
    return y.detach().float().cpu().numpy().astype(np.float64) if y.dtype != t.int16 else \
        W.from_bits(host16(y), dt).astype(np.float64)


def tol(layer: dict) -> float:
    return TOL[layer["w_dtype"]]


def ctx(max_layers=1, max_batch=8) -> pi.Context:
    ensure_built()
    return pi.Context(0, max_layers=max_layers, max_batch=max_batch)


def predict_checked(c: pi.Context, slot: int, layer_host: dict, xhat: np.ndarray, perm=None):
    """GPU predictor vs oracle: ascending physical list, bit-exact set."""
    t = torch()
    n = layer_host["n"]
    idx, cnt = c.predict(slot, dev16(xhat))
    c.check()
    m = int(cnt.item())
    gidx = idx[:m].cpu().numpy()
    assert np.all(np.diff(gidx) > 0), "index list not strictly ascending"
    assert gidx.size == 0 or (gidx.min() >= 0 and gidx.max() < n)
    ref = O.layer_predict(layer_host, xhat)
    oidx = O.union(ref["mask"])
    orig = gidx if perm is None else np.asarray(perm)[gidx]
    assert np.array_equal(np.sort(orig), oidx), (
        f"predicted sets differ: gpu {gidx.size} vs oracle {oidx.size}; "
        f"min |z64| among mismatches: {np.abs(ref['z64']).min():.3g}")
    return idx, cnt, oidx


def ffn_checked(c: pi.Context, slot: int, layer_host: dict, xhat: np.ndarray, idx, cnt, oidx):
    y = c.sparse_ffn(slot, dev16(xhat), idx, cnt)
    c.check()
    got = y_to_f64(y, layer_host["act_dtype"])
    want = O.masked_ffn(layer_host, xhat, oidx)
    err = max_rel_err(got, want)
    assert err <= tol(layer_host), f"max rel err {err:.3g} > {tol(layer_host)}"
    return err
