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


def predict_checked(c: pi.Context, slot: int, layer_host: dict, xhat: np.ndarray, perm=None, hot=None):
    """GPU predictor vs oracle: ascending physical list, bit-exact set.
    ``hot``: original ids of the neurons the loaded layer keeps always active."""
    t = torch()
    n = layer_host["n"]
    idx, cnt = c.predict(slot, dev16(xhat))
    c.check()
    m = int(cnt.item())
    gidx = idx[:m].cpu().numpy()
    assert np.all(np.diff(gidx) > 0), "index list not strictly ascending"
    assert gidx.size == 0 or (gidx.min() >= 0 and gidx.max() < n)
    ref = O.layer_predict(layer_host, xhat, hot=hot)
    oidx = O.union(ref["mask"])
    orig = gidx if perm is None else np.asarray(perm)[gidx]
    assert np.array_equal(np.sort(orig), oidx), (
        f"predicted sets differ: gpu {gidx.size} vs oracle {oidx.size}; "
        f"min |z64| among mismatches: {np.abs(ref['z64']).min():.3g}")
    return idx, cnt, oidx


def tc_error_bound(layer: dict, xhat: np.ndarray, idx) -> np.ndarray:
    """Per-output bound on the tensor-core FFN's error, from its arithmetic
    (an extra check beside the max relative error of 1e-2).

    The path passes every activation to the down-projection as two parts in
    the weights' 16-bit type, hi = round(a) and lo = round(a - hi) (a 16-bit
    tensor-core product takes both operands in one type), so a reaches it
    within u^2 |a|, and rounds y to the 16-bit type.  With u the type's unit
    roundoff (2^-8 bf16, 2^-11 f16) and M_j = sum_i |a_i| |W_down[j, i]|:
    |y_tc - y| <= 2 u^2 M_j + u |y_j| + g M_j, where g = (m + d) 2^-23 covers
    the fp32 sums of the up-projection (d terms, entering a squared
    activation at most twice) and of the down-projection (2 m terms)."""
    from tests._helpers import layer_dense_f64
    u = 2.0 ** -8 if layer["act_dtype"] == W.BF16 else 2.0 ** -11
    a = O.ffn_act(layer["w_up"], layer.get("w_gate"), layer["b"], xhat, layer["act"], layer["w_dtype"],
                  layer["act_dtype"])
    wd = layer_dense_f64(layer)[3]
    sel = np.asarray(idx, dtype=np.int64)
    mag = np.abs(a[:, sel]) @ np.abs(wd[:, sel]).T
    y = O.masked_ffn(layer, xhat, np.asarray(idx, dtype=np.int32))
    g = (2 * sel.size + layer["d"]) * 2.0 ** -23
    return (2 * u * u + g) * mag + u * np.abs(y) + 1e-6


def ffn_checked(c: pi.Context, slot: int, layer_host: dict, xhat: np.ndarray, idx, cnt, oidx):
    y = c.sparse_ffn(slot, dev16(xhat), idx, cnt)
    c.check()
    got = y_to_f64(y, layer_host["act_dtype"])
    want = O.masked_ffn(layer_host, xhat, oidx)
    err = max_rel_err(got, want)
    assert err <= tol(layer_host), f"max rel err {err:.3g} > {tol(layer_host)}"
    return err
