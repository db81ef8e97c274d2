"""Shared test helpers: golden fixtures, tolerances, layer permutation."""
from __future__ import annotations

import json
import os

import numpy as np

from activation_sparse_decode_sigmoid_gb300 import workload as W

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load_golden(name: str) -> dict:
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def worked_example_layer(dt: int = W.F16) -> tuple[dict, np.ndarray, dict]:
    """The {3,4,5} worked example as a layer dict + x_hat [1,d] + expected."""
    g = load_golden("worked_example_345.json")
    d, n, r = g["d"], g["n"], g["r"]
    w_down = np.zeros((d, n), np.float32)
    for i, col in enumerate(g["w_down_columns"]):
        w_down[: len(col), i] = col
    w1 = np.zeros((r, d), np.float32)
    w1[0] = g["p_w1_row0"]
    w2 = np.zeros((n, r), np.float32)
    w2[:, 0] = g["p_w2_col0"]
    layer = {
        "d": d, "n": n, "r": r, "act": W.RELU, "w_dtype": dt, "act_dtype": dt,
        "w_up": W.to_bits(np.array(g["w_up"], np.float32), dt),
        "w_gate": None,
        "b": W.to_bits(np.array(g["b"], np.float32), dt),
        "w_down": W.to_bits(w_down, dt),
        "b_down": W.to_bits(np.array(g["b_down"], np.float32), dt),
        "p_w1": W.to_bits(w1, dt), "p_b1": None,
        "p_w2": W.to_bits(w2, dt), "p_b2": None,
    }
    x = W.to_bits(np.array([g["x_hat"]], np.float32), dt)
    return layer, x, g["expected"]


def permute_layer(layer: dict, perm: np.ndarray) -> dict:
    """Relabel neurons: physical neuron p is original neuron perm[p]."""
    out = dict(layer)
    out["w_up"] = layer["w_up"][perm]
    if layer.get("w_gate") is not None:
        out["w_gate"] = layer["w_gate"][perm]
    out["b"] = layer["b"][perm]
    if layer["w_dtype"] == W.Q4_0:
        out["w_down"] = layer["w_down"][perm]
    else:
        out["w_down"] = np.ascontiguousarray(layer["w_down"][:, perm])
    out["p_w2"] = layer["p_w2"][perm]
    if layer.get("p_b2") is not None:
        out["p_b2"] = layer["p_b2"][perm]
    return out


def max_rel_err(y, ref) -> float:
    """max_k |y_k - ref_k| / max(|ref_k|, rms(ref)) over the whole array."""
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    den = np.maximum(np.abs(ref), rms)
    den = np.where(den == 0, 1.0, den)
    return float(np.max(np.abs(y - ref) / den)) if ref.size else 0.0


def dequant_q4_numpy(blocks: np.ndarray) -> np.ndarray:
    """Independent numpy decode of Q4_0 rows [rows, nb*18] -> float64 [rows, nb*32]."""
    rows = blocks.shape[0]
    b = blocks.reshape(rows, -1, 18)
    s = b[..., 0:2].copy().view(np.float16)[..., 0].astype(np.float64)
    qs = b[..., 2:18]
    lo = (qs & 15).astype(np.float64) - 8
    hi = (qs >> 4).astype(np.float64) - 8
    q = np.concatenate([lo, hi], axis=-1)
    return (q * s[..., None]).reshape(rows, -1)


def layer_dense_f64(layer: dict):
    """float64 numpy matrices of a host layer (independent of the oracle)."""
    dt = layer["act_dtype"]
    if layer["w_dtype"] == W.Q4_0:
        wu = dequant_q4_numpy(layer["w_up"])
        wg = None if layer.get("w_gate") is None else dequant_q4_numpy(layer["w_gate"])
        wd = dequant_q4_numpy(layer["w_down"]).T  # stored transposed
    else:
        wu = W.from_bits(layer["w_up"], layer["w_dtype"]).astype(np.float64)
        wg = None if layer.get("w_gate") is None else W.from_bits(layer["w_gate"], layer["w_dtype"]).astype(np.float64)
        wd = W.from_bits(layer["w_down"], layer["w_dtype"]).astype(np.float64)
    b = W.from_bits(layer["b"], dt).astype(np.float64)
    bd = None if layer.get("b_down") is None else W.from_bits(layer["b_down"], dt).astype(np.float64)
    return wu, wg, b, wd, bd
