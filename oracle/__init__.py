"""CPU oracle for the predictor -> neuron-aware sparse FFN decode step.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package.  The CUDA library never
loads it and shares no code with it.  The arithmetic lives in ``oracle.c``
(plain C, fp64 FFN, canonical-order fp32 predictor); this module only builds
that file with gcc and marshals numpy arrays into it.

What each function follows (PowerInfer: Fast LLM Serving with a Consumer-grade
GPU; blog.csdn.net QbitAI/IPADS article and de.news.hada.io summary):

* ``predict``      -- the per-layer routing predictor ("充分利用模型和硬件特点"):
  a small MLP decides which neurons fire; here d -> r -> n with ReLU, then
  sigmoid(z) > 0.5, i.e. z > 0, evaluated in the canonical fp32 order CDOT.
* ``union``        -- the batch's active set: union of the per-token sets.
* ``predict(..., hot=ids)`` -- the one-device reading of the hot/cold split
  ("CPU/GPU混合推理设计"): the hot neurons (the first ones of the calibrated
  order) are active for every token, the rest as predicted.
* ``ffn_act``      -- ReLU / ReGLU / squared-ReLU activations of every neuron
  (fp64; the three families the pages name, de.news.hada.io summary,
  "Einschränkungen und FAQ").
* ``ffn_down``     -- only the listed neurons' columns of W_down are summed
  (neuron-aware sparse operator); merging partial results over any partition
  of the list gives the whole ("CPU/GPU混合推理设计" worked example {3,4,5}).
* ``rmsnorm``      -- weightless RMSNorm of the residual stream between layers.
* ``perm_from_counts`` -- offline hot/cold profiling turned into a neuron
  permutation by descending activation count.
* ``q4_dequant``   -- Q4_0 blocks ("Quantisierung und Kompatibilität").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")

F16, BF16, Q4_0 = 0, 1, 2
RELU, REGLU, SQRELU = 0, 1, 2

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into oracle/_build/liboracle.so (gcc, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + ".tmp.%d" % os.getpid()
        cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11",
               "-D_GNU_SOURCE", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm", "-lpthread"]
        subprocess.check_call(cmd)
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32, f64 = ctypes.c_int, ctypes.c_double
            lib.or_to_double.restype = f64
            lib.or_to_double.argtypes = [ctypes.c_uint16, i32]
            lib.or_round.restype = ctypes.c_uint16
            lib.or_round.argtypes = [f64, i32]
            lib.or_cdot.restype = ctypes.c_float
            lib.or_cdot.argtypes = [P, i32, P, i32]
            lib.or_q4_dequant.restype = None
            lib.or_q4_dequant.argtypes = [P, ctypes.c_long, P]
            lib.or_predict.restype = i32
            lib.or_predict.argtypes = [i32, i32, i32, i32, P, P, P, P, P, i32, P, P, P, P, i32]
            lib.or_force_active.restype = i32
            lib.or_force_active.argtypes = [P, i32, i32, P, i32]
            lib.or_union.restype = i32
            lib.or_union.argtypes = [P, i32, i32, P, P]
            lib.or_ffn_act.restype = i32
            lib.or_ffn_act.argtypes = [i32, i32, i32, i32, i32, P, P, P, P, i32, P, i32]
            lib.or_ffn_down.restype = i32
            lib.or_ffn_down.argtypes = [i32, i32, i32, i32, P, P, P, i32, P, i32, P, i32]
            lib.or_rmsnorm.restype = i32
            lib.or_rmsnorm.argtypes = [P, i32, i32, i32, f64, P]
            lib.or_perm_from_counts.restype = i32
            lib.or_perm_from_counts.argtypes = [P, i32, P]
            _lib = lib
    return _lib


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _u16(a):
    return None if a is None else np.ascontiguousarray(a).view(np.uint16)


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what}: invalid arguments (rc={rc})")


# ---------------------------------------------------------------- formats
def to_double(bits, dt: int) -> np.ndarray:
    """Exact value of 16-bit float bit patterns (F16 or BF16) as float64."""
    lib = _load()
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return np.array([lib.or_to_double(int(v), dt) for v in b.ravel()], dtype=np.float64).reshape(b.shape)


def round_to(values, dt: int) -> np.ndarray:
    """Round float64 values to F16/BF16 (nearest, ties to even); bit patterns."""
    lib = _load()
    v = np.ascontiguousarray(values, dtype=np.float64)
    return np.array([lib.or_round(float(x), dt) for x in v.ravel()], dtype=np.uint16).reshape(v.shape)


def q4_dequant(blocks) -> np.ndarray:
    """Q4_0 blocks (uint8, 18 bytes each) -> float64 weights, 32 per block."""
    lib = _load()
    b = np.ascontiguousarray(blocks, dtype=np.uint8).ravel()
    assert b.size % 18 == 0
    out = np.empty(b.size // 18 * 32, dtype=np.float64)
    lib.or_q4_dequant(_p(b), b.size // 18, _p(out))
    return out


# ---------------------------------------------------------------- predictor
def cdot(w, dt: int, v) -> np.float32:
    """Canonical fp32 dot product of a 16-bit row with an fp32 vector."""
    lib = _load()
    w = _u16(w)
    v = np.ascontiguousarray(v, dtype=np.float32)
    assert w.size == v.size
    return np.float32(lib.or_cdot(_p(w), dt, _p(v), w.size))


def predict(W1, b1, W2, b2, xhat, dt: int, nthreads: int | None = None, hot=None):
    """Per-token predicted masks.

    W1 [r,d], b1 [r] or None, W2 [n,r], b2 [n] or None, xhat [B,d] as 16-bit
    bit patterns (uint16) of dtype ``dt``.  Returns dict with ``mask`` (bool
    [B,n]), ``z`` (fp32 canonical logits), ``z64`` (fp64 logits), ``h`` (fp32
    hidden [B,r]).  ``hot``: ids of hot neurons, active for every token
    whatever their logits (``z`` still holds those)."""
    lib = _load()
    W1, W2, xhat = _u16(W1), _u16(W2), _u16(xhat)
    b1, b2 = _u16(b1), _u16(b2)
    r, d = W1.shape
    n = W2.shape[0]
    assert W2.shape[1] == r
    xhat = xhat.reshape(-1, d)
    B = xhat.shape[0]
    h = np.empty((B, r), np.float32)
    z = np.empty((B, n), np.float32)
    z64 = np.empty((B, n), np.float64)
    mask = np.empty((B, n), np.uint8)
    rc = lib.or_predict(d, n, r, dt, _p(W1), _p(b1), _p(W2), _p(b2), _p(xhat), B,
                        _p(h), _p(z), _p(z64), _p(mask), nthreads or default_threads())
    _check(rc, "predict")
    if hot is not None:
        ids = np.ascontiguousarray(hot, dtype=np.int32)
        _check(lib.or_force_active(_p(mask), B, n, _p(ids) if ids.size else None, int(ids.size)), "force_active")
    return {"mask": mask.astype(bool), "z": z, "z64": z64, "h": h}


def union(mask) -> np.ndarray:
    """Ascending list of neurons active for any token of the batch."""
    lib = _load()
    m = np.ascontiguousarray(mask, dtype=np.uint8)
    if m.ndim == 1:
        m = m[None]
    B, n = m.shape
    idx = np.empty(n, np.int32)
    cnt = np.zeros(1, np.int32)
    _check(lib.or_union(_p(m), B, n, _p(idx), _p(cnt)), "union")
    return idx[: int(cnt[0])].copy()


# ---------------------------------------------------------------- FFN
def ffn_act(Wup, Wgate, b, xhat, act: int, wdt: int, adt: int, nthreads: int | None = None):
    """fp64 activations a[B,n] of every neuron (ReLU, ReGLU or squared ReLU)."""
    lib = _load()
    xhat = _u16(xhat)
    if wdt == Q4_0:
        Wup = np.ascontiguousarray(Wup, dtype=np.uint8)
        Wgate = None if Wgate is None else np.ascontiguousarray(Wgate, dtype=np.uint8)
        n = Wup.shape[0]
        d = Wup.shape[1] // 18 * 32
    else:
        Wup, Wgate = _u16(Wup), _u16(Wgate)
        n, d = Wup.shape
    xhat = xhat.reshape(-1, d)
    B = xhat.shape[0]
    a = np.empty((B, n), np.float64)
    rc = lib.or_ffn_act(d, n, act, wdt, adt, _p(Wup), _p(Wgate), _p(_u16(b)), _p(xhat), B, _p(a),
                        nthreads or default_threads())
    _check(rc, "ffn_act")
    return a


def ffn_down(Wdown, bdown, a, idx, wdt: int, adt: int, nthreads: int | None = None):
    """y[B,d] = sum over listed neurons of a[:,i] * W_down[:,i] (+ b_down), fp64.

    Dense W_down is the model's [d,n] matrix; a Q4_0 W_down is given transposed
    as [n] rows of Q4_0 blocks along d."""
    lib = _load()
    a = np.ascontiguousarray(a, dtype=np.float64)
    if a.ndim == 1:
        a = a[None]
    B, n = a.shape
    if wdt == Q4_0:
        Wdown = np.ascontiguousarray(Wdown, dtype=np.uint8)
        assert Wdown.shape[0] == n
        d = Wdown.shape[1] // 18 * 32
    else:
        Wdown = _u16(Wdown)
        d = Wdown.shape[0]
        assert Wdown.shape[1] == n
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    y = np.empty((B, d), np.float64)
    rc = lib.or_ffn_down(d, n, wdt, adt, _p(Wdown), _p(_u16(bdown)), _p(a), B,
                         _p(idx) if idx.size else None, int(idx.size), _p(y), nthreads or default_threads())
    _check(rc, "ffn_down")
    return y


def masked_ffn(layer: dict, xhat, idx, nthreads: int | None = None):
    """Masked FFN of a layer dict (see ``workload``) on the neurons of ``idx``."""
    a = ffn_act(layer["w_up"], layer.get("w_gate"), layer["b"], xhat, layer["act"],
                layer["w_dtype"], layer["act_dtype"], nthreads)
    return ffn_down(layer["w_down"], layer.get("b_down"), a, idx, layer["w_dtype"],
                    layer["act_dtype"], nthreads)


def layer_predict(layer: dict, xhat, nthreads: int | None = None, hot=None):
    return predict(layer["p_w1"], layer.get("p_b1"), layer["p_w2"], layer.get("p_b2"), xhat,
                   layer["act_dtype"], nthreads, hot)


# ---------------------------------------------------------------- stack / load
def rmsnorm(x, dt: int, eps: float = 1e-5) -> np.ndarray:
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float32)
    if x.ndim == 1:
        x = x[None]
    B, d = x.shape
    out = np.empty((B, d), np.uint16)
    _check(lib.or_rmsnorm(_p(x), B, d, dt, eps, _p(out)), "rmsnorm")
    return out


def perm_from_counts(counts) -> np.ndarray:
    """Physical order of neurons: descending count, ties to the lower id."""
    lib = _load()
    c = np.ascontiguousarray(counts, dtype=np.int32)
    perm = np.empty(c.size, np.int32)
    _check(lib.or_perm_from_counts(_p(c), c.size, _p(perm)), "perm_from_counts")
    return perm
