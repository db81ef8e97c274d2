"""Thin Python binding of libpi (include/pi.h): same entry-point names,
argument marshalling only.  Every step of the hot path runs in the library's
CUDA kernels; there is no CPU fallback.  If ``_build/libpi.so`` is missing this
module raises on first use -- build it with
``python -m activation_sparse_decode_sigmoid_gb300.build``.

Tensors are torch tensors on the context's device (PyTorch supplies device
memory and streams only).  16-bit data may be passed as float16 / bfloat16 or
as int16 / uint16 views of the bit patterns.  Every compute call is issued on
torch's current CUDA stream.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libpi.so")

PI_OK = 0
PI_ERR_ARG, PI_ERR_SHAPE, PI_ERR_CUDA, PI_ERR_OOM = -1, -2, -3, -4
PI_ERR_NOT_LOADED, PI_ERR_TIMEOUT, PI_ERR_DEVICE_FLAG, PI_ERR_UNSUPPORTED = -5, -6, -7, -8
PI_RELU, PI_REGLU, PI_SQRELU = 0, 1, 2
PI_F16, PI_BF16, PI_Q4_0 = 0, 1, 2

# every symbol include/pi.h declares
EXPORTS = ("pi_create", "pi_destroy", "pi_set_stream", "pi_load_layer", "pi_layer_counts",
           "pi_perm_from_counts", "pi_predict", "pi_sparse_ffn", "pi_dense_ffn", "pi_decode_step",
           "pi_decode_step_host",
           "pi_dense_step", "pi_set_trace", "pi_sync_status", "pi_last_error", "pi_grid_size",
           "pi_debug_set_wait_limit", "pi_debug_barrier_extra", "pi_debug_set_timeline",
           "pi_debug_set_tuning", "pi_debug_copy_hidden", "pi_debug_set_mma_min_batch",
           "pi_sparse_ffn_noalloc", "pi_set_hot_prefix", "pi_hot_prefix_crossover", "pi_choose_hot_prefix",
           "pi_layerwise_min_batch", "pi_load_layer_shard", "pi_layer_shard", "pi_layer_partial",
           "pi_residual_add")


class PiError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"libpi status {status}: {msg}")
        self.status = status


class pi_layer_desc(ctypes.Structure):
    _fields_ = [("d_model", ctypes.c_int32), ("d_ffn", ctypes.c_int32), ("rank", ctypes.c_int32),
                ("act", ctypes.c_int32), ("w_dtype", ctypes.c_int32), ("act_dtype", ctypes.c_int32)]


class pi_ffn_rows(ctypes.Structure):
    _fields_ = [("d_model", ctypes.c_int32), ("d_ffn", ctypes.c_int32), ("act", ctypes.c_int32),
                ("act_dtype", ctypes.c_int32), ("up", ctypes.c_void_p), ("gate", ctypes.c_void_p),
                ("down_rows", ctypes.c_void_p), ("b", ctypes.c_void_p), ("b_down", ctypes.c_void_p)]


class pi_layer_weights(ctypes.Structure):
    _fields_ = [("w_up", ctypes.c_void_p), ("w_gate", ctypes.c_void_p), ("b", ctypes.c_void_p),
                ("w_down", ctypes.c_void_p), ("b_down", ctypes.c_void_p), ("p_w1", ctypes.c_void_p),
                ("p_b1", ctypes.c_void_p), ("p_w2", ctypes.c_void_p), ("p_b2", ctypes.c_void_p),
                ("on_device", ctypes.c_int32)]


_lib = None


def load_library(path: str = LIB_PATH):
    """Load libpi.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"libpi.so not built ({path}); run python -m activation_sparse_decode_sigmoid_gb300.build")
    lib = ctypes.CDLL(path)
    P, I32, st = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32
    sig = {
        "pi_create": (st, [ctypes.POINTER(P), I32, P, I32, I32]),
        "pi_destroy": (st, [P]),
        "pi_set_stream": (st, [P, P]),
        "pi_load_layer": (st, [P, I32, ctypes.POINTER(pi_layer_desc), ctypes.POINTER(pi_layer_weights), P]),
        "pi_layer_counts": (st, [P, I32, P, I32, P]),
        "pi_perm_from_counts": (st, [P, I32, P]),
        "pi_predict": (st, [P, I32, P, I32, P, P]),
        "pi_sparse_ffn": (st, [P, I32, P, I32, P, P, P]),
        "pi_dense_ffn": (st, [P, I32, P, I32, P]),
        "pi_decode_step": (st, [P, P, I32]),
        "pi_decode_step_host": (st, [P, P, P, I32]),
        "pi_dense_step": (st, [P, P, I32]),
        "pi_set_trace": (st, [P, P, P, P, P]),
        "pi_sync_status": (st, [P]),
        "pi_last_error": (ctypes.c_char_p, [P]),
        "pi_grid_size": (I32, [P]),
        "pi_debug_set_wait_limit": (st, [P, ctypes.c_uint64]),
        "pi_debug_barrier_extra": (st, [P, I32]),
        "pi_debug_set_timeline": (st, [P, P, I32]),
        "pi_debug_set_tuning": (st, [P, I32, I32, I32, I32]),
        "pi_debug_copy_hidden": (st, [P, P, I32]),
        "pi_debug_set_mma_min_batch": (st, [P, I32]),
        "pi_sparse_ffn_noalloc": (st, [ctypes.POINTER(pi_ffn_rows), P, I32, P, P, P, P, P]),
        "pi_set_hot_prefix": (st, [P, I32, I32]),
        "pi_layerwise_min_batch": (st, [P, I32, P]),
        "pi_hot_prefix_crossover": (st, [P, I32, I32, I32, ctypes.c_double, ctypes.c_double, P]),
        "pi_choose_hot_prefix": (st, [P, I32, P, I32, I32, P]),
        "pi_load_layer_shard": (st, [P, I32, ctypes.POINTER(pi_layer_desc), ctypes.POINTER(pi_layer_weights), P,
                                     I32, I32]),
        "pi_layer_shard": (st, [P, I32, P, P]),
        "pi_layer_partial": (st, [P, I32, P, I32, P]),
        "pi_residual_add": (st, [P, P, P, I32]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return t.data_ptr()


def _stream_ptr(device) -> int:
    import torch
    return torch.cuda.current_stream(device).cuda_stream


# ---------------------------------------------------------------- same-named calls
def pi_create(device: int = 0, stream: int | None = None, max_layers: int = 1, max_batch: int = 1) -> int:
    lib = load_library()
    h = ctypes.c_void_p()
    rc = lib.pi_create(ctypes.byref(h), device, stream, max_layers, max_batch)
    if rc:
        raise PiError(rc, "pi_create failed")
    return h.value


def _check(ctx, rc, what):
    if rc:
        msg = load_library().pi_last_error(ctx)
        raise PiError(rc, f"{what}: {msg.decode() if msg else ''}")


def pi_destroy(ctx: int) -> None:
    _check(ctx, load_library().pi_destroy(ctx), "pi_destroy")


def pi_set_stream(ctx: int, stream: int | None) -> None:
    _check(ctx, load_library().pi_set_stream(ctx, stream), "pi_set_stream")


def pi_load_layer(ctx: int, layer: int, desc: pi_layer_desc, weights: pi_layer_weights, perm=None) -> None:
    perm_arr = None if perm is None else np.ascontiguousarray(perm, dtype=np.int32)
    rc = load_library().pi_load_layer(ctx, layer, ctypes.byref(desc), ctypes.byref(weights), _ptr(perm_arr))
    _check(ctx, rc, "pi_load_layer")


def pi_load_layer_shard(ctx: int, layer: int, desc: pi_layer_desc, weights: pi_layer_weights, perm, shard: int,
                        nshards: int) -> None:
    perm_arr = None if perm is None else np.ascontiguousarray(perm, dtype=np.int32)
    rc = load_library().pi_load_layer_shard(ctx, layer, ctypes.byref(desc), ctypes.byref(weights), _ptr(perm_arr),
                                            shard, nshards)
    _check(ctx, rc, "pi_load_layer_shard")


def pi_layer_shard(ctx: int, layer: int) -> tuple[int, int]:
    v = np.zeros(2, np.int32)
    _check(ctx, load_library().pi_layer_shard(ctx, layer, _ptr(v[0:1]), _ptr(v[1:2])), "pi_layer_shard")
    return int(v[0]), int(v[1])


def pi_layer_partial(ctx: int, layer: int, x, B: int, u) -> None:
    _check(ctx, load_library().pi_layer_partial(ctx, layer, _ptr(x), B, _ptr(u)), "pi_layer_partial")


def pi_residual_add(ctx: int, x, u, B: int) -> None:
    _check(ctx, load_library().pi_residual_add(ctx, _ptr(x), _ptr(u), B), "pi_residual_add")


def pi_layer_counts(ctx: int, layer: int, x_hat, T: int, counts) -> None:
    _check(ctx, load_library().pi_layer_counts(ctx, layer, _ptr(x_hat), T, _ptr(counts)), "pi_layer_counts")


def pi_perm_from_counts(counts) -> np.ndarray:
    c = np.ascontiguousarray(counts, dtype=np.int32)
    perm = np.empty(c.size, np.int32)
    rc = load_library().pi_perm_from_counts(_ptr(c), c.size, _ptr(perm))
    if rc:
        raise PiError(rc, "pi_perm_from_counts")
    return perm


def pi_set_hot_prefix(ctx: int, layer: int, hot: int) -> None:
    _check(ctx, load_library().pi_set_hot_prefix(ctx, layer, hot), "pi_set_hot_prefix")


def pi_hot_prefix_crossover(counts, T: int, B: int, pred_bytes: float, ffn_bytes: float) -> int:
    c = np.ascontiguousarray(counts, dtype=np.int32)
    hot = np.zeros(1, np.int32)
    rc = load_library().pi_hot_prefix_crossover(_ptr(c), c.size, T, B, pred_bytes, ffn_bytes, _ptr(hot))
    if rc:
        raise PiError(rc, "pi_hot_prefix_crossover")
    return int(hot[0])


def pi_choose_hot_prefix(ctx: int, layer: int, counts, T: int, B: int) -> int:
    c = np.ascontiguousarray(counts, dtype=np.int32)
    hot = np.zeros(1, np.int32)
    _check(ctx, load_library().pi_choose_hot_prefix(ctx, layer, _ptr(c), T, B, _ptr(hot)), "pi_choose_hot_prefix")
    return int(hot[0])


def pi_predict(ctx: int, layer: int, x_hat, B: int, idx, count) -> None:
    _check(ctx, load_library().pi_predict(ctx, layer, _ptr(x_hat), B, _ptr(idx), _ptr(count)), "pi_predict")


def pi_sparse_ffn(ctx: int, layer: int, x_hat, B: int, idx, count, y) -> None:
    rc = load_library().pi_sparse_ffn(ctx, layer, _ptr(x_hat), B, _ptr(idx), _ptr(count), _ptr(y))
    _check(ctx, rc, "pi_sparse_ffn")


def pi_sparse_ffn_noalloc(rows: pi_ffn_rows, x_hat, B: int, idx, count, y, dev_status=None,
                          stream: int | None = None) -> int:
    """Context-free sparse FFN that allocates nothing (for callers that may
    not call cudaMalloc); scratch lives in a fixed per-GPU array inside the
    library.  Returns the status instead of raising.  `stream` defaults to
    torch's current stream."""
    if stream is None:
        import torch
        stream = torch.cuda.current_stream().cuda_stream
    return load_library().pi_sparse_ffn_noalloc(ctypes.byref(rows), _ptr(x_hat), B, _ptr(idx), _ptr(count),
                                                 _ptr(y), _ptr(dev_status), stream)


def pi_dense_ffn(ctx: int, layer: int, x_hat, B: int, y) -> None:
    _check(ctx, load_library().pi_dense_ffn(ctx, layer, _ptr(x_hat), B, _ptr(y)), "pi_dense_ffn")


def pi_decode_step(ctx: int, x, B: int) -> None:
    _check(ctx, load_library().pi_decode_step(ctx, _ptr(x), B), "pi_decode_step")


def pi_decode_step_host(ctx: int, x_in, x_out, B: int) -> None:
    """x_in / x_out: host fp32 [B][d] (numpy arrays or CPU tensors, ideally pinned)."""
    _check(ctx, load_library().pi_decode_step_host(ctx, _ptr(x_in), _ptr(x_out), B), "pi_decode_step_host")


def pi_dense_step(ctx: int, x, B: int) -> None:
    _check(ctx, load_library().pi_dense_step(ctx, _ptr(x), B), "pi_dense_step")


def pi_set_trace(ctx: int, x_trace=None, xhat_trace=None, idx_trace=None, count_trace=None) -> None:
    rc = load_library().pi_set_trace(ctx, _ptr(x_trace), _ptr(xhat_trace), _ptr(idx_trace), _ptr(count_trace))
    _check(ctx, rc, "pi_set_trace")


def pi_sync_status(ctx: int) -> int:
    """Returns the status (0 = OK) instead of raising, so callers can test it."""
    return load_library().pi_sync_status(ctx)


def pi_last_error(ctx: int) -> str:
    m = load_library().pi_last_error(ctx)
    return m.decode() if m else ""


def pi_grid_size(ctx: int) -> int:
    return load_library().pi_grid_size(ctx)


def pi_debug_set_wait_limit(ctx: int, ns: int) -> None:
    _check(ctx, load_library().pi_debug_set_wait_limit(ctx, ns), "pi_debug_set_wait_limit")


def pi_debug_set_timeline(ctx: int, stamps=None, per_cta: int = 0) -> None:
    _check(ctx, load_library().pi_debug_set_timeline(ctx, _ptr(stamps), per_cta), "pi_debug_set_timeline")


def pi_debug_set_tuning(ctx: int, prefetch: int, prefetch_ns: int, lookahead: int, rows_ahead: int = 0) -> None:
    rc = load_library().pi_debug_set_tuning(ctx, prefetch, prefetch_ns, lookahead, rows_ahead)
    _check(ctx, rc, "pi_debug_set_tuning")


def pi_debug_copy_hidden(ctx: int, dst, count: int) -> None:
    _check(ctx, load_library().pi_debug_copy_hidden(ctx, _ptr(dst), count), "pi_debug_copy_hidden")


def pi_debug_set_mma_min_batch(ctx: int, min_batch: int) -> None:
    _check(ctx, load_library().pi_debug_set_mma_min_batch(ctx, min_batch), "pi_debug_set_mma_min_batch")


def pi_layerwise_min_batch(ctx: int, layer: int) -> int:
    mb = np.zeros(1, np.int32)
    _check(ctx, load_library().pi_layerwise_min_batch(ctx, layer, _ptr(mb)), "pi_layerwise_min_batch")
    return int(mb[0])


def pi_debug_barrier_extra(ctx: int, extra: int) -> None:
    _check(ctx, load_library().pi_debug_barrier_extra(ctx, extra), "pi_debug_barrier_extra")


# ---------------------------------------------------------------- convenience wrapper
class Context:
    """Owns a pi_ctx; every call runs on torch's current stream of `device`."""

    def __init__(self, device: int = 0, max_layers: int = 1, max_batch: int = 1):
        import torch
        self.device = device
        self.torch_device = torch.device("cuda", device)
        self.max_layers, self.max_batch = max_layers, max_batch
        self.handle = pi_create(device, _stream_ptr(self.torch_device), max_layers, max_batch)
        self.descs: dict[int, pi_layer_desc] = {}
        self.hot: dict[int, int] = {}  # each layer's always-active prefix

    def close(self):
        if self.handle:
            pi_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _s(self):
        pi_set_stream(self.handle, _stream_ptr(self.torch_device))

    @property
    def grid(self) -> int:
        return pi_grid_size(self.handle)

    # -- loading
    def load_layer(self, layer: int, lw: dict, perm=None) -> None:
        """Load a layer dict as drawn by ``workload.make_layer`` (numpy, host)
        or ``workload.make_layer_device`` (torch, device)."""
        desc, w, keep = self._weights(lw)
        self._s()
        pi_load_layer(self.handle, layer, desc, w, perm)
        self.descs[layer] = desc
        self.hot[layer] = 0
        del keep

    def _weights(self, lw: dict):
        """(descriptor, weight pointers, the buffers they point into) of a layer dict."""
        desc = pi_layer_desc(lw["d"], lw["n"], lw["r"], lw["act"], lw["w_dtype"], lw["act_dtype"])
        keys = ("w_up", "w_gate", "b", "w_down", "b_down", "p_w1", "p_b1", "p_w2", "p_b2")
        vals = [lw.get(k) for k in keys]
        on_dev = any(v is not None and not isinstance(v, np.ndarray) for v in vals)
        keep = []
        ptrs = []
        for v in vals:
            if v is None:
                ptrs.append(None)
                continue
            if on_dev and isinstance(v, np.ndarray):
                import torch
                v = torch.from_numpy(np.ascontiguousarray(v).view(np.int16) if v.dtype == np.uint16 else
                                     np.ascontiguousarray(v)).to(self.torch_device)
            elif isinstance(v, np.ndarray):
                v = np.ascontiguousarray(v)
            else:
                v = v.contiguous()
            keep.append(v)
            ptrs.append(_ptr(v))
        w = pi_layer_weights(*ptrs, 1 if on_dev else 0)
        return desc, w, keep

    def load_layer_shard(self, layer: int, lw: dict, shard: int, nshards: int, perm=None) -> None:
        """Load shard `shard` of `nshards` of a layer dict (its physical
        neurons shard, shard + nshards, ...)."""
        desc, w, keep = self._weights(lw)
        self._s()
        pi_load_layer_shard(self.handle, layer, desc, w, perm, shard, nshards)
        n = lw["n"]
        desc.d_ffn = (n - shard + nshards - 1) // nshards
        self.descs[layer] = desc
        self.hot[layer] = 0
        del keep

    def layer_partial(self, layer: int, x, u=None):
        """The layer's fp32 update of the residual x ([B][d]), not added."""
        import torch
        if u is None:
            u = torch.empty_like(x)
        self._s()
        pi_layer_partial(self.handle, layer, x, x.shape[0], u)
        return u

    def residual_add(self, x, u) -> None:
        self._s()
        pi_residual_add(self.handle, x, u, x.shape[0])

    def layer_counts(self, layer: int, x_hat):
        import torch
        n = self.descs[layer].d_ffn
        counts = torch.zeros(n, dtype=torch.int32, device=self.torch_device)
        self._s()
        pi_layer_counts(self.handle, layer, x_hat, x_hat.shape[0], counts)
        return counts

    def set_hot_prefix(self, layer: int, hot: int) -> None:
        self._s()
        pi_set_hot_prefix(self.handle, layer, hot)
        self.hot[layer] = hot

    def choose_hot_prefix(self, layer: int, counts, T: int, B: int) -> int:
        """Crossover prefix length from calibration counts (host or device, physical order)."""
        if not isinstance(counts, np.ndarray):
            counts = counts.cpu().numpy()
        return pi_choose_hot_prefix(self.handle, layer, counts, T, B)

    # -- hot path
    def predict(self, layer: int, x_hat, idx=None, count=None):
        import torch
        n = self.descs[layer].d_ffn
        if idx is None:
            idx = torch.empty(n, dtype=torch.int32, device=self.torch_device)
        if count is None:
            count = torch.empty(1, dtype=torch.int32, device=self.torch_device)
        self._s()
        pi_predict(self.handle, layer, x_hat, x_hat.shape[0], idx, count)
        return idx, count

    def _y(self, layer, B, y):
        import torch
        if y is None:
            d = self.descs[layer]
            dt = torch.bfloat16 if d.act_dtype == PI_BF16 else torch.float16
            y = torch.empty((B, d.d_model), dtype=dt, device=self.torch_device)
        return y

    def sparse_ffn(self, layer: int, x_hat, idx, count, y=None):
        y = self._y(layer, x_hat.shape[0], y)
        self._s()
        pi_sparse_ffn(self.handle, layer, x_hat, x_hat.shape[0], idx, count, y)
        return y

    def dense_ffn(self, layer: int, x_hat, y=None):
        y = self._y(layer, x_hat.shape[0], y)
        self._s()
        pi_dense_ffn(self.handle, layer, x_hat, x_hat.shape[0], y)
        return y

    def decode_step(self, x) -> None:
        self._s()
        pi_decode_step(self.handle, x, x.shape[0])

    def decode_step_host(self, x_in, x_out) -> None:
        self._s()
        pi_decode_step_host(self.handle, x_in, x_out, x_in.shape[0])

    def dense_step(self, x) -> None:
        self._s()
        pi_dense_step(self.handle, x, x.shape[0])

    def set_trace(self, x_trace=None, xhat_trace=None, idx_trace=None, count_trace=None) -> None:
        pi_set_trace(self.handle, x_trace, xhat_trace, idx_trace, count_trace)

    def sync_status(self) -> int:
        self._s()
        return pi_sync_status(self.handle)

    def check(self) -> None:
        rc = self.sync_status()
        if rc:
            raise PiError(rc, pi_last_error(self.handle))
