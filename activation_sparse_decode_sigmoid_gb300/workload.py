"""Seeded synthetic workloads: power-law-sparse FFN layers with predictors.

This module only draws inputs.  It holds none of the method's arithmetic and
serves both the CUDA library's callers and the CPU oracle, which always work on
the same bytes.

Shapes follow the models the PowerInfer pages evaluate (OPT-30B, LLaMA(ReGLU)-
70B, Falcon(ReLU)-40B; blog.csdn.net QbitAI/IPADS article, "推理速度最高11倍")
and the power-law activation statistics they report (section
"稀疏激活带来的推理局部性": a few hot neurons fire for most inputs; about 10% of
an OPT FFN's neurons suffice, section "何谓'稀疏激活'").  No checkpoints,
predictor weights or calibration corpora exist here; these layers stand in.

Recipe (per layer, all seeded):
  * activation probability of the neuron with popularity rank k:
    p = min(0.9, c * k**-alpha), c solved by bisection so that mean(p) = rho;
    the p values are assigned to neurons by a seeded shuffle;
  * W_up, W_gate ~ N(0, 1/d_model), W_down ~ N(0, 1/d_ffn), predictor
    W1 ~ N(0, 1/d_model), W2 ~ N(0, 1/rank) (fan-in scaling);
  * FFN bias (on the gate for ReGLU) b = Phi^-1(p), so that with a unit-RMS
    input P(neuron fires) = p;
  * predictor output bias b2 = Phi^-1(p) / sqrt(2) (std of W2 h is 1/sqrt(2)),
    so that the random predictor selects about rho of the neurons;
  * b1 = 0 and b_down = 0 unless a test asks for random ones;
  * decode inputs x ~ N(0, 1) in fp32; calibration inputs x_hat ~ N(0, 1)
    rounded to the activation dtype, from seed + 1.
"""
from __future__ import annotations

import hashlib
import math
from dataclasses import dataclass, field, replace

import numpy as np

F16, BF16, Q4_0 = 0, 1, 2
RELU, REGLU, SQRELU = 0, 1, 2
DTYPE_NAMES = {F16: "f16", BF16: "bf16", Q4_0: "q4_0"}


@dataclass(frozen=True)
class LayerConfig:
    name: str
    d: int                 # d_model
    n: int                 # d_ffn (neurons)
    r: int                 # predictor rank
    L: int                 # layers in the stack
    act: int               # RELU / REGLU / SQRELU
    w_dtype: int           # F16 / BF16 / Q4_0 (FFN matrices)
    act_dtype: int         # F16 / BF16 (activations, predictor, biases)
    alpha: float           # Zipf exponent of the activation probabilities
    rho: float = 0.10      # mean activation probability
    batches: tuple = (1,)
    tokens: int = 64
    prompt: int = 0
    cfg_id: int = 0
    notes: str = field(default="", compare=False)

    def scaled(self, **kw) -> "LayerConfig":
        return replace(self, **kw)


CONFIGS = {
    # one OPT-style ReLU layer, fp16
    "opt_1layer_relu_f16": LayerConfig("opt_1layer_relu_f16", 1024, 4096, 128, 1, RELU, F16, F16,
                                       alpha=0.8, batches=(1,), tokens=64, cfg_id=1),
    # OPT-30B-shaped ReLU stack, fp16
    "opt30b_relu_f16": LayerConfig("opt30b_relu_f16", 7168, 28672, 1024, 48, RELU, F16, F16,
                                   alpha=1.0, batches=(1,), tokens=128, cfg_id=2),
    # LLaMA-70B-shaped ReGLU stack, bf16
    "llama70b_reglu_bf16": LayerConfig("llama70b_reglu_bf16", 8192, 28672, 1024, 80, REGLU, BF16, BF16,
                                       alpha=0.7, batches=(1, 8), tokens=64, cfg_id=3),
    # Falcon-40B(ReLU)-shaped stack, fp16, batch sweep
    "falcon40b_relu_f16": LayerConfig("falcon40b_relu_f16", 8192, 32768, 1024, 60, RELU, F16, F16,
                                      alpha=0.9, batches=(1, 4, 16, 32), tokens=64, cfg_id=4),
    # Falcon-40B-shaped stack with Q4_0 FFN weights, fp16 predictor
    "falcon40b_relu_q4": LayerConfig("falcon40b_relu_q4", 8192, 32768, 1024, 60, RELU, Q4_0, F16,
                                     alpha=0.9, batches=(64, 1), tokens=128, prompt=64, cfg_id=5),
    # the third activation family on OPT-30B shapes: squared ReLU, fp16 (measurement of that
    # family; the pages name no model for it)
    "opt30b_sqrelu_f16": LayerConfig("opt30b_sqrelu_f16", 7168, 28672, 1024, 48, SQRELU, F16, F16,
                                     alpha=1.0, batches=(1, 8), tokens=128, cfg_id=6),
}

# tensor ids for keyed random streams
_T = {"p": 1, "w_up": 2, "w_gate": 3, "w_down": 4, "p_w1": 5, "p_w2": 6, "b1": 7, "bdown": 8,
      "x": 9, "cal": 10}


def _key(seed: int, cfg_id: int, layer: int, tensor: str) -> list:
    return [int(seed), int(cfg_id), int(layer), _T[tensor]]


def rng_for(seed: int, cfg_id: int, layer: int, tensor: str) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(_key(seed, cfg_id, layer, tensor))))


def torch_seed_for(seed: int, cfg_id: int, layer: int, tensor: str) -> int:
    h = hashlib.sha256(repr(_key(seed, cfg_id, layer, tensor)).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


# ------------------------------------------------------------------ probabilities
def zipf_scale(n: int, alpha: float, rho: float, pmax: float = 0.9) -> float:
    """c such that mean(min(pmax, c * k**-alpha)), k = 1..n, equals rho."""
    k = np.arange(1, n + 1, dtype=np.float64) ** (-alpha)
    lo, hi = 0.0, 1.0
    while np.minimum(pmax, hi * k).mean() < rho:
        hi *= 2.0
        if hi > 1e30:
            raise ValueError("rho not reachable")
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        if np.minimum(pmax, mid * k).mean() < rho:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


def activation_probs(cfg: LayerConfig, layer: int, seed: int = 0) -> np.ndarray:
    """Per-neuron activation probabilities (original neuron order)."""
    c = zipf_scale(cfg.n, cfg.alpha, cfg.rho)
    p_sorted = np.minimum(0.9, c * np.arange(1, cfg.n + 1, dtype=np.float64) ** (-cfg.alpha))
    order = rng_for(seed, cfg.cfg_id, layer, "p").permutation(cfg.n)
    p = np.empty(cfg.n)
    p[order] = p_sorted
    return p


def probit(p: np.ndarray) -> np.ndarray:
    from scipy.special import ndtri
    return ndtri(p)


# ------------------------------------------------------------------ 16-bit encodings
def to_bits(values: np.ndarray, dt: int) -> np.ndarray:
    """float -> 16-bit bit patterns, round to nearest even."""
    v = np.asarray(values)
    if dt == F16:
        return v.astype(np.float16).view(np.uint16)
    if dt == BF16:
        u = np.ascontiguousarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
        nan = np.isnan(np.asarray(v, dtype=np.float32))
        r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
        r[nan] = 0x7FC0
        return r
    raise ValueError(dt)


def from_bits(bits: np.ndarray, dt: int) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    if dt == F16:
        return b.view(np.float16).astype(np.float32)
    if dt == BF16:
        return (b.astype(np.uint32) << 16).view(np.float32)
    raise ValueError(dt)


# ------------------------------------------------------------------ Q4_0 packing (test data)
def q4_quantize(w: np.ndarray) -> np.ndarray:
    """Rows of float weights [rows, cols] -> Q4_0 blocks [rows, cols/32*18] (uint8).

    Block of 32: m = the signed value of largest magnitude, s = m / -8 stored
    as fp16, q = clamp(round_half_even(w / s) + 8, 0, 15); s = 0 gives q = 8.
    Element j < 16 goes to the low nibble of byte j, j >= 16 to the high
    nibble of byte j - 16."""
    w = np.asarray(w, dtype=np.float32)
    rows, cols = w.shape
    assert cols % 32 == 0
    blk = w.reshape(rows, cols // 32, 32)
    amax_i = np.abs(blk).argmax(axis=2)
    m = np.take_along_axis(blk, amax_i[..., None], axis=2)[..., 0]
    s = m / -8.0
    s16 = s.astype(np.float16)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(s[..., None] != 0, np.rint(blk / np.where(s == 0, 1, s)[..., None]) + 8, 8)
    q = np.clip(q, 0, 15).astype(np.uint8)
    out = np.empty((rows, cols // 32, 18), np.uint8)
    out[..., 0:2] = s16.view(np.uint8).reshape(rows, cols // 32, 2)
    out[..., 2:18] = q[..., :16] | (q[..., 16:] << 4)
    return out.reshape(rows, cols // 32 * 18)


# ------------------------------------------------------------------ host layers
def make_layer(cfg: LayerConfig, layer: int = 0, seed: int = 0, *, random_b1: bool = False,
               random_bdown: bool = False) -> dict:
    """One layer as host numpy arrays (16-bit bit patterns as uint16, Q4_0 as uint8).

    Keys: w_up [n,d], w_gate [n,d] (ReGLU), b [n], w_down [d,n] (Q4_0: the
    transposed matrix as [n] rows of blocks along d), b_down [d] or None,
    p_w1 [r,d], p_b1 [r] or None, p_w2 [n,r], p_b2 [n], p (probabilities)."""
    d, n, r = cfg.d, cfg.n, cfg.r
    adt = cfg.act_dtype
    p = activation_probs(cfg, layer, seed)
    bias = probit(p)

    def normal(tensor, shape, std):
        g = rng_for(seed, cfg.cfg_id, layer, tensor)
        return g.standard_normal(shape, dtype=np.float32) * np.float32(std)

    out = {"d": d, "n": n, "r": r, "act": cfg.act, "w_dtype": cfg.w_dtype, "act_dtype": adt, "p": p}
    w_up = normal("w_up", (n, d), 1.0 / math.sqrt(d))
    w_gate = normal("w_gate", (n, d), 1.0 / math.sqrt(d)) if cfg.act == REGLU else None
    w_down = normal("w_down", (d, n), 1.0 / math.sqrt(n))
    if cfg.w_dtype == Q4_0:
        out["w_up"] = q4_quantize(w_up)
        out["w_gate"] = None if w_gate is None else q4_quantize(w_gate)
        out["w_down"] = q4_quantize(np.ascontiguousarray(w_down.T))
    else:
        out["w_up"] = to_bits(w_up, cfg.w_dtype)
        out["w_gate"] = None if w_gate is None else to_bits(w_gate, cfg.w_dtype)
        out["w_down"] = to_bits(w_down, cfg.w_dtype)
    out["b"] = to_bits(bias.astype(np.float32), adt)
    out["b_down"] = to_bits(normal("bdown", (d,), 0.1), adt) if random_bdown else None
    out["p_w1"] = to_bits(normal("p_w1", (r, d), 1.0 / math.sqrt(d)), adt)
    out["p_b1"] = to_bits(normal("b1", (r,), 0.1), adt) if random_b1 else None
    out["p_w2"] = to_bits(normal("p_w2", (n, r), 1.0 / math.sqrt(r)), adt)
    out["p_b2"] = to_bits((bias / math.sqrt(2.0)).astype(np.float32), adt)
    return out


def decode_inputs(cfg: LayerConfig, T: int, seed: int = 0) -> np.ndarray:
    """T residual-stream inputs x ~ N(0,1), fp32 [T, d]."""
    return rng_for(seed, cfg.cfg_id, 0, "x").standard_normal((T, cfg.d), dtype=np.float32)


def xhat_inputs(cfg: LayerConfig, T: int, seed: int = 0, layer: int = 0) -> np.ndarray:
    """T normalised-scale layer inputs x_hat ~ N(0,1) as 16-bit patterns [T, d]."""
    g = rng_for(seed, cfg.cfg_id, layer, "x")
    return to_bits(g.standard_normal((T, cfg.d), dtype=np.float32), cfg.act_dtype)


def calibration_inputs(cfg: LayerConfig, layer: int, seed: int = 0, T: int = 256) -> np.ndarray:
    """Calibration x_hat for the offline activation-frequency profile (seed + 1)."""
    g = rng_for(seed + 1, cfg.cfg_id, layer, "cal")
    return to_bits(g.standard_normal((T, cfg.d), dtype=np.float32), cfg.act_dtype)


# ------------------------------------------------------------------ device layers (large stacks)
def make_layer_device(cfg: LayerConfig, layer: int, seed: int, device, chunk_rows: int = 4096):
    """Same recipe as :func:`make_layer`, drawn on the GPU with torch (for the
    multi-GB stacks).  Returns torch tensors; the oracle copies back the bytes
    of any layer it checks.  16-bit tensors are returned as int16 views."""
    import torch

    d, n, r = cfg.d, cfg.n, cfg.r
    adt = cfg.act_dtype
    tdt = {F16: torch.float16, BF16: torch.bfloat16}

    def normal(tensor, shape, std, dt):
        g = torch.Generator(device=device)
        g.manual_seed(torch_seed_for(seed, cfg.cfg_id, layer, tensor))
        out = torch.empty(shape, dtype=dt, device=device)
        rows = shape[0]
        for r0 in range(0, rows, chunk_rows):
            r1 = min(rows, r0 + chunk_rows)
            tmp = torch.randn((r1 - r0,) + tuple(shape[1:]), generator=g, device=device, dtype=torch.float32)
            out[r0:r1] = (tmp * std).to(dt)
        return out

    p = activation_probs(cfg, layer, seed)
    bias = probit(p)
    out = {"d": d, "n": n, "r": r, "act": cfg.act, "w_dtype": cfg.w_dtype, "act_dtype": adt, "p": p}
    if cfg.w_dtype == Q4_0:
        f32 = torch.float32
        out["w_up"] = q4_quantize_torch(normal("w_up", (n, d), 1.0 / math.sqrt(d), f32))
        out["w_gate"] = (q4_quantize_torch(normal("w_gate", (n, d), 1.0 / math.sqrt(d), f32))
                         if cfg.act == REGLU else None)
        wd = normal("w_down", (d, n), 1.0 / math.sqrt(n), f32)
        out["w_down"] = q4_quantize_torch(wd.t().contiguous())
        del wd
    else:
        wdt = tdt[cfg.w_dtype]
        out["w_up"] = normal("w_up", (n, d), 1.0 / math.sqrt(d), wdt).view(torch.int16)
        out["w_gate"] = (normal("w_gate", (n, d), 1.0 / math.sqrt(d), wdt).view(torch.int16)
                         if cfg.act == REGLU else None)
        out["w_down"] = normal("w_down", (d, n), 1.0 / math.sqrt(n), wdt).view(torch.int16)
    out["b"] = torch.from_numpy(to_bits(bias.astype(np.float32), adt).view(np.int16)).to(device)
    out["b_down"] = None
    out["p_w1"] = normal("p_w1", (r, d), 1.0 / math.sqrt(d), tdt[adt]).view(torch.int16)
    out["p_b1"] = None
    out["p_w2"] = normal("p_w2", (n, r), 1.0 / math.sqrt(r), tdt[adt]).view(torch.int16)
    out["p_b2"] = torch.from_numpy(to_bits((bias / math.sqrt(2.0)).astype(np.float32), adt)
                                   .view(np.int16)).to(device)
    return out


def q4_quantize_torch(w, chunk_rows: int = 4096):
    """Device version of :func:`q4_quantize` (same rule, torch ops)."""
    import torch

    rows, cols = w.shape
    assert cols % 32 == 0
    out = torch.empty((rows, cols // 32, 18), dtype=torch.uint8, device=w.device)
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        blk = w[r0:r1].float().reshape(r1 - r0, cols // 32, 32)
        amax_i = blk.abs().argmax(dim=2, keepdim=True)
        m = torch.gather(blk, 2, amax_i)[..., 0]
        s = m / -8.0
        safe = torch.where(s == 0, torch.ones_like(s), s)
        q = torch.where(s[..., None] != 0, torch.round(blk / safe[..., None]) + 8, torch.full_like(blk, 8))
        q = q.clamp(0, 15).to(torch.uint8)
        out[r0:r1, :, 0:2] = s.to(torch.float16).view(torch.uint8).reshape(r1 - r0, cols // 32, 2)
        out[r0:r1, :, 2:18] = q[..., :16] | (q[..., 16:] << 4)
    return out.reshape(rows, cols // 32 * 18)


def layer_to_host(layer: dict) -> dict:
    """Copy a device layer (torch tensors) to host numpy arrays for the oracle."""
    out = {}
    for k, v in layer.items():
        if hasattr(v, "detach"):
            a = v.detach().cpu().numpy()
            out[k] = a.view(np.uint16) if a.dtype == np.int16 else a
        else:
            out[k] = v
    return out
