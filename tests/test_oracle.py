"""Pins of the CPU oracle against facts that do not come from the oracle itself:
the golden worked example, closed forms, exact integer arithmetic, textbook
library routines (numpy float64 matmul, sort), brute force, error bounds."""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np
import pytest

import oracle as O
from activation_sparse_decode_sigmoid_gb300 import workload as W
from tests._helpers import (dequant_q4_numpy, layer_dense_f64, permute_layer,
                            worked_example_layer)

SMALL = W.LayerConfig("small", 256, 384, 64, 1, W.RELU, W.F16, W.F16, alpha=0.8, cfg_id=101)
SMALL_REGLU = W.LayerConfig("small_reglu", 256, 320, 32, 1, W.REGLU, W.BF16, W.BF16, alpha=0.7, cfg_id=102)
SMALL_Q4 = W.LayerConfig("small_q4", 256, 256, 64, 1, W.RELU, W.Q4_0, W.F16, alpha=0.9, cfg_id=103)
SMALL_SQ = W.LayerConfig("small_sqrelu", 256, 288, 64, 1, W.SQRELU, W.BF16, W.BF16, alpha=0.8, cfg_id=105)


# ------------------------------------------------------------------ number formats
def test_f16_decode_all_patterns():
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = O.to_double(bits, O.F16)
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.array_equal(got[~both_nan], ref[~both_nan])


def test_bf16_decode_all_patterns():
    bits = np.arange(65536, dtype=np.uint16)
    with np.errstate(invalid="ignore"):
        ref = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    got = O.to_double(bits, O.BF16)
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.array_equal(got[~both_nan], ref[~both_nan])


def _nearest_even(v: float, table_vals: list, table_bits: list) -> int:
    """Brute-force round-to-nearest-even over a sorted table of finite values."""
    import bisect
    fv = Fraction(v)
    i = bisect.bisect_left(table_vals, fv)
    cands = [j for j in (i - 1, i) if 0 <= j < len(table_vals)]
    best = min(cands, key=lambda j: (abs(table_vals[j] - fv), table_bits[j] & 1))
    return table_bits[best]


@pytest.mark.parametrize("dt", [O.F16, O.BF16])
def test_round_matches_bruteforce(dt):
    bits = np.arange(0, 0x7C00 if dt == O.F16 else 0x7F80, dtype=np.uint16)  # positive finite
    vals = O.to_double(bits, dt)
    table = sorted(zip((Fraction(float(v)) for v in vals), (int(b) for b in bits)))
    tv, tb = [t[0] for t in table], [t[1] for t in table]
    rng = np.random.default_rng(5)
    lo, hi = (-20, 15) if dt == O.F16 else (-120, 120)
    samples = np.ldexp(rng.uniform(1, 2, 400), rng.integers(lo, hi, 400))
    # exact half-way points between neighbours (ties go to the even pattern)
    mids = [(float(tv[k]) + float(tv[k + 1])) / 2 for k in rng.integers(1, len(tv) - 2, 200)]
    for v in list(samples) + mids:
        want = _nearest_even(float(v), tv, tb)
        got = int(O.round_to(np.array([v]), dt)[0])
        assert got == want, (v, hex(got), hex(want))
        assert int(O.round_to(np.array([-v]), dt)[0]) == want | 0x8000


def test_round_f16_matches_numpy():
    rng = np.random.default_rng(1)
    v = rng.standard_normal(5000) * np.exp(rng.uniform(-12, 11, 5000))
    with np.errstate(over="ignore"):
        want = v.astype(np.float16).view(np.uint16)
    assert np.array_equal(O.round_to(v, O.F16), want)


# ------------------------------------------------------------------ Q4_0
def test_q4_grid_closed_form():
    """Weights on the grid (q-8)*s, hand-packed: dequantise exactly."""
    rng = np.random.default_rng(2)
    for _ in range(20):
        q = rng.integers(0, 16, 32)
        s = np.float16(rng.uniform(-3, 3))
        blk = np.zeros(18, np.uint8)
        blk[0:2] = np.array([s], np.float16).view(np.uint8)
        for j in range(16):
            blk[2 + j] = q[j] | (q[j + 16] << 4)
        want = (q.astype(np.float64) - 8) * float(s)
        assert np.array_equal(O.q4_dequant(blk), want)


def test_q4_quantiser_error_bound():
    rng = np.random.default_rng(3)
    w = rng.standard_normal((8, 256)).astype(np.float32)
    blocks = W.q4_quantize(w)
    deq = O.q4_dequant(blocks).reshape(8, 256)
    assert np.array_equal(deq, dequant_q4_numpy(blocks))
    s = np.abs(dequant_q4_numpy(blocks).reshape(8, 8, 32)).max(axis=2) / 8.0  # |s|
    err = np.abs(deq - w).reshape(8, 8, 32)
    # codes span [-8, 7]: values rounding to +8 are clipped to 7 (error <= |s|),
    # everything else is within half a step (+ the fp16 rounding of s)
    assert np.all(err.max(axis=2) <= s * (1 + 1e-2))
    assert np.mean(err <= s[..., None] * 0.51) > 0.95


# ------------------------------------------------------------------ canonical dot (CDOT)
@pytest.mark.parametrize("K", [1, 7, 8, 13, 255, 256, 257, 1024, 2049, 7168])
@pytest.mark.parametrize("dt", [O.F16, O.BF16])
def test_cdot_integer_exact(K, dt):
    """Small integers: every partial sum is exact in fp32, so any summation
    order gives the exact dot product (catches dropped or repeated terms)."""
    rng = np.random.default_rng(K)
    w = rng.integers(-8, 9, K)
    v = rng.integers(-16, 17, K)
    want = int(np.dot(w.astype(np.int64), v.astype(np.int64)))
    got = O.cdot(W.to_bits(w.astype(np.float32), dt), dt, v.astype(np.float32))
    assert float(got) == float(want)


@pytest.mark.parametrize("K", [64, 1024, 7168, 8192])
def test_cdot_error_bound(K):
    """|CDOT - exact| <= gamma_k * sum|w v| with k = the longest rounding chain."""
    rng = np.random.default_rng(K + 7)
    w = W.to_bits(rng.standard_normal(K).astype(np.float32), O.F16)
    v = rng.standard_normal(K).astype(np.float32)
    wv = O.to_double(w, O.F16)
    prods = [float(a) * float(b) for a, b in zip(wv, v.astype(np.float64))]  # exact in fp64
    exact = math.fsum(prods)
    chain = 8 * math.ceil(K / 256) + 5
    u = 2.0 ** -24
    gamma = chain * u / (1 - chain * u)
    got = float(O.cdot(w, O.F16, v))
    assert abs(got - exact) <= gamma * math.fsum(abs(p) for p in prods)


def test_cdot_order_hand_example():
    """K = 264: lane 0 holds elements 0..7 and 256..263, lane 16 holds 128..135.
    w*v = 2^24 at 0, -2^24 at 128, 1 at 256 and 257.  Lane 0: 2^24 + 1 rounds
    to 2^24 (tie to even) twice, lane 16 = -2^24; the butterfly adds lane 16 to
    lane 0 first, giving 0.  (A left-to-right sum would give 2.)"""
    K = 264
    w = np.zeros(K, np.float32)
    v = np.zeros(K, np.float32)
    w[0], v[0] = 4096, 4096
    w[128], v[128] = -4096, 4096
    w[256], v[256] = 1, 1
    w[257], v[257] = 1, 1
    assert float(O.cdot(W.to_bits(w, O.F16), O.F16, v)) == 0.0
    # moving the +1s into lane 1 (elements 8, 9) keeps them out of lane 0's chain:
    # lane 0 + lane 16 = 0 at m=16, lane 1 + lane 17 = 2, then 0 + 2 at m=1.
    w2, v2 = w.copy(), v.copy()
    w2[256] = w2[257] = 0
    w2[8], v2[8], w2[9], v2[9] = 1, 1, 1, 1
    assert float(O.cdot(W.to_bits(w2, O.F16), O.F16, v2)) == 2.0


# ------------------------------------------------------------------ predictor
def _int_predictor(seed, d=48, r=16, n=40):
    rng = np.random.default_rng(seed)
    W1 = rng.integers(-3, 4, (r, d)).astype(np.float32)
    b1 = rng.integers(-4, 5, r).astype(np.float32)
    W2 = rng.integers(-3, 4, (n, r)).astype(np.float32)
    b2 = rng.integers(-10, 11, n).astype(np.float32)
    x = rng.integers(-2, 3, (3, d)).astype(np.float32)
    # exact zeros: two all-zero rows, and one row whose bias cancels token 0's
    # logit exactly (strict threshold: z == 0 is inactive)
    W2[0:2] = 0
    b2[0:2] = 0
    h0 = np.maximum(x[0].astype(np.int64) @ W1.astype(np.int64).T + b1.astype(np.int64), 0)
    W2[2] = np.where(np.arange(r) % 2 == 0, 1, 0)
    b2[2] = -float(h0 @ W2[2].astype(np.int64))
    return W1, b1, W2, b2, x


@pytest.mark.parametrize("dt", [O.F16, O.BF16])
def test_predict_integer_exact(dt):
    W1, b1, W2, b2, x = _int_predictor(11)
    res = O.predict(W.to_bits(W1, dt), W.to_bits(b1, dt), W.to_bits(W2, dt), W.to_bits(b2, dt),
                    W.to_bits(x, dt), dt)
    xi, W1i, W2i = x.astype(np.int64), W1.astype(np.int64), W2.astype(np.int64)
    h = np.maximum(xi @ W1i.T + b1.astype(np.int64), 0)
    z = h @ W2i.T + b2.astype(np.int64)
    assert np.array_equal(res["h"], h.astype(np.float32))
    assert np.array_equal(res["z"], z.astype(np.float32))
    assert np.array_equal(res["mask"], z > 0)
    assert (z == 0).any(), "fixture must contain exact zeros (threshold is strict)"


def test_predict_zero_and_nan_are_inactive():
    d, r, n = 16, 8, 4
    W1 = np.ones((r, d), np.float32)
    W2 = np.zeros((n, r), np.float32)
    W2[1, 0] = 1.0      # z1 = h0 > 0
    W2[2, 0] = -1.0     # z2 < 0
    b2 = np.zeros(n, np.float32)
    x = np.ones((1, d), np.float32)
    w2b = W.to_bits(W2, O.F16)
    w2b[3, 0] = 0x7E00  # NaN weight -> NaN logit
    res = O.predict(W.to_bits(W1, O.F16), None, w2b, W.to_bits(b2, O.F16), W.to_bits(x, O.F16), O.F16)
    assert res["z"][0, 0] == 0.0 and np.isnan(res["z"][0, 3])
    assert res["mask"][0].tolist() == [False, True, False, False]


@pytest.mark.parametrize("cfg", [SMALL, SMALL_REGLU])
def test_predict_sign_matches_numpy_fp64(cfg):
    layer = W.make_layer(cfg, 0, 0, random_b1=True)
    x = W.xhat_inputs(cfg, 8, 0)
    res = O.layer_predict(layer, x)
    dt = cfg.act_dtype
    xf = W.from_bits(x, dt).astype(np.float64)
    h = np.maximum(xf @ W.from_bits(layer["p_w1"], dt).astype(np.float64).T
                   + W.from_bits(layer["p_b1"], dt).astype(np.float64), 0)
    z = h @ W.from_bits(layer["p_w2"], dt).astype(np.float64).T + W.from_bits(layer["p_b2"], dt)
    assert np.allclose(res["h"], h, rtol=1e-5, atol=1e-5)
    assert np.allclose(res["z64"], z, rtol=1e-9, atol=1e-9)
    clear = np.abs(z) > 1e-4
    assert np.array_equal(res["mask"][clear], (z > 0)[clear])
    assert 0.02 < res["mask"].mean() < 0.3


def test_union_matches_flatnonzero():
    rng = np.random.default_rng(4)
    m = rng.random((7, 300)) < 0.05
    assert np.array_equal(O.union(m), np.flatnonzero(m.any(0)))
    assert O.union(np.zeros((3, 10), bool)).size == 0


@pytest.mark.parametrize("cfg", [SMALL, SMALL_REGLU])
def test_hot_neurons_are_active_for_every_token_and_the_rest_as_predicted(cfg):
    """Hot neurons (the hot/cold split mapped to one device): the forced ids
    are on for every token, every other bit is the plain prediction, and the
    logits are untouched; every neuron hot is the dense FFN's list."""
    layer = W.make_layer(cfg, 0, 0, random_b1=True)
    x = W.xhat_inputs(cfg, 5, 3)
    plain = O.layer_predict(layer, x)
    rng = np.random.default_rng(8)
    for hot in (np.arange(0), np.arange(1), np.arange(33), rng.permutation(cfg.n)[:50], np.arange(cfg.n)):
        res = O.layer_predict(layer, x, hot=hot)
        assert res["mask"][:, hot].all()
        rest = np.setdiff1d(np.arange(cfg.n), hot)
        assert np.array_equal(res["mask"][:, rest], plain["mask"][:, rest])
        assert np.array_equal(res["z"], plain["z"])
        # the batch's list is the hot ids together with the union of the predictions (brute force)
        assert np.array_equal(O.union(res["mask"]), np.union1d(hot, np.flatnonzero(plain["mask"].any(0))))
    assert np.array_equal(O.union(O.layer_predict(layer, x, hot=np.arange(cfg.n))["mask"]), np.arange(cfg.n))
    with pytest.raises(ValueError):
        O.layer_predict(layer, x, hot=np.array([cfg.n], np.int32))


# ------------------------------------------------------------------ FFN
@pytest.mark.parametrize("cfg", [SMALL, SMALL_REGLU, SMALL_Q4, SMALL_SQ])
def test_dense_ffn_matches_numpy(cfg):
    layer = W.make_layer(cfg, 0, 0, random_bdown=True)
    x = W.xhat_inputs(cfg, 3, 0)
    a = O.ffn_act(layer["w_up"], layer.get("w_gate"), layer["b"], x, cfg.act, cfg.w_dtype, cfg.act_dtype)
    wu, wg, b, wd, bd = layer_dense_f64(layer)
    xf = W.from_bits(x, cfg.act_dtype).astype(np.float64)
    if cfg.act == W.REGLU:
        a_ref = np.maximum(xf @ wg.T + b, 0) * (xf @ wu.T)
    elif cfg.act == W.SQRELU:
        a_ref = np.square(np.maximum(xf @ wu.T + b, 0))
    else:
        a_ref = np.maximum(xf @ wu.T + b, 0)
    assert np.allclose(a, a_ref, rtol=1e-12, atol=1e-12)
    y = O.ffn_down(layer["w_down"], layer["b_down"], a, np.arange(cfg.n), cfg.w_dtype, cfg.act_dtype)
    y_ref = a_ref @ wd.T + bd
    assert np.allclose(y, y_ref, rtol=1e-11, atol=1e-11)


@pytest.mark.parametrize("cfg", [SMALL, SMALL_REGLU, SMALL_Q4, SMALL_SQ])
def test_masked_ffn_invariants(cfg):
    layer = W.make_layer(cfg, 0, 0, random_bdown=True)
    x = W.xhat_inputs(cfg, 2, 0)
    a = O.ffn_act(layer["w_up"], layer.get("w_gate"), layer["b"], x, cfg.act, cfg.w_dtype, cfg.act_dtype)
    allidx = np.arange(cfg.n, dtype=np.int32)
    dense = O.ffn_down(layer["w_down"], layer["b_down"], a, allidx, cfg.w_dtype, cfg.act_dtype)
    fired = np.flatnonzero((a != 0).any(0))
    rng = np.random.default_rng(0)
    extra = rng.choice(np.setdiff1d(allidx, fired), size=10, replace=False)
    superset = np.union1d(fired, extra).astype(np.int32)
    # a superset of the fired neurons adds only exact zeros
    assert np.array_equal(O.ffn_down(layer["w_down"], layer["b_down"], a, superset, cfg.w_dtype, cfg.act_dtype), dense)
    # the empty list leaves b_down
    bd = W.from_bits(layer["b_down"], cfg.act_dtype).astype(np.float64)
    empty = O.ffn_down(layer["w_down"], layer["b_down"], a, np.zeros(0, np.int32), cfg.w_dtype, cfg.act_dtype)
    assert np.array_equal(empty, np.broadcast_to(bd, empty.shape))
    # merging the partial results of a partition equals the whole
    part = rng.random(superset.size) < 0.5
    y1 = O.ffn_down(layer["w_down"], None, a, superset[part], cfg.w_dtype, cfg.act_dtype)
    y2 = O.ffn_down(layer["w_down"], None, a, superset[~part], cfg.w_dtype, cfg.act_dtype)
    assert np.allclose(y1 + y2 + bd, dense, rtol=1e-12, atol=1e-12)
    # a strict subset of the fired set differs
    drop = fired[: max(1, fired.size // 4)]
    sub = np.setdiff1d(fired, drop).astype(np.int32)
    assert not np.allclose(O.ffn_down(layer["w_down"], layer["b_down"], a, sub, cfg.w_dtype, cfg.act_dtype), dense)


@pytest.mark.parametrize("dt", [O.F16, O.BF16])
def test_golden_worked_example(dt):
    layer, x, exp = worked_example_layer(dt)
    res = O.layer_predict(layer, x)
    idx = O.union(res["mask"])
    assert idx.tolist() == exp["predicted"]
    a = O.ffn_act(layer["w_up"], None, layer["b"], x, W.RELU, dt, dt)
    assert a[0].tolist() == exp["activations"]
    y = O.ffn_down(layer["w_down"], layer["b_down"], a, idx, dt, dt)
    assert y[0].tolist() == exp["y_masked"]
    cpu = O.ffn_down(layer["w_down"], None, a, np.array([4], np.int32), dt, dt)
    gpu = O.ffn_down(layer["w_down"], None, a, np.array([3, 5], np.int32), dt, dt)
    assert cpu[0].tolist() == exp["y_part_cpu_neuron4_no_bias"]
    assert gpu[0].tolist() == exp["y_part_gpu_neurons35_no_bias"]
    dense = O.ffn_down(layer["w_down"], layer["b_down"], a, np.arange(8, dtype=np.int32), dt, dt)
    assert dense[0].tolist() == exp["y_dense"]


def test_squared_relu_is_the_relu_activation_squared():
    """Squared ReLU fires exactly where ReLU does, with the ReLU value squared
    (the ReLU path is pinned on its own above); Q4_0 rows included."""
    for cfg in (SMALL, SMALL_Q4):
        layer = W.make_layer(cfg, 0, 0)
        x = W.xhat_inputs(cfg, 3, 2)
        relu = O.ffn_act(layer["w_up"], None, layer["b"], x, W.RELU, cfg.w_dtype, cfg.act_dtype)
        sq = O.ffn_act(layer["w_up"], None, layer["b"], x, W.SQRELU, cfg.w_dtype, cfg.act_dtype)
        assert np.array_equal(sq, relu * relu)
        assert np.array_equal(sq != 0, relu != 0) and (relu != 0).any() and (relu == 0).any()


def test_bruteforce_tiny_layer_exact_rationals():
    """Pure-Python exact arithmetic on a tiny layer: the fp64 oracle agrees to
    rounding, for ReLU, ReGLU and squared ReLU."""
    for act in (W.RELU, W.REGLU, W.SQRELU):
        cfg = W.LayerConfig("tiny", 16, 12, 8, 1, act, W.F16, W.F16, alpha=0.5, rho=0.3, cfg_id=104)
        layer = W.make_layer(cfg, 0, 3, random_bdown=True)
        x = W.xhat_inputs(cfg, 1, 3)
        xv = [Fraction(float(v)) for v in W.from_bits(x[0], W.F16)]
        wu = [[Fraction(float(v)) for v in row] for row in W.from_bits(layer["w_up"], W.F16)]
        wg = None if act != W.REGLU else [[Fraction(float(v)) for v in row] for row in W.from_bits(layer["w_gate"], W.F16)]
        b = [Fraction(float(v)) for v in W.from_bits(layer["b"], W.F16)]
        wd = [[Fraction(float(v)) for v in row] for row in W.from_bits(layer["w_down"], W.F16)]
        bd = [Fraction(float(v)) for v in W.from_bits(layer["b_down"], W.F16)]
        a_exact = []
        for i in range(cfg.n):
            up = sum(wu[i][k] * xv[k] for k in range(cfg.d))
            if act == W.RELU:
                a_exact.append(max(up + b[i], Fraction(0)))
            elif act == W.SQRELU:
                a_exact.append(max(up + b[i], Fraction(0)) ** 2)
            else:
                g = sum(wg[i][k] * xv[k] for k in range(cfg.d)) + b[i]
                a_exact.append(max(g, Fraction(0)) * up)
        idx = np.array([0, 2, 3, 5, 7, 11], np.int32)
        y_exact = [sum(a_exact[i] * wd[j][i] for i in idx) + bd[j] for j in range(cfg.d)]
        a = O.ffn_act(layer["w_up"], layer.get("w_gate"), layer["b"], x, act, W.F16, W.F16)
        y = O.ffn_down(layer["w_down"], layer["b_down"], a, idx, W.F16, W.F16)
        assert np.allclose(a[0], [float(v) for v in a_exact], rtol=1e-14, atol=1e-15)
        assert np.allclose(y[0], [float(v) for v in y_exact], rtol=1e-13, atol=1e-15)


# ------------------------------------------------------------------ between layers / load
@pytest.mark.parametrize("dt", [O.F16, O.BF16])
def test_rmsnorm_matches_numpy(dt):
    rng = np.random.default_rng(9)
    x = (rng.standard_normal((4, 1000)) * rng.uniform(0.1, 5, (4, 1))).astype(np.float32)
    got = O.rmsnorm(x, dt)
    xf = x.astype(np.float64)
    ref = xf / np.sqrt((xf * xf).sum(1, keepdims=True) / xf.shape[1] + 1e-5)
    want = W.to_bits(ref.astype(np.float32), dt) if dt == O.BF16 else ref.astype(np.float16).view(np.uint16)
    ulp = np.abs(got.astype(np.int32) - want.astype(np.int32))
    assert ulp.max() <= 1 and (ulp == 0).mean() > 0.999


def test_perm_from_counts_is_stable_descending():
    rng = np.random.default_rng(6)
    c = rng.integers(0, 20, 5000).astype(np.int32)
    assert np.array_equal(O.perm_from_counts(c), np.argsort(-c, kind="stable"))


def test_permutation_invariance():
    cfg = SMALL
    layer = W.make_layer(cfg, 0, 0, random_bdown=True)
    x = W.xhat_inputs(cfg, 4, 0)
    perm = np.random.default_rng(8).permutation(cfg.n).astype(np.int32)
    pl = permute_layer(layer, perm)
    m0 = O.layer_predict(layer, x)["mask"]
    m1 = O.layer_predict(pl, x)["mask"]
    assert np.array_equal(m1, m0[:, perm])  # bit-identical decisions
    idx0 = O.union(m0)
    idx1 = O.union(m1)
    assert np.array_equal(np.sort(perm[idx1]), idx0)
    y0 = O.masked_ffn(layer, x, idx0)
    y1 = O.masked_ffn(pl, x, idx1)
    assert np.allclose(y0, y1, rtol=1e-12, atol=1e-12)
