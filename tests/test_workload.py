"""The synthetic workload matches its stated recipe (generator diagnostics)."""
from __future__ import annotations

import numpy as np
import pytest
from scipy.special import ndtr

import oracle as O
from activation_sparse_decode_sigmoid_gb300 import workload as W


@pytest.mark.parametrize("name", list(W.CONFIGS))
def test_zipf_mean_is_rho(name):
    cfg = W.CONFIGS[name]
    c = W.zipf_scale(cfg.n, cfg.alpha, cfg.rho)
    p = np.minimum(0.9, c * np.arange(1, cfg.n + 1, dtype=np.float64) ** (-cfg.alpha))
    assert abs(p.mean() - cfg.rho) < 1e-9
    assert p.max() <= 0.9 and np.all(np.diff(p) <= 0)


def test_probit_bias_gives_p():
    cfg = W.CONFIGS["opt_1layer_relu_f16"]
    p = W.activation_probs(cfg, 0, 0)
    assert np.allclose(ndtr(W.probit(p)), p, rtol=1e-12, atol=1e-15)
    # the shuffle is seeded and a permutation of the sorted profile
    p2 = W.activation_probs(cfg, 0, 0)
    assert np.array_equal(p, p2)
    assert not np.array_equal(p, W.activation_probs(cfg, 1, 0))


def test_one_layer_density_matches_rho():
    """True firing rate and predicted rate of the one-layer fp16 workload are
    ~10% (binomial error over 64 tokens x 4096 neurons)."""
    cfg = W.CONFIGS["opt_1layer_relu_f16"]
    layer = W.make_layer(cfg, 0, 0)
    x = O.rmsnorm(W.decode_inputs(cfg, 64, 0), cfg.act_dtype)
    a = O.ffn_act(layer["w_up"], None, layer["b"], x, cfg.act, cfg.w_dtype, cfg.act_dtype)
    fired = (a > 0).mean()
    # per-neuron probabilities vary, so the binomial variance is at most rho(1-rho)/N
    sd = np.sqrt(cfg.rho * (1 - cfg.rho) / a.size)
    assert abs(fired - cfg.rho) < 0.01 + 6 * sd
    pred = O.layer_predict(layer, x)["mask"].mean()
    assert 0.07 < pred < 0.13


def test_bf16_encoding_round_to_nearest_even():
    v = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 3.0e38, 1e-40], np.float32)
    bits = W.to_bits(v, W.BF16)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7 -> even (1.0); 1 + 3*2^-8 -> 1 + 2^-6
    assert W.from_bits(bits, W.BF16)[:3].tolist() == [1.0, 1.0, 1.0 + 2 ** -6]
    assert W.from_bits(bits, W.BF16)[3] == -2.5
    assert np.array_equal(O.round_to(v.astype(np.float64), O.BF16)[:4], bits[:4])


def test_make_layer_shapes_and_determinism():
    cfg = W.CONFIGS["falcon40b_relu_q4"].scaled(d=256, n=512, r=64)
    l1 = W.make_layer(cfg, 2, 0)
    l2 = W.make_layer(cfg, 2, 0)
    assert l1["w_up"].shape == (512, 256 // 32 * 18) and l1["w_down"].shape == (512, 256 // 32 * 18)
    assert l1["p_w1"].shape == (64, 256) and l1["p_w2"].shape == (512, 64)
    for k in ("w_up", "w_down", "p_w1", "p_w2", "b", "p_b2"):
        assert np.array_equal(l1[k], l2[k])
