"""Host-side logic of the benchmark: the algorithmic byte count behind the
roofline figure and the L2-flush rule.  No GPU needed."""
from __future__ import annotations

import bench
from activation_sparse_decode_sigmoid_gb300 import workload as W


def test_algorithmic_bytes_per_layer_follow_the_formula():
    cfg = W.CONFIGS["opt30b_relu_f16"]
    d, n, r = cfg.d, cfg.n, cfg.r
    m = [2899, 3000]
    got = bench.algorithmic_bytes(cfg, 2, 1, m)
    # predictor weights and biases, then W_up row + bias + W_down^T row per listed neuron,
    # then x_hat (2 bytes) and the residual read and written (4 + 4) per element
    want = sum(r * d * 2 + n * r * 2 + (r + n) * 2 + k * (2 * d * 2 + 2) + d * 10 for k in m)
    assert got == want


def test_hot_prefix_removes_its_predictor_rows_only():
    cfg = W.CONFIGS["llama70b_reglu_bf16"]
    m = [5000, 5100, 4900]
    plain = bench.algorithmic_bytes(cfg, 3, 4, m)
    assert bench.algorithmic_bytes(cfg, 3, 4, m, [0, 0, 0]) == plain
    hot = [100, 0, 37]
    # each hot neuron's W2 row (2r bytes) and b2 entry (2 bytes) are not read
    assert plain - bench.algorithmic_bytes(cfg, 3, 4, m, hot) == sum(h * (2 * cfg.r + 2) for h in hot)


def test_reglu_and_q4_rows():
    for name, per_neuron in (("llama70b_reglu_bf16", lambda c: 3 * c.d * 2 + 2),
                             ("falcon40b_relu_q4", lambda c: 2 * c.d * 18 / 32 + 2)):
        cfg = W.CONFIGS[name]
        a = bench.algorithmic_bytes(cfg, 1, 1, [10])
        b = bench.algorithmic_bytes(cfg, 1, 1, [11])
        assert b - a == per_neuron(cfg)


def test_l2_flush_only_for_stacks_that_fit_in_l2():
    assert bench.needs_l2_flush(W.CONFIGS["opt_1layer_relu_f16"], 1)
    assert not bench.needs_l2_flush(W.CONFIGS["opt30b_relu_f16"], 48)
    assert not bench.needs_l2_flush(W.CONFIGS["opt30b_relu_f16"], 4)

