"""Offline predictor distillation (the adaptive predictor without real data):
its labels and its evaluation agree with the oracle, training beats the
random predictor, recall grows with the rank, and the rank choice keeps the
smallest rank that reaches the target.  CPU only (torch on the host)."""
from __future__ import annotations

import numpy as np
import pytest

import oracle as O
from activation_sparse_decode_sigmoid_gb300 import distill as D
from activation_sparse_decode_sigmoid_gb300 import workload as W

pytest.importorskip("torch")

TINY = W.LayerConfig("tiny", 64, 200, 16, 1, W.RELU, W.F16, W.F16, alpha=0.8, cfg_id=401)
TINY_REGLU = W.LayerConfig("tiny_reglu", 64, 160, 16, 1, W.REGLU, W.BF16, W.BF16, alpha=0.8, cfg_id=402)
TINY_Q4 = W.LayerConfig("tiny_q4", 64, 96, 16, 1, W.RELU, W.Q4_0, W.F16, alpha=0.8, cfg_id=403)


@pytest.mark.parametrize("cfg", [TINY, TINY_REGLU, TINY_Q4])
def test_fired_sets_are_the_oracles_nonzero_activations(cfg):
    layer = W.make_layer(cfg, 0, 0)
    x = W.xhat_inputs(cfg, 64, 3)
    fired = D.fired_sets(layer, x)
    a = O.ffn_act(layer["w_up"], layer.get("w_gate"), layer["b"], x, cfg.act, cfg.w_dtype, cfg.act_dtype)
    if cfg.act == W.REGLU:
        # a = relu(g) * v: nonzero where the gate fires (and v is not exactly 0)
        nz = a != 0
        assert not np.any(nz & ~fired)
        assert np.mean(fired & ~nz) < 1e-3
    else:
        # fp32 labels vs the fp64 oracle: they may differ only where u is within rounding of 0
        assert np.mean(fired != (a > 0)) < 1e-3


@pytest.mark.parametrize("cfg", [TINY, TINY_REGLU])
def test_predicted_sets_are_the_oracles_predictions(cfg):
    layer = W.make_layer(cfg, 0, 0, random_b1=True)
    x = W.xhat_inputs(cfg, 64, 4)
    ref = O.layer_predict(layer, x)
    got = D.predicted_sets(layer, x)
    clear = np.abs(ref["z64"]) > 1e-4
    assert np.array_equal(got[clear], ref["mask"][clear])


def test_quality_counts():
    fired = np.array([[1, 1, 0, 0], [1, 0, 0, 1]], bool)
    pred = np.array([[1, 0, 1, 0], [1, 0, 0, 1]], bool)
    q = D.set_quality(pred, fired)
    assert q["recall"] == 3 / 4 and q["precision"] == 3 / 4
    assert q["predicted_density"] == 4 / 8 and q["fired_density"] == 4 / 8


def test_distilled_predictor_beats_the_random_one_and_keeps_the_format():
    layer = W.make_layer(TINY, 0, 0)
    xtr = W.calibration_inputs(TINY, 0, 0, T=2048)
    xte = W.xhat_inputs(TINY, 256, 9)
    fired = D.fired_sets(layer, xte)
    before = D.set_quality(D.predicted_sets(layer, xte), fired)
    out = D.distill(layer, xtr, 32, steps=400)
    after = D.set_quality(D.predicted_sets(out, xte), fired)
    assert after["recall"] > before["recall"] + 0.2
    assert out["r"] == 32 and out["p_w1"].shape == (32, 64) and out["p_w2"].shape == (200, 32)
    assert out["p_w1"].dtype == np.uint16 and out["p_b2"].shape == (200,)
    # the FFN weights are the layer's own
    assert out["w_up"] is layer["w_up"] and out["w_down"] is layer["w_down"]
    # seeded: the same call gives the same bytes
    again = D.distill(layer, xtr, 32, steps=400)
    assert np.array_equal(again["p_w2"], out["p_w2"])


def test_recall_grows_with_rank_and_the_rank_choice_stops_at_the_first_that_reaches_the_target():
    layer = W.make_layer(TINY, 0, 0)
    xtr = W.calibration_inputs(TINY, 0, 0, T=2048)
    xte = W.xhat_inputs(TINY, 256, 9)
    _, tried = D.adaptive_rank(layer, xtr, xte, [4, 16, 64], target_recall=1.01, steps=400)
    recalls = [q["recall"] for _, q in tried]
    assert [r for r, _ in tried] == [4, 16, 64]
    assert recalls[0] < recalls[1] < recalls[2]
    target = (recalls[0] + recalls[1]) / 2  # reached first at rank 16
    chosen, tried2 = D.adaptive_rank(layer, xtr, xte, [64, 4, 16], target_recall=target, steps=400)
    assert [r for r, _ in tried2] == [4, 16] and chosen["r"] == 16
