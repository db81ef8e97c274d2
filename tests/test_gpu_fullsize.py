"""GPU parity at the full sizes of the five workloads.

Each full-size layer is drawn on the GPU, calibrated and loaded exactly as the
benchmark does; the oracle works on the same bytes copied back.  Index lists
are compared bit-exactly for the whole batch; FFN outputs for every token when
the batch is small, else for sampled tokens (the oracle computes them one by
one).  The OPT-30B-, LLaMA-70B- and Falcon-40B-shaped stacks (the last also
with Q4_0 weights) run whole in the benchmark's launch configuration (one
persistent launch per token at one token, layer by layer for batches) and are
checked on sampled layers with teacher forcing from the trace."""
from __future__ import annotations

import numpy as np
import pytest

import oracle as O
from activation_sparse_decode_sigmoid_gb300 import workload as W
from activation_sparse_decode_sigmoid_gb300.calibrate import calibrate_and_load, load_synthetic_stack
from tests import _gpu as G
from tests._helpers import max_rel_err

pytestmark = pytest.mark.gpu

FULL = {
    "opt30b_relu_f16": [1, 3],
    "llama70b_reglu_bf16": [1, 8],
    "falcon40b_relu_f16": [1, 4, 16, 32],
    "falcon40b_relu_q4": [1, 64],
    "opt_1layer_relu_f16": [1, 8],
}

# whole stacks decoded as the benchmark runs them, checked on sampled layers:
# the batches of each workload (the Q4_0 one: its 64-token prompt, then
# one-token decode on the same context)
STACKS = {
    "opt30b_relu_f16": [1],
    "llama70b_reglu_bf16": [1, 8],
    "falcon40b_relu_f16": [1, 16],
    "falcon40b_relu_q4": [64, 1],
}


@pytest.mark.parametrize("name", list(FULL))
def test_full_size_layer(name):
    t = G.torch()
    cfg = W.CONFIGS[name]
    batches = FULL[name]
    c = G.ctx(max_layers=1, max_batch=max(batches))
    dev = t.device("cuda", 0)
    lw = W.make_layer_device(cfg, 0, 0, dev)
    cal = t.from_numpy(W.calibration_inputs(cfg, 0, 0).view(np.int16)).to(dev)
    perm = calibrate_and_load(c, 0, lw, cal)
    host = W.layer_to_host(lw)
    del lw
    for B in batches:
        x = W.xhat_inputs(cfg, B, 21)
        idx, cnt, oidx = G.predict_checked(c, 0, host, x, perm)
        frac = oidx.size / cfg.n
        assert 0.02 < frac < 0.999, frac
        y = c.sparse_ffn(0, G.dev16(x), idx, cnt)
        c.check()
        got = G.y_to_f64(y, cfg.act_dtype)
        toks = range(B) if B <= 8 else [0, B // 2, B - 1]
        for tok in toks:
            want = O.masked_ffn(host, x[tok: tok + 1], oidx)
            err = max_rel_err(got[tok: tok + 1], want)
            assert err <= G.tol(host), f"B={B} token {tok}: {err:.3g}"
    c.close()


@pytest.mark.parametrize("name", list(STACKS))
def test_full_stack_decode_sampled_layers(name):
    """The whole stack in the benchmark's launch configuration (one
    persistent launch per token at 1 token, layer by layer for batches),
    teacher-forced on the first, middle and last layer: the GPU's x_hat
    within one unit in the last place of the oracle's RMSNorm of the traced
    residual, the list equal to the oracle's on that x_hat, and the layer's
    update within the tolerance (every token up to 8, else three)."""
    t = G.torch()
    cfg = W.CONFIGS[name]
    L, d, n = cfg.L, cfg.d, cfg.n
    sample = (0, L // 2, L - 1)
    c, host = load_synthetic_stack(cfg, L, 0, 0, max(STACKS[name]), keep_host=sample)
    for B in STACKS[name]:
        x0 = W.decode_inputs(cfg, B, 3 + B)
        x = t.from_numpy(x0.copy()).cuda()
        tx = t.zeros((L, B, d), dtype=t.float32, device="cuda")
        txh = t.zeros((L, B, d), dtype=t.int16, device="cuda")
        tidx = t.full((L, n), -1, dtype=t.int32, device="cuda")
        tcnt = t.zeros(L, dtype=t.int32, device="cuda")
        c.set_trace(tx, txh, tidx, tcnt)
        c.decode_step(x)
        c.check()
        c.set_trace(None, None, None, None)
        xs = np.concatenate([tx.cpu().numpy(), x.cpu().numpy()[None]], 0).astype(np.float64)
        assert np.array_equal(xs[0], x0.astype(np.float64))
        xh = G.host16(txh)
        counts = tcnt.cpu().numpy()
        assert np.all(counts > 0.03 * n) and np.all(counts <= n), counts
        toks = list(range(B)) if B <= 8 else [0, B // 2, B - 1]
        for l in sample:
            lw, perm = host[l]
            want = O.rmsnorm(xs[l].astype(np.float32), cfg.act_dtype)
            assert np.abs(xh[l].astype(np.int32) - want.astype(np.int32)).max() <= 1
            gidx = tidx[l, : counts[l]].cpu().numpy()
            oidx = O.union(O.layer_predict(lw, xh[l])["mask"])
            assert np.array_equal(np.sort(perm[gidx]), oidx), f"B={B} layer {l}"
            for tok in toks:
                err = max_rel_err(xs[l + 1][tok: tok + 1] - xs[l][tok: tok + 1],
                                  O.masked_ffn(lw, xh[l][tok: tok + 1], oidx))
                assert err <= G.tol(lw), f"B={B} layer {l} token {tok}: {err:.3g}"
    c.close()


# every dimension at the library's limit: d_model 8192, d_ffn 65536, rank 2048,
# ReGLU (three 1 GiB matrices), 64 tokens
MAX = W.LayerConfig("max_sizes", 8192, 65536, 2048, 1, W.REGLU, W.BF16, W.BF16, alpha=0.9, cfg_id=7)


def test_maximum_sizes():
    """Predictor lists bit-exact for 1 and 64 tokens; the FFN and a decode
    step (one launch at 1 token, layer by layer at 64) match the oracle on
    sampled tokens, with every dimension at its limit."""
    t = G.torch()
    cfg = MAX
    c = G.ctx(max_layers=1, max_batch=64)
    dev = t.device("cuda", 0)
    lw = W.make_layer_device(cfg, 0, 0, dev)
    cal = t.from_numpy(W.calibration_inputs(cfg, 0, 0).view(np.int16)).to(dev)
    perm = calibrate_and_load(c, 0, lw, cal)
    host = W.layer_to_host(lw)
    del lw
    for B in (1, 64):
        x = W.xhat_inputs(cfg, B, 43)
        idx, cnt, oidx = G.predict_checked(c, 0, host, x, perm)
        y = c.sparse_ffn(0, G.dev16(x), idx, cnt)
        c.check()
        got = G.y_to_f64(y, cfg.act_dtype)
        for tok in ([0] if B == 1 else [0, 37, 63]):
            xt = x[tok: tok + 1]
            want = O.masked_ffn(host, xt, oidx)
            assert max_rel_err(got[tok: tok + 1], want) <= G.tol(host)
            if B > 1:  # the tensor-core path: also within the bound of its arithmetic
                assert np.all(np.abs(got[tok: tok + 1] - want) <= G.tc_error_bound(host, xt, oidx))
        # a decode step on the residual: x_hat, list and update against the oracle
        x0 = W.decode_inputs(cfg, B, 44)
        xd = t.from_numpy(x0.copy()).cuda()
        txh = t.zeros((1, B, cfg.d), dtype=t.int16, device="cuda")
        tidx = t.full((1, cfg.n), -1, dtype=t.int32, device="cuda")
        tcnt = t.zeros(1, dtype=t.int32, device="cuda")
        c.set_trace(None, txh, tidx, tcnt)
        c.decode_step(xd)
        c.check()
        c.set_trace(None, None, None, None)
        xh = G.host16(txh)[0]
        want_xh = O.rmsnorm(x0.astype(np.float32), cfg.act_dtype)
        assert np.abs(xh.astype(np.int32) - want_xh.astype(np.int32)).max() <= 1
        m = int(tcnt[0].item())
        sel = np.sort(perm[tidx[0, :m].cpu().numpy()])
        assert np.array_equal(sel, O.union(O.layer_predict(host, xh)["mask"]))
        upd = xd.cpu().numpy().astype(np.float64) - x0.astype(np.float64)
        for tok in ([0] if B == 1 else [0, 63]):
            xt = xh[tok: tok + 1]
            want = O.masked_ffn(host, xt, sel)
            assert max_rel_err(upd[tok: tok + 1], want) <= G.tol(host)
            if B > 1:
                assert np.all(np.abs(upd[tok: tok + 1] - want) <= G.tc_error_bound(host, xt, sel))
    c.close()
