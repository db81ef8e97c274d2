"""The allocation-free sparse FFN entry point against the CPU oracle and the
context-based entry point.

pi_sparse_ffn_noalloc serves callers that may not allocate device memory
(pre-allocated buffers only, a fixed memory budget, a server-owned pool): it
keeps its scratch in a fixed array inside the library.  Here its output must
match the oracle's masked FFN on the same list and the output of
pi_sparse_ffn (max relative error within 1e-2, the tolerance of the other
parity tests) on two calls in a row, since every call reuses what the
previous one left in that array.  This file is collected last so that a run
stopping at its first failure has run everything else already."""
from __future__ import annotations

import numpy as np
import pytest

import oracle as O
from activation_sparse_decode_sigmoid_gb300 import pi
from activation_sparse_decode_sigmoid_gb300 import workload as W
from tests import _gpu as G
from tests._helpers import max_rel_err

pytestmark = pytest.mark.gpu

CFGS = {
    "relu_f16": W.LayerConfig("nz_relu_f16", 1024, 3000, 64, 1, W.RELU, W.F16, W.F16, alpha=0.8, cfg_id=301),
    "reglu_bf16": W.LayerConfig("nz_reglu_bf16", 520, 1777, 32, 1, W.REGLU, W.BF16, W.BF16, alpha=0.7, cfg_id=302),
}


def _rows(layer: dict, keep: list) -> pi.pi_ffn_rows:
    """Device rows in the library's layout: W_up, W_gate, W_down transposed."""
    def dev(a):
        if a is None:
            return None
        t = G.dev16(np.ascontiguousarray(a))
        keep.append(t)
        return t.data_ptr()
    return pi.pi_ffn_rows(layer["d"], layer["n"], layer["act"], layer["act_dtype"], dev(layer["w_up"]),
                          dev(layer.get("w_gate")), dev(layer["w_down"].T), dev(layer["b"]),
                          dev(layer.get("b_down")))


@pytest.mark.parametrize("name", list(CFGS))
def test_noalloc_matches_oracle_and_context_path_on_consecutive_calls(name):
    t = G.torch()
    cfg = CFGS[name]
    layer = W.make_layer(cfg, 0, 0, random_bdown=True)
    c = G.ctx(max_layers=1, max_batch=8)
    c.load_layer(0, layer)  # identity permutation: physical ids = original ids
    keep: list = []
    rows = _rows(layer, keep)
    for call, B in enumerate((3, 1)):
        xh = W.xhat_inputs(cfg, B, 40 + call)
        x = G.dev16(xh)
        idx, cnt = c.predict(0, x)
        y_ref = c.sparse_ffn(0, x, idx, cnt)
        c.check()
        y = t.empty_like(y_ref)
        status = t.full((1,), 12345, dtype=t.int32, device="cuda")
        rc = pi.pi_sparse_ffn_noalloc(rows, x, B, idx, cnt, y, status)
        assert rc == pi.PI_OK, rc
        t.cuda.synchronize()
        assert int(status.item()) == 0
        got = G.y_to_f64(y, cfg.act_dtype)
        oidx = np.sort(idx[: int(cnt.item())].cpu().numpy())
        err_o = max_rel_err(got, O.masked_ffn(layer, xh, oidx))
        assert err_o <= 1e-2, f"call {call}: max rel err vs the oracle {err_o:.3g}"
        err = max_rel_err(got, G.y_to_f64(y_ref, cfg.act_dtype))
        assert err <= 1e-2, f"call {call}: max rel err vs pi_sparse_ffn {err:.3g}"
    c.close()


def test_noalloc_rejects_sizes_beyond_its_scratch():
    t = G.torch()
    G.ensure_built()
    cfg = W.LayerConfig("nz_big", 8192, 64, 8, 1, W.RELU, W.F16, W.F16, alpha=0.8, cfg_id=303)
    layer = W.make_layer(cfg, 0, 0)
    keep: list = []
    rows = _rows(layer, keep)
    B = 64  # 64 tokens x 8192 columns of partials per SM cannot fit the fixed scratch
    x = t.zeros((B, cfg.d), dtype=t.int16, device="cuda")
    idx = t.zeros(1, dtype=t.int32, device="cuda")
    cnt = t.zeros(1, dtype=t.int32, device="cuda")
    y = t.empty((B, cfg.d), dtype=t.int16, device="cuda")
    assert pi.pi_sparse_ffn_noalloc(rows, x, B, idx, cnt, y) == pi.PI_ERR_SHAPE
