"""GPU parity: the CUDA path through the C ABI against the CPU oracle on the
same seeded inputs.  Index lists bit-exact; fp16/bf16 outputs within a max
relative error of 1e-2 and Q4_0 within 2e-2 (max_k |y-ref| / max(|ref|, rms))."""
from __future__ import annotations

import numpy as np
import pytest

import oracle as O
from activation_sparse_decode_sigmoid_gb300 import pi
from activation_sparse_decode_sigmoid_gb300 import workload as W
from tests import _gpu as G
from tests._helpers import max_rel_err, worked_example_layer

pytestmark = pytest.mark.gpu

# pi_debug_set_mma_min_batch: the library's own choice of the smallest batch
# that runs layer by layer (2 tokens for 16-bit layers, 3 for Q4_0 layers)
AUTO = -1

# small layers spanning several tiles with ragged tails (n not a multiple of
# 32, d not a multiple of 256), every activation / weight kind
CFGS = {
    "relu_f16": W.LayerConfig("relu_f16", 256, 1000, 64, 3, W.RELU, W.F16, W.F16, alpha=0.8, cfg_id=201),
    "reglu_bf16": W.LayerConfig("reglu_bf16", 264, 777, 32, 3, W.REGLU, W.BF16, W.BF16, alpha=0.7, cfg_id=202),
    "relu_q4": W.LayerConfig("relu_q4", 512, 640, 64, 3, W.RELU, W.Q4_0, W.F16, alpha=0.9, cfg_id=203),
    # the third activation family: squared ReLU
    "sqrelu_bf16": W.LayerConfig("sqrelu_bf16", 320, 900, 64, 3, W.SQRELU, W.BF16, W.BF16, alpha=0.8, cfg_id=206),
    "opt_1layer": W.CONFIGS["opt_1layer_relu_f16"],
    # enough W1 / W2 rows per SM that both static-ring passes wrap several times
    "ring_wrap": W.LayerConfig("ring_wrap", 4096, 12000, 2048, 2, W.RELU, W.F16, W.F16, alpha=0.9, cfg_id=205),
    # wide ReGLU rows: the few-token row kernel's ring holds only 4 to 6 neurons
    "reglu_wide": W.LayerConfig("reglu_wide", 8192, 16384, 64, 1, W.REGLU, W.BF16, W.BF16, alpha=0.7, cfg_id=207),
    # ReGLU with Q4_0 rows; d not a multiple of 256: a partial last super-stage of 8 blocks
    "reglu_q4": W.LayerConfig("reglu_q4", 416, 700, 32, 3, W.REGLU, W.Q4_0, W.F16, alpha=0.7, cfg_id=208),
}


@pytest.fixture(scope="module")
def c64():
    c = G.ctx(max_layers=4, max_batch=64)
    yield c
    c.close()


def _layer(name, random_bias=True):
    cfg = CFGS[name]
    return cfg, W.make_layer(cfg, 0, 0, random_b1=random_bias, random_bdown=random_bias)


@pytest.mark.parametrize("name", list(CFGS))
@pytest.mark.parametrize("B", [1, 3, 8])
def test_predict_and_sparse_ffn(c64, name, B):
    cfg, layer = _layer(name)
    perm = np.random.default_rng(1).permutation(cfg.n).astype(np.int32)
    c64.load_layer(0, layer, perm)
    x = W.xhat_inputs(cfg, B, 7)
    idx, cnt, oidx = G.predict_checked(c64, 0, layer, x, perm)
    assert oidx.size > 0
    G.ffn_checked(c64, 0, layer, x, idx, cnt, oidx)


@pytest.mark.parametrize("name", ["relu_f16", "reglu_bf16", "relu_q4", "reglu_q4", "sqrelu_bf16"])
@pytest.mark.parametrize("B", [1, 2, 3, 4, 7, 9, 64])
@pytest.mark.parametrize("path", ["default", "step kernel"], indirect=True)
def test_batch_sizes(c64, name, B, path):
    """Every batch size on the default path (layer by layer from 2 or 3
    tokens; up to 4 tokens the up/gate rows stream whole on the CUDA cores,
    from 5 through the tensor cores) and on the persistent step kernel (its
    token groups of 1, 2 and 4)."""
    cfg, layer = _layer(name)
    c64.load_layer(0, layer)
    x = W.xhat_inputs(cfg, B, 11)
    idx, cnt, oidx = G.predict_checked(c64, 0, layer, x)
    G.ffn_checked(c64, 0, layer, x, idx, cnt, oidx)


@pytest.fixture
def path(c64, request):
    """Run a test on the default path, or with every batch on the step kernel."""
    if request.param == "step kernel":
        pi.pi_debug_set_mma_min_batch(c64.handle, 0)
    yield request.param
    pi.pi_debug_set_mma_min_batch(c64.handle, AUTO)


@pytest.mark.parametrize("name", ["ring_wrap", "reglu_wide"])
@pytest.mark.parametrize("B", [2, 3, 4])
def test_few_token_row_kernel_wraps_its_ring(c64, name, B):
    """Up to 4 tokens the up/gate rows stream whole through a ring of stages
    with one consumer warp per stage slot; with far more neurons per SM than
    slots (16 slots of 8 KB rows; 4 to 6 slots of 32 KB ReGLU rows) every
    slot is refilled many times, and the FFN still matches the oracle."""
    cfg, layer = _layer(name)
    c64.load_layer(0, layer)
    x = W.xhat_inputs(cfg, B, 61 + B)
    try:
        pi.pi_debug_set_mma_min_batch(c64.handle, 2)
        idx, cnt, oidx = G.predict_checked(c64, 0, layer, x)
        assert oidx.size > 4 * c64.grid  # many neurons per SM
        G.ffn_checked(c64, 0, layer, x, idx, cnt, oidx)
    finally:
        pi.pi_debug_set_mma_min_batch(c64.handle, AUTO)


@pytest.mark.parametrize("name", ["relu_f16", "reglu_bf16", "relu_q4", "reglu_q4", "sqrelu_bf16"])
@pytest.mark.parametrize("path", ["default", "step kernel"], indirect=True)
def test_dense_ffn(c64, name, path):
    cfg, layer = _layer(name)
    c64.load_layer(0, layer)
    x = W.xhat_inputs(cfg, 4, 3)
    y = c64.dense_ffn(0, G.dev16(x))
    c64.check()
    want = O.masked_ffn(layer, x, np.arange(cfg.n, dtype=np.int32))
    assert max_rel_err(G.y_to_f64(y, cfg.act_dtype), want) <= G.tol(layer)


@pytest.mark.parametrize("name", ["relu_f16", "relu_q4"])
@pytest.mark.parametrize("path", ["default", "step kernel"], indirect=True)
def test_edge_lists(c64, name, path):
    """Empty list -> b_down; full list -> dense; an unordered subset."""
    t = G.torch()
    cfg, layer = _layer(name)
    c64.load_layer(0, layer)
    x = W.xhat_inputs(cfg, 2, 5)
    bd = W.from_bits(layer["b_down"], cfg.act_dtype).astype(np.float64)
    for ids in (np.zeros(0, np.int32), np.arange(cfg.n, dtype=np.int32),
                np.random.default_rng(2).permutation(cfg.n)[:37].astype(np.int32)):
        idx = t.from_numpy(np.concatenate([ids, np.zeros(1, np.int32)])).cuda()
        cnt = t.tensor([ids.size], dtype=t.int32, device="cuda")
        y = c64.sparse_ffn(0, G.dev16(x), idx, cnt)
        c64.check()
        got = G.y_to_f64(y, cfg.act_dtype)
        want = O.masked_ffn(layer, x, np.sort(ids))
        if ids.size == 0:
            assert np.array_equal(got, np.broadcast_to(
                W.from_bits(W.to_bits(bd.astype(np.float32), cfg.act_dtype), cfg.act_dtype), got.shape))
        else:
            assert max_rel_err(got, want) <= G.tol(layer)


def test_golden_worked_example_on_gpu(c64):
    """The {3,4,5} example: predicted set and merged output, exact."""
    layer, x, exp = worked_example_layer(W.F16)
    c64.load_layer(0, layer)
    idx, cnt = c64.predict(0, G.dev16(x))
    c64.check()
    assert idx[: int(cnt.item())].cpu().tolist() == exp["predicted"]
    y = c64.sparse_ffn(0, G.dev16(x), idx, cnt)
    c64.check()
    assert G.y_to_f64(y, W.F16)[0].tolist() == exp["y_masked"]
    yd = c64.dense_ffn(0, G.dev16(x))
    c64.check()
    assert G.y_to_f64(yd, W.F16)[0].tolist() == exp["y_dense"]


def test_zero_logits_are_inactive(c64):
    """Integer predictor: every logit is exact, including exact zeros."""
    cfg = W.LayerConfig("intpred", 64, 200, 16, 1, W.RELU, W.F16, W.F16, alpha=0.8, cfg_id=204)
    layer = W.make_layer(cfg, 0, 0)
    rng = np.random.default_rng(3)
    w1 = rng.integers(-2, 3, (16, 64)).astype(np.float32)
    w2 = rng.integers(-2, 3, (200, 16)).astype(np.float32)
    w2[:40] = 0                      # z = b2 = 0 exactly for these rows
    b2 = rng.integers(-4, 5, 200).astype(np.float32)
    b2[:40] = 0
    layer.update(p_w1=W.to_bits(w1, W.F16), p_w2=W.to_bits(w2, W.F16), p_b2=W.to_bits(b2, W.F16), p_b1=None)
    x = W.to_bits(rng.integers(-2, 3, (3, 64)).astype(np.float32), W.F16)
    c64.load_layer(0, layer)
    idx, cnt, oidx = G.predict_checked(c64, 0, layer, x)
    assert not np.any(idx[: int(cnt.item())].cpu().numpy() < 40)


def test_layer_counts_and_calibrated_permutation(c64):
    t = G.torch()
    cfg, layer = _layer("relu_f16")
    c64.load_layer(0, layer)
    cal = W.calibration_inputs(cfg, 0, 0, T=150)  # > max_batch: several launches
    counts = c64.layer_counts(0, G.dev16(cal))
    c64.check()
    ref = O.layer_predict(layer, cal)["mask"].sum(0).astype(np.int32)
    assert np.array_equal(counts.cpu().numpy(), ref)
    perm = pi.pi_perm_from_counts(ref)
    assert np.array_equal(perm, O.perm_from_counts(ref))
    c64.load_layer(0, layer, perm)
    counts2 = c64.layer_counts(0, G.dev16(cal))
    assert np.array_equal(counts2.cpu().numpy(), ref[perm])  # hot neurons first
    assert np.all(np.diff(counts2.cpu().numpy()) <= 0)
    x = W.xhat_inputs(cfg, 1, 9)
    G.predict_checked(c64, 0, layer, x, perm)
    del t


@pytest.mark.parametrize("name", ["relu_f16", "reglu_bf16", "relu_q4", "sqrelu_bf16"])
@pytest.mark.parametrize("B", [1, 3, 8, 16])
@pytest.mark.parametrize("dense", [False, True])
@pytest.mark.parametrize("layerwise", [True, False])
def test_decode_stack_teacher_forced(name, B, dense, layerwise):
    """Three-layer stack, on the default path (batches layer by layer) or all
    in one persistent launch: per layer the oracle consumes the GPU's x_hat
    (trace) and must give the same list and the same update."""
    t = G.torch()
    cfg = CFGS[name]
    c = G.ctx(max_layers=3, max_batch=max(8, B))
    if not layerwise:
        pi.pi_debug_set_mma_min_batch(c.handle, 0)
    layers, perms = [], []
    for l in range(3):
        lw = W.make_layer(cfg, l, 0, random_b1=True, random_bdown=True)
        c.load_layer(l, lw)
        cal = W.calibration_inputs(cfg, l, 0, T=64)
        perm = pi.pi_perm_from_counts(c.layer_counts(l, G.dev16(cal)).cpu().numpy())
        c.load_layer(l, lw, perm)
        layers.append(lw)
        perms.append(perm)
    L, d, n = 3, cfg.d, cfg.n
    x0 = W.decode_inputs(cfg, B, 4)
    x = t.from_numpy(x0.copy()).cuda()
    tx = t.zeros((L, B, d), dtype=t.float32, device="cuda")
    txh = t.zeros((L, B, d), dtype=t.int16, device="cuda")
    tidx = t.full((L, n), -1, dtype=t.int32, device="cuda")
    tcnt = t.zeros(L, dtype=t.int32, device="cuda")
    c.set_trace(tx, txh, tidx, tcnt)
    (c.dense_step if dense else c.decode_step)(x)
    c.check()
    xs = np.concatenate([tx.cpu().numpy(), x.cpu().numpy()[None]], 0).astype(np.float64)
    assert np.array_equal(xs[0], x0.astype(np.float64))
    xh = G.host16(txh)
    for l in range(L):
        # the GPU's RMSNorm is within one unit in the last place of the fp64 one
        want = O.rmsnorm(xs[l].astype(np.float32), cfg.act_dtype)
        assert np.abs(xh[l].astype(np.int32) - want.astype(np.int32)).max() <= 1
        m = int(tcnt[l].item())
        gidx = tidx[l, :m].cpu().numpy()
        if dense:
            assert m == n and np.array_equal(gidx, np.arange(n))
            oidx = np.arange(n, dtype=np.int32)
        else:
            oidx = O.union(O.layer_predict(layers[l], xh[l])["mask"])
            assert np.array_equal(np.sort(perms[l][gidx]), oidx)
        y_ref = O.masked_ffn(layers[l], xh[l], oidx)
        err = max_rel_err(xs[l + 1] - xs[l], y_ref)
        assert err <= G.tol(layers[l]), f"layer {l}: {err:.3g}"
    c.close()


def test_decode_step_host_buffers_match_device_step():
    """The host-buffer step (copy in, step, copy out, synchronise) gives the
    device step's result bit for bit, from pinned and from pageable memory."""
    t = G.torch()
    cfg, layer = _layer("relu_f16")
    c = G.ctx(max_layers=1, max_batch=4)
    c.load_layer(0, layer)
    x0 = W.decode_inputs(cfg, 3, 5)
    xd = t.from_numpy(x0.copy()).cuda()
    c.decode_step(xd)
    c.check()
    want = xd.cpu().numpy()
    pinned_in = t.from_numpy(x0.copy()).pin_memory()
    pinned_out = t.empty_like(pinned_in).pin_memory()
    c.decode_step_host(pinned_in, pinned_out)
    assert np.array_equal(pinned_out.numpy(), want)
    pageable = x0.copy()
    c.decode_step_host(pageable, pageable)  # in place
    assert np.array_equal(pageable, want)
    c.close()


@pytest.mark.parametrize("name", list(CFGS))
@pytest.mark.parametrize("path", ["default", "step kernel"], indirect=True)
def test_predictor_hidden_layer_bit_exact(c64, name, path):
    """h = max(CDOT(W1, x_hat) + b1, 0) of every token equals the oracle's
    canonical fp32 h bit for bit (the mixed-precision fma of the kernel
    widens both 16-bit operands exactly and rounds once per step)."""
    t = G.torch()
    cfg, layer = _layer(name)
    c64.load_layer(0, layer)
    B = 4
    x = W.xhat_inputs(cfg, B, 17)
    idx, cnt = c64.predict(0, G.dev16(x))
    h = t.zeros(B * cfg.r, dtype=t.float32, device="cuda")
    pi.pi_debug_copy_hidden(c64.handle, h, B * cfg.r)
    c64.check()
    want = O.layer_predict(layer, x)["h"].astype(np.float32)
    got = h.cpu().numpy().reshape(B, cfg.r)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("name", ["relu_f16", "reglu_bf16", "sqrelu_bf16"])
@pytest.mark.parametrize("B", [8, 16, 40, 64])
def test_tensor_core_ffn_matches_oracle_and_cuda_core_path(c64, name, B):
    """Batches of several tokens run the FFN as a gather-GEMM on tcgen05 (A^T
    passed between the two GEMMs as hi and lo 16-bit parts); it must match
    the oracle within the usual tolerance (and within the error bound of its
    arithmetic, output by output), and the CUDA-core path of the step kernel
    on the same list within twice the tolerance -- for every activation
    family, the dense variant included."""
    t = G.torch()
    cfg, layer = _layer(name)
    c64.load_layer(0, layer)
    x = W.xhat_inputs(cfg, B, 23 + B)
    xd = G.dev16(x)
    idx, cnt = c64.predict(0, xd)
    y_tc = c64.sparse_ffn(0, xd, idx, cnt)
    c64.check()
    pi.pi_debug_set_mma_min_batch(c64.handle, 0)
    y_cc = c64.sparse_ffn(0, xd, idx, cnt)
    c64.check()
    pi.pi_debug_set_mma_min_batch(c64.handle, AUTO)
    m = int(cnt.item())
    oidx = np.sort(idx[:m].cpu().numpy())
    got = G.y_to_f64(y_tc, cfg.act_dtype)
    want = O.masked_ffn(layer, x, oidx)
    assert max_rel_err(got, want) <= G.tol(layer)
    # within the error bound of the path's arithmetic, output by output
    assert np.all(np.abs(got - want) <= G.tc_error_bound(layer, x, oidx))
    assert max_rel_err(got, G.y_to_f64(y_cc, cfg.act_dtype)) <= 2 * G.tol(layer)
    # the dense variant (every neuron) on the same path
    yd = c64.dense_ffn(0, xd)
    c64.check()
    every = np.arange(cfg.n)
    got_d, want_d = G.y_to_f64(yd, cfg.act_dtype), O.masked_ffn(layer, x, every)
    assert max_rel_err(got_d, want_d) <= G.tol(layer)
    assert np.all(np.abs(got_d - want_d) <= G.tc_error_bound(layer, x, every))


@pytest.mark.parametrize("name", ["relu_q4", "reglu_q4"])
@pytest.mark.parametrize("B", [3, 8, 64])
def test_q4_tensor_core_ffn_matches_oracle_and_cuda_core_path(c64, name, B):
    """Q4_0 batches dequantise their listed rows in the tensor-core kernels'
    shared memory, w = (q - 8) * s rounded to f16 on its way to the MMA (no
    dequantised copy goes back to HBM); the FFN must match the oracle (exact
    fp64 dequantisation) within the Q4_0 tolerance and the step kernel's
    CUDA-core path (fp32 products) within twice it, sparse and dense."""
    cfg, layer = _layer(name)
    c64.load_layer(0, layer)
    x = W.xhat_inputs(cfg, B, 81 + B)
    xd = G.dev16(x)
    idx, cnt, oidx = G.predict_checked(c64, 0, layer, x)
    y_tc = c64.sparse_ffn(0, xd, idx, cnt)
    c64.check()
    pi.pi_debug_set_mma_min_batch(c64.handle, 0)
    y_cc = c64.sparse_ffn(0, xd, idx, cnt)
    yd_cc = c64.dense_ffn(0, xd)
    c64.check()
    pi.pi_debug_set_mma_min_batch(c64.handle, AUTO)
    got = G.y_to_f64(y_tc, cfg.act_dtype)
    assert max_rel_err(got, O.masked_ffn(layer, x, oidx)) <= G.tol(layer)
    assert max_rel_err(got, G.y_to_f64(y_cc, cfg.act_dtype)) <= 2 * G.tol(layer)
    yd = c64.dense_ffn(0, xd)
    c64.check()
    got_d = G.y_to_f64(yd, cfg.act_dtype)
    assert max_rel_err(got_d, O.masked_ffn(layer, x, np.arange(cfg.n, dtype=np.int32))) <= G.tol(layer)
    assert max_rel_err(got_d, G.y_to_f64(yd_cc, cfg.act_dtype)) <= 2 * G.tol(layer)


# tall layers: so many neurons that a CTA of the tensor-core up kernel makes
# more than one pass over K on 152 SMs (16-bit rows: 263 rows per SM, a
# 256-row pass then a short one; Q4_0 ReLU, two CTAs per SM: 132 rows per CTA,
# two 128-row passes; Q4_0 ReGLU, one CTA per SM: 132 rows)
TALL = {
    "tall_relu_f16": W.LayerConfig("tall_relu_f16", 128, 40000, 32, 1, W.RELU, W.F16, W.F16, alpha=0.8, cfg_id=211),
    "tall_reglu_bf16": W.LayerConfig("tall_reglu_bf16", 128, 40000, 32, 1, W.REGLU, W.BF16, W.BF16, alpha=0.7,
                                     cfg_id=212),
    "tall_relu_q4": W.LayerConfig("tall_relu_q4", 160, 40000, 32, 1, W.RELU, W.Q4_0, W.F16, alpha=0.8, cfg_id=213),
    "tall_reglu_q4": W.LayerConfig("tall_reglu_q4", 96, 20000, 32, 1, W.REGLU, W.Q4_0, W.F16, alpha=0.7, cfg_id=214),
}


@pytest.mark.parametrize("name", list(TALL))
@pytest.mark.parametrize("B", [8, 64])
def test_tensor_core_ffn_several_passes_per_cta(c64, name, B):
    """Dense FFN of a tall layer on the tensor cores (every neuron listed, so
    each up-kernel CTA runs more than one pass over K): the oracle within the
    stated tolerance, the step kernel's CUDA-core path within twice it."""
    _dense_tc_matches(c64, TALL[name], B)


# wide layers: the down-projection splits each 256-column block's list into
# shares, 24 blocks x 6 shares at d = 6144 (a d that is no power of two),
# 32 x 4 at d = 8192; with 200 neurons (4 K steps of 64) most shares hold
# one step
WIDE = {
    "wide_relu_f16": W.LayerConfig("wide_relu_f16", 6144, 2000, 32, 1, W.RELU, W.F16, W.F16, alpha=0.8, cfg_id=215),
    "wide_reglu_bf16": W.LayerConfig("wide_reglu_bf16", 8192, 1500, 32, 1, W.REGLU, W.BF16, W.BF16, alpha=0.7,
                                     cfg_id=216),
    "wide_relu_q4": W.LayerConfig("wide_relu_q4", 8192, 1200, 32, 1, W.RELU, W.Q4_0, W.F16, alpha=0.8, cfg_id=217),
    "wide_short_bf16": W.LayerConfig("wide_short_bf16", 8192, 200, 32, 1, W.RELU, W.BF16, W.BF16, alpha=0.8,
                                     cfg_id=218),
}


@pytest.mark.parametrize("name", list(WIDE))
@pytest.mark.parametrize("B", [8, 24])
def test_tensor_core_ffn_wide_layers(c64, name, B):
    """Dense FFN of a wide layer on the tensor cores, the down-projection's
    share partials merged in order: the oracle within the stated tolerance,
    the CUDA-core path within twice it."""
    _dense_tc_matches(c64, WIDE[name], B)


def _dense_tc_matches(c64, cfg, B):
    layer = W.make_layer(cfg, 0, 0, random_b1=True, random_bdown=True)
    c64.load_layer(0, layer)
    x = W.xhat_inputs(cfg, B, 91 + B)
    xd = G.dev16(x)
    y_tc = c64.dense_ffn(0, xd)
    c64.check()
    try:
        pi.pi_debug_set_mma_min_batch(c64.handle, 0)
        y_cc = c64.dense_ffn(0, xd)
        c64.check()
    finally:
        pi.pi_debug_set_mma_min_batch(c64.handle, AUTO)
    got = G.y_to_f64(y_tc, cfg.act_dtype)
    assert max_rel_err(got, O.masked_ffn(layer, x, np.arange(cfg.n, dtype=np.int32))) <= G.tol(layer)
    assert max_rel_err(got, G.y_to_f64(y_cc, cfg.act_dtype)) <= 2 * G.tol(layer)


@pytest.mark.parametrize("name", ["relu_f16", "reglu_bf16", "ring_wrap", "opt_1layer"])
@pytest.mark.parametrize("B", [2, 5, 8, 9, 16, 17, 40, 64])
def test_batched_predictor_matches_oracle_and_step_kernel(c64, name, B):
    """Layer by layer (forced from 2 tokens here) the predictor runs as
    register-tiled launches (8-token blocks, a halving butterfly over R x 8
    dot products per warp); its lists equal the oracle's and, entry for
    entry, the step kernel's on the same x_hat (one, two and several token
    blocks; r = 2048 takes the narrow output tile that shares mask words
    between CTAs)."""
    cfg, layer = _layer(name)
    c64.load_layer(0, layer)
    x = W.xhat_inputs(cfg, B, 31 + B)
    try:
        pi.pi_debug_set_mma_min_batch(c64.handle, 2)
        idx, cnt, _ = G.predict_checked(c64, 0, layer, x)
        pi.pi_debug_set_mma_min_batch(c64.handle, 0)
        idx2, cnt2 = c64.predict(0, G.dev16(x))
        c64.check()
    finally:
        pi.pi_debug_set_mma_min_batch(c64.handle, AUTO)
    m = int(cnt.item())
    assert m == int(cnt2.item())
    assert np.array_equal(idx[:m].cpu().numpy(), idx2[:m].cpu().numpy())


@pytest.mark.parametrize("name", ["relu_f16", "reglu_bf16", "relu_q4", "ring_wrap"])
@pytest.mark.parametrize("B", [1, 3, 8, 64])
@pytest.mark.parametrize("path", ["default", "step kernel"], indirect=True)
def test_hot_prefix_lists_and_ffn_match_oracle(c64, name, B, path):
    """Neurons [0, hot) of the physical order are always active and their
    predictor rows are skipped: the list equals the oracle's with those
    neurons forced on, for a prefix inside a mask word, on a word boundary,
    past whole output tiles of the batched predictor, and all but one or
    every neuron; the FFN on that list matches."""
    cfg, layer = _layer(name)
    if name == "ring_wrap" and B == 64:
        pytest.skip("the oracle's predictor at r = 2048 and 64 tokens is slow; B <= 8 covers the narrow tile")
    perm = np.random.default_rng(5).permutation(cfg.n).astype(np.int32)
    c64.load_layer(0, layer, perm)
    x = W.xhat_inputs(cfg, B, 41 + B)
    try:
        for hot in (0, 1, 31, 32, 33, 200, cfg.n - 1, cfg.n):
            c64.set_hot_prefix(0, hot)
            idx, cnt, oidx = G.predict_checked(c64, 0, layer, x, perm, hot=perm[:hot])
            assert np.array_equal(idx[:hot].cpu().numpy(), np.arange(hot))
            if hot == 200:
                G.ffn_checked(c64, 0, layer, x, idx, cnt, oidx)
    finally:
        c64.set_hot_prefix(0, 0)
    with pytest.raises(pi.PiError):
        c64.set_hot_prefix(0, cfg.n + 1)


@pytest.mark.parametrize("layerwise", [True, False])
def test_decode_stack_with_crossover_hot_prefix(layerwise):
    """A three-layer stack whose hot prefixes come from the calibration
    counts at the crossover for the batch (pi_choose_hot_prefix): every layer's
    list equals the oracle's with the calibrated order's first neurons forced
    on, and the update matches."""
    t = G.torch()
    cfg = CFGS["relu_f16"]
    B, L, T = 8, 3, 64
    c = G.ctx(max_layers=L, max_batch=B)
    if not layerwise:
        pi.pi_debug_set_mma_min_batch(c.handle, 0)
    layers, perms, hots = [], [], []
    for l in range(L):
        lw = W.make_layer(cfg, l, 0, random_b1=True, random_bdown=True)
        c.load_layer(l, lw)
        cal = W.calibration_inputs(cfg, l, 0, T=T)
        perm = pi.pi_perm_from_counts(c.layer_counts(l, G.dev16(cal)).cpu().numpy())
        c.load_layer(l, lw, perm)
        counts = c.layer_counts(l, G.dev16(cal)).cpu().numpy()  # physical order, descending
        hot = c.choose_hot_prefix(l, counts, T, B)
        assert 0 < hot < cfg.n
        # the layer's bytes: W2 row and b2 predicted; W_up row, bias and W_down^T row computed
        assert hot == pi.pi_hot_prefix_crossover(counts, T, B, 2.0 * cfg.r + 2, 2 * cfg.d * 2.0 + 2)
        c.set_hot_prefix(l, hot)
        layers.append(lw)
        perms.append(perm)
        hots.append(hot)
    assert len(set(hots)) > 1 or hots[0] > 32
    x0 = W.decode_inputs(cfg, B, 6)
    x = t.from_numpy(x0.copy()).cuda()
    tx = t.zeros((L, B, cfg.d), dtype=t.float32, device="cuda")
    txh = t.zeros((L, B, cfg.d), dtype=t.int16, device="cuda")
    tidx = t.full((L, cfg.n), -1, dtype=t.int32, device="cuda")
    tcnt = t.zeros(L, dtype=t.int32, device="cuda")
    c.set_trace(tx, txh, tidx, tcnt)
    c.decode_step(x)
    c.check()
    xs = np.concatenate([tx.cpu().numpy(), x.cpu().numpy()[None]], 0).astype(np.float64)
    xh = G.host16(txh)
    for l in range(L):
        m = int(tcnt[l].item())
        gidx = tidx[l, :m].cpu().numpy()
        assert np.array_equal(gidx[:hots[l]], np.arange(hots[l]))
        oidx = O.union(O.layer_predict(layers[l], xh[l], hot=perms[l][:hots[l]])["mask"])
        assert np.array_equal(np.sort(perms[l][gidx]), oidx)
        err = max_rel_err(xs[l + 1] - xs[l], O.masked_ffn(layers[l], xh[l], oidx))
        assert err <= G.tol(layers[l]), f"layer {l}: {err:.3g}"
    c.close()


@pytest.mark.parametrize("B", [1, 2, 8])
def test_distilled_predictor_runs_unchanged_on_the_gpu(c64, B):
    """A predictor fitted offline to the layer's fired sets (another rank than
    the layer's own) loads like any other: the lists equal the oracle's."""
    pytest.importorskip("torch")
    from activation_sparse_decode_sigmoid_gb300 import distill as D
    cfg, layer = _layer("relu_f16")
    fitted = D.distill(layer, W.calibration_inputs(cfg, 0, 0, T=1024), 48, steps=100)
    c64.load_layer(0, fitted)
    x = W.xhat_inputs(cfg, B, 51 + B)
    idx, cnt, oidx = G.predict_checked(c64, 0, fitted, x)
    G.ffn_checked(c64, 0, fitted, x, idx, cnt, oidx)


@pytest.mark.parametrize("B", [1, 2, 8])
def test_stack_with_a_rank_per_layer(B):
    """Distilled predictors of different ranks per layer (16, 48, 32) in one
    stack: each layer's list equals the oracle's on the GPU's x_hat, and the
    update matches."""
    pytest.importorskip("torch")
    from activation_sparse_decode_sigmoid_gb300 import distill as D
    t = G.torch()
    cfg = CFGS["relu_f16"]
    L = 3
    c = G.ctx(max_layers=L, max_batch=8)
    layers = []
    for l, rank in enumerate((16, 48, 32)):
        lw = W.make_layer(cfg, l, 0, random_bdown=True)
        fitted = D.distill(lw, W.calibration_inputs(cfg, l, 0, T=512), rank, steps=50, seed=l)
        c.load_layer(l, fitted)
        layers.append(fitted)
    x0 = W.decode_inputs(cfg, B, 12)
    x = t.from_numpy(x0.copy()).cuda()
    tx = t.zeros((L, B, cfg.d), dtype=t.float32, device="cuda")
    txh = t.zeros((L, B, cfg.d), dtype=t.int16, device="cuda")
    tidx = t.full((L, cfg.n), -1, dtype=t.int32, device="cuda")
    tcnt = t.zeros(L, dtype=t.int32, device="cuda")
    c.set_trace(tx, txh, tidx, tcnt)
    c.decode_step(x)
    c.check()
    xs = np.concatenate([tx.cpu().numpy(), x.cpu().numpy()[None]], 0).astype(np.float64)
    xh = G.host16(txh)
    for l in range(L):
        m = int(tcnt[l].item())
        oidx = O.union(O.layer_predict(layers[l], xh[l])["mask"])
        assert np.array_equal(tidx[l, :m].cpu().numpy(), oidx)
        err = max_rel_err(xs[l + 1] - xs[l], O.masked_ffn(layers[l], xh[l], oidx))
        assert err <= G.tol(layers[l]), f"layer {l}: {err:.3g}"
    c.close()


def test_large_batch_decode_x_hat_and_list_match_fused_kernel():
    """A batch of 8 decodes layer by layer (RMSNorm launch, batched
    predictor, tensor-core FFN); with the tensor cores off the same batch
    runs in the persistent step kernel.  Both compute x_hat in one reduction
    order and the lists by the same dot products: layer 0's x_hat and list
    are bit-identical (later layers see slightly different FFN sums)."""
    t = G.torch()
    cfg = CFGS["relu_f16"]
    B, L = 8, 2
    c = G.ctx(max_layers=L, max_batch=B)
    for l in range(L):
        c.load_layer(l, W.make_layer(cfg, l, 0, random_b1=True, random_bdown=True))
    x0 = W.decode_inputs(cfg, B, 8)
    out = []
    for mma in (2, 0):
        pi.pi_debug_set_mma_min_batch(c.handle, mma)
        x = t.from_numpy(x0.copy()).cuda()
        tx = t.zeros((L, B, cfg.d), dtype=t.float32, device="cuda")
        txh = t.zeros((L, B, cfg.d), dtype=t.int16, device="cuda")
        tidx = t.full((L, cfg.n), -1, dtype=t.int32, device="cuda")
        tcnt = t.zeros(L, dtype=t.int32, device="cuda")
        c.set_trace(tx, txh, tidx, tcnt)
        c.decode_step(x)
        c.check()
        c.set_trace(None, None, None, None)
        m = int(tcnt[0].item())
        out.append((txh[0].cpu().numpy(), tidx[0, :m].cpu().numpy(), tx[0].cpu().numpy()))
    assert np.array_equal(out[0][2], out[1][2]) and np.array_equal(out[0][2], x0)
    assert np.array_equal(out[0][0], out[1][0])
    assert np.array_equal(out[0][1], out[1][1])
    c.close()


def test_layerwise_threshold_follows_the_layer_kind():
    """By default a 16-bit layer runs layer by layer from 2 tokens, a Q4_0
    layer from 3; a set threshold overrides both until -1 restores them."""
    c = G.ctx(max_layers=3, max_batch=8)
    c.load_layer(0, _layer("relu_f16")[1])
    c.load_layer(1, _layer("reglu_bf16")[1])
    c.load_layer(2, _layer("relu_q4")[1])
    ls = (0, 1, 2)
    assert [pi.pi_layerwise_min_batch(c.handle, l) for l in ls] == [2, 2, 3]
    pi.pi_debug_set_mma_min_batch(c.handle, 0)
    assert [pi.pi_layerwise_min_batch(c.handle, l) for l in ls] == [0, 0, 0]
    pi.pi_debug_set_mma_min_batch(c.handle, 5)
    assert [pi.pi_layerwise_min_batch(c.handle, l) for l in ls] == [5, 5, 5]
    pi.pi_debug_set_mma_min_batch(c.handle, AUTO)
    assert [pi.pi_layerwise_min_batch(c.handle, l) for l in ls] == [2, 2, 3]
    with pytest.raises(pi.PiError):
        pi.pi_debug_set_mma_min_batch(c.handle, -2)
    c.close()


def test_layerwise_decode_step_replays_from_a_cuda_graph():
    """Batches that run layer by layer depend on no host state that changes
    between calls, so a decode step captured once into a CUDA graph replays
    on new inputs with the eager step's results, bit for bit."""
    t = G.torch()
    cfg = CFGS["reglu_bf16"]
    B, L = 8, 2
    c = G.ctx(max_layers=L, max_batch=B)
    for l in range(L):
        c.load_layer(l, W.make_layer(cfg, l, 0, random_b1=True, random_bdown=True))
    xs = [t.from_numpy(W.decode_inputs(cfg, B, s)).cuda() for s in (11, 12, 13)]
    want = []
    for x in xs:
        y = x.clone()
        c.decode_step(y)
        c.check()
        want.append(y)
    buf = xs[0].clone()
    side = t.cuda.Stream()
    side.wait_stream(t.cuda.current_stream())
    with t.cuda.stream(side):  # warm-up on the capture's side stream
        c.decode_step(buf)
    t.cuda.current_stream().wait_stream(side)
    t.cuda.synchronize()
    g = t.cuda.CUDAGraph()
    with t.cuda.graph(g):
        c.decode_step(buf)
    for x, w in zip(xs, want):
        buf.copy_(x)
        g.replay()
        t.cuda.synchronize()
        c.check()
        assert t.equal(buf, w)
    c.close()


@pytest.mark.parametrize("knobs", [(0, 0, 0, 0), (1, 0, 2, 4), (2, 400, 4, 0), (3, 800, 3, 8), (3, 0, 16, 64)])
def test_tuning_knobs_do_not_change_results(knobs):
    """Prefetch modes, the FFN lookahead and row prefetch only move data
    earlier: a 3-layer decode step is bit-identical under every setting."""
    t = G.torch()
    cfg = CFGS["relu_f16"]
    c = G.ctx(max_layers=3, max_batch=4)
    pi.pi_debug_set_mma_min_batch(c.handle, 0)  # the knobs tune the step kernel
    for l in range(3):
        c.load_layer(l, W.make_layer(cfg, l, 0, random_b1=True, random_bdown=True))
    x0 = t.from_numpy(W.decode_inputs(cfg, 2, 6)).cuda()
    ref = x0.clone()
    c.decode_step(ref)
    c.check()
    pi.pi_debug_set_tuning(c.handle, *knobs)
    got = x0.clone()
    c.decode_step(got)
    c.check()
    assert t.equal(got, ref)
    c.close()


def test_timeout_is_reported_and_context_recovers():
    """A grid barrier that can never complete (one phantom arrival expected)
    must time out, report PI_ERR_TIMEOUT and leave the context usable."""
    t = G.torch()
    cfg, layer = _layer("relu_f16")
    c = G.ctx(max_layers=1, max_batch=1)
    c.load_layer(0, layer)
    x = t.from_numpy(W.decode_inputs(cfg, 1, 0)).cuda()
    ref = x.clone()
    c.decode_step(ref)
    c.check()
    pi.pi_debug_set_wait_limit(c.handle, 50_000_000)  # 50 ms
    pi.pi_debug_barrier_extra(c.handle, 1)
    bad = x.clone()
    c.decode_step(bad)
    assert c.sync_status() == pi.PI_ERR_TIMEOUT
    pi.pi_debug_barrier_extra(c.handle, 0)
    again = x.clone()
    c.decode_step(again)
    c.check()
    assert t.equal(again, ref)  # deterministic and unaffected by the failed launch
    c.close()


def _until_timeout(run, c, tries=5):
    """Run `run` (a call under a one-nanosecond wait limit) until a bounded
    wait runs out; returns the last status."""
    st = pi.PI_OK
    for _ in range(tries):
        run()
        st = c.sync_status()
        if st == pi.PI_ERR_TIMEOUT:
            break
    return st


@pytest.mark.parametrize("call", ["sparse_ffn", "decode_step"])
def test_layerwise_timeout_is_reported_and_next_call_is_unchanged(call):
    """Eight tokens run layer by layer: the batched predictor's launches and
    the tensor-core FFN (ffn_up_mma, ffn_down_mma).  With a wait limit of one
    nanosecond every bounded wait that has to spin runs out: the call reports
    PI_ERR_TIMEOUT, and every CTA lets its own bulk copies and MMAs finish
    before it exits (the producers that stopped early complete the stages
    they skipped).  The same call afterwards gives the clean result bit for
    bit."""
    t = G.torch()
    cfg = CFGS["ring_wrap"]  # d 4096: 64 pipeline stages per row pass, waits are not instant
    B, L = 8, 2
    c = G.ctx(max_layers=L, max_batch=B)
    for l in range(L):
        c.load_layer(l, W.make_layer(cfg, l, 0, random_b1=True, random_bdown=True))
    assert pi.pi_layerwise_min_batch(c.handle, 0) <= B
    if call == "sparse_ffn":
        x = G.dev16(W.xhat_inputs(cfg, B, 71))
        idx, cnt = c.predict(0, x)
        ref = c.sparse_ffn(0, x, idx, cnt)
        c.check()
        run = lambda: c.sparse_ffn(0, x, idx, cnt)  # noqa: E731
        again = lambda: c.sparse_ffn(0, x, idx, cnt)  # noqa: E731
    else:
        x0 = t.from_numpy(W.decode_inputs(cfg, B, 72)).cuda()
        ref = x0.clone()
        c.decode_step(ref)
        c.check()

        def run():
            c.decode_step(x0.clone())

        def again():
            y = x0.clone()
            c.decode_step(y)
            return y
    pi.pi_debug_set_wait_limit(c.handle, 1)  # 1 ns
    try:
        st = _until_timeout(run, c)
    finally:
        pi.pi_debug_set_wait_limit(c.handle, 2_000_000_000)
    assert st == pi.PI_ERR_TIMEOUT
    got = again()
    c.check()
    assert t.equal(got, ref)
    c.close()


def test_out_of_range_index_is_flagged(c64):
    t = G.torch()
    cfg, layer = _layer("relu_f16")
    c64.load_layer(0, layer)
    x = G.dev16(W.xhat_inputs(cfg, 1, 0))
    idx = t.tensor([3, cfg.n + 5, 7], dtype=t.int32, device="cuda")
    cnt = t.tensor([3], dtype=t.int32, device="cuda")
    c64.sparse_ffn(0, x, idx, cnt)
    assert c64.sync_status() == pi.PI_ERR_DEVICE_FLAG
    cnt_bad = t.tensor([cfg.n + 1], dtype=t.int32, device="cuda")
    c64.sparse_ffn(0, x, idx, cnt_bad)
    assert c64.sync_status() == pi.PI_ERR_DEVICE_FLAG
    ok_idx = t.tensor([3, 7], dtype=t.int32, device="cuda")
    c64.sparse_ffn(0, x, ok_idx, t.tensor([2], dtype=t.int32, device="cuda"))
    c64.check()


def test_host_side_errors(c64):
    cfg, layer = _layer("relu_f16")
    bad = dict(layer, d=260)  # not a multiple of 8
    with pytest.raises(pi.PiError) as e:
        c64.load_layer(1, bad)
    assert e.value.status == pi.PI_ERR_SHAPE
    with pytest.raises(pi.PiError) as e:
        c64.load_layer(0, layer, perm=np.zeros(cfg.n, np.int32))
    assert e.value.status == pi.PI_ERR_ARG
    with pytest.raises(pi.PiError) as e:
        pi.pi_predict(c64.handle, 3, None, 1, None, None)
    assert e.value.status in (pi.PI_ERR_NOT_LOADED, pi.PI_ERR_ARG)
