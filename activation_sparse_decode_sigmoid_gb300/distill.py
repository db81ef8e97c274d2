"""Offline predictor distillation and per-layer rank choice (the "adaptive
predictor" of the pages, without real data).

PowerInfer runs the model offline on general inputs, records which neurons
each layer's input activates, and trains a small routing predictor per layer
on those pairs (blog.csdn.net QbitAI/IPADS article, "充分利用模型和硬件特点");
its predictors are adaptive in size (de.news.hada.io summary,
"CPU/GPU-Hybrid-Inferenzansatz").  Here the layers are synthetic, so the
training pairs come from the layer itself: for inputs x_hat the fired set is
{i : W_up[i] . x_hat + b_i > 0} (the gate row for ReGLU), and the predictor
h = relu(W1 x_hat + b1), z = W2 h + b2 is fitted to it with a weighted
logistic loss.  The fitted weights are rounded to the layer's 16-bit type and
replace p_w1, p_b1, p_w2, p_b2; the hot path runs them unchanged.

Training is offline plumbing in plain PyTorch (CPU or GPU); nothing here runs
on the decode path.
"""
from __future__ import annotations

import numpy as np

from . import workload as W


def _rows_f32(rows, w_dtype: int, d: int) -> np.ndarray:
    """16-bit rows [n, d] (bit patterns) or Q4_0 rows [n, d/32*18] as float32."""
    if w_dtype != W.Q4_0:
        return W.from_bits(rows, w_dtype).astype(np.float32)
    blocks = np.ascontiguousarray(rows, dtype=np.uint8).reshape(rows.shape[0], d // 32, 18)
    scale = blocks[:, :, :2].copy().view(np.float16).astype(np.float32)  # [n, nb, 1]
    q = blocks[:, :, 2:]
    lo = (q & 15).astype(np.int32) - 8
    hi = (q >> 4).astype(np.int32) - 8
    vals = np.concatenate([lo, hi], axis=2).astype(np.float32) * scale
    return vals.reshape(rows.shape[0], d)


def fired_sets(layer: dict, xhat_bits) -> np.ndarray:
    """bool [T, n]: the neurons whose activation is nonzero for each input
    (pre-activation of the ReLU, i.e. of the gate for ReGLU, above zero), in
    fp32.  These are the labels the predictor is trained on."""
    import torch
    d = layer["d"]
    x = torch.from_numpy(W.from_bits(np.asarray(xhat_bits).reshape(-1, d), layer["act_dtype"]).astype(np.float32))
    rows = layer["w_gate"] if layer["act"] == W.REGLU else layer["w_up"]
    w = torch.from_numpy(_rows_f32(rows, layer["w_dtype"], d))
    b = torch.from_numpy(W.from_bits(layer["b"], layer["act_dtype"]).astype(np.float32))
    return ((x @ w.T) + b > 0).numpy()


def predicted_sets(layer: dict, xhat_bits) -> np.ndarray:
    """bool [T, n]: z > 0 for the layer's predictor, evaluated in fp32 with
    torch (the order of the sums differs from the kernels', which decides
    only logits within rounding of zero)."""
    import torch
    dt, d = layer["act_dtype"], layer["d"]
    f = lambda a: torch.from_numpy(W.from_bits(a, dt).astype(np.float32))
    x = f(np.asarray(xhat_bits).reshape(-1, d))
    h = x @ f(layer["p_w1"]).T
    if layer.get("p_b1") is not None:
        h = h + f(layer["p_b1"])
    z = torch.relu(h) @ f(layer["p_w2"]).T + f(layer["p_b2"])
    return (z > 0).numpy()


def set_quality(pred: np.ndarray, fired: np.ndarray) -> dict:
    """Recall (fired neurons predicted), precision, and the predicted and
    fired densities, pooled over all inputs."""
    tp = float(np.logical_and(pred, fired).sum())
    return {"recall": tp / max(1.0, float(fired.sum())), "precision": tp / max(1.0, float(pred.sum())),
            "predicted_density": float(pred.mean()), "fired_density": float(fired.mean())}


def distill(layer: dict, x_train, rank: int, *, steps: int = 300, lr: float = 3e-3, pos_weight: float = 4.0,
            batch: int = 1024, seed: int = 0, device: str = "cpu") -> dict:
    """A copy of `layer` whose predictor (rank `rank`) is fitted to the layer's
    fired sets on the inputs x_train (16-bit bit patterns [T, d]).

    Loss: logistic loss of z against the fired labels, fired neurons weighted
    pos_weight (> 1 trades precision for recall: a missed neuron changes the
    output, a spurious one only costs its rows).  Adam, `steps` minibatches
    of `batch` inputs, seeded.  Initial b2 = the logit of each neuron's fired
    rate, so training starts from the frequency prior."""
    import torch
    dt, d, n = layer["act_dtype"], layer["d"], layer["n"]
    g = torch.Generator(device="cpu").manual_seed(seed)
    x = torch.from_numpy(W.from_bits(np.asarray(x_train).reshape(-1, d), dt).astype(np.float32))
    y = torch.from_numpy(fired_sets(layer, x_train).astype(np.float32))
    T = x.shape[0]
    rate = y.mean(0).clamp(1.0 / (T + 1), 1.0 - 1.0 / (T + 1))
    w1 = (torch.randn(rank, d, generator=g) / d ** 0.5).to(device).requires_grad_()
    b1 = torch.zeros(rank, device=device, requires_grad=True)
    w2 = (torch.randn(n, rank, generator=g) / rank ** 0.5).to(device).requires_grad_()
    b2 = torch.log(rate / (1 - rate)).to(device).requires_grad_()
    x, y = x.to(device), y.to(device)
    opt = torch.optim.Adam([w1, b1, w2, b2], lr=lr)
    loss_fn = torch.nn.BCEWithLogitsLoss(pos_weight=torch.full((n,), float(pos_weight), device=device))
    for _ in range(steps):
        sel = torch.randint(0, T, (min(batch, T),), generator=g).to(device)
        z = torch.relu(x[sel] @ w1.T + b1) @ w2.T + b2
        loss = loss_fn(z, y[sel])
        opt.zero_grad()
        loss.backward()
        opt.step()
    out = dict(layer)
    out["r"] = rank
    bits = lambda t: W.to_bits(t.detach().cpu().numpy().astype(np.float32), dt)
    out["p_w1"], out["p_b1"], out["p_w2"], out["p_b2"] = bits(w1), bits(b1), bits(w2), bits(b2)
    return out


def adaptive_rank(layer: dict, x_train, x_test, ranks, target_recall: float, **kw):
    """Distil one predictor per rank (ascending) and keep the smallest whose
    recall on x_test reaches target_recall (else the largest).  Returns
    (chosen layer, [(rank, quality dict), ...])."""
    fired = fired_sets(layer, x_test)
    tried, chosen = [], None
    for r in sorted(ranks):
        cand = distill(layer, x_train, r, **kw)
        q = set_quality(predicted_sets(cand, x_test), fired)
        tried.append((r, q))
        chosen = cand
        if q["recall"] >= target_recall:
            break
    return chosen, tried
