#!/usr/bin/env python3
"""Benchmark of the predictor -> neuron-aware sparse FFN decode step on GB300.

Default workload: the largest of the five workloads, the LLaMA-70B-shaped
ReGLU FFN stack in bf16 (80 layers, d_model 8192, d_ffn 28672, predictor rank
1024), seeded synthetic Zipf-sparse weights drawn on the device, neurons
permuted by a 256-token calibration profile, batch 1.  One step = one decode
token through all 80 layers = one launch of the persistent step kernel.
Every step streams ~17 GB of distinct weights, far more than the 129 MB L2,
so no flush is needed between steps.  --config selects another workload.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  --impl reference times the CPU oracle on the
host cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sparse-FFN decode tokens/s (1 GB300) and effective HBM GB/s vs 8 TB/s roofline"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="llama70b_reglu_bf16")
    ap.add_argument("--batch", type=int, default=1)
    ap.add_argument("--layers", type=int, default=0, help="override the stack depth (0 = the config's)")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-extras", action="store_true", help="skip dense, e2e and CPU legs")
    ap.add_argument("--hot-prefix", action="store_true",
                    help="give every layer its always-active prefix at the byte crossover for the batch")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="CPU-oracle sample budget")
    ap.add_argument("--mode", choices=["step", "ffn", "sequence"], default="step",
                    help="step: the decode step over the stack (the headline); ffn: the sparse FFN of one "
                         "full-size layer alone, for per-kernel numbers; sequence: the workload's prompt "
                         "(one step of its prompt length) followed by its decode tokens one at a time")
    return ap.parse_args()


# ------------------------------------------------------------------ distributed plumbing
def dist_init(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def allreduce_max(world, v: float, device) -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ peaks, clocks, profiles
def measured_hbm():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.path = tempfile.mktemp(prefix="clocks_", suffix=".csv")
        self.proc = None
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(device_index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        self.t0 = self.t1 = None

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        try:
            sm = [float(r[1]) for r in rows]
            mx = max(float(r[2]) for r in rows)
        except ValueError:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        loaded = [s for s in sm if s > 0.5 * mx] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": mx, "reasons": reasons, "samples": len(rows)}


ACT_NAMES = ("ReLU", "ReGLU", "squared ReLU")  # by the workload's activation ids 0, 1, 2

# The sources the persistent step kernel is built from, with the host plan
# that sizes its rings (pi_api.cu): a profile's DRAM counters stand for the
# kernel only while these files are unchanged.
STEP_SOURCES = ("pi_api.cu", "pi_device.cuh", "pi_kernels.h", "pi_step.cuh", "pi_step_bf16.cu", "pi_step_f16.cu",
                "pi_step_q4.cu")


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "activation_sparse_decode_sigmoid_gb300", "csrc")
    files = sorted(os.path.join(csrc, f) for f in STEP_SOURCES)
    for p in files:
        with open(p, "rb") as f:
            h.update(os.path.basename(p).encode() + f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per launch of the step kernel from a committed ncu summary,
    if it was taken on the current kernel sources (else None)."""
    for p in glob.glob(os.path.join(ROOT, "profiles", "*.md")):
        kv = {}
        with open(p) as f:
            for line in f:
                if line.startswith("- ") and ":" in line:
                    k, v = line[2:].split(":", 1)
                    kv[k.strip()] = v.strip().strip("`")
        if kv.get("workload") == workload and kv.get("kernel_source_hash") == kernel_source_hash():
            try:
                return float(kv["traffic_bytes_per_launch"])
            except (KeyError, ValueError):
                pass
    return None


# ------------------------------------------------------------------ workload
def algorithmic_bytes(cfg, L, B, counts, hot=None):
    """Bytes a step must move: predictor weights + biases (the rows of the
    neurons past each layer's hot prefix), the rows of the active neurons
    (W_up [+ W_gate] + W_down^T + bias), x_hat / x traffic."""
    from activation_sparse_decode_sigmoid_gb300 import workload as W
    d, n, r = cfg.d, cfg.n, cfg.r
    rows = 3 if cfg.act == W.REGLU else 2
    row = d * 18 / 32 if cfg.w_dtype == W.Q4_0 else d * 2
    total = 0.0
    for l, m in enumerate(counts):
        h = hot[l] if hot else 0
        pred = r * d * 2 + (n - h) * r * 2 + (r + n - h) * 2
        total += pred + m * (rows * row + 2) + B * d * (2 + 4 + 4)
    return total


def cpu_oracle_sample(cfg, L, host_layers, seed, budget_s, hot=None):
    """Time the oracle (as it stands, all host cores) on layer-token pairs of
    the workload until the budget is used; returns tokens/s for the stack."""
    import numpy as np
    import oracle as O
    from activation_sparse_decode_sigmoid_gb300 import workload as W

    threads = O.default_threads()
    xs = W.xhat_inputs(cfg, 8, seed + 7)
    times, pairs = [], 0
    t_start = time.perf_counter()
    for tok in range(8):
        for l, (lw, perm) in host_layers.items():
            x = xs[tok: tok + 1]
            h = hot.get(l, 0) if hot else 0
            t0 = time.perf_counter()
            res = O.layer_predict(lw, x, threads, hot=perm[:h] if h else None)
            idx = O.union(res["mask"])
            O.masked_ffn(lw, x, idx, threads)
            times.append(time.perf_counter() - t0)
            pairs += 1
            if time.perf_counter() - t_start > budget_s:
                break
        if time.perf_counter() - t_start > budget_s:
            break
    per_layer = sum(times) / len(times)
    return {"value": 1.0 / (per_layer * L), "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{pairs} (layer, token) pairs of the full-size workload (layers {sorted(host_layers)}), "
                      f"mean {per_layer:.3f} s per layer, scaled to the {L}-layer stack"}


def host_layers_numpy(cfg, layers, seed):
    from activation_sparse_decode_sigmoid_gb300 import workload as W
    return {l: (W.make_layer(cfg, l, seed), None) for l in layers}


# ------------------------------------------------------------------ arms
def run_reference(args, world, rank):
    """The oracle on the host cores, same config/metric, bounded per step."""
    import oracle as O
    from activation_sparse_decode_sigmoid_gb300 import workload as W

    if rank != 0:
        return
    O.build()
    cfg = W.CONFIGS[args.config]
    L = args.layers or cfg.L
    hl = host_layers_numpy(cfg, [0, 1], args.seed)
    threads = O.default_threads()
    xs = W.xhat_inputs(cfg, args.steps + args.warmup, args.seed + 7)
    keys = sorted(hl)

    def step(i):
        lw = hl[keys[i % len(keys)]][0]
        x = xs[i: i + 1]
        res = O.layer_predict(lw, x, threads)
        O.masked_ffn(lw, x, O.union(res["mask"]), threads)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i)
    el = time.perf_counter() - t0
    per_layer = el / args.steps
    value = args.batch / (per_layer * L)
    # a step of this arm is one (layer, token) pair: ms_per_step is its
    # measured time; the token through the whole stack is that time x L
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_layer * 1e3,
        "ms_per_token_scaled": per_layer * L * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_block(cfg, L, args.batch),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": f"each step = one (layer, token) pair of the full-size stack (ms_per_step is "
                                   f"its measured time); tokens/s = 1 / (that time x {L} layers)"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


L2_BYTES = 129 * 2 ** 20  # GB300's L2


def stack_weight_bytes(cfg, L) -> float:
    """Bytes of every weight of an L-layer stack (predictor and FFN)."""
    from activation_sparse_decode_sigmoid_gb300 import workload as W
    rows = 3 if cfg.act == W.REGLU else 2
    row = cfg.d * 18 / 32 if cfg.w_dtype == W.Q4_0 else cfg.d * 2
    return L * (cfg.r * cfg.d * 2 + cfg.n * cfg.r * 2 + cfg.n * rows * row)


def needs_l2_flush(cfg, L) -> bool:
    """A stack that fits twice in L2 would be timed from L2, not HBM."""
    return stack_weight_bytes(cfg, L) < 2 * L2_BYTES


def config_block(cfg, L, B, hot=None):
    from activation_sparse_decode_sigmoid_gb300 import workload as W
    l2 = ("flushed: the stack fits in L2, so a buffer of twice the L2 size is written before every "
          "timed step, outside that step's CUDA events" if needs_l2_flush(cfg, L)
          else "no flush: each step streams the whole stack (GBs) through the 129 MB L2")
    return {"workload": f"{cfg.name}: {L} layers, d_model {cfg.d}, d_ffn {cfg.n}, predictor rank {cfg.r}, "
                        f"{ACT_NAMES[cfg.act]}, weights {W.DTYPE_NAMES[cfg.w_dtype]}, "
                        f"Zipf alpha {cfg.alpha}, mean activation {cfg.rho}",
            "batch": B, "seq_len": 1, "parallelism": "replicas (one independent stack per GPU)",
            "l2": l2, "seed": 0,
            **({"hot_prefix": f"neurons [0, H) always active, H at the byte crossover for {B} tokens: "
                              f"mean H {sum(hot) / len(hot):.0f} of {cfg.n} (min {min(hot)}, max {max(hot)})"}
               if hot and any(hot) else {})}


def run_ours(args, world, rank, local):
    import numpy as np
    import torch
    from activation_sparse_decode_sigmoid_gb300 import build as libbuild
    from activation_sparse_decode_sigmoid_gb300 import pi
    from activation_sparse_decode_sigmoid_gb300 import workload as W

    libbuild.build()
    device = local
    torch.cuda.set_device(device)
    cfg = W.CONFIGS[args.config]
    L = args.layers or cfg.L
    B = args.batch
    K, Wm = args.steps, args.warmup
    do_extras = not args.no_extras
    do_cpu = do_extras and rank == 0 and world == 1
    from activation_sparse_decode_sigmoid_gb300.calibrate import load_synthetic_stack
    ctx, host = load_synthetic_stack(cfg, L, args.seed, device, max(B, 1), keep_host=(0, L // 2) if do_cpu else (),
                                     hot_batch=B if args.hot_prefix else 0)
    hot = [ctx.hot.get(l, 0) for l in range(L)]
    d = cfg.d
    xbuf = torch.from_numpy(W.decode_inputs(cfg, (K + Wm) * B, args.seed)).cuda(device).view(K + Wm, B, d)
    cnt = torch.zeros((K + Wm, L), dtype=torch.int32, device=device)
    stream = torch.cuda.current_stream(device)

    clocks = ClockSampler(device) if rank == 0 else None
    for i in range(Wm):
        ctx.set_trace(None, None, None, cnt[i])
        ctx.decode_step(xbuf[i])
    ctx.check()
    flush = needs_l2_flush(cfg, L)
    if flush:  # twice the device's L2, written before every timed step
        l2 = torch.cuda.get_device_properties(device).L2_cache_size
        flush_buf = torch.empty(2 * l2, dtype=torch.uint8, device=device)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(K + 1)]
    ev_start = [torch.cuda.Event(enable_timing=True) for _ in range(K)] if flush else None
    torch.cuda.synchronize(device)
    barrier(world)
    if clocks:
        clocks.mark_start()
    torch.cuda.nvtx.range_push("timed")
    ev[0].record(stream)
    for k in range(K):
        ctx.set_trace(None, None, None, cnt[Wm + k])
        if flush:
            flush_buf.zero_()
            ev_start[k].record(stream)
        ctx.decode_step(xbuf[Wm + k])
        ev[k + 1].record(stream)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize(device)
    if clocks:
        clocks.mark_end()
    barrier(world)
    st = ctx.sync_status()
    if st:
        raise RuntimeError(f"device status {st}: {pi.pi_last_error(ctx.handle)}")
    if flush:  # the steps alone, without the flushes between them
        per_launch = [ev_start[k].elapsed_time(ev[k + 1]) for k in range(K)]
        ms = sum(per_launch)
    else:
        per_launch = [ev[k].elapsed_time(ev[k + 1]) for k in range(K)]
        ms = ev[0].elapsed_time(ev[K])
    ms = allreduce_max(world, ms, torch.device("cuda", device))
    counts = cnt[Wm:].cpu().numpy()  # [K][L] active neurons per layer
    bytes_per_step = [algorithmic_bytes(cfg, L, B, counts[k], hot) for k in range(K)]
    mean_launch_s = statistics.mean(per_launch) / 1e3
    achieved = statistics.mean(bytes_per_step) / mean_launch_s / 1e9
    peak, peak_kind = measured_hbm()
    value = world * K * B / (ms / 1e3)
    # batches from the library's layer-by-layer threshold on run per layer: RMSNorm, the
    # predictor's hidden layer, output layer and compaction, the FFN's up and down kernels
    # (Q4_0: with the rows dequantised in shared memory) and the share merge; smaller ones
    # are one persistent launch per step
    mb = pi.pi_layerwise_min_batch(ctx.handle, 0)
    layerwise = 0 < mb <= B
    q4 = cfg.w_dtype == W.Q4_0
    ffn = ("FFN up/gate and down (tcgen05, Q4_0 rows dequantised in shared memory), share merge" if q4 else
           "FFN up/gate (whole rows on the CUDA cores up to 4 tokens, else tcgen05), down (tcgen05), share merge")
    kernel = (f"per-layer launches: RMSNorm, batched predictor (3), {ffn}" if layerwise
              else "step_kernel (one persistent launch per step)")
    launches_per_step = 7 * L if layerwise else 1

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": Wm,
        "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": W.DTYPE_NAMES[cfg.w_dtype], "data": "synthetic", "config": config_block(cfg, L, B, hot),
        "effective_hbm_gbs": achieved, "frac_of_nominal_8tbs": achieved / NOMINAL_HBM_GBS,
        "mean_active_neurons_per_layer": float(counts.mean()), "mean_active_fraction": float(counts.mean() / cfg.n),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": f"{peak_kind} copy bandwidth (hbm_gbs)",
                     "traffic": None if layerwise else profiled_traffic(cfg.name + f"/L{L}/B{B}"),
                     "kernel": kernel},
        "gpu_launches": K * launches_per_step,
    }

    if do_extras:
        # dense baseline: the same stack, every neuron, same kernel family
        nd = max(2, min(5, K))
        xd = xbuf[:nd].clone()
        ctx.set_trace(None, None, None, None)
        ctx.dense_step(xd[0])
        torch.cuda.synchronize(device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(1, nd):
            ctx.dense_step(xd[i])
        e1.record(stream)
        torch.cuda.synchronize(device)
        dense_ms = e0.elapsed_time(e1) / (nd - 1)
        row = d * 18 / 32 if cfg.w_dtype == W.Q4_0 else d * 2
        dense_bytes = L * cfg.n * ((3 if cfg.act == W.REGLU else 2) * row + 2)
        line["dense_baseline"] = {"tokens_per_s": B / (dense_ms / 1e3), "ms_per_step": dense_ms,
                                  "effective_hbm_gbs": dense_bytes / (dense_ms / 1e3) / 1e9,
                                  "what": ("every neuron, no predictor, layer by layer on the tensor-core FFN" if layerwise
                                           else "same persistent kernel over every neuron, no predictor (cuBLAS-free dense GEMV)")}
        # end to end through the public API: one pi_decode_step_host call per
        # step (pinned host x in, H2D, the step, D2H, stream synchronised),
        # timed by the host clock
        ne = K
        xh_in = torch.from_numpy(W.decode_inputs(cfg, ne * B, args.seed + 3)).view(ne, B, d).pin_memory()
        xh_out = torch.empty_like(xh_in).pin_memory()
        for i in range(min(2, ne)):
            ctx.decode_step_host(xh_in[i], xh_out[i])
        torch.cuda.synchronize(device)
        barrier(world)
        t0 = time.perf_counter()
        for i in range(ne):
            ctx.decode_step_host(xh_in[i], xh_out[i])
        e2e_ms = (time.perf_counter() - t0) * 1e3
        e2e_ms = allreduce_max(world, e2e_ms, torch.device("cuda", device))
        line["e2e"] = {"value": world * ne * B / (e2e_ms / 1e3), "unit": "tokens/s",
                       "h2d_bytes_per_step": B * d * 4, "d2h_bytes_per_step": B * d * 4,
                       "call": "pi_decode_step_host (host buffers, copies and sync inside)"}
        ctx.check()
    if clocks:
        line["clocks"] = clocks.stop()
    if do_cpu:
        line["cpu_baseline"] = cpu_oracle_sample(cfg, L, host, args.seed, args.cpu_seconds, dict(enumerate(hot)))
    ctx.close()
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_ffn(args, world, rank, local):
    """pi_sparse_ffn on one calibrated full-size layer with the tokens' predicted
    union list: batches from the layer-by-layer threshold on run the
    tensor-core kernels, smaller ones the step kernel's FFN phase.  Bytes =
    the rows of the listed neurons."""
    import numpy as np
    import torch
    from activation_sparse_decode_sigmoid_gb300 import build as libbuild
    from activation_sparse_decode_sigmoid_gb300 import pi
    from activation_sparse_decode_sigmoid_gb300 import workload as W
    from activation_sparse_decode_sigmoid_gb300.calibrate import calibrate_and_load

    libbuild.build()
    torch.cuda.set_device(local)
    cfg = W.CONFIGS[args.config]
    B, K, Wm = args.batch, args.steps, args.warmup
    ctx = pi.Context(local, max_layers=1, max_batch=max(B, 1))
    dev = torch.device("cuda", local)
    lw = W.make_layer_device(cfg, 0, args.seed, dev)
    cal = torch.from_numpy(W.calibration_inputs(cfg, 0, args.seed).view(np.int16)).to(dev)
    calibrate_and_load(ctx, 0, lw, cal)
    del lw
    x = torch.from_numpy(W.xhat_inputs(cfg, B, args.seed + 5).view(np.int16)).to(dev)
    idx, cnt = ctx.predict(0, x)
    y = ctx.sparse_ffn(0, x, idx, cnt)
    for _ in range(Wm):
        ctx.sparse_ffn(0, x, idx, cnt, y)
    stream = torch.cuda.current_stream(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    barrier(world)
    e0.record(stream)
    for _ in range(K):
        ctx.sparse_ffn(0, x, idx, cnt, y)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ctx.check()
    ms = allreduce_max(world, e0.elapsed_time(e1) / K, dev)
    m = int(cnt.item())
    mb = pi.pi_layerwise_min_batch(ctx.handle, 0)
    tc = 0 < mb <= B  # the tensor-core FFN: up, down, merge
    rows = 3 if cfg.act == W.REGLU else 2
    row = cfg.d * 18 / 32 if cfg.w_dtype == W.Q4_0 else cfg.d * 2
    byts = m * (rows * row + 2) + B * cfg.d * 4
    gbs = byts / (ms / 1e3) / 1e9
    peak, kind = measured_hbm()
    ctx.close()
    if rank == 0:
        print(json.dumps({
            "metric": "sparse FFN of one layer, effective HBM GB/s", "value": gbs * world, "unit": "GB/s",
            "n_gpus": world, "steps": K, "warmup": Wm, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": W.DTYPE_NAMES[cfg.w_dtype], "data": "synthetic",
            "config": {"workload": f"{cfg.name}: one layer, d_model {cfg.d}, d_ffn {cfg.n}, batch {B}, "
                                   f"{m} listed neurons ({m / cfg.n:.3f} of d_ffn)",
                       "path": "tensor cores (tcgen05)" if tc else "step kernel"},
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                         "peak_source": f"{kind} copy bandwidth (hbm_gbs)", "traffic": None},
            "gpu_launches": K * (3 if tc else 1)}), flush=True)


def run_sequence(args, world, rank, local):
    """A prompt of cfg.prompt tokens (one batched step through the stack, the
    union of their predicted neurons) followed by cfg.tokens one-token decode
    steps, as the Falcon-40B-shaped Q4_0 workload defines it; each timed
    sequence is that whole run.  Tokens/s counts prompt and decode tokens."""
    import torch
    from activation_sparse_decode_sigmoid_gb300 import build as libbuild
    from activation_sparse_decode_sigmoid_gb300 import workload as W
    from activation_sparse_decode_sigmoid_gb300.calibrate import load_synthetic_stack

    libbuild.build()
    torch.cuda.set_device(local)
    cfg = W.CONFIGS[args.config]
    if cfg.prompt < 1:
        raise SystemExit(f"{cfg.name} has no prompt phase")
    L = args.layers or cfg.L
    P, T, K, Wm = cfg.prompt, cfg.tokens, args.steps, args.warmup
    ctx, _ = load_synthetic_stack(cfg, L, args.seed, local, P)
    d = cfg.d
    xp = torch.from_numpy(W.decode_inputs(cfg, (K + Wm) * P, args.seed)).cuda(local).view(K + Wm, P, d)
    xd = torch.from_numpy(W.decode_inputs(cfg, (K + Wm) * T, args.seed + 1)).cuda(local).view(K + Wm, T, 1, d)
    stream = torch.cuda.current_stream(local)

    def sequence(i, ev=None):
        ctx.decode_step(xp[i])
        if ev is not None:
            ev.record(stream)
        for t in range(T):
            ctx.decode_step(xd[i, t])

    for i in range(Wm):
        sequence(i)
    ctx.check()
    e = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    torch.cuda.synchronize(local)
    barrier(world)
    for k in range(K):
        e[k][0].record(stream)
        sequence(Wm + k, e[k][1])
        e[k][2].record(stream)
    torch.cuda.synchronize(local)
    ctx.check()
    ms = sum(a.elapsed_time(c) for a, _, c in e)
    ms_prompt = sum(a.elapsed_time(b) for a, b, _ in e) / K
    ms = allreduce_max(world, ms, torch.device("cuda", local))
    from activation_sparse_decode_sigmoid_gb300 import pi
    mb = pi.pi_layerwise_min_batch(ctx.handle, 0)
    per_prompt = 7 * L if 0 < mb <= P else 1
    ctx.close()
    if rank == 0:
        print(json.dumps({
            "metric": "prompt + decode tokens/s of the workload's sequence", "value": world * K * (P + T) / (ms / 1e3),
            "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": Wm, "ms_per_step": ms / K,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": W.DTYPE_NAMES[cfg.w_dtype],
            "data": "synthetic",
            "config": {"workload": f"{cfg.name}: {L} layers, a {P}-token prompt step then {T} one-token steps",
                       "seq_len": P + T},
            "prompt_ms": ms_prompt, "prompt_tokens_per_s": P / (ms_prompt / 1e3),
            "decode_ms_per_token": (ms / K - ms_prompt) / T,
            "decode_tokens_per_s": T / ((ms / K - ms_prompt) / 1e3),
            "gpu_launches": K * (per_prompt + T)}), flush=True)


def main():
    args = parse_args()
    world, rank, local = dist_init(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
    elif args.mode == "ffn":
        run_ffn(args, world, rank, local)
    elif args.mode == "sequence":
        run_sequence(args, world, rank, local)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
