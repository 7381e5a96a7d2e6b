#!/usr/bin/env python3
"""Benchmark of the IndexCache hot path on one B300 (or N replicas under torchrun).

Headline workload (one step = one pass of the whole hot path):
  47 layers, Full layers at 0, 4, ..., 44 (12 F / 35 S), batch 1, L = 32768
  causal, indexer H_I = 64, d_I = 128 (bf16 keys), k = 2048; core attention
  32 query heads sharing one K/V head of dim 128, bf16.  Each step is one
  ic_forward_pattern call: the fused indexer + top-k on the 12 F layers and
  sparse attention on all 47.  Inputs are seeded synthetic tensors resident
  in HBM; every layer's q_I (512 MiB) and Q (256 MiB) exceed the 126 MB L2.

Also reported: the same stack all-Full (standard DSA), the same 1/4-F stack
with e4m3 indexer keys, the end-to-end figure through host buffers, the
decode workload (32 sequences at context 131072, 64 steps, fp8 keys) with
its kernels against HBM bandwidth, per-kernel roofline fractions from live
CUDA events, and the CPU oracle timed on a bounded sample (a reported
baseline, not a target).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from cross_layer_top_indexer_b300 import synth  # noqa: E402

METRIC = "prefill tok/s (47-layer 1/4-F stack, L=32K); decode tok/s; % of roofline"
PEAKS_FALLBACK = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


# ---------------------------------------------------------------------------
# small helpers
# ---------------------------------------------------------------------------


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        d["_source"] = "measured"
        return d
    d = dict(PEAKS_FALLBACK)
    d["_source"] = "fallback"
    return d


class ClockSampler:
    """nvidia-smi samples (200 ms) while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        power = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "power_w_max": max(power) if power else None}


def indexer_flops(T, q_pos0, H, D):
    # 2*H*D flops per causal (query, key) pair
    pairs = sum_causal(T, q_pos0)
    return 2.0 * H * D * pairs


def sum_causal(T, q_pos0):
    # sum over rows of (q_pos0 + t + 1)
    return T * (q_pos0 + 1) + T * (T - 1) // 2


def attn_flops(T, q_pos0, Hq, Dh, k):
    # 4*Hq*Dh flops per (query, selected row): QK^T and PV
    n = 0
    for_t_small = max(0, min(T, k - q_pos0))      # rows with fewer than k causal keys
    n += sum(q_pos0 + t + 1 for t in range(for_t_small))
    n += (T - for_t_small) * k
    return 4.0 * Hq * Dh * n


def launches_per_forward(pattern, B, T, k):
    # the library's dispatch: decode indexer (<= 8 rows) = 2 kernels, prefill = 1;
    # attention splits over the k rows (2 kernels) when fewer than 296 rows
    n_f = pattern.count("F")
    idx = 2 if T <= 8 else 1
    rows = B * T
    attn = 1
    if rows < 296:
        n_chunks = (k + 63) // 64
        want = (4 * 148 + rows - 1) // rows
        attn = 2 if min(want, n_chunks) > 1 else 1
    return n_f * idx + len(pattern) * attn


# ---------------------------------------------------------------------------
# timed runs
# ---------------------------------------------------------------------------


def make_prefill_layers(cfg, seed, dev, indexer_layers):
    torch.cuda.synchronize()
    layers = synth.make_stack(cfg, seed, dev, indexer_layers=indexer_layers)
    for L in layers:
        L["O"] = torch.empty_like(L["Q"])
    torch.cuda.synchronize()
    return layers


def time_forward(binding, fwd, steps, warmup, n_layers, gpu_index, trace=True):
    """W untimed + K timed forwards on the current stream, CUDA events around
    the K; per-layer kernel times from the library's trace events."""
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        fwd(stream)
    torch.cuda.synchronize()
    tr = binding.Trace(n_layers, steps) if trace else None
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    with ClockSampler(gpu_index) as clk:
        torch.cuda.synchronize()
        start.record(stream)
        for _ in range(steps):
            fwd(stream, trace=tr)
        stop.record(stream)
        torch.cuda.synchronize()
    binding.stream_status()
    total_ms = start.elapsed_time(stop)
    per = None
    if tr is not None:
        n, idx_ms, attn_ms = tr.read()
        tr.close()
        per = {"n": n, "indexer_ms": idx_ms, "attn_ms": attn_ms}
    return total_ms, per, clk.summary()


def kernel_roofline(per, pattern, cfg, peaks, steps):
    """Per-kernel achieved rate from the traced events (averaged over launches)."""
    n_f = pattern.count("F")
    idx_launch_ms = sum(per["indexer_ms"]) / max(1, steps * n_f)
    attn_launch_ms = sum(per["attn_ms"]) / max(1, steps * len(pattern))
    peak_tf = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])
    fl_i = indexer_flops(cfg.T, cfg.q_pos0, cfg.H, cfg.D) * cfg.B
    fl_a = attn_flops(cfg.T, cfg.q_pos0, cfg.Hq, cfg.Dh, cfg.k) * cfg.B
    out = {}
    if n_f:
        ach = fl_i / (idx_launch_ms * 1e-3) / 1e12
        out["indexer_topk"] = {"bound": "tensor", "achieved": ach, "peak": peak_tf, "unit": "TFLOP/s",
                               "frac": ach / peak_tf, "launch_ms": idx_launch_ms, "flops_per_launch": fl_i,
                               "total_ms_per_step": idx_launch_ms * n_f}
    ach = fl_a / (attn_launch_ms * 1e-3) / 1e12
    out["sparse_attn"] = {"bound": "tensor", "achieved": ach, "peak": peak_tf, "unit": "TFLOP/s",
                          "frac": ach / peak_tf, "launch_ms": attn_launch_ms, "flops_per_launch": fl_a,
                          "total_ms_per_step": attn_launch_ms * len(pattern)}
    return out


def run_e2e(binding, layers, cfg, pattern, steps, warmup):
    """Same metric through the public API with HOST buffers: every step copies
    each layer's inputs host->device (pinned), runs the forward, and reads
    every layer's output back to host."""
    dev = layers[0]["Q"].device
    kinds = ["q", "kI", "w", "Q", "K", "V"]
    host = {}
    for kd in kinds:
        src = next(L[kd] for L in layers if L.get(kd) is not None)
        host[kd] = torch.empty(src.shape, dtype=src.dtype, pin_memory=True)
        host[kd].copy_(src.cpu())
    o_host = torch.empty(layers[0]["Q"].shape, dtype=torch.bfloat16, pin_memory=True)
    fwd = binding.Forward(pattern, layers, cfg.k, cfg.q_pos0, cfg.S)
    stream = torch.cuda.current_stream()
    h2d = d2h = 0

    def step():
        nonlocal h2d, d2h
        h2d = d2h = 0
        for l, L in enumerate(layers):
            for kd in kinds:
                if L.get(kd) is not None and (kd not in ("q", "kI", "w") or pattern[l] == "F"):
                    L[kd].copy_(host[kd], non_blocking=True)
                    h2d += L[kd].numel() * L[kd].element_size()
        fwd(stream)
        for L in layers:
            o_host.copy_(L["O"], non_blocking=True)
            d2h += L["O"].numel() * L["O"].element_size()

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    binding.stream_status()
    ms = t0.elapsed_time(t1) / steps
    del host, o_host
    return {"value": cfg.B * cfg.T / (ms * 1e-3), "unit": "tok/s", "ms_per_step": ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps, "warmup": warmup}


def run_decode(binding, pattern, steps_tok, seed, dev, gpu_index):
    """The decode workload: 32 sequences with 131072 cached tokens, one new
    query per sequence per step; step i sees S = 131073 + i keys."""
    cfg = synth.DECODE.with_(pattern=pattern)
    S_cap = cfg.q_pos0 + cfg.steps
    torch.cuda.synchronize()
    layers = synth.make_stack(cfg, seed, dev, T=1, S=S_cap, indexer_layers="pattern")
    for L in layers:
        L["O"] = torch.empty_like(L["Q"])
    ws_need = binding.workspace_size(binding.make_dims(cfg.B, 1, S_cap, cfg.H, cfg.D, cfg.k, cfg.Hq, cfg.Dh,
                                                       S_cap - 1, binding.IC_E4M3, S_cap))
    ws = torch.empty(max(ws_need, 1), dtype=torch.uint8, device=dev)
    cache = torch.empty((cfg.B, 1, cfg.k), dtype=torch.int32, device=dev)
    fwds = [binding.Forward(pattern, layers, cfg.k, cfg.q_pos0 + i, cfg.q_pos0 + i + 1, index_cache=cache, ws=ws)
            for i in range(steps_tok)]
    stream = torch.cuda.current_stream()
    for f in fwds[:3]:
        f(stream)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(gpu_index) as clk:
        t0.record(stream)
        for f in fwds:
            f(stream)
        t1.record(stream)
        torch.cuda.synchronize()
    binding.stream_status()
    ms = t0.elapsed_time(t1)
    clocks = clk.summary()
    # the same 64 steps replayed from CUDA graphs (one graph per step, captured
    # before the timed region): the kernels and the work are the same, the
    # host launch gaps between ~140 short kernels per step are gone
    graph = None
    try:
        cs = torch.cuda.Stream()
        graphs = []
        torch.cuda.synchronize()
        for f in fwds:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cs):
                f(cs)
            graphs.append(g)
        torch.cuda.synchronize()
        for g in graphs[:3]:
            g.replay()
        torch.cuda.synchronize()
        g0 = torch.cuda.Event(enable_timing=True)
        g1 = torch.cuda.Event(enable_timing=True)
        with ClockSampler(gpu_index) as clk_g:
            g0.record()
            for g in graphs:
                g.replay()
            g1.record()
            torch.cuda.synchronize()
        binding.stream_status()
        ms_g = g0.elapsed_time(g1)
        graph = {"value": cfg.B * steps_tok / (ms_g * 1e-3), "unit": "tok/s", "ms_per_token_step": ms_g / steps_tok,
                 "clocks": clk_g.summary()}
        del graphs
    except Exception as ex:  # capture refused: report it, the stream-launched figure stands
        graph = {"unavailable": ("%s: %s" % (type(ex).__name__, ex))[:240]}
    # per-call breakdown at the last context length: each call alone, repeated,
    # CUDA events on the stream (a traced step would also count launch gaps)
    q_last = cfg.q_pos0 + steps_tok - 1
    L0 = layers[0]

    def call_ms(fn, reps):
        fn()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    idx_layer_ms = call_ms(lambda: binding.indexer_topk(L0["q"], L0["kI"], L0["w"], cfg.k, q_last,
                                                        kscale=L0["kscale"], S=q_last + 1, idx_out=cache, ws=ws,
                                                        stream=stream), 10)
    # one attention call (~25 us of device time) is shorter than its launch from
    # Python, so its share is derived from the step: the step time less the
    # indexer calls, over the layers
    attn_layer_ms = max(0.0, ms / steps_tok - pattern.count("F") * idx_layer_ms) / len(pattern)
    binding.stream_status()
    del layers, fwds, ws
    torch.cuda.empty_cache()
    # algorithmic HBM bytes of one layer at the traced context S = S_cap:
    # indexer: every cached key once (d_I e4m3 bytes + its fp32 scale) plus q, w
    # and the index row; attention: the k selected K and V rows (bf16) plus Q, O
    S = S_cap
    idx_bytes = cfg.B * (S * (cfg.D + 4) + cfg.H * cfg.D * 2 + cfg.H * 4 + cfg.k * 4)
    attn_bytes = cfg.B * (cfg.k * 2 * cfg.Dh * 2 + 2 * cfg.Hq * cfg.Dh * 2 + cfg.k * 4)
    hbm = load_peaks()["hbm_gbs"]
    roof = {}
    for name, nbytes, t_ms in (("indexer_topk", idx_bytes, idx_layer_ms), ("sparse_attn", attn_bytes, attn_layer_ms)):
        if t_ms > 0:
            ach = nbytes / (t_ms * 1e-3) / 1e9
            roof[name] = {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
                          "bytes_per_launch": nbytes, "launch_ms": t_ms}
    return {"value": cfg.B * steps_tok / (ms * 1e-3), "unit": "tok/s", "ms_per_token_step": ms / steps_tok,
            "steps": steps_tok, "batch": cfg.B, "context": cfg.q_pos0, "pattern": pattern,
            "indexer_ms_per_F_layer": idx_layer_ms, "attn_ms_per_layer": attn_layer_ms,
            "kernels": roof, "clocks": clocks, "graph_replay": graph}


# ---------------------------------------------------------------------------
# CPU oracle baseline (bounded sample)
# ---------------------------------------------------------------------------


def cpu_baseline(cfg, layers_f, layers_any, budget_s=15.0, seed=0):
    """Time the fp64 oracle on sampled query rows of one F layer (indexer +
    top-k) and of one layer's attention; extrapolate to whole-stack tok/s."""
    import numpy as np

    import oracle
    try:
        from threadpoolctl import threadpool_info
        threads = max([p.get("num_threads", 1) for p in threadpool_info()] or [1])
    except Exception:
        threads = os.cpu_count()
    rng = np.random.default_rng(seed)
    L = layers_f
    kI = oracle.bf16_to_f64(synth.bf16_bits(L["kI"][0]))
    K = oracle.bf16_to_f64(synth.bf16_bits(layers_any["K"][0]))
    V = oracle.bf16_to_f64(synth.bf16_bits(layers_any["V"][0]))
    t_idx = []
    t_att = []
    t_begin = time.perf_counter()
    rows_done = []
    while time.perf_counter() - t_begin < budget_s:
        t = int(rng.integers(0, cfg.T))
        q = oracle.bf16_to_f64(synth.bf16_bits(L["q"][0, t:t + 1]))
        w = L["w"][0, t:t + 1].double().cpu().numpy()
        Q = oracle.bf16_to_f64(synth.bf16_bits(layers_any["Q"][0, t:t + 1]))
        a = time.perf_counter()
        idx = oracle.indexer_topk(q, kI[: cfg.q_pos0 + t + 1], w, cfg.k, q_pos0=cfg.q_pos0 + t)
        b = time.perf_counter()
        oracle.sparse_attention(Q, K, V, idx, cfg.scale)
        c = time.perf_counter()
        t_idx.append(b - a)
        t_att.append(c - b)
        rows_done.append(t)
    n_f = cfg.pattern.count("F")
    per_token = n_f * statistics.mean(t_idx) + cfg.n_layers * statistics.mean(t_att)
    return {"value": 1.0 / per_token, "unit": "tok/s", "cores": threads, "kind": "oracle",
            "sample": "%d query rows drawn uniformly from the %d of one F layer (indexer+top-k) and one layer's "
                      "attention, fp64 NumPy, extrapolated to %d F + %d attention layers per token"
                      % (len(rows_done), cfg.T, n_f, cfg.n_layers),
            "seconds": time.perf_counter() - t_begin, "host_cpus": os.cpu_count()}


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def reduce_max(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def reference_arm(args, world, rank):
    """The oracle as it stands, on host cores, on this workload (bounded
    sample per step): the slow program the driver divides by."""
    if rank != 0:
        return
    cfg = synth.PREFILL_32K
    dev = "cpu"
    L = {}
    L["q"], L["kI"], _, L["w"] = synth.make_indexer_inputs(cfg, 0, 1234, dev)
    L["Q"], L["K"], L["V"] = synth.make_attn_inputs(cfg, 0, 1234, dev)
    per_step_budget = max(1.0, min(20.0, 150.0 / max(1, args.steps + args.warmup)))
    vals = []
    for i in range(args.warmup + args.steps):
        r = cpu_baseline(cfg, L, L, budget_s=per_step_budget, seed=i)
        if i >= args.warmup:
            vals.append(r)
    value = statistics.mean(v["value"] for v in vals)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": cfg.T / value * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": "prefill32k: 47 layers, F at 0,4,..,44, B=1, L=32768, H_I=64, d_I=128, "
                                   "k=2048, 32 q heads / 1 KV head, dim 128, bf16 inputs",
                       "impl": "fp64 NumPy oracle on host cores (bounded sample per step)"},
            "cpu_baseline": {"value": value, "unit": "tok/s", "kind": "oracle", "cores": vals[0]["cores"],
                             "sample": vals[0]["sample"] + " (per step)"},
            "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def ours_arm(args, world, rank, local):
    from cross_layer_top_indexer_b300 import binding
    binding.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    gpu_index = int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[local]) \
        if os.environ.get("CUDA_VISIBLE_DEVICES") else local
    peaks = load_peaks()
    cfg = synth.CONFIGS[args.config]
    seed = 1000 + 7919 * rank
    quarter = cfg.pattern
    allf = "F" * cfg.n_layers

    # ---- headline: 1/4-F prefill, inputs resident ----
    layers = make_prefill_layers(cfg, seed, dev, "all" if not args.no_allf else "pattern")
    fwd = binding.Forward(quarter, layers, cfg.k)
    barrier(world)
    total_ms, per, clocks = time_forward(binding, fwd, args.steps, args.warmup, cfg.n_layers, gpu_index)
    total_ms = reduce_max(total_ms, world)
    ms_step = total_ms / args.steps
    value = world * cfg.B * cfg.T / (ms_step * 1e-3)
    kern = kernel_roofline(per, quarter, cfg, peaks, args.steps)

    allf_res = None
    if not args.no_allf:
        fwd_f = binding.Forward(allf, layers, cfg.k)
        barrier(world)
        t_f, per_f, clk_f = time_forward(binding, fwd_f, max(2, args.steps // 2), max(1, args.warmup // 2),
                                         cfg.n_layers, gpu_index)
        t_f = reduce_max(t_f, world)
        k_f = max(2, args.steps // 2)
        ms_f = t_f / k_f
        allf_res = {"pattern": "all-F (47 F)", "ms_per_step": ms_f,
                    "value": world * cfg.B * cfg.T / (ms_f * 1e-3), "unit": "tok/s", "steps": k_f,
                    "kernels": kernel_roofline(per_f, allf, cfg, peaks, k_f), "clocks": clk_f}

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(binding, layers, cfg, quarter, max(1, min(args.steps, 3)), 1)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_baseline(cfg, next(L for L, c in zip(layers, quarter) if c == "F"), layers[0],
                           budget_s=args.cpu_seconds)
    del layers, fwd
    torch.cuda.empty_cache()

    # ---- the same 1/4-F stack with e4m3 indexer keys (per-key fp32 scale) ----
    e4 = None
    if not args.no_e4m3:
        cfg8 = cfg.with_(k_dtype="e4m3")
        layers8 = make_prefill_layers(cfg8, seed + 3, dev, "pattern")
        fwd8 = binding.Forward(quarter, layers8, cfg.k)
        barrier(world)
        k8 = max(2, args.steps // 2)
        t8, per8, clk8 = time_forward(binding, fwd8, k8, max(1, args.warmup // 2), cfg.n_layers, gpu_index)
        t8 = reduce_max(t8, world)
        ms8 = t8 / k8
        e4 = {"pattern": quarter, "k_dtype": "e4m3", "ms_per_step": ms8,
              "value": world * cfg.B * cfg.T / (ms8 * 1e-3), "unit": "tok/s", "steps": k8,
              "kernels": kernel_roofline(per8, quarter, cfg, peaks, k8), "clocks": clk8}
        del layers8, fwd8
        torch.cuda.empty_cache()

    decode = None
    if not args.no_decode:
        dq = run_decode(binding, synth.DECODE.pattern, args.decode_steps, seed + 1, dev, gpu_index)
        df = run_decode(binding, "F" * 47, args.decode_steps, seed + 2, dev, gpu_index) if not args.no_allf else None
        decode = {"quarter_f": dq, "all_f": df}
        if df:
            decode["speedup_quarter_vs_allf"] = dq["value"] / df["value"]

    dom_name = max(kern, key=lambda n: kern[n]["total_ms_per_step"])
    dom = kern[dom_name]
    traffic = None
    prof = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(prof):
        try:
            with open(prof) as f:
                traffic = json.load(f).get(dom_name)
        except Exception:
            traffic = None
    roofline = {"kernel": dom_name, "bound": dom["bound"], "achieved": dom["achieved"], "peak": dom["peak"],
                "unit": dom["unit"], "frac": dom["frac"], "traffic": traffic,
                "peak_source": "%s (bf16_tflops_sustained: kernel timed inside a long step)" % peaks["_source"]}
    if rank != 0:
        return
    line = {"metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": ("prefill32k: 47 layers, F at 0,4,..,44 (12 F / 35 S), B=1, L=32768 causal, "
                                    "H_I=64, d_I=128, bf16 keys, k=2048; 32 q heads / 1 KV head, dim 128, bf16")
                       if args.config == "prefill32k" else
                       ("short: 8 layers FSSSFSSS, B=1, L=8192, H_I=64, d_I=128, bf16 keys, k=2048; "
                        "32 q heads / 1 KV head, dim 128"),
                       "pattern": quarter, "seq_len": cfg.T, "global_batch": cfg.B * world,
                       "parallelism": "replicas" if world > 1 else "single GPU",
                       "l2": "inputs larger than L2 (per layer q_I 512 MiB, Q 256 MiB; 126 MB L2), no flush"},
            "roofline": roofline, "kernels": kern, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": args.steps * launches_per_forward(quarter, cfg.B, cfg.T, cfg.k),
            "clocks": clocks, "all_f": allf_res, "e4m3_keys": e4,
            "speedup_quarter_vs_allf": (value / allf_res["value"]) if allf_res else None,
            "decode": decode, "peaks": {k: v for k, v in peaks.items() if not k.startswith("_") and
                                        isinstance(v, (int, float))}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-allf", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-e4m3", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--decode-steps", type=int, default=64)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--config", default="prefill32k", choices=["prefill32k", "short"],
                    help="prefill32k: the headline 47-layer stack; short: the 8-layer L=8192 stack (profiling)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        print("note: fewer than 3 warm-up steps", file=sys.stderr)
    world, rank, local = dist_setup()
    if args.impl == "reference":
        reference_arm(args, world, rank)
    else:
        ours_arm(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
