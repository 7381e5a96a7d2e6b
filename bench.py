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


# names of this library's kernels (substrings of the CUDA kernel names)
OUR_KERNELS = ("indexer_prefill_tc_kernel", "indexer_prefill_kernel", "widen_e4m3_keys_kernel",
               "indexer_decode_tc_kernel", "decode_scores_kernel", "select_cluster_kernel",
               "decode_select_kernel", "sparse_attn_tc_kernel", "sparse_attn_kernel", "attn_combine_kernel",
               "decode_append_kernel", "overlap_kernel")


def observed_launches(fwd):
    """This library's kernels launched by one call of fwd, counted from the
    CUDA activity records of torch's profiler (None if it is unavailable).
    Runs outside every timed region."""
    try:
        from torch.profiler import ProfilerActivity, profile
        torch.cuda.synchronize()
        with profile(activities=[ProfilerActivity.CUDA]) as prof:
            fwd()
            torch.cuda.synchronize()
        return sum(1 for e in prof.events() if any(t in e.name for t in OUR_KERNELS))
    except Exception:   # no CUPTI activity records on this setup
        return None


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


def run_fp8q_indexer(binding, cfg, seed, dev, peaks, reps=5):
    """The fused indexer + top-k of one Full layer of this workload with e4m3
    queries and keys as stored (ic_indexer_topk_fp8, kind::f8f6f4 tensor
    cores), timed alone with CUDA events.  Its peak is the fp8 dense rate:
    the measured bf16 figure times the nominal fp8 / bf16 ratio of 2."""
    q8, qs, k8, ks, w = synth.make_fp8_indexer_inputs(cfg, 0, seed, dev)
    out = torch.empty((cfg.B, cfg.T, cfg.k), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()
    binding.indexer_topk_fp8(q8, qs, k8, ks, w, cfg.k, idx_out=out, stream=stream)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(reps):
        binding.indexer_topk_fp8(q8, qs, k8, ks, w, cfg.k, idx_out=out, stream=stream)
    b.record(stream)
    torch.cuda.synchronize()
    binding.stream_status()
    ms = a.elapsed_time(b) / reps
    fl = indexer_flops(cfg.T, cfg.q_pos0, cfg.H, cfg.D) * cfg.B
    peak = 2.0 * peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])
    ach = fl / (ms * 1e-3) / 1e12
    del q8, qs, k8, ks, w, out
    torch.cuda.empty_cache()
    return {"bound": "tensor", "launch_ms": ms, "achieved": ach, "peak": peak, "unit": "TFLOP/s", "frac": ach / peak,
            "flops_per_launch": fl, "peak_source": "2 x measured bf16 sustained (nominal fp8/bf16 dense ratio)",
            "inputs": "q_I and k_I e4m3 (amax/448 scale per query head / key row), w fp32"}


def adjacent_overlap(binding, layers, cfg):
    """Top-k overlap of adjacent layers in the all-F stack (deep-read page,
    "相邻层重叠很高…": Overlap(l, l-1) = |I_l ∩ I_(l-1)| / k, averaged over the
    query rows), through ic_indexer_topk and ic_overlap.  The synthetic layers
    are independent draws, so the expected overlap is that of unrelated
    top-k sets (about k / L per row on long rows), far below the pages' 0.7-1.0
    for a trained model; the figure checks the measurement path."""
    bufs = [torch.empty((cfg.B, cfg.T, cfg.k), dtype=torch.int32, device=layers[0]["Q"].device) for _ in range(2)]
    out = []
    for l, L in enumerate(layers):
        binding.indexer_topk(L["q"], L["kI"], L["w"], cfg.k, kscale=L.get("kscale"), idx_out=bufs[l & 1])
        if l:
            out.append(float(binding.overlap(bufs[l & 1], bufs[(l - 1) & 1]).mean().item()))
    binding.stream_status()
    return {"mean": statistics.mean(out), "min": min(out), "max": max(out), "per_pair": out}


def run_e2e(binding, layers, cfg, pattern, steps, warmup):
    """Same metric through the public per-layer API with HOST buffers.  Every
    step copies each layer's inputs from pinned host memory (q_I/k_I/w on F
    layers; Q/K/V on all layers), runs the layer (ic_indexer_topk on F layers,
    ic_sparse_attn on all), and reads every layer's O back.  Uploads run on
    one copy stream, downloads on another, the layers on the compute stream;
    events order them, so layer l+1's uploads overlap layer l's compute."""
    dev = layers[0]["Q"].device
    kinds = ["q", "kI", "w", "Q", "K", "V"]
    host = {}
    for kd in kinds:
        src = next(L[kd] for L in layers if L.get(kd) is not None)
        host[kd] = torch.empty(src.shape, dtype=src.dtype, pin_memory=True)
        host[kd].copy_(src.cpu())
    n = len(layers)
    o_host = [torch.empty(layers[0]["Q"].shape, dtype=torch.bfloat16, pin_memory=True) for _ in range(2)]
    comp = torch.cuda.current_stream()
    up = torch.cuda.Stream()
    down = torch.cuda.Stream()
    up_done = [torch.cuda.Event() for _ in range(n)]
    comp_done = [torch.cuda.Event() for _ in range(n)]
    for e in comp_done:
        e.record(comp)
    cache = torch.empty((cfg.B, cfg.T, cfg.k), dtype=torch.int32, device=dev)
    counts = {"h2d": 0, "d2h": 0}

    def step():
        counts["h2d"] = counts["d2h"] = 0
        for l, L in enumerate(layers):
            up.wait_event(comp_done[l])          # the previous step is done with this layer's buffers
            with torch.cuda.stream(up):
                for kd in kinds:
                    if L.get(kd) is not None and (kd not in ("q", "kI", "w") or pattern[l] == "F"):
                        L[kd].copy_(host[kd], non_blocking=True)
                        counts["h2d"] += L[kd].numel() * L[kd].element_size()
            up_done[l].record(up)
        for l, L in enumerate(layers):
            comp.wait_event(up_done[l])
            if pattern[l] == "F":
                binding.indexer_topk(L["q"], L["kI"], L["w"], cfg.k, kscale=L.get("kscale"), idx_out=cache,
                                     stream=comp)
            binding.sparse_attn(L["Q"], L["K"], L["V"], cache, O=L["O"], stream=comp)
            comp_done[l].record(comp)
            down.wait_event(comp_done[l])
            with torch.cuda.stream(down):
                o_host[l & 1].copy_(L["O"], non_blocking=True)
            counts["d2h"] += L["O"].numel() * L["O"].element_size()

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(comp)
    up.wait_event(t0)
    for _ in range(steps):
        step()
    comp.wait_stream(down)
    comp.wait_stream(up)
    t1.record(comp)
    torch.cuda.synchronize()
    binding.stream_status()
    ms = t0.elapsed_time(t1) / steps
    del host, o_host
    return {"value": cfg.B * cfg.T / (ms * 1e-3), "unit": "tok/s", "ms_per_step": ms,
            "h2d_bytes_per_step": counts["h2d"], "d2h_bytes_per_step": counts["d2h"], "steps": steps,
            "warmup": warmup, "api": "ic_indexer_topk / ic_sparse_attn per layer, host pinned buffers",
            "overlap": "uploads and downloads on their own streams, ordered by events"}


def graph_time_ms(fn, reps, stream):
    """Device time of one call of ``fn`` (launches on ``stream``): ``reps``
    calls captured in one CUDA graph, replayed, timed with CUDA events, so
    host launch gaps do not count."""
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(reps):
            fn()
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    with torch.cuda.stream(stream):
        g.replay()
    b.record(stream)
    torch.cuda.synchronize()
    del g
    return a.elapsed_time(b) / reps


def run_decode(binding, pattern, steps_tok, seed, dev, gpu_index):
    """The decode workload: 32 sequences with 131072 cached tokens, one new
    token per sequence per step.  Step i appends the new token's indexer key
    (Full layers) and K/V rows at position 131072 + i of every layer
    (ic_decode_append, one launch), then runs the stack for the query at
    that position over S = 131073 + i keys (ic_forward_pattern)."""
    cfg = synth.DECODE.with_(pattern=pattern)
    S_cap = cfg.q_pos0 + cfg.steps
    torch.cuda.synchronize()
    layers = synth.make_stack(cfg, seed, dev, T=1, S=S_cap, indexer_layers="pattern")
    for L in layers:
        L["O"] = torch.empty_like(L["Q"])
    # the new tokens' rows of every step, drawn before the timed region
    new_rows = []
    for i in range(steps_tok):
        rows = []
        for l, c in enumerate(pattern):
            R = {}
            if c == "F":
                _, kI1, ks1, _ = synth.make_indexer_inputs(cfg, l, seed + 7 + 1000003 * (i + 1), dev, T=1, S=1)
                R["kI"] = kI1[:, 0].contiguous()
                R["kscale"] = ks1[:, 0].contiguous() if ks1 is not None else None
            _, K1, V1 = synth.make_attn_inputs(cfg, l, seed + 7 + 1000003 * (i + 1), dev, T=1, S=1)
            R["K"], R["V"] = K1[:, 0].contiguous(), V1[:, 0].contiguous()
            rows.append(R)
        new_rows.append(rows)
    kd = binding.IC_E4M3 if cfg.k_dtype == "e4m3" else binding.IC_BF16
    appends = [binding.DecodeAppend(pattern, layers, new_rows[i], kd) for i in range(steps_tok)]
    ws_need = binding.workspace_size(binding.make_dims(cfg.B, 1, S_cap, cfg.H, cfg.D, cfg.k, cfg.Hq, cfg.Dh,
                                                       S_cap - 1, kd, S_cap))
    ws = torch.empty(max(ws_need, 1), dtype=torch.uint8, device=dev)
    cache = torch.empty((cfg.B, 1, cfg.k), dtype=torch.int32, device=dev)
    fwds = [binding.Forward(pattern, layers, cfg.k, cfg.q_pos0 + i, cfg.q_pos0 + i + 1, index_cache=cache, ws=ws)
            for i in range(steps_tok)]
    stream = torch.cuda.current_stream()

    def step(i, st):
        appends[i](cfg.q_pos0 + i, stream=st)
        fwds[i](st)

    for i in range(3):
        step(i, stream)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(gpu_index) as clk:
        t0.record(stream)
        for i in range(steps_tok):
            step(i, stream)
        t1.record(stream)
        torch.cuda.synchronize()
    binding.stream_status()
    ms = t0.elapsed_time(t1)
    clocks = clk.summary()
    # the same 64 steps replayed from CUDA graphs (one graph per step,
    # captured before the timed region): same kernels and work, without the
    # host launch gaps between the short kernels of a step
    graph = None
    try:
        cs = torch.cuda.Stream()
        graphs = []
        torch.cuda.synchronize()
        for i in range(steps_tok):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cs):
                step(i, cs)
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
    # per-call device times at the last context, each call alone, measured
    # from CUDA-graph replays of repeated calls (no host launch gaps)
    q_last = cfg.q_pos0 + steps_tok - 1
    L0 = layers[0]
    cs = torch.cuda.Stream()
    idx_layer_ms = graph_time_ms(lambda: binding.indexer_topk(L0["q"], L0["kI"], L0["w"], cfg.k, q_last,
                                                              kscale=L0["kscale"], S=q_last + 1, idx_out=cache,
                                                              ws=ws, stream=cs), 10, cs)
    attn_layer_ms = graph_time_ms(lambda: binding.sparse_attn(L0["Q"], L0["K"], L0["V"], cache, S=q_last + 1,
                                                              O=L0["O"], ws=ws, stream=cs), 20, cs)
    append_ms = graph_time_ms(lambda: appends[-1](q_last, stream=cs), 20, cs)
    binding.stream_status()
    del layers, fwds, ws, appends, new_rows
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
                          "bytes_per_launch": nbytes, "launch_ms": t_ms, "timing": "CUDA-graph replay of repeated calls"}
    step_bytes = pattern.count("F") * idx_bytes + len(pattern) * attn_bytes
    step_ms = (graph or {}).get("ms_per_token_step") or ms / steps_tok
    return {"value": cfg.B * steps_tok / (ms * 1e-3), "unit": "tok/s", "ms_per_token_step": ms / steps_tok,
            "steps": steps_tok, "batch": cfg.B, "context": cfg.q_pos0, "pattern": pattern,
            "appends": "timed: one ic_decode_append launch per step (new token's k_I/scale on F layers, K/V on all)",
            "indexer_ms_per_F_layer": idx_layer_ms, "attn_ms_per_layer": attn_layer_ms, "append_ms_per_step": append_ms,
            "step_hbm_bytes": step_bytes,
            "step_hbm_frac": step_bytes / (step_ms * 1e-3) / 1e9 / hbm,
            "kernels": roof, "clocks": clocks, "graph_replay": graph}


def run_long(binding, pattern, seed, dev, gpu_index, peaks, n_chunks=None):
    """The long-prefill workload: 47 layers, L = 204800 tokens prefilled in
    chunks of 8192 query rows, each chunk over its whole causal prefix
    (q_pos0 = 8192 c, S = 8192 (c + 1)), e4m3 indexer keys.  The key caches
    (k_I + scale on the Full layers, K/V on all) are resident for the whole
    run; each chunk's query-side inputs (q_I, w, Q) are drawn before its timed
    forward.  Time = the sum over chunks of the ic_forward_pattern times."""
    cfg = synth.LONG.with_(pattern=pattern)
    L, C = cfg.S, cfg.chunk
    n_chunks = L // C if n_chunks is None else n_chunks
    n = cfg.n_layers
    torch.cuda.synchronize()
    caches = []
    for l in range(n):
        d = {}
        if pattern[l] == "F":
            _, d["kI"], d["kscale"], _ = synth.make_indexer_inputs(cfg, l, seed, dev, T=1, S=L)
        _, d["K"], d["V"] = synth.make_attn_inputs(cfg, l, seed, dev, T=1, S=L)
        caches.append(d)
    O = [torch.empty((1, C, cfg.Hq, cfg.Dh), dtype=torch.bfloat16, device=dev) for _ in range(n)]
    cache = torch.empty((1, C, cfg.k), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()

    def chunk_layers(c):
        layers = []
        for l in range(n):
            d = dict(caches[l])
            if pattern[l] == "F":
                d["q"], _, _, d["w"] = synth.make_indexer_inputs(cfg, l, seed, dev, T=C, S=1, t0=c * C)
            d["Q"], _, _ = synth.make_attn_inputs(cfg, l, seed, dev, T=C, S=1, t0=c * C)
            d["O"] = O[l]
            layers.append(d)
        return layers

    # warm-up: the first and the last chunk once, untimed
    for c in (0, n_chunks - 1):
        f = binding.Forward(pattern, chunk_layers(c), cfg.k, c * C, (c + 1) * C, index_cache=cache)
        f(stream)
    torch.cuda.synchronize()
    total_ms = 0.0
    idx_ms = [0.0] * n
    attn_ms = [0.0] * n
    with ClockSampler(gpu_index) as clk:
        for c in range(n_chunks):
            layers = chunk_layers(c)
            f = binding.Forward(pattern, layers, cfg.k, c * C, (c + 1) * C, index_cache=cache)
            tr = binding.Trace(n, 1)
            torch.cuda.synchronize()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            f(stream, trace=tr)
            b.record(stream)
            torch.cuda.synchronize()
            total_ms += a.elapsed_time(b)
            _, im, am = tr.read()
            tr.close()
            idx_ms = [x + y for x, y in zip(idx_ms, im)]
            attn_ms = [x + y for x, y in zip(attn_ms, am)]
            del layers, f
    binding.stream_status()
    clocks = clk.summary()
    del caches, O, cache
    torch.cuda.empty_cache()
    Lp = n_chunks * C
    n_f = pattern.count("F")
    peak_tf = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])
    fl_i = 2.0 * cfg.H * cfg.D * (Lp * (Lp + 1) // 2)       # per F layer, all chunks
    fl_a = sum(attn_flops(C, c * C, cfg.Hq, cfg.Dh, cfg.k) for c in range(n_chunks))
    kern = {}
    if n_f:
        t = sum(idx_ms) / n_f
        kern["indexer_topk"] = {"bound": "tensor", "achieved": fl_i / (t * 1e-3) / 1e12, "peak": peak_tf,
                                "unit": "TFLOP/s", "frac": fl_i / (t * 1e-3) / 1e12 / peak_tf,
                                "ms_per_F_layer_all_chunks": t, "flops_per_F_layer": fl_i}
    t = sum(attn_ms) / n
    kern["sparse_attn"] = {"bound": "tensor", "achieved": fl_a / (t * 1e-3) / 1e12, "peak": peak_tf,
                           "unit": "TFLOP/s", "frac": fl_a / (t * 1e-3) / 1e12 / peak_tf,
                           "ms_per_layer_all_chunks": t, "flops_per_layer": fl_a,
                           "gathered_TB_per_s": fl_a / (4 * cfg.Hq * cfg.Dh) * 512 / (t * 1e-3) / 1e12}
    return {"pattern": pattern, "tokens": Lp, "chunks": n_chunks, "chunk": C, "k_dtype": cfg.k_dtype,
            "ms": total_ms, "value": Lp / (total_ms * 1e-3), "unit": "tok/s", "kernels": kern, "clocks": clocks}


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
    launches_seen = observed_launches(fwd)

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
        if not args.no_overlap:
            allf_res["overlap_adjacent"] = adjacent_overlap(binding, layers, cfg)

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

    fp8q = None
    if not args.no_e4m3:
        fp8q = run_fp8q_indexer(binding, cfg, seed + 4, dev, peaks)

    decode = None
    if not args.no_decode:
        dq = run_decode(binding, synth.DECODE.pattern, args.decode_steps, seed + 1, dev, gpu_index)
        df = run_decode(binding, "F" * 47, args.decode_steps, seed + 2, dev, gpu_index) if not args.no_allf else None
        decode = {"quarter_f": dq, "all_f": df}
        if df:
            decode["speedup_quarter_vs_allf"] = dq["value"] / df["value"]

    long_res = None
    if not args.no_long:
        lq = run_long(binding, synth.LONG.pattern, seed + 5, dev, gpu_index, peaks)
        lf = run_long(binding, "F" * 47, seed + 6, dev, gpu_index, peaks) if not args.no_allf else None
        long_res = {"workload": "long: 47 layers, L=204800 prefilled in 25 chunks of 8192 query rows over the "
                                "causal prefix, e4m3 indexer keys, H_I=64, d_I=128, k=2048; 32 q heads / 1 KV head, "
                                "dim 128", "quarter_f": lq, "all_f": lf}
        if lf:
            long_res["speedup_quarter_vs_allf"] = lq["value"] / lf["value"]

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
            "gpu_launches": args.steps * (launches_seen if launches_seen is not None
                                          else launches_per_forward(quarter, cfg.B, cfg.T, cfg.k)),
            "gpu_launches_source": ("this library's kernels in the CUDA activity of one forward (torch profiler), "
                                    "times the timed steps") if launches_seen is not None
                                   else "computed from the library's dispatch",
            "clocks": clocks, "all_f": allf_res, "e4m3_keys": e4,
            "speedup_quarter_vs_allf": (value / allf_res["value"]) if allf_res else None,
            "fp8_indexer": fp8q, "decode": decode, "long": long_res, "peaks": {k: v for k, v in peaks.items() if not k.startswith("_") and
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
    ap.add_argument("--no-long", action="store_true")
    ap.add_argument("--no-overlap", action="store_true")
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
