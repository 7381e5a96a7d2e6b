"""Seeded synthetic inputs shaped like the IndexCache workloads.

This module only draws random tensors and stores them in the layouts the
library expects; it holds none of the method's arithmetic (no scores, no
selection, no attention).  The same generators feed the CUDA path and, after a
copy to host memory, the CPU oracle.

Layouts (row-major, innermost axis last):
  q   [B, T, H, D]   bf16   indexer queries, query row t at position q_pos0 + t
  kI  [B, S, D]      bf16, or e4m3 bytes with kscale [B, S] fp32 (> 0)
  w   [B, T, H]      fp32   indexer head weights
  Q   [B, T, Hq, Dh] bf16   core-attention queries
  K,V [B, S, Dh]     bf16   the single K/V head
  O   [B, T, Hq, Dh] bf16   core-attention output

Seeds: the tensor with id ``tid`` of layer ``l`` is drawn from a generator
seeded with ``base + 1000 * l + tid``.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch

TID_Q, TID_KI, TID_W, TID_QA, TID_K, TID_V = 1, 2, 3, 4, 5, 6

E4M3_MAX = 448.0


def quarter_f_pattern(n_layers: int) -> str:
    """Full layer at 0, 4, 8, ... and Shared elsewhere (one Full layer in four)."""
    return "".join("F" if i % 4 == 0 else "S" for i in range(n_layers))


@dataclass(frozen=True)
class StackConfig:
    """One workload: a stack of layers over one batch of sequences."""

    name: str
    n_layers: int
    pattern: str
    B: int
    T: int             # query rows per sequence in one call
    S: int             # causal key rows visible to the last query (>= q_pos0 + T)
    H: int             # indexer heads
    D: int             # indexer feature dim
    k: int             # top-k
    Hq: int            # core-attention query heads (one shared K/V head)
    Dh: int            # core-attention head dim
    k_dtype: str = "bf16"   # "bf16" or "e4m3"
    dist: str = "normal"    # "int" (values in {-2..2}) or "normal"
    q_pos0: int = 0
    chunk: int = 0          # >0: prefill is issued in chunks of this many query rows
    steps: int = 0          # >0: decode steps (T = 1 per step)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.Dh)

    def with_(self, **kw) -> "StackConfig":
        return replace(self, **kw)


# The five workloads (tiny, short, 30B-shaped, decode, long).
TINY = StackConfig("tiny", 4, "FSSF", 1, 256, 256, 4, 32, 16, 4, 64, "bf16", "int")
SHORT = StackConfig("short", 8, "FSSSFSSS", 1, 8192, 8192, 64, 128, 2048, 32, 128)
PREFILL_32K = StackConfig("prefill32k", 47, quarter_f_pattern(47), 1, 32768, 32768, 64, 128, 2048, 32, 128)
DECODE = StackConfig("decode", 47, quarter_f_pattern(47), 32, 1, 131073, 64, 128, 2048, 32, 128,
                     "e4m3", "normal", q_pos0=131072, steps=64)
LONG = StackConfig("long", 47, quarter_f_pattern(47), 1, 204800, 204800, 64, 128, 2048, 32, 128,
                   "e4m3", "normal", chunk=8192)

CONFIGS = {c.name: c for c in (TINY, SHORT, PREFILL_32K, DECODE, LONG)}


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _draw(shape, dist: str, std: float, seed: int, device) -> torch.Tensor:
    g = _gen(device, seed)
    if dist == "int":
        return torch.randint(-2, 3, shape, generator=g, device=device, dtype=torch.int32).to(torch.float32)
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std


def quantize_e4m3(k: torch.Tensor):
    """Per-row e4m3 storage of key features: scale = amax / 448 (1 if the row is 0).

    Returns (e4m3 bytes as torch.float8_e4m3fn, fp32 scale per row).  Only the
    stored bytes and scales matter downstream; both sides read them as given.
    """
    amax = k.abs().amax(dim=-1)
    scale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax)).to(torch.float32)
    q8 = (k / scale.unsqueeze(-1)).clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)
    return q8, scale


def make_indexer_inputs(cfg: StackConfig, layer: int, base_seed: int, device, T: int | None = None,
                        S: int | None = None, t0: int = 0):
    """q [B,T,H,D] bf16, kI [B,S,D] (bf16 or e4m3), kscale [B,S] fp32 or None, w [B,T,H] fp32.

    ``t0`` offsets the query rows drawn (rows t0 .. t0+T-1 of the full draw are
    reproduced exactly only when T and t0 cover whole seeds; chunked users draw
    per chunk with their own seed offset instead).
    """
    T = cfg.T if T is None else T
    S = cfg.S if S is None else S
    s0 = base_seed + 1000 * layer
    std_q = 1.0 / math.sqrt(cfg.D)
    std_w = 1.0 / math.sqrt(cfg.H)
    q = _draw((cfg.B, T, cfg.H, cfg.D), cfg.dist, std_q, s0 + TID_Q + 100 * t0, device).to(torch.bfloat16)
    w = _draw((cfg.B, T, cfg.H), cfg.dist, std_w, s0 + TID_W + 100 * t0, device)
    kf = _draw((cfg.B, S, cfg.D), cfg.dist, std_q, s0 + TID_KI, device)
    if cfg.k_dtype == "e4m3":
        kI, kscale = quantize_e4m3(kf)
    else:
        kI, kscale = kf.to(torch.bfloat16), None
    return q, kI, kscale, w


def make_fp8_indexer_inputs(cfg: StackConfig, layer: int, base_seed: int, device, T: int | None = None,
                            S: int | None = None, t0: int = 0, codes: bool = False):
    """Indexer inputs with e4m3 queries AND keys: q8 [B,T,H,D] e4m3, q_scale
    [B,T,H] fp32, k8 [B,S,D] e4m3, k_scale [B,S] fp32, w [B,T,H] fp32.

    Default: the same draws as ``make_indexer_inputs``, each query head and
    key row stored as e4m3 with scale amax/448.  ``codes``: q and k are the
    integers {-2..2} (exact e4m3 codes) with power-of-two scales in
    [2^-3, 2^3], so every score is exact in fp32."""
    T = cfg.T if T is None else T
    S = cfg.S if S is None else S
    s0 = base_seed + 1000 * layer
    std_q = 1.0 / math.sqrt(cfg.D)
    std_w = 1.0 / math.sqrt(cfg.H)
    if codes:
        q = _draw((cfg.B, T, cfg.H, cfg.D), "int", 1.0, s0 + TID_Q + 100 * t0, device)
        kf = _draw((cfg.B, S, cfg.D), "int", 1.0, s0 + TID_KI, device)
        w = _draw((cfg.B, T, cfg.H), "int", 1.0, s0 + TID_W + 100 * t0, device)
        gq = _gen(device, s0 + 77 + 100 * t0)
        gk = _gen(device, s0 + 78)
        q_scale = torch.pow(2.0, torch.randint(-3, 4, (cfg.B, T, cfg.H), generator=gq, device=device).float())
        k_scale = torch.pow(2.0, torch.randint(-3, 4, (cfg.B, S), generator=gk, device=device).float())
        return q.to(torch.float8_e4m3fn), q_scale, kf.to(torch.float8_e4m3fn), k_scale, w
    q = _draw((cfg.B, T, cfg.H, cfg.D), cfg.dist, std_q, s0 + TID_Q + 100 * t0, device)
    w = _draw((cfg.B, T, cfg.H), cfg.dist, std_w, s0 + TID_W + 100 * t0, device)
    kf = _draw((cfg.B, S, cfg.D), cfg.dist, std_q, s0 + TID_KI, device)
    q8, q_scale = quantize_e4m3(q)
    k8, k_scale = quantize_e4m3(kf)
    return q8, q_scale, k8, k_scale, w


def make_attn_inputs(cfg: StackConfig, layer: int, base_seed: int, device, T: int | None = None,
                     S: int | None = None, t0: int = 0):
    """Q [B,T,Hq,Dh], K [B,S,Dh], V [B,S,Dh], all bf16."""
    T = cfg.T if T is None else T
    S = cfg.S if S is None else S
    s0 = base_seed + 1000 * layer
    Q = _draw((cfg.B, T, cfg.Hq, cfg.Dh), cfg.dist, 1.0, s0 + TID_QA + 100 * t0, device).to(torch.bfloat16)
    K = _draw((cfg.B, S, cfg.Dh), cfg.dist, 1.0, s0 + TID_K, device).to(torch.bfloat16)
    V = _draw((cfg.B, S, cfg.Dh), cfg.dist, 1.0, s0 + TID_V, device).to(torch.bfloat16)
    return Q, K, V


def make_stack(cfg: StackConfig, base_seed: int, device, T: int | None = None, S: int | None = None,
               indexer_layers: str = "pattern"):
    """All layers of a stack.  Shared layers get no indexer inputs unless
    ``indexer_layers == "all"`` (needed to run the same stack all-Full)."""
    layers = []
    for layer in range(cfg.n_layers):
        need = indexer_layers == "all" or cfg.pattern[layer] == "F"
        d = {}
        if need:
            d["q"], d["kI"], d["kscale"], d["w"] = make_indexer_inputs(cfg, layer, base_seed, device, T, S)
        else:
            d["q"] = d["kI"] = d["kscale"] = d["w"] = None
        d["Q"], d["K"], d["V"] = make_attn_inputs(cfg, layer, base_seed, device, T, S)
        layers.append(d)
    return layers


# ---------------------------------------------------------------------------
# Host copies for the CPU side (raw bit patterns, no arithmetic).
# ---------------------------------------------------------------------------


def bf16_bits(t: torch.Tensor):
    """Raw uint16 bit patterns of a bf16 tensor as a NumPy array."""
    import numpy as np
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def e4m3_bits(t: torch.Tensor):
    """Raw uint8 bit patterns of an e4m3 tensor as a NumPy array."""
    import numpy as np
    return t.detach().contiguous().cpu().view(torch.uint8).numpy().astype(np.uint8)


def f32_values(t: torch.Tensor):
    return t.detach().contiguous().cpu().numpy()
