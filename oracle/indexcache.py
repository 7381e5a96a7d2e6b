"""Plain float64 CPU oracle of the IndexCache hot path.

TEST INFRASTRUCTURE ONLY: used by the tests, by the smoke check and by the
CPU-baseline leg of the benchmark, never by the product path.  It is slow on
purpose and follows the definitions step by step; a NumPy matmul, sort or
exponential is the only library help it takes.

Sources (web pages on "IndexCache: Accelerating Sparse Attention via
Cross-Layer Index Reuse", arXiv 2603.12201):

* notes page (joezjh.github.io, "NLP--IndexCache"), section "背景 & 问题提出"
  (background): a lightning indexer scores, for every query, all previous
  tokens; core attention then runs only on the top-k (k = 2048) of them.
* same notes page, section "IndexCache 方法" (method): roles c_l in {F, S};
  a Shared layer reuses the indices of f(l) = max{j < l : c_j = F}.
* deep-read page (wineandchord.com, "IndexCache：跨层复用稀疏注意力的索引"),
  section "从 DSA 的成本分解开始" (cost decomposition): the executable
  refresh/share schedule, its argument checks and its worked example.
* same deep-read page, section "相邻层重叠很高…" (overlap): the overlap metric
  |I_l ∩ I_j| / k; section "Training-free…": the greedy layer selection.

The pages name the lightning indexer but do not print its score.  The score
used here is the DeepSeek-Sparse-Attention indexer score

    I[t, s] = sum_h w[t, h] * ReLU(q_I[t, h, :] . k_I[s, :]),   s <= pos(t)

Readings taken where the pages are silent (each is also listed in the design
notes of the repository):

* causal includes the query's own position (s <= pos(t));
* when fewer than k positions are causal, all of them are returned and the
  row is padded with -1;
* ties in score go to the lower position; positions come back in ascending
  order (the pages' own example is order-invariant);
* the pattern alphabet is 'F'/'S' and the whole pattern is validated before
  any work;
* core attention: scale 1/sqrt(Dh) unless given, every query head reads the
  single K/V head, a row whose index list is all -1 yields a zero output.

Parity pins: every function here is pinned in ``tests/test_oracle.py`` by the
pages' worked example, closed forms, invariants, brute force or a special case
that reduces to an independent library routine.
"""

from __future__ import annotations

import math
from typing import Callable, Sequence

import numpy as np

# ---------------------------------------------------------------------------
# Step C1: decoding the stored number formats (exact).
# ---------------------------------------------------------------------------


def bf16_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64, exactly.

    bfloat16 is the upper half of an IEEE-754 binary32: shift the 16 bits
    into the high half of a 32-bit word and read it as float32.
    """
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def e4m3_to_f64(bits) -> np.ndarray:
    """OCP FP8 E4M3 ("e4m3fn") bit patterns (uint8) -> float64, exactly.

    Layout s.eeee.mmm, exponent bias 7, no infinities:
      e == 0          : (-1)^s * 2^-6 * m/8         (subnormal)
      e == 15, m == 7 : NaN
      otherwise       : (-1)^s * 2^(e-7) * (1 + m/8)
    """
    b = np.asarray(bits, dtype=np.uint8).astype(np.int64)
    s = (b >> 7) & 1
    e = (b >> 3) & 0xF
    m = b & 0x7
    sign = np.where(s == 1, -1.0, 1.0)
    normal = sign * np.ldexp(1.0 + m / 8.0, e - 7)
    subnormal = sign * np.ldexp(m / 8.0, -6)
    out = np.where(e == 0, subnormal, normal)
    return np.where((e == 15) & (m == 7), np.nan, out)


def dequantize_e4m3(bits, scale) -> np.ndarray:
    """e4m3 codes times their positive scale, one scale per vector of the
    last axis (a key row, or a query head): the value the fp8 inputs stand
    for, exactly, in float64."""
    return e4m3_to_f64(bits) * np.asarray(scale, dtype=np.float64)[..., None]


# ---------------------------------------------------------------------------
# Step C2: indexer scores.
# ---------------------------------------------------------------------------


def indexer_scores(q, kI, w, q_pos0: int = 0, rows: Sequence[int] | None = None) -> np.ndarray:
    """Lightning-indexer scores of one sequence, float64.

    q  : [T, H, D] query features of the indexer (query row t sits at
         absolute position q_pos0 + t)
    kI : [S, D]    key features of the indexer (already dequantised)
    w  : [T, H]    per-query head weights
    rows : optional subset of query rows to evaluate (default: all T)

    Returns I with shape [len(rows), S]; entries for non-causal keys
    (s > q_pos0 + t) are -inf.
    """
    q = np.asarray(q, dtype=np.float64)
    kI = np.asarray(kI, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    T, H, D = q.shape
    S = kI.shape[0]
    if kI.shape[1] != D or w.shape != (T, H):
        raise ValueError("shape mismatch between q, kI and w")
    if q_pos0 < 0 or q_pos0 + T > S:
        raise ValueError("every query position must have its own key: need q_pos0 + T <= S")
    rows = list(range(T)) if rows is None else list(rows)
    out = np.full((len(rows), S), -np.inf)
    for i, t in enumerate(rows):
        n = q_pos0 + t + 1                      # keys 0 .. pos(t), self included
        per_head = q[t] @ kI[:n].T              # [H, n]: q_I[t,h,:] . k_I[s,:]
        out[i, :n] = w[t] @ np.maximum(per_head, 0.0)   # sum_h w[t,h] * ReLU(.)
    return out


# ---------------------------------------------------------------------------
# Step C3: top-k of one causal score row.
# ---------------------------------------------------------------------------


def topk_positions(scores, k: int) -> np.ndarray:
    """Top-k positions of one score row in which every entry is causal.

    Order of preference: higher score first, then lower position.  The first
    min(k, n) positions of that order are returned sorted ascending and padded
    with -1 up to length k.
    """
    scores = np.asarray(scores, dtype=np.float64)
    if k < 1:
        raise ValueError("k must be >= 1")
    n = scores.shape[0]
    pos = np.arange(n)
    order = np.lexsort((pos, -scores))          # primary -score, secondary position
    keep = np.sort(order[: min(k, n)])
    out = np.full(k, -1, dtype=np.int32)
    out[: keep.shape[0]] = keep
    return out


def indexer_topk(q, kI, w, k: int, q_pos0: int = 0, rows: Sequence[int] | None = None) -> np.ndarray:
    """Scores (C2) then top-k (C3) for the query rows of one sequence: [R, k] int32."""
    T = np.asarray(q).shape[0]
    rows = list(range(T)) if rows is None else list(rows)
    scores = indexer_scores(q, kI, w, q_pos0, rows)
    out = np.empty((len(rows), k), dtype=np.int32)
    for i, t in enumerate(rows):
        out[i] = topk_positions(scores[i, : q_pos0 + t + 1], k)
    return out


# ---------------------------------------------------------------------------
# Step C4: the F/S schedule.
# ---------------------------------------------------------------------------


class PatternError(ValueError):
    """Raised for a pattern the schedule refuses (same family as the pages' ValueError)."""


def validate_pattern(pattern, n_layers: int) -> None:
    """Whole-pattern check done before any layer runs.

    The deep-read page's schedule refuses a pattern whose length differs from
    the number of layers or whose first role is not F (a Shared layer needs an
    earlier Full layer to copy from), and any role other than F or S.
    """
    if not isinstance(pattern, str) or len(pattern) == 0:
        raise PatternError("pattern must be a non-empty string of 'F'/'S'")
    if len(pattern) != n_layers:
        raise PatternError("pattern length must equal the number of layers")
    if pattern[0] != "F":
        raise PatternError("the first layer must be a Full layer")
    for c in pattern:
        if c not in ("F", "S"):
            raise PatternError("every role must be 'F' or 'S'")


def schedule(pattern: str, n_layers: int, topk_of_layer: Callable[[int], np.ndarray]):
    """Refresh-on-F / share-on-S state machine.

    A Full layer runs its own indexer (``topk_of_layer(l)``) and overwrites
    the single cached index tensor; a Shared layer runs nothing and takes a
    copy of the cache, i.e. the indices of the nearest preceding Full layer.
    Returns (per-layer index tensors, number of indexer calls).
    """
    validate_pattern(pattern, n_layers)
    cache = None
    calls = 0
    selected = []
    for layer, role in enumerate(pattern):
        if role == "F":
            cache = np.array(topk_of_layer(layer), dtype=np.int32, copy=True)
            calls += 1
        selected.append(cache.copy())
    return selected, calls


def schedule_rows(score_rows, pattern: str, k: int):
    """The schedule applied to raw score rows, as in the pages' worked example.

    ``score_rows[l]`` is a [R, n] array of indexer outputs for layer l; every
    one of the n positions is treated as causal (the query sits at the last
    position), so each row's top-k is ``topk_positions(row, k)``.
    """
    rows = [np.atleast_2d(np.asarray(r, dtype=np.float64)) for r in score_rows]

    def topk_of_layer(layer):
        return np.stack([topk_positions(r, k) for r in rows[layer]])

    return schedule(pattern, len(rows), topk_of_layer)


# ---------------------------------------------------------------------------
# Step C5: sparse core attention over the selected rows.
# ---------------------------------------------------------------------------


def sparse_attention(Q, K, V, idx, scale: float | None = None) -> np.ndarray:
    """Softmax attention of every query head over its selected K/V rows, float64.

    Q   : [T, Hq, Dh] query heads; all of them read the single K/V head
    K,V : [S, Dh]
    idx : [T, k] selected positions, -1 = empty slot
    O[t, h] = sum_j softmax_j(scale * Q[t,h] . K[idx_j]) * V[idx_j] over the
    valid j.  A row with no valid index gives a zero output.
    """
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    idx = np.asarray(idx)
    T, Hq, Dh = Q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(Dh)
    O = np.zeros((T, Hq, Dh))
    for t in range(T):
        sel = idx[t][idx[t] >= 0]
        if sel.shape[0] == 0:
            continue
        z = scale * (Q[t] @ K[sel].T)            # [Hq, n]
        z = z - z.max(axis=1, keepdims=True)
        p = np.exp(z)
        p = p / p.sum(axis=1, keepdims=True)
        O[t] = p @ V[sel]
    return O


# ---------------------------------------------------------------------------
# The whole stack: schedule + attention on every layer.
# ---------------------------------------------------------------------------


def forward_pattern(pattern: str, layers, k: int, q_pos0: int = 0, scale: float | None = None,
                    rows: Sequence[int] | None = None):
    """Run the F/S stack of one batch of sequences.

    ``layers[l]`` is a dict of float64 arrays with a leading batch axis:
    ``q`` [B,T,H,D], ``kI`` [B,S,D], ``w`` [B,T,H], ``Q`` [B,T,Hq,Dh],
    ``K``/``V`` [B,S,Dh].  (S-layers need no ``q``/``kI``/``w``.)
    ``rows`` restricts the work to a subset of query rows.
    Returns (idx per layer [B,R,k], O per layer [B,R,Hq,Dh], indexer calls).
    """
    n_layers = len(layers)
    validate_pattern(pattern, n_layers)
    B = np.asarray(layers[0]["Q"]).shape[0]
    T = np.asarray(layers[0]["Q"]).shape[1]
    rows = list(range(T)) if rows is None else list(rows)

    def topk_of_layer(layer):
        L = layers[layer]
        return np.stack([indexer_topk(L["q"][b], L["kI"][b], L["w"][b], k, q_pos0, rows)
                         for b in range(B)])

    selected, calls = schedule(pattern, n_layers, topk_of_layer)
    outs = []
    for layer in range(n_layers):
        L = layers[layer]
        outs.append(np.stack([
            sparse_attention(np.asarray(L["Q"][b])[rows], L["K"][b], L["V"][b], selected[layer][b], scale)
            for b in range(B)]))
    return selected, outs, calls


# ---------------------------------------------------------------------------
# Cross-layer metrics and the greedy layer search (next-step items).
# ---------------------------------------------------------------------------


def overlap(idx_a, idx_b, k: int) -> np.ndarray:
    """Per-row Overlap(a, b) = |I_a ∩ I_b| / k (deep-read page, overlap section).

    -1 slots are ignored.  Returns float64 [R].
    """
    a = np.atleast_2d(np.asarray(idx_a))
    b = np.atleast_2d(np.asarray(idx_b))
    out = np.empty(a.shape[0])
    for r in range(a.shape[0]):
        sa = set(int(x) for x in a[r] if x >= 0)
        sb = set(int(x) for x in b[r] if x >= 0)
        out[r] = len(sa & sb) / float(k)
    return out


def greedy_full_layers(num_layers: int, removals: int, evaluate_loss: Callable[[str], float]) -> str:
    """Training-free layer selection (notes page, "核心算法：Greedy Layer Selection").

    Start from all-Full; layer 0 is never a candidate.  Each of ``removals``
    rounds tries turning every remaining Full layer into Shared, evaluates the
    loss of each trial pattern and keeps the flip with the lowest loss (ties:
    the lower layer index).
    """
    if removals < 0 or removals > num_layers - 1:
        raise ValueError("removals must lie in [0, num_layers - 1]")
    roles = ["F"] * num_layers
    remaining = list(range(1, num_layers))
    for _ in range(removals):
        best = None
        for layer in remaining:
            trial = list(roles)
            trial[layer] = "S"
            loss = float(evaluate_loss("".join(trial)))
            if best is None or (loss, layer) < best:
                best = (loss, layer)
        roles[best[1]] = "S"
        remaining.remove(best[1])
    return "".join(roles)
