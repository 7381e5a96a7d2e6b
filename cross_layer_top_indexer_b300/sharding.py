"""Query-row sharding of a causal prefill across ranks.

Every query row's top-k and its sparse attention depend only on that row's
own inputs and on the keys at positions <= its own (notes page
"NLP--IndexCache", "背景 & 问题提出": the indexer scores, for each query, the
tokens before it; core attention then runs on the k selected ones).  Rows
therefore split across ranks with no merge of results: each rank keeps its
rows' indices and outputs.  The one exchange is the key side: a rank needs
the indexer keys (and their scales) and the K/V rows of the whole causal
prefix of its rows, so each layer's key rows, produced where their tokens
live, are all-gathered once.

The split is zig-zag: the L rows form 2N chunks, and rank r takes chunks r
and 2N-1-r, so every rank gets one early (cheap) and one late (expensive)
chunk and the causal work balances.  Each chunk runs as one
``ic_forward_pattern`` call with ``q_pos0`` at the chunk start and
``S = q_pos0 + T``.  Positions are absolute, so the concatenated per-rank
results equal the unsharded run exactly.
"""

from __future__ import annotations

from typing import List, Sequence, Tuple

import torch


def zigzag_chunks(L: int, world: int) -> List[Tuple[int, int]]:
    """The 2*world chunks (start, length) of rows 0..L-1, in order; the first
    L % (2*world) chunks are one row longer."""
    n = 2 * world
    if L < n:
        raise ValueError("need at least two rows per rank (L=%d, world=%d)" % (L, world))
    base, extra = divmod(L, n)
    out, start = [], 0
    for c in range(n):
        length = base + (1 if c < extra else 0)
        out.append((start, length))
        start += length
    return out


def rank_rows(L: int, world: int, rank: int) -> List[Tuple[int, int]]:
    """Row ranges (q_pos0, T) of `rank`: chunks rank and 2*world-1-rank."""
    if not 0 <= rank < world:
        raise ValueError("rank %d outside [0, %d)" % (rank, world))
    ch = zigzag_chunks(L, world)
    return [ch[rank], ch[2 * world - 1 - rank]]


def causal_pairs(ranges: Sequence[Tuple[int, int]]) -> int:
    """Causal (query, key) pairs of the rows in `ranges`: the indexer's work."""
    return sum(T * (q0 + 1) + T * (T - 1) // 2 for q0, T in ranges)


def all_gather_rows(local: torch.Tensor, L: int, world: int, rank: int, group=None) -> torch.Tensor:
    """The exchange step: `local` holds this rank's key-side rows, the rows of
    its two chunks concatenated along dim 1 ([B, rows, ...]); returns the
    [B, L, ...] tensor of all rows in position order, on every rank.  One
    all-gather (NCCL on GPUs, gloo on CPU); chunk lengths may differ by one,
    so every rank pads its block to the longest."""
    import torch.distributed as dist

    ranges = [rank_rows(L, world, r) for r in range(world)]
    counts = [sum(T for _, T in rr) for rr in ranges]
    width = max(counts)
    if local.shape[1] != counts[rank]:
        raise ValueError("rank %d holds %d rows, its chunks have %d" % (rank, local.shape[1], counts[rank]))
    pad = list(local.shape)
    pad[1] = width
    send = local.new_zeros(pad)
    send[:, : counts[rank]] = local
    recv = [torch.empty_like(send) for _ in range(world)]
    dist.all_gather(recv, send, group=group)
    full_shape = list(local.shape)
    full_shape[1] = L
    out = local.new_empty(full_shape)
    for r in range(world):
        off = 0
        for q0, T in ranges[r]:
            out[:, q0:q0 + T] = recv[r][:, off:off + T]
            off += T
    return out


def take_rows(full: torch.Tensor, ranges: Sequence[Tuple[int, int]]) -> torch.Tensor:
    """The rows of `ranges` of a [B, L, ...] tensor, concatenated along dim 1."""
    return torch.cat([full[:, q0:q0 + T] for q0, T in ranges], dim=1).contiguous()


def forward_rows(binding, pattern: str, layers: Sequence[dict], k: int, ranges: Sequence[Tuple[int, int]],
                 stream=None):
    """Run the F/S stack for the query rows of `ranges` (this rank's share).

    ``layers[l]`` holds the full-prefix key side (kI, kscale, K, V: [B, L, ...])
    and the full query side (q, w, Q); each range runs as one
    ic_forward_pattern call over its rows with ``q_pos0`` at the range start.
    Returns, per range, (index cache [B, T, k], outputs per layer [B, T, Hq, Dh])."""
    results = []
    for q0, T in ranges:
        sub = []
        for L in layers:
            d = {"kI": L.get("kI"), "kscale": L.get("kscale"), "K": L["K"], "V": L["V"]}
            d["q"] = L["q"][:, q0:q0 + T].contiguous() if L.get("q") is not None else None
            d["w"] = L["w"][:, q0:q0 + T].contiguous() if L.get("w") is not None else None
            d["Q"] = L["Q"][:, q0:q0 + T].contiguous()
            d["O"] = torch.empty_like(d["Q"])
            sub.append(d)
        cache, _ = binding.forward_pattern(pattern, sub, k, q_pos0=q0, S=q0 + T, stream=stream)
        results.append((cache, [d["O"] for d in sub]))
    return results
