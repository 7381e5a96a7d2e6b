"""Helpers that compare the CUDA path with the CPU oracle on the same inputs."""

from __future__ import annotations

import numpy as np
import torch

import oracle
from cross_layer_top_indexer_b300 import synth

# Tolerances of the parity contract.
SCORE_REL_TOL = 1e-3       # a selected position may fall below the k-th score by this much (relative, floor 1)
RECALL_MIN = 0.999         # set recall against the oracle's own top-k
ATTN_MAX_ABS = 2e-2        # bf16 output against the fp64 oracle on the GPU's own indices


def to_f64(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return oracle.bf16_to_f64(synth.bf16_bits(t))
    if t.dtype == torch.float8_e4m3fn:
        return oracle.e4m3_to_f64(synth.e4m3_bits(t))
    return t.detach().cpu().to(torch.float64).numpy()


def keys_f64(kI: torch.Tensor, kscale) -> np.ndarray:
    k = to_f64(kI)
    if kscale is not None:
        k = k * to_f64(kscale)[..., None]
    return k


def check_topk(gpu_idx: np.ndarray, q64, k64, w64, k: int, q_pos0: int, rows, exact: bool, stats=None):
    """Check GPU index rows (one sequence) against the oracle for ``rows``.

    exact: the index sets must be identical (integer inputs).
    otherwise: the tolerance rule (every selected position scores at least
    the k-th oracle score minus 1e-3*max(1,|k-th|); recall accumulated in
    ``stats``).
    """
    rows = list(rows)
    scores = oracle.indexer_scores(q64, k64, w64, q_pos0, rows)
    if stats is None:
        stats = {"hit": 0, "tot": 0}
    for i, t in enumerate(rows):
        pos = q_pos0 + t
        n = pos + 1
        want = oracle.topk_positions(scores[i, :n], k)
        got = gpu_idx[t]
        nv = min(k, n)
        # layout: nv valid ascending positions in [0, pos], then -1
        assert np.all(got[nv:] == -1), (t, got[nv:][:8])
        valid = got[:nv]
        assert np.all(valid >= 0) and np.all(valid <= pos), (t, valid.min(), valid.max(), pos)
        assert np.all(np.diff(valid) > 0), ("not strictly ascending", t)
        if exact:
            assert np.array_equal(got, want), (t, np.setdiff1d(want, got)[:8], np.setdiff1d(got, want)[:8])
        else:
            row = scores[i, :n]
            kth = np.sort(row)[::-1][nv - 1]
            floor = kth - SCORE_REL_TOL * max(1.0, abs(kth))
            assert np.all(row[valid] >= floor), (t, row[valid].min(), kth)
            stats["hit"] += len(np.intersect1d(valid, want[:nv]))
            stats["tot"] += nv
    return stats


def check_recall(stats):
    assert stats["tot"] > 0
    rec = stats["hit"] / stats["tot"]
    assert rec >= RECALL_MIN, rec
    return rec


def check_attention(O_gpu: torch.Tensor, Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, idx: torch.Tensor,
                    scale: float, rows=None, tol: float = ATTN_MAX_ABS):
    """O (one sequence, [T,Hq,Dh] bf16) against the oracle on the GPU's own indices."""
    T = Q.shape[0]
    rows = list(range(T)) if rows is None else list(rows)
    Q64 = to_f64(Q[rows])
    want = oracle.sparse_attention(Q64, to_f64(K), to_f64(V), idx[rows].cpu().numpy(), scale)
    got = to_f64(O_gpu[rows])
    err = float(np.abs(got - want).max()) if got.size else 0.0
    assert err <= tol, err
    return err
