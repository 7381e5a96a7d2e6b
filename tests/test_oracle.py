"""Pins for the CPU oracle (no GPU).

Each test ties the oracle to something other than itself: the pages' worked
example, closed forms, hand-computed cases, brute force by a different
mechanism, invariants, or a special case that reduces to an independent
library routine (torch's own dtype decoders, torch's dense attention).
"""

import math
import os
import random

import numpy as np
import pytest
import torch

import oracle
from oracle import indexcache as oc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_worked_example():
    rows, expect, same, differ = {}, {}, [], []
    pattern = k = calls = None
    with open(os.path.join(GOLDEN, "worked_example.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            tok = line.split()
            if tok[0] == "pattern":
                pattern = tok[1]
            elif tok[0] == "k":
                k = int(tok[1])
            elif tok[0] == "row":
                rows[int(tok[1])] = [float(x) for x in tok[2:]]
            elif tok[0] == "calls":
                calls = int(tok[1])
            elif tok[0] == "same":
                same.append((int(tok[1]), int(tok[2])))
            elif tok[0] == "differ":
                differ.append((int(tok[1]), int(tok[2])))
            elif tok[0] == "expect":
                expect[(tok[1], int(tok[2]))] = [int(x) for x in tok[3:]]
    return pattern, k, [rows[i] for i in sorted(rows)], calls, same, differ, expect


# ---------------------------------------------------------------------------
# The pages' worked example.
# ---------------------------------------------------------------------------


def test_worked_example_page_asserts():
    pattern, k, rows, calls, same, differ, expect = _read_worked_example()
    selected, n_calls = oracle.schedule_rows(rows, pattern, k)
    assert n_calls == calls
    for a, b in same:
        assert np.array_equal(selected[a], selected[b])
    for a, b in differ:
        assert not np.array_equal(selected[a], selected[b])
    for layer in range(4):
        assert selected[layer][0].tolist() == expect[(pattern, layer)]


def test_worked_example_all_full_recomputes():
    pattern, k, rows, _, _, _, expect = _read_worked_example()
    selected, n_calls = oracle.schedule_rows(rows, "FFFF", k)
    assert n_calls == 4
    for layer in range(4):
        assert selected[layer][0].tolist() == expect[("FFFF", layer)]
    # layer 2 is where reuse and recomputation disagree
    assert selected[2][0].tolist() != expect[("FSSF", 2)]


# ---------------------------------------------------------------------------
# Pattern validation (the page's schedule refuses these).
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("pattern,n", [
    ("", 0), ("FSS", 4), ("FSSFS", 4), ("SFFF", 4), ("FSXF", 4), ("1001", 4), ("fssf", 4), ("F SF", 4),
])
def test_pattern_rejected(pattern, n):
    with pytest.raises(oracle.PatternError):
        oracle.validate_pattern(pattern, n)
    with pytest.raises(ValueError):
        oracle.schedule_rows([[0.0, 1.0]] * max(n, 1), pattern, 1)


def test_pattern_accepted():
    for p in ("F", "FS", "FSSF", "FFFF", "F" + "S" * 46):
        oracle.validate_pattern(p, len(p))


# ---------------------------------------------------------------------------
# Top-k (C3) against brute force by a different mechanism.
# ---------------------------------------------------------------------------


def _brute_topk(row, k):
    n = len(row)
    best = sorted(range(n), key=lambda s: (-row[s], s))[:k]
    best = sorted(best)
    return best + [-1] * (k - len(best))


def test_topk_brute_force_with_ties():
    rng = random.Random(7)
    for _ in range(300):
        n = rng.randint(1, 60)
        k = rng.randint(1, 70)
        row = [float(rng.randint(-3, 3)) for _ in range(n)]   # many exact ties
        assert oracle.topk_positions(row, k).tolist() == _brute_topk(row, k)


def test_topk_short_row_returns_all_positions():
    for n in range(1, 20):
        out = oracle.topk_positions(np.random.default_rng(n).normal(size=n), 32).tolist()
        assert out == list(range(n)) + [-1] * (32 - n)


def test_topk_negative_zero_ties_with_zero():
    # -0.0 and +0.0 are the same score: the lower position wins
    assert oracle.topk_positions([0.0, -0.0, 0.0], 1).tolist() == [0]
    assert oracle.topk_positions([-0.0, 0.0], 1).tolist() == [0]


# ---------------------------------------------------------------------------
# Scores (C2): hand values, textbook special case, identities, invariances.
# ---------------------------------------------------------------------------


def test_scores_hand_computed():
    # H = 2, D = 2; one key.  Head 0: q.k = 3 (kept), head 1: q.k = -2 (ReLU -> 0).
    q = np.array([[[1.0, 1.0], [-1.0, 0.0]]])      # [T=1, H=2, D=2]
    kI = np.array([[1.0, 2.0]])                    # [S=1, D=2]
    w = np.array([[2.0, -5.0]])                    # [T=1, H=2]
    # I = 2 * ReLU(3) + (-5) * ReLU(-1) = 6
    assert oracle.indexer_scores(q, kI, w)[0, 0] == 6.0
    # a negative weight on a positive head lowers the score: w = [-1, 4], q.k = [3, 2]
    q2 = np.array([[[1.0, 1.0], [0.0, 1.0]]])
    w2 = np.array([[-1.0, 4.0]])
    assert oracle.indexer_scores(q2, kI, w2)[0, 0] == -1.0 * 3 + 4.0 * 2


def test_scores_single_head_nonnegative_is_textbook_matmul():
    rng = np.random.default_rng(3)
    T, S, D = 5, 9, 4
    q = rng.integers(0, 4, size=(T, 1, D)).astype(float)
    kI = rng.integers(0, 4, size=(S, D)).astype(float)
    w = np.ones((T, 1))
    got = oracle.indexer_scores(q, kI, w, q_pos0=S - T)
    for t in range(T):
        for s in range(S):
            if s <= S - T + t:
                ref = sum(q[t, 0, d] * kI[s, d] for d in range(D))   # plain dot product
                assert got[t, s] == ref
            else:
                assert got[t, s] == -np.inf


def test_scores_relu_difference_identity():
    # ReLU(x) - ReLU(-x) = x, so I(q) - I(-q) is the bilinear form sum_h w q.k
    rng = np.random.default_rng(4)
    T, H, D = 6, 3, 5
    q = rng.normal(size=(T, H, D))
    kI = rng.normal(size=(T, D))
    w = rng.normal(size=(T, H))
    diff = oracle.indexer_scores(q, kI, w) - oracle.indexer_scores(-q, kI, w)
    bil = np.einsum("th,thd,sd->ts", w, q, kI)
    mask = np.tril(np.ones((T, T), bool))
    assert np.allclose(diff[mask], bil[mask], rtol=1e-12, atol=1e-12)


def test_scores_invariances():
    rng = np.random.default_rng(5)
    T, H, D = 7, 4, 6
    q = rng.normal(size=(T, H, D))
    kI = rng.normal(size=(T + 3, D))
    w = rng.normal(size=(T, H))
    base = oracle.indexer_scores(q, kI, w, q_pos0=3)
    perm = rng.permutation(H)
    assert np.allclose(oracle.indexer_scores(q[:, perm], kI, w[:, perm], q_pos0=3), base)
    assert np.allclose(oracle.indexer_scores(q, kI, 2.5 * w, q_pos0=3), 2.5 * base)
    assert np.allclose(oracle.indexer_scores(3.0 * q, kI, w, q_pos0=3), 3.0 * base)
    w2 = rng.normal(size=(T, H))
    assert np.allclose(oracle.indexer_scores(q, kI, w + w2, q_pos0=3),
                       base + oracle.indexer_scores(q, kI, w2, q_pos0=3))
    # keys past a row's position never influence that row
    k_alt = kI.copy()
    k_alt[-1] += 100.0
    alt = oracle.indexer_scores(q, k_alt, w, q_pos0=3)
    assert np.array_equal(alt[:-1], base[:-1])


def test_integer_scores_are_exact():
    rng = np.random.default_rng(6)
    T, H, D = 16, 4, 32
    q = rng.integers(-2, 3, size=(T, H, D)).astype(float)
    kI = rng.integers(-2, 3, size=(T, D)).astype(float)
    w = rng.integers(-2, 3, size=(T, H)).astype(float)
    I = oracle.indexer_scores(q, kI, w)
    fin = I[np.isfinite(I)]
    assert np.array_equal(fin, np.round(fin))
    assert np.abs(fin).max() <= 4 * 2 * (4 * D)


# ---------------------------------------------------------------------------
# Number formats (C1) against torch's own decoders.
# ---------------------------------------------------------------------------


def test_bf16_decode_all_codes():
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.bf16_to_f64(codes)
    ref = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_e4m3_decode_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_to_f64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert nan.sum() == 2 and np.isnan(ours[0x7F]) and np.isnan(ours[0xFF])
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9


def test_e4m3_dequantise_closed_form():
    # codes of 1, -2, 0.5 and the smallest subnormal 2^-9, one scale per row
    codes = np.array([[0x38, 0xC0, 0x30, 0x01], [0x38, 0xC0, 0x30, 0x01]], dtype=np.uint8)
    scale = np.array([0.25, 8.0])
    want = np.array([[0.25, -0.5, 0.125, 2.0 ** -11], [8.0, -16.0, 4.0, 2.0 ** -6]])
    assert np.array_equal(oracle.dequantize_e4m3(codes, scale), want)
    # a scale per query head of a [T, H, D] tensor broadcasts over D only
    rng = np.random.default_rng(4)
    c = rng.integers(0, 256, (3, 5, 7)).astype(np.uint8)
    c[c == 0x7F] = 0x7E
    c[c == 0xFF] = 0xFE
    sc = rng.uniform(0.1, 4.0, (3, 5))
    ref = torch.from_numpy(c).view(torch.float8_e4m3fn).to(torch.float64).numpy() * sc[..., None]
    assert np.array_equal(oracle.dequantize_e4m3(c, sc), ref)


# ---------------------------------------------------------------------------
# Sparse attention (C5).
# ---------------------------------------------------------------------------


def test_attention_all_causal_equals_dense_causal():
    rng = np.random.default_rng(8)
    T, Hq, Dh, k = 24, 3, 16, 32
    Q = rng.normal(size=(T, Hq, Dh))
    K = rng.normal(size=(T, Dh))
    V = rng.normal(size=(T, Dh))
    idx = np.stack([oracle.topk_positions(np.zeros(t + 1), k) for t in range(T)])  # all causal
    ours = oracle.sparse_attention(Q, K, V, idx, 1.0 / math.sqrt(Dh))
    q_t = torch.from_numpy(Q).permute(1, 0, 2)[None]        # [1, Hq, T, Dh]
    k_t = torch.from_numpy(K)[None, None].expand(1, Hq, T, Dh)
    v_t = torch.from_numpy(V)[None, None].expand(1, Hq, T, Dh)
    ref = torch.nn.functional.scaled_dot_product_attention(q_t, k_t, v_t, is_causal=True)
    ref = ref[0].permute(1, 0, 2).numpy()
    assert np.allclose(ours, ref, rtol=1e-12, atol=1e-12)


def test_attention_permutation_and_padding_invariant():
    rng = np.random.default_rng(9)
    T, Hq, Dh, S = 4, 2, 8, 40
    Q = rng.normal(size=(T, Hq, Dh))
    K = rng.normal(size=(S, Dh))
    V = rng.normal(size=(S, Dh))
    idx = np.stack([rng.choice(S, size=6, replace=False) for _ in range(T)])
    base = oracle.sparse_attention(Q, K, V, idx, 0.3)
    shuffled = np.stack([rng.permutation(r) for r in idx])
    padded = np.concatenate([np.full((T, 3), -1), idx, np.full((T, 2), -1)], axis=1)
    assert np.allclose(oracle.sparse_attention(Q, K, V, shuffled, 0.3), base, rtol=1e-13, atol=1e-13)
    assert np.allclose(oracle.sparse_attention(Q, K, V, padded, 0.3), base, rtol=1e-13, atol=1e-13)


def test_attention_closed_forms():
    rng = np.random.default_rng(10)
    Q = rng.normal(size=(1, 2, 4))
    K = rng.normal(size=(5, 4))
    V = rng.normal(size=(5, 4))
    # one selected row: the output is that V row
    assert np.allclose(oracle.sparse_attention(Q, K, V, np.array([[3, -1]]), 1.0)[0], V[3])
    # zero scale: plain mean of the selected V rows
    out = oracle.sparse_attention(Q, K, V, np.array([[0, 2, 4]]), 0.0)[0]
    assert np.allclose(out, V[[0, 2, 4]].mean(axis=0))
    # two rows: softmax of two logits is a logistic weight
    z = Q[0] @ K[[1, 2]].T * 0.5
    a = 1.0 / (1.0 + np.exp(z[:, 1] - z[:, 0]))
    want = a[:, None] * V[1] + (1 - a)[:, None] * V[2]
    assert np.allclose(oracle.sparse_attention(Q, K, V, np.array([[1, 2]]), 0.5)[0], want)
    # no valid row: zero output
    assert np.all(oracle.sparse_attention(Q, K, V, np.array([[-1, -1]]), 1.0) == 0.0)


# ---------------------------------------------------------------------------
# Schedule (C4): reuse rule and invariants on random patterns.
# ---------------------------------------------------------------------------


def test_schedule_reuse_rule_and_call_count():
    rng = random.Random(11)
    for _ in range(50):
        n = rng.randint(1, 12)
        pattern = "F" + "".join(rng.choice("FS") for _ in range(n - 1))
        rows = [np.random.default_rng(rng.randint(0, 10**6)).normal(size=(3, 9)) for _ in range(n)]
        sel, calls = oracle.schedule_rows(rows, pattern, 4)
        allf, calls_f = oracle.schedule_rows(rows, "F" * n, 4)
        assert calls == pattern.count("F") and calls_f == n
        for layer in range(n):
            f = max(j for j in range(layer + 1) if pattern[j] == "F")   # f(l), or l itself if F
            assert np.array_equal(sel[layer], allf[f])


def test_forward_pattern_all_full_is_independent_per_layer():
    rng = np.random.default_rng(12)
    B, T, H, D, Hq, Dh, k = 2, 10, 2, 4, 2, 8, 3
    layers = []
    for _ in range(3):
        layers.append(dict(q=rng.normal(size=(B, T, H, D)), kI=rng.normal(size=(B, T, D)),
                           w=rng.normal(size=(B, T, H)), Q=rng.normal(size=(B, T, Hq, Dh)),
                           K=rng.normal(size=(B, T, Dh)), V=rng.normal(size=(B, T, Dh))))
    sel, outs, calls = oracle.forward_pattern("FFF", layers, k)
    assert calls == 3
    for l, L in enumerate(layers):
        for b in range(B):
            assert np.array_equal(sel[l][b], oracle.indexer_topk(L["q"][b], L["kI"][b], L["w"][b], k))
            assert np.allclose(outs[l][b], oracle.sparse_attention(L["Q"][b], L["K"][b], L["V"][b], sel[l][b]))
    sel2, outs2, calls2 = oracle.forward_pattern("FSF", layers, k)
    assert calls2 == 2 and np.array_equal(sel2[1], sel2[0]) and np.array_equal(sel2[2], sel[2])


# ---------------------------------------------------------------------------
# Chunked prefill and decode rows (C6).
# ---------------------------------------------------------------------------


def test_chunked_rows_equal_unchunked():
    rng = np.random.default_rng(13)
    T, H, D, k = 40, 3, 6, 8
    q = rng.normal(size=(T, H, D))
    kI = rng.normal(size=(T, D))
    w = rng.normal(size=(T, H))
    full = oracle.indexer_topk(q, kI, w, k)
    for c0 in (0, 8, 16, 24, 32):
        part = oracle.indexer_topk(q[c0:c0 + 8], kI[: c0 + 8], w[c0:c0 + 8], k, q_pos0=c0)
        assert np.array_equal(part, full[c0:c0 + 8])
    # a decode query at position p sees keys 0..p, like prefill row p
    p = 29
    dec = oracle.indexer_topk(q[p:p + 1], kI[: p + 1], w[p:p + 1], k, q_pos0=p)
    assert np.array_equal(dec[0], full[p])


def test_causal_positions_never_exceed_query():
    rng = np.random.default_rng(14)
    T, H, D, k = 30, 2, 4, 8
    idx = oracle.indexer_topk(rng.normal(size=(T, H, D)), rng.normal(size=(T, D)), rng.normal(size=(T, H)), k)
    for t in range(T):
        valid = idx[t][idx[t] >= 0]
        assert len(valid) == min(k, t + 1)
        assert valid.max() <= t and np.all(np.diff(valid) > 0)


# ---------------------------------------------------------------------------
# Next-step items: overlap metric and greedy layer search.
# ---------------------------------------------------------------------------


def test_overlap_metric():
    a = np.array([[0, 1, 2, 3], [5, 6, -1, -1]])
    b = np.array([[2, 3, 4, 5], [5, 6, -1, -1]])
    assert oracle.overlap(a, b, 4).tolist() == [0.5, 0.5]
    assert oracle.overlap(a[:1], a[:1], 4).tolist() == [1.0]


def test_greedy_toy_and_forward_count():
    # deep-read page, "Training-free" section: five layers, importance per layer,
    # the loss is the total importance of the Shared layers; two removals.
    importance = [99.0, 3.0, 0.2, 2.0, 0.1]
    evaluated = []

    def loss(pattern):
        evaluated.append(pattern)
        return sum(x for role, x in zip(pattern, importance) if role == "S")

    assert oracle.greedy_full_layers(5, 2, loss) == "FFSFS"
    N, K = 5, 2
    assert len(evaluated) == K * (N - 1) - K * (K - 1) // 2
    evaluated.clear()
    out = oracle.greedy_full_layers(N, N - 1, loss)
    assert out == "F" + "S" * (N - 1) and len(evaluated) == N * (N - 1) // 2
