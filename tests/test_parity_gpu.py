"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Integer-valued inputs must give bit-identical index sets; random inputs are
held to the tolerance rule in ``parity_util``; attention outputs to a max-abs
error of 2e-2 against the fp64 oracle evaluated on the GPU's own indices.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from cross_layer_top_indexer_b300 import binding as B
from cross_layer_top_indexer_b300 import synth
from tests import parity_util as pu

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.load()


def _idx64(t):
    return t.cpu().numpy()


# ---------------------------------------------------------------------------
# The pages' worked example, realised through the real indexer kernels.
# ---------------------------------------------------------------------------

WORKED_ROWS = [[0.1, 0.9, 0.3, 0.2], [0.2, 0.7, 0.4, 0.1], [0.6, 0.1, 0.5, 0.3], [0.8, 0.1, 0.2, 0.7]]


def _worked_layers(T):
    """Layer l: one indexer head, query row 3 = e_0, key s = 10*score_l[s] e_0, w = 1.
    Scores of row 3 are then exactly 10x the page's row (integers, exact in bf16)."""
    D = 32
    layers = []
    g = torch.Generator(device="cpu").manual_seed(5)
    for l in range(4):
        q = torch.zeros(1, T, 1, D)
        q[0, 3, 0, 0] = 1.0
        kI = torch.zeros(1, T, D)
        for s in range(4):
            kI[0, s, 0] = round(10 * WORKED_ROWS[l][s])
        w = torch.ones(1, T, 1)
        Q = torch.randn(1, T, 4, 64, generator=g)
        K = torch.randn(1, T, 64, generator=g)
        V = torch.randn(1, T, 64, generator=g)
        layers.append(dict(q=q.to(DEV, torch.bfloat16), kI=kI.to(DEV, torch.bfloat16), kscale=None,
                           w=w.to(DEV), Q=Q.to(DEV, torch.bfloat16), K=K.to(DEV, torch.bfloat16),
                           V=V.to(DEV, torch.bfloat16)))
    return layers


@pytest.mark.parametrize("T", [16, 4])    # 16 rows: prefill kernel; 4 rows: decode kernels
def test_worked_example_through_kernels(T):
    layers = _worked_layers(T)
    expect_row3 = {"F": [1, 2], "FS": [1, 2], "FSS": [1, 2], "FSSF": [0, 3], "FFF": [0, 2], "FFFF": [0, 3]}
    for pattern, want in expect_row3.items():
        cache, calls = B.forward_pattern(pattern, layers[: len(pattern)], k=2)
        torch.cuda.synchronize()
        assert calls == pattern.count("F")
        c = _idx64(cache)[0]
        assert c[3].tolist() == want, (pattern, c[3])
        assert c[0].tolist() == [0, -1] and c[1].tolist() == [0, 1]
    # outputs of the FSSF run: layers 1 and 2 attend over layer 0's indices
    cache, calls = B.forward_pattern("FSSF", layers, k=2)
    torch.cuda.synchronize()
    sel, _ = oracle.schedule_rows(WORKED_ROWS, "FSSF", 2)
    for l in range(4):
        idx = torch.full((T, 2), -1, dtype=torch.int32)
        idx[:3] = torch.tensor([[0, -1], [0, 1], [0, 1]], dtype=torch.int32)
        idx[3] = torch.from_numpy(sel[l][0])
        if T > 4:   # rows past 3 have all-zero scores: the lowest positions win
            idx[4:] = torch.tensor([0, 1], dtype=torch.int32)
        L = layers[l]
        pu.check_attention(L["O"][0], L["Q"][0], L["K"][0], L["V"][0], idx, 1.0 / 8.0, rows=range(4))


# ---------------------------------------------------------------------------
# Tiny stack: integer inputs, bit-exact indices.
# ---------------------------------------------------------------------------


def test_tiny_stack_bit_exact():
    cfg = synth.TINY
    layers = synth.make_stack(cfg, 1234, DEV)
    per_layer = {}
    for l, c in enumerate(cfg.pattern):
        if c == "F":
            L = layers[l]
            idx = B.indexer_topk(L["q"], L["kI"], L["w"], cfg.k)
            torch.cuda.synchronize()
            want = oracle.indexer_topk(pu.to_f64(L["q"][0]), pu.to_f64(L["kI"][0]), pu.to_f64(L["w"][0]), cfg.k)
            got = _idx64(idx)[0]
            assert np.array_equal(got, want), np.argwhere(got != want)[:5]
            per_layer[l] = want
    cache, calls = B.forward_pattern(cfg.pattern, layers, cfg.k)
    torch.cuda.synchronize()
    assert calls == cfg.pattern.count("F")
    assert np.array_equal(_idx64(cache)[0], per_layer[3])
    f = 0
    for l, c in enumerate(cfg.pattern):
        f = l if c == "F" else f
        L = layers[l]
        idx = torch.from_numpy(per_layer[f])
        pu.check_attention(L["O"][0], L["Q"][0], L["K"][0], L["V"][0], idx, cfg.scale)


# ---------------------------------------------------------------------------
# Indexer on random and adversarial inputs (prefill kernel).
# ---------------------------------------------------------------------------

CASES = [
    # B, T, S, q_pos0, H, D, k, dist, kdtype
    (1, 1000, 1000, 0, 64, 128, 64, "normal", "bf16"),       # ragged tail, one compaction
    (2, 333, 1333, 1000, 64, 128, 256, "normal", "bf16"),    # query chunk at an offset, batch 2
    (1, 700, 700, 0, 16, 64, 2048, "normal", "bf16"),        # k above every causal count
    (1, 517, 517, 0, 64, 128, 1, "normal", "bf16"),          # k = 1
    (1, 3000, 3000, 0, 64, 128, 2048, "normal", "bf16"),     # k = 2048 with compactions
    (1, 600, 600, 0, 8, 32, 100, "int", "bf16"),             # heavy ties, bit-exact
    (1, 1500, 1500, 0, 64, 128, 256, "normal", "e4m3"),      # fp8 keys (tensor-core path)
    (2, 700, 1700, 1000, 64, 128, 2048, "normal", "e4m3"),   # fp8 keys, chunk at an offset, batch 2
    (1, 900, 900, 0, 16, 64, 64, "normal", "e4m3"),          # fp8 keys, mma.sync path
    (1, 1029, 1029, 0, 4, 32, 16, "int", "bf16"),            # tiny head shape, ragged
    (1, 777, 777, 0, 64, 128, 100, "int", "bf16"),           # tensor-core path, integer: bit-exact
    (2, 2600, 2600, 0, 64, 128, 2048, "int", "bf16"),        # tensor-core path, ties across cuts
    (1, 4099, 4099, 0, 64, 128, 333, "normal", "bf16"),      # tensor-core path, many cuts, ragged
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B%d_T%d_S%d_p%d_H%d_D%d_k%d_%s_%s" % c)
def test_indexer_prefill_cases(case):
    Bn, T, S, q_pos0, H, D, k, dist, kd = case
    cfg = synth.StackConfig("case", 1, "F", Bn, T, S, H, D, k, 4, 64, kd, dist, q_pos0)
    q, kI, ks, w = synth.make_indexer_inputs(cfg, 0, 77, DEV)
    idx = B.indexer_topk(q, kI, w, k, q_pos0, kscale=ks, S=S)
    torch.cuda.synchronize()
    got = _idx64(idx)
    stats = {"hit": 0, "tot": 0}
    for b in range(Bn):
        pu.check_topk(got[b], pu.to_f64(q[b]), pu.keys_f64(kI[b], None if ks is None else ks[b]),
                      pu.to_f64(w[b]), k, q_pos0, range(T), exact=(dist == "int"), stats=stats)
    if dist != "int":
        pu.check_recall(stats)


@pytest.mark.parametrize("T,k,mode", [(900, 100, "int"), (1283, 512, "codes")])
def test_prefill_e4m3_every_code(T, k, mode):
    # e4m3 keys through the tensor-core prefill kernel: integer codes with
    # power-of-two key scales (exact products and sums: bit-exact sets), or
    # every code but NaN with random scales (tolerance rule)
    g = torch.Generator(device="cpu").manual_seed(T)
    if mode == "int":
        ints = torch.tensor([0x00, 0x38, 0x40, 0x44, 0xB8, 0xC0, 0xC4], dtype=torch.uint8)   # 0, 1, 2, 3, -1, -2, -3
        kb = ints[torch.randint(0, len(ints), (1, T, 128), generator=g)]
        q = torch.randint(-2, 3, (1, T, 64, 128), generator=g).float()
        w = torch.randint(-2, 3, (1, T, 64), generator=g).float()
        ks = 2.0 ** torch.randint(-1, 2, (1, T), generator=g).float()
    else:
        codes = torch.tensor([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=torch.uint8)
        kb = codes[torch.randint(0, len(codes), (1, T, 128), generator=g)]
        q = torch.randn(1, T, 64, 128, generator=g) / 11.3
        w = torch.randn(1, T, 64, generator=g) / 8
        ks = torch.rand(1, T, generator=g) * 0.01 + 1e-3
    kI = kb.view(torch.float8_e4m3fn).to(DEV)
    q, w, ks = q.to(DEV, torch.bfloat16), w.to(DEV), ks.to(DEV)
    got = _idx64(B.indexer_topk(q, kI, w, k, kscale=ks))
    torch.cuda.synchronize()
    stats = {"hit": 0, "tot": 0}
    pu.check_topk(got[0], pu.to_f64(q[0]), pu.keys_f64(kI[0], ks[0]), pu.to_f64(w[0]), k, 0, range(T),
                  exact=(mode == "int"), stats=stats)
    if mode != "int":
        pu.check_recall(stats)


@pytest.mark.parametrize("H,D", [(1, 32), (64, 128)])    # mma.sync kernel, tensor-core kernel
def test_indexer_monotone_scores_many_compactions(H, D):
    # score grows with position in bf16 steps (with exact ties): every key
    # beats the threshold, so the candidate list is cut back again and again
    T, k = 2600, 300
    q = torch.zeros(1, T, H, D)
    q[:, :, 0, 0] = 1.0
    kI = torch.zeros(1, T, D)
    kI[0, :, 0] = torch.arange(T, dtype=torch.float32) * 0.01
    w = torch.ones(1, T, H)
    q, kI, w = q.to(DEV, torch.bfloat16), kI.to(DEV, torch.bfloat16), w.to(DEV)
    idx = B.indexer_topk(q, kI, w, k)
    torch.cuda.synchronize()
    pu.check_topk(_idx64(idx)[0], pu.to_f64(q[0]), pu.to_f64(kI[0]), pu.to_f64(w[0]), k, 0, range(T), exact=True)


@pytest.mark.parametrize("H,D", [(2, 32), (64, 128)])
def test_indexer_constant_scores_lowest_positions(H, D):
    T, k = 1100, 200
    q = torch.zeros(1, T, H, D, device=DEV, dtype=torch.bfloat16)
    kI = torch.ones(1, T, D, device=DEV, dtype=torch.bfloat16)
    w = torch.ones(1, T, H, device=DEV)
    idx = _idx64(B.indexer_topk(q, kI, w, k))[0]
    for t in (0, 5, 199, 200, 1099):
        n = min(k, t + 1)
        assert idx[t].tolist() == list(range(n)) + [-1] * (k - n)


# ---------------------------------------------------------------------------
# Decode path (few rows): score rows in the workspace + radix select.
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("Bn,T,S,S_cap,q_pos0,k,kd", [
    (4, 1, 5000, 5000, 4999, 2048, "bf16"),
    (4, 1, 5000, 5100, 4999, 2048, "e4m3"),
    (2, 3, 4003, 4100, 4000, 16, "bf16"),
    (3, 1, 100, 100, 99, 2048, "bf16"),      # fewer causal keys than k
    (1, 8, 3008, 3008, 3000, 500, "e4m3"),
    (2, 1, 2049, 2100, 2048, 2048, "e4m3"),  # one key more than k: a cut of one, 4-CTA clusters of ~512 keys
])
def test_indexer_decode_path(Bn, T, S, S_cap, q_pos0, k, kd):
    cfg = synth.StackConfig("dec", 1, "F", Bn, T, S, 64, 128, k, 32, 128, kd, "normal", q_pos0)
    q, kI, ks, w = synth.make_indexer_inputs(cfg, 0, 91, DEV, S=S_cap)
    idx = B.indexer_topk(q, kI, w, k, q_pos0, kscale=ks, S=S)
    torch.cuda.synchronize()
    got = _idx64(idx)
    stats = {"hit": 0, "tot": 0}
    for b in range(Bn):
        pu.check_topk(got[b], pu.to_f64(q[b]), pu.keys_f64(kI[b, :S], None if ks is None else ks[b, :S]),
                      pu.to_f64(w[b]), k, q_pos0, range(T), exact=False, stats=stats)
    pu.check_recall(stats)


@pytest.mark.parametrize("Bn,S,k,mode", [(3, 1300, 256, "codes"), (2, 777, 100, "int"), (5, 4099, 2048, "codes")])
def test_decode_e4m3_every_code(Bn, S, k, mode):
    # decode keys drawn from every e4m3 code but NaN (zeros, subnormals, the
    # largest magnitudes) exercise the exact widening to bf16 in the kernel
    g = torch.Generator(device="cpu").manual_seed(17)
    codes = torch.tensor([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=torch.uint8)
    kb = codes[torch.randint(0, len(codes), (Bn, S, 128), generator=g)]
    if mode == "int":
        # small integers: exact products, bit-exact selection
        ints = torch.tensor([0x00, 0x38, 0x40, 0x44, 0xB8, 0xC0, 0xC4], dtype=torch.uint8)   # 0, 1, 2, 3, -1, -2, -3
        kb = ints[torch.randint(0, len(ints), (Bn, S, 128), generator=g)]
        q = torch.randint(-2, 3, (Bn, 1, 64, 128), generator=g).float()
        w = torch.randint(-2, 3, (Bn, 1, 64), generator=g).float()
        ks = torch.ones(Bn, S)
    else:
        q = torch.randn(Bn, 1, 64, 128, generator=g) / 11.3
        w = torch.randn(Bn, 1, 64, generator=g) / 8
        ks = torch.rand(Bn, S, generator=g) * 0.01 + 1e-3
    kI = kb.view(torch.float8_e4m3fn).to(DEV)
    q, w, ks = q.to(DEV, torch.bfloat16), w.to(DEV), ks.to(DEV)
    idx = B.indexer_topk(q, kI, w, k, S - 1, kscale=ks, S=S)
    torch.cuda.synchronize()
    got = _idx64(idx)
    stats = {"hit": 0, "tot": 0}
    for b in range(Bn):
        pu.check_topk(got[b], pu.to_f64(q[b]), pu.keys_f64(kI[b], ks[b]), pu.to_f64(w[b]), k, S - 1, [0],
                      exact=(mode == "int"), stats=stats)
    if mode != "int":
        pu.check_recall(stats)


@pytest.mark.parametrize("S,n_top,top_val", [
    (20000, 0, 0.0),        # every score equal: the threshold bin holds the whole row
    (6000, 2500, 1.0),      # more tied top scores than k, all within the candidate buffer
    (30000, 9000, 2.0),     # more tied top scores than the candidate buffer holds
])
def test_decode_select_ties(S, n_top, top_val):
    # score = ReLU(kI[s, 0]) through head 0 only; ties go to the lower positions
    k, Bn = 2048, 2
    g = torch.Generator(device="cpu").manual_seed(S)
    q = torch.zeros(Bn, 1, 64, 128)
    q[:, 0, 0, 0] = 1.0
    kI = torch.zeros(Bn, S, 128)
    for b in range(Bn):
        kI[b, torch.randperm(S, generator=g)[:n_top], 0] = top_val
        kI[b, torch.randperm(S, generator=g)[:S // 3], 1] = 0.5     # head 0 ignores feature 1
    w = torch.zeros(Bn, 1, 64)
    w[:, 0, 0] = 1.0
    q, kI, w = q.to(DEV, torch.bfloat16), kI.to(DEV, torch.bfloat16), w.to(DEV)
    got = _idx64(B.indexer_topk(q, kI, w, k, S - 1, S=S))
    torch.cuda.synchronize()
    for b in range(Bn):
        pu.check_topk(got[b], pu.to_f64(q[b]), pu.to_f64(kI[b]), pu.to_f64(w[b]), k, S - 1, [0], exact=True)


@pytest.mark.parametrize("S", [40000, 300007])
def test_decode_select_paths_agree(S):
    # the clustered select (workspace with the histogram) and
    # the one-CTA select (workspace of the score rows only) pick the same rows;
    # at 300007 keys each CTA of a cluster copies and lists its quarter of the
    # row in three passes, the last one ragged
    dc = synth.DECODE.with_(B=3)
    q, kI, ks, w = synth.make_indexer_inputs(dc, 0, 23, DEV, T=1, S=S)
    full = _idx64(B.indexer_topk(q, kI, w, 2048, S - 1, kscale=ks, S=S))
    small_ws = torch.empty(3 * ((S + 3) // 4) * 4 * 4, dtype=torch.uint8, device=DEV)
    small = _idx64(B.indexer_topk(q, kI, w, 2048, S - 1, kscale=ks, S=S, ws=small_ws))
    torch.cuda.synchronize()
    assert np.array_equal(full, small)
    stats = {"hit": 0, "tot": 0}
    for b in range(3):
        pu.check_topk(full[b], pu.to_f64(q[b]), pu.keys_f64(kI[b], ks[b]), pu.to_f64(w[b]), 2048, S - 1, [0],
                      exact=False, stats=stats)
    pu.check_recall(stats)


def test_decode_matches_prefill_row():
    # the decode kernels at position p give the prefill kernel's row p
    cfg = synth.StackConfig("x", 1, "F", 1, 1200, 1200, 64, 128, 128, 32, 128)
    q, kI, _, w = synth.make_indexer_inputs(cfg, 0, 5, DEV)
    full = _idx64(B.indexer_topk(q, kI, w, 128))[0]
    for p in (0, 127, 128, 700, 1199):
        dec = _idx64(B.indexer_topk(q[:, p:p + 1].contiguous(), kI, w[:, p:p + 1].contiguous(), 128, p, S=p + 1))
        assert np.array_equal(dec[0, 0], full[p])


# ---------------------------------------------------------------------------
# Sparse attention.
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("Bn,T,S,Hq,Dh,k", [
    (1, 400, 3000, 32, 128, 2048),   # many rows: one CTA per row
    (2, 300, 900, 4, 64, 100),
    (32, 1, 5000, 32, 128, 2048),    # few rows: split over the k rows + merge
    (3, 2, 700, 16, 64, 333),
])
def test_sparse_attention(Bn, T, S, Hq, Dh, k):
    g = torch.Generator(device=DEV).manual_seed(3)
    Q = torch.randn(Bn, T, Hq, Dh, device=DEV, generator=g).to(torch.bfloat16)
    K = torch.randn(Bn, S, Dh, device=DEV, generator=g).to(torch.bfloat16)
    V = torch.randn(Bn, S, Dh, device=DEV, generator=g).to(torch.bfloat16)
    idx = torch.stack([torch.stack([torch.randperm(S, device=DEV, generator=g)[:k] for _ in range(T)])
                       for _ in range(Bn)]).to(torch.int32)
    # -1 holes, a short row and an empty row
    idx[:, :, ::7] = -1
    if T > 1:
        idx[0, 1, 5:] = -1
        idx[0, 0, :] = -1
    O = B.sparse_attn(Q, K, V, idx)
    torch.cuda.synchronize()
    for b in range(Bn):
        pu.check_attention(O[b], Q[b], K[b], V[b], idx[b], 1.0 / math.sqrt(Dh))
    if T > 1:
        assert torch.all(O[0, 0] == 0)


def _attn_case(Bn, T, S, S_cap, k, mode, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    Q = torch.randn(Bn, T, 32, 128, device=DEV, generator=g)
    K = torch.randn(Bn, S_cap, 128, device=DEV, generator=g)
    V = torch.randn(Bn, S_cap, 128, device=DEV, generator=g)
    idx = torch.stack([torch.stack([torch.sort(torch.randperm(S, device=DEV, generator=g)[:k]).values
                                    for _ in range(T)]) for _ in range(Bn)]).to(torch.int32)
    if mode == "growing":
        # key magnitude grows with position: later tiles beat the running max by
        # far more than the lazy-rescale threshold, again and again
        K = K * torch.linspace(0.05, 4.0, S_cap, device=DEV)[None, :, None]
    elif mode == "spike":
        # one late key aligned with every head's query dominates the softmax
        sel = idx[:, :, -1].long()
        for b in range(Bn):
            K[b, sel[b]] = Q[b].mean(1) * 6.0
    elif mode == "masked_head":
        # the first tile of every row is empty, the rest valid, some rows empty
        idx[:, :, :128] = -1
        idx[:, ::9, :] = -1
        idx[:, 1::5, 200:260] = S + 7    # outside [0, S): empty slots too
    return Q.to(torch.bfloat16), K.to(torch.bfloat16), V.to(torch.bfloat16), idx


@pytest.mark.parametrize("Bn,T,S,S_cap,k,mode", [
    (32, 1, 5000, 5100, 2048, "normal"),      # the decode workload's shape: 32 rows, k = 2048
    (5, 2, 3000, 3000, 333, "normal"),        # k not a multiple of the 64-position chunk, two rows per sequence
    (3, 1, 700, 700, 100, "spike"),           # one dominant key
    (4, 1, 2000, 2000, 1024, "growing"),      # later splits hold the larger scores
    (6, 1, 3000, 3000, 512, "masked_head"),   # an empty first chunk, empty rows, out-of-range slots
    (3, 1, 4000, 4000, 1152, "growing"),      # 9 tiles of 128 keys shared 3 + 3 + 3 among CTAs
    (7, 1, 2500, 2600, 644, "spike"),         # 6 tiles, the last with 4 keys, shared 2 + 2 + 2
    (8, 1, 3000, 3000, 2048, "growing"),      # 16 tiles shared by a cluster of 8 CTAs, 2 each
    (30, 2, 2500, 2500, 2048, "normal"),      # 60 rows: clusters of 2 CTAs, 8 tiles each
])
def test_decode_attention_split_cases(Bn, T, S, S_cap, k, mode):
    # few rows: the k positions are split across CTAs and the splits merged
    # (in a thread block cluster per row: clusters of 2, 3, 4 and 8 CTAs here)
    Q, K, V, idx = _attn_case(Bn, T, S, S_cap, k, mode, 19)
    O = B.sparse_attn(Q, K, V, idx, S=S)
    torch.cuda.synchronize()
    B.stream_status()
    idx_o = torch.where((idx >= 0) & (idx < S), idx, torch.full_like(idx, -1))
    for b in range(Bn):
        pu.check_attention(O[b], Q[b], K[b, :S], V[b, :S], idx_o[b], 1.0 / math.sqrt(128))
    if mode == "masked_head":
        assert torch.all(O[:, ::9] == 0)


@pytest.mark.parametrize("Bn,T,S,S_cap,k,mode", [
    (1, 296, 5000, 5000, 2048, "normal"),     # tensor-core path at its smallest row count
    (2, 200, 3000, 3100, 300, "normal"),      # k not a multiple of the 128-key tile, S_cap > S
    (1, 400, 6000, 6000, 2048, "growing"),    # the reference max rises tile after tile
    (1, 300, 4000, 4000, 1024, "spike"),      # one dominant late key
    (2, 160, 3000, 3000, 512, "masked_head"), # leading empty tile, empty rows, out-of-range slots
])
def test_sparse_attention_tensor_core_cases(Bn, T, S, S_cap, k, mode):
    Q, K, V, idx = _attn_case(Bn, T, S, S_cap, k, mode, 11)
    O = B.sparse_attn(Q, K, V, idx, S=S)
    torch.cuda.synchronize()
    B.stream_status()
    rows = sorted(set([0, 1, 2, T - 1] + list(range(3, T, max(1, T // 40)))))
    # the C ABI treats any index outside [0, S) as an empty slot, i.e. as -1
    idx_o = torch.where((idx >= 0) & (idx < S), idx, torch.full_like(idx, -1))
    for b in range(Bn):
        pu.check_attention(O[b], Q[b], K[b, :S], V[b, :S], idx_o[b], 1.0 / math.sqrt(128), rows=rows)
    if mode == "masked_head":
        assert torch.all(O[:, ::9] == 0)


# ---------------------------------------------------------------------------
# Whole stacks.
# ---------------------------------------------------------------------------


def _stack_check(cfg, layers, sample_rows, base_seed, q_pos0=0, S=None):
    """Per-F-layer indices through ic_indexer_topk + the forward through
    ic_forward_pattern; sampled rows against the oracle."""
    S = cfg.S if S is None else S
    per_f = {}
    stats = {"hit": 0, "tot": 0}
    for l, c in enumerate(cfg.pattern):
        if c != "F":
            continue
        L = layers[l]
        idx = B.indexer_topk(L["q"], L["kI"], L["w"], cfg.k, q_pos0, kscale=L["kscale"], S=S)
        torch.cuda.synchronize()
        per_f[l] = idx.clone()
        for b in range(cfg.B):
            pu.check_topk(_idx64(idx)[b], pu.to_f64(L["q"][b]),
                          pu.keys_f64(L["kI"][b, :S], None if L["kscale"] is None else L["kscale"][b, :S]),
                          pu.to_f64(L["w"][b]), cfg.k, q_pos0, sample_rows, exact=(cfg.dist == "int"),
                          stats=stats)
    if cfg.dist != "int":
        pu.check_recall(stats)
    cache, calls = B.forward_pattern(cfg.pattern, layers, cfg.k, q_pos0, S)
    torch.cuda.synchronize()
    assert calls == cfg.pattern.count("F")
    last_f = max(per_f)
    assert torch.equal(cache, per_f[last_f])
    f = 0
    for l, c in enumerate(cfg.pattern):
        f = l if c == "F" else f
        L = layers[l]
        for b in range(cfg.B):
            pu.check_attention(L["O"][b], L["Q"][b], L["K"][b, :S], L["V"][b, :S], per_f[f][b], cfg.scale,
                               rows=sample_rows)


def _sample_rows(T, k, n_rand, seed):
    rng = np.random.default_rng(seed)
    fixed = [0, 1, k - 2, k - 1, k, k + 1, T - 2, T - 1]
    rows = sorted(set([r for r in fixed if 0 <= r < T] + rng.integers(0, T, n_rand).tolist()))
    return rows


def test_short_stack_sampled():
    cfg = synth.SHORT
    layers = synth.make_stack(cfg, 2024, DEV)
    _stack_check(cfg, layers, _sample_rows(cfg.T, cfg.k, 24, 1), 2024)


@pytest.mark.slow
@pytest.mark.parametrize("kd", ["bf16", "e4m3"])
def test_prefill32k_full_size_sampled(kd):
    # the 30B-shaped workload's sizes (L = 32768, H_I = 64, d_I = 128, k = 2048,
    # 32 query heads of dim 128) and launch configuration, on five of its layers
    cfg = synth.PREFILL_32K.with_(n_layers=5, pattern="FSSSF", k_dtype=kd)
    layers = synth.make_stack(cfg, 31337, DEV)
    _stack_check(cfg, layers, _sample_rows(cfg.T, cfg.k, 10, 2), 31337)


@pytest.mark.slow
def test_decode_full_size_sampled():
    # 32 sequences at context 131072 (plus the new token), fp8 keys; checks 4 sequences
    cfg = synth.DECODE.with_(n_layers=2, pattern="FS")
    S = cfg.S
    layers = synth.make_stack(cfg, 4242, DEV, T=1, S=S)
    idx = B.indexer_topk(layers[0]["q"], layers[0]["kI"], layers[0]["w"], cfg.k, cfg.q_pos0,
                         kscale=layers[0]["kscale"], S=S)
    torch.cuda.synchronize()
    got = _idx64(idx)
    stats = {"hit": 0, "tot": 0}
    for b in (0, 9, 20, 31):
        L = layers[0]
        pu.check_topk(got[b], pu.to_f64(L["q"][b]), pu.keys_f64(L["kI"][b], L["kscale"][b]), pu.to_f64(L["w"][b]),
                      cfg.k, cfg.q_pos0, [0], exact=False, stats=stats)
    pu.check_recall(stats)
    cache, calls = B.forward_pattern(cfg.pattern, layers, cfg.k, cfg.q_pos0, S)
    torch.cuda.synchronize()
    assert calls == 1 and torch.equal(cache, idx)
    for l in range(2):
        L = layers[l]
        for b in (0, 31):
            pu.check_attention(L["O"][b], L["Q"][b], L["K"][b], L["V"][b], idx[b], cfg.scale)


@pytest.mark.slow
@pytest.mark.parametrize("chunk", [0, 12, 24])
def test_long_chunk_sampled(chunk):
    # the first, a middle and the last 8192-query chunk of the 204800-token
    # prefill (queries over the whole causal prefix), fp8 keys
    cfg = synth.LONG.with_(n_layers=2, pattern="FS", T=8192)
    q_pos0 = chunk * 8192
    layers = synth.make_stack(cfg, 555 + chunk, DEV, T=8192, S=204800)
    rows = _sample_rows(8192, 2048 if chunk == 0 else 0, 6, 3 + chunk)
    _stack_check(cfg, layers, rows, 555 + chunk, q_pos0=q_pos0, S=204800)


def test_bad_pattern_launches_nothing():
    cfg = synth.TINY
    layers = synth.make_stack(cfg, 1, DEV)
    for L in layers:
        L["O"] = torch.full_like(L["Q"], 7.0)
    cache = torch.full((1, cfg.T, cfg.k), 12345, dtype=torch.int32, device=DEV)
    for bad in ("SSSF", "FSX F"[:4], "FS", "1001"):
        with pytest.raises(ValueError):
            B.forward_pattern(bad, layers, cfg.k, index_cache=cache)
    torch.cuda.synchronize()
    assert torch.all(cache == 12345)
    assert all(torch.all(L["O"] == 7.0) for L in layers)
    B.stream_status()
