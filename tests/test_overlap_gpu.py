"""ic_overlap (cross-layer top-k overlap, deep-read page section
"相邻层重叠很高，但“重叠率”不是搜索目标") against the oracle's set-based
Overlap(a, b) = |I_a ∩ I_b| / k: exact counts on the indexer's own index
tensors (integer inputs with ties, an all-F run) and on hand-made rows with
-1 slots, repeats and any order."""

import numpy as np
import pytest
import torch

import oracle
from cross_layer_top_indexer_b300 import binding as B
from cross_layer_top_indexer_b300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.load()


def _check(a, b, k):
    ratio, cnt = B.overlap(a, b, k, counts=True)
    torch.cuda.synchronize()
    an = a.reshape(-1, a.shape[-1]).cpu().numpy()
    bn = b.reshape(-1, b.shape[-1]).cpu().numpy()
    want = oracle.overlap(an, bn, k)
    want_cnt = np.rint(want * k).astype(np.int64)
    got_cnt = cnt.reshape(-1).cpu().numpy().astype(np.int64)
    assert np.array_equal(got_cnt, want_cnt)
    got = ratio.reshape(-1).cpu().numpy().astype(np.float64)
    assert np.array_equal(got, (want_cnt / k).astype(np.float32).astype(np.float64))


def test_adjacent_layers_of_an_all_f_tiny_stack():
    cfg = synth.TINY
    idx = []
    for layer in range(cfg.n_layers):
        q, kI, ks, w = synth.make_indexer_inputs(cfg, layer, 21, DEV)
        idx.append(B.indexer_topk(q, kI, w, cfg.k, kscale=ks))
    for l in range(1, cfg.n_layers):
        _check(idx[l], idx[l - 1], cfg.k)
    _check(idx[0], idx[0], cfg.k)   # a layer with itself: every valid slot


@pytest.mark.parametrize("R,k,n_pos,seed", [(1, 1, 3, 0), (37, 16, 40, 1), (513, 100, 300, 2),
                                            (2000, 2048, 5000, 3), (64, 2048, 2100, 4)])
def test_unsorted_repeated_and_padded_rows(R, k, n_pos, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    a = torch.randint(-1, n_pos, (R, k), generator=g, dtype=torch.int32)
    b = torch.randint(-1, n_pos, (R, k), generator=g, dtype=torch.int32)
    a[:, : k // 3] = b[:, : k // 3].flip(-1)     # shared part, in another order
    a[0, :] = -1                                 # an empty row
    _check(a.to(DEV), b.to(DEV), k)
    # rows as the indexer writes them: ascending, -1 padded at the end
    sa = torch.sort(torch.where(a < 0, torch.full_like(a, 1 << 30), a), dim=-1).values
    sa = torch.where(sa == (1 << 30), torch.full_like(sa, -1), sa)
    _check(sa.to(DEV), b.to(DEV), k)


def test_full_size_prefill_layers_sampled():
    cfg = synth.SHORT
    k = cfg.k
    q0, kI0, _, w0 = synth.make_indexer_inputs(cfg, 0, 31, DEV)
    i0 = B.indexer_topk(q0, kI0, w0, k)
    q1, kI1, _, w1 = synth.make_indexer_inputs(cfg, 1, 31, DEV)
    i1 = B.indexer_topk(q1, kI1, w1, k)
    ratio, cnt = B.overlap(i0, i1, counts=True)
    torch.cuda.synchronize()
    rows = np.r_[0, 1, 2046, 2047, 2048, 4095, cfg.T - 1, np.random.default_rng(5).integers(0, cfg.T, 120)]
    a = i0[0].cpu().numpy()[rows]
    b = i1[0].cpu().numpy()[rows]
    want = np.rint(oracle.overlap(a, b, k) * k).astype(np.int64)
    assert np.array_equal(cnt[0].cpu().numpy()[rows].astype(np.int64), want)
    # rows below k select every causal key in both layers: overlap = (t + 1) / k
    t = np.arange(64)
    assert np.array_equal(cnt[0, :64].cpu().numpy(), t + 1)


def test_argument_errors():
    lib = B.load()
    a = torch.zeros((4, 16), dtype=torch.int32, device=DEV)
    r = torch.empty(4, dtype=torch.float32, device=DEV)
    assert lib.ic_overlap(0, 16, a.data_ptr(), a.data_ptr(), r.data_ptr(), None, None) == B.IC_ERR_ARG
    assert lib.ic_overlap(4, 4096, a.data_ptr(), a.data_ptr(), r.data_ptr(), None, None) == B.IC_ERR_UNSUPPORTED
    assert lib.ic_overlap(4, 16, a.data_ptr(), None, r.data_ptr(), None, None) == B.IC_ERR_ARG
