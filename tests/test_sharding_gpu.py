"""Query-row sharding on one GPU: the per-rank row ranges of a zig-zag
split, each run as its own ic_forward_pattern call (q_pos0 at the range
start), give bit for bit the index cache and every layer's output of the
unsharded forward on those rows."""

import pytest
import torch

from cross_layer_top_indexer_b300 import binding as B
from cross_layer_top_indexer_b300 import sharding
from cross_layer_top_indexer_b300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.load()


@pytest.mark.parametrize("kd,world", [("bf16", 2), ("e4m3", 4)])
def test_sharded_rows_equal_unsharded(kd, world):
    # the short workload's shapes (tensor-core indexer and attention), 4 layers FSSF
    cfg = synth.SHORT.with_(n_layers=4, pattern="FSSF", T=4096, S=4096, k_dtype=kd)
    layers = synth.make_stack(cfg, 808, DEV)
    cache, _ = B.forward_pattern(cfg.pattern, layers, cfg.k)
    torch.cuda.synchronize()
    want_idx = cache.clone()
    want_O = [L["O"].clone() for L in layers]
    for r in range(world):
        ranges = sharding.rank_rows(cfg.T, world, r)
        res = sharding.forward_rows(B, cfg.pattern, layers, cfg.k, ranges)
        torch.cuda.synchronize()
        for (q0, T), (idx, outs) in zip(ranges, res):
            assert torch.equal(idx, want_idx[:, q0:q0 + T]), (r, q0)
            for l in range(cfg.n_layers):
                assert torch.equal(outs[l], want_O[l][:, q0:q0 + T]), (r, q0, l)
    B.stream_status()
