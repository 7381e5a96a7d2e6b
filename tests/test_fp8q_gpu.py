"""ic_indexer_topk_fp8: e4m3 queries and keys as stored on the f8f6f4 tensor
cores, against the oracle on the dequantised inputs (q8 * q_scale per
query head, k8 * k_scale per key row): bit-exact index sets on integer
codes with power-of-two scales, the tolerance rule and recall on quantised
random data, and the refusals."""

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
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.load()


def _deq(t8, scale):
    return oracle.dequantize_e4m3(synth.e4m3_bits(t8), scale.detach().cpu().numpy())


def _check(cfg, codes, seed, rows, q_pos0=0, S=None):
    S = cfg.S if S is None else S
    q8, qs, k8, ks, w = synth.make_fp8_indexer_inputs(cfg, 0, seed, DEV, S=S, codes=codes)
    idx = B.indexer_topk_fp8(q8, qs, k8, ks, w, cfg.k, q_pos0, S=S)
    torch.cuda.synchronize()
    B.stream_status()
    stats = {"hit": 0, "tot": 0}
    for b in range(cfg.B):
        pu.check_topk(idx[b].cpu().numpy().astype(np.int64), _deq(q8[b], qs[b]), _deq(k8[b], ks[b]),
                      pu.to_f64(w[b]), cfg.k, q_pos0, rows, exact=codes, stats=stats)
    if not codes:
        pu.check_recall(stats)


@pytest.mark.parametrize("T,k", [(512, 64), (1100, 300)])
def test_fp8q_integer_codes_bit_exact(T, k):
    cfg = synth.StackConfig("fp8q", 1, "F", 1, T, T, 64, 128, k, 32, 128, "e4m3", "int")
    rows = sorted(set([0, 1, k - 1, k, k + 1, T - 1] + list(range(7, T, max(1, T // 24)))))
    _check(cfg, True, 5, rows)


def test_fp8q_quantised_random_tolerance():
    cfg = synth.StackConfig("fp8q", 1, "F", 2, 2048, 2048, 64, 128, 256, 32, 128, "e4m3", "normal")
    rows = sorted(set([0, 255, 256, 1000, 2047] + np.random.default_rng(1).integers(0, 2048, 30).tolist()))
    _check(cfg, False, 6, rows)


def test_fp8q_short_workload_sampled_chunk():
    # the short workload's sizes, one 8192-row prefill chunk at q_pos0 = 8192 over a 16384-key prefix
    cfg = synth.SHORT.with_(T=8192, S=16384)
    rows = [0, 1, 4095, 8190, 8191] + np.random.default_rng(2).integers(0, 8192, 12).tolist()
    _check(cfg, False, 7, sorted(set(rows)), q_pos0=8192, S=16384)


def test_fp8q_refusals():
    lib = B.load()
    cfg = synth.StackConfig("fp8q", 1, "F", 1, 8, 64, 64, 128, 16, 32, 128, "e4m3", "int")
    q8, qs, k8, ks, w = synth.make_fp8_indexer_inputs(cfg, 0, 1, DEV, codes=True)
    out = torch.full((1, 8, 16), -7, dtype=torch.int32, device=DEV)
    args = lambda T, H, qsp: (1, T, 64, 64, H, 128, 16, 0, q8.data_ptr(), qsp, k8.data_ptr(), ks.data_ptr(),
                              w.data_ptr(), out.data_ptr(), None)
    assert lib.ic_indexer_topk_fp8(*args(8, 64, qs.data_ptr())) == B.IC_ERR_UNSUPPORTED     # decode rows
    assert lib.ic_indexer_topk_fp8(*args(8, 32, qs.data_ptr())) == B.IC_ERR_UNSUPPORTED
    assert lib.ic_indexer_topk_fp8(*args(8, 64, None)) == B.IC_ERR_ARG
    torch.cuda.synchronize()
    assert torch.all(out == -7)
