"""The allocation-free indexer entry point, ic_indexer_topk_noalloc.

It is meant for callers that cannot call cudaMalloc where they run the
indexer (a server whose memory manager owns all free device memory, a plugin
without its host's allocator, a loop that must not take cudaMalloc's device
synchronisation).  Its scratch is a fixed device array inside the library, so
this test checks, through the C ABI:

* every case runs twice in a row, after a decoy call of other sizes that
  leaves different scores in the shared array, and both calls give exactly
  the indices of ic_indexer_topk with a caller workspace;
* one case on integer inputs is exact against the CPU oracle as well;
* a case near the array's limit (the score rows fit, the score-key
  histogram of the clustered select does not) takes the select path that
  histograms the score row itself;
* sizes past the array are refused without touching the output.

Kept in its own file, collected last, so a failure here never hides the
other tests' results; it passes alone in a fresh process or after them.
"""

import numpy as np
import pytest
import torch

from cross_layer_top_indexer_b300 import binding as B
from cross_layer_top_indexer_b300 import synth
from tests import parity_util as pu

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _inputs(Bn, T, S, S_cap, q_pos0, k, kd, seed, dist="normal"):
    cfg = synth.StackConfig("noalloc", 1, "F", Bn, T, S, 64, 128, k, 32, 128, kd, dist, q_pos0)
    return synth.make_indexer_inputs(cfg, 0, seed, DEV, S=S_cap)


def _noalloc(lib, q, kI, ks, w, k, q_pos0, S, out):
    Bn, T, H, D = q.shape
    kd = B.IC_E4M3 if kI.dtype == torch.float8_e4m3fn else B.IC_BF16
    return lib.ic_indexer_topk_noalloc(Bn, T, S, kI.shape[1], H, D, k, q_pos0, q.data_ptr(), kI.data_ptr(), kd,
                                       None if ks is None else ks.data_ptr(), w.data_ptr(), out.data_ptr(),
                                       torch.cuda.current_stream().cuda_stream)


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return B.load()


CASES = [
    # B, T, S, S_cap, q_pos0, k, key dtype, seed
    (8, 1, 30001, 30100, 30000, 2048, "e4m3", 11),
    (3, 2, 9002, 9002, 9000, 512, "bf16", 12),
    (32, 1, 261000, 261000, 260999, 2048, "e4m3", 15),   # the score rows fit, the histogram does not
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B%d_T%d_S%d" % (c[0], c[1], c[2]))
def test_noalloc_matches_workspace_entry_twice_in_a_row(lib, case):
    Bn, T, S, S_cap, q_pos0, k, kd, seed = case
    q, kI, ks, w = _inputs(Bn, T, S, S_cap, q_pos0, k, kd, seed)
    want = B.indexer_topk(q, kI, w, k, q_pos0, kscale=ks, S=S)
    # decoy: other sizes and values, so the array holds different scores
    dq, dk, dks, dw = _inputs(4, 1, 7001, 7001, 7000, 300, "bf16", seed + 100)
    dout = torch.empty((4, 1, 300), dtype=torch.int32, device=DEV)
    assert _noalloc(lib, dq, dk, dks, dw, 300, 7000, 7001, dout) == B.IC_OK, lib.ic_last_error()
    for _ in range(2):
        got = torch.full_like(want, -7)
        assert _noalloc(lib, q, kI, ks, w, k, q_pos0, S, got) == B.IC_OK, lib.ic_last_error()
        torch.cuda.synchronize()
        assert torch.equal(got, want)
    B.stream_status()


def test_noalloc_exact_against_the_oracle(lib):
    Bn, T, S, q_pos0, k = 2, 1, 3000, 2999, 256
    q, kI, ks, w = _inputs(Bn, T, S, S, q_pos0, k, "bf16", 16, dist="int")
    out = torch.full((Bn, T, k), -7, dtype=torch.int32, device=DEV)
    assert _noalloc(lib, q, kI, ks, w, k, q_pos0, S, out) == B.IC_OK, lib.ic_last_error()
    torch.cuda.synchronize()
    for b in range(Bn):
        pu.check_topk(out[b].cpu().numpy().astype(np.int64), pu.to_f64(q[b]), pu.keys_f64(kI[b], None),
                      pu.to_f64(w[b]), k, q_pos0, [0], exact=True)


def test_noalloc_refuses_sizes_past_the_array(lib):
    q, kI, ks, w = _inputs(32, 1, 300000, 300000, 299999, 2048, "e4m3", 13)   # 38.4 MB of score rows
    out = torch.full((32, 1, 2048), -7, dtype=torch.int32, device=DEV)
    code = _noalloc(lib, q, kI, ks, w, 2048, 299999, 300000, out)
    assert code == B.IC_ERR_UNSUPPORTED
    assert b"scratch" in lib.ic_last_error()
    q9, kI9, ks9, w9 = _inputs(1, 9, 1009, 1009, 1000, 64, "bf16", 14)
    out9 = torch.full((1, 9, 64), -7, dtype=torch.int32, device=DEV)
    assert _noalloc(lib, q9, kI9, ks9, w9, 64, 1000, 1009, out9) == B.IC_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.all(out == -7) and torch.all(out9 == -7)
