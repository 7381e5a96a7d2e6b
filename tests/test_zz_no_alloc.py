"""The allocation-free indexer entry point, ic_indexer_topk_noalloc.

It is meant for callers that cannot call cudaMalloc where they run the
indexer (a server whose memory manager owns all free device memory, a plugin
without its host's allocator, a loop that must not take cudaMalloc's device
synchronisation).  Its scratch is a fixed device array inside the library, so
this test checks, through the C ABI, that two calls in a row give exactly the
indices of ic_indexer_topk with a caller workspace, that the second call is
not disturbed by what the first left in the shared array, and that sizes past
the array are refused without touching the output.

Kept in its own file, collected last, so a failure here never hides the
other tests' results; it passes alone in a fresh process or after them.
"""

import ctypes

import pytest
import torch

from cross_layer_top_indexer_b300 import binding as B
from cross_layer_top_indexer_b300 import synth

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _inputs(Bn, T, S, S_cap, q_pos0, k, kd, seed):
    cfg = synth.StackConfig("noalloc", 1, "F", Bn, T, S, 64, 128, k, 32, 128, kd, "normal", q_pos0)
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


def test_noalloc_matches_workspace_entry_twice_in_a_row(lib):
    cases = [
        # B, T, S, S_cap, q_pos0, k, key dtype, seed
        (8, 1, 30001, 30100, 30000, 2048, "e4m3", 11),
        (3, 2, 9002, 9002, 9000, 512, "bf16", 12),   # smaller: stale scores of call 1 remain past S
    ]
    for Bn, T, S, S_cap, q_pos0, k, kd, seed in cases:
        q, kI, ks, w = _inputs(Bn, T, S, S_cap, q_pos0, k, kd, seed)
        want = B.indexer_topk(q, kI, w, k, q_pos0, kscale=ks, S=S)
        got = torch.full_like(want, -7)
        assert _noalloc(lib, q, kI, ks, w, k, q_pos0, S, got) == B.IC_OK, lib.ic_last_error()
        torch.cuda.synchronize()
        assert torch.equal(got, want)


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
