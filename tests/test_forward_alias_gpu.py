"""A Shared layer whose query buffer is the previous layer's output.

The forward lets a Shared layer's attention read its inputs before the
previous layer's attention has finished, unless that layer's output overlaps
them.  Here layer 1 takes layer 0's output O as its Q, so it must wait: the
forward has to give, bit for bit, what the two attention calls give one after
the other."""

import pytest
import torch

from cross_layer_top_indexer_b300 import binding as B
from cross_layer_top_indexer_b300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.load()


@pytest.mark.parametrize("Bn,T,S,k", [
    (8, 1, 4096, 512),       # decode shape: rows shared by the CTAs of a cluster
    (1, 320, 2048, 256),     # prefill shape: whole rows per CTA
])
def test_shared_layer_reads_previous_output(Bn, T, S, k):
    cfg = synth.StackConfig("alias", 2, "FS", Bn, T, S, 64, 128, k, 32, 128, "bf16", "normal", q_pos0=S - T)
    layers = synth.make_stack(cfg, 5, DEV, T=T, S=S)
    layers[0]["O"] = torch.empty_like(layers[0]["Q"])
    layers[1]["Q"] = layers[0]["O"]            # layer 1's query is layer 0's output
    layers[1]["O"] = torch.empty_like(layers[1]["Q"])
    for _ in range(3):                          # the race, were there one, need not show the first time
        fwd = B.Forward("FS", layers, k, q_pos0=S - T, S=S)
        fwd()
        torch.cuda.synchronize()
        B.stream_status()
        idx = fwd.index_cache
        o0 = B.sparse_attn(layers[0]["Q"], layers[0]["K"], layers[0]["V"], idx, S=S)
        o1 = B.sparse_attn(o0, layers[1]["K"], layers[1]["V"], idx, S=S)
        torch.cuda.synchronize()
        assert torch.equal(layers[0]["O"].view(torch.int16), o0.view(torch.int16))
        assert torch.equal(layers[1]["O"].view(torch.int16), o1.view(torch.int16))
