"""Decode steps captured in a CUDA graph give, bit for bit, what the same
calls give launched one by one: three steps of (append the new token's rows,
forward the FSSF stack at the new position).  The decode kernels start early
on the stream (programmatic dependent launch) and read their inputs only
after the kernel before them has completed; the graph keeps those edges."""

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


def _new_rows(cfg, pattern, seed):
    rows = []
    for l in range(len(pattern)):
        src = synth.make_indexer_inputs(cfg, l, seed, DEV, T=1, S=1)
        kv = synth.make_attn_inputs(cfg, l, seed, DEV, T=1, S=1)
        rows.append({
            "kI": src[1][:, 0].contiguous() if pattern[l] == "F" else None,
            "kscale": src[2][:, 0].contiguous() if (pattern[l] == "F" and src[2] is not None) else None,
            "K": kv[1][:, 0].contiguous(),
            "V": kv[2][:, 0].contiguous(),
        })
    return rows


@pytest.mark.parametrize("kd", ["e4m3", "bf16"])
def test_decode_steps_graph_equals_eager(kd):
    pattern, steps = "FSSF", 3
    Bn, S_cap, pos0, k = 4, 4096, 3000, 512
    cfg = synth.StackConfig("graph", 4, pattern, Bn, 1, S_cap, 64, 128, k, 32, 128, kd, "normal", q_pos0=pos0)
    layers = synth.make_stack(cfg, 77, DEV, T=1, S=S_cap)
    for L in layers:
        L["O"] = torch.empty_like(L["Q"])
    cached = ("kI", "kscale", "K", "V")
    start = [{n: (L[n].clone() if L.get(n) is not None else None) for n in cached} for L in layers]
    kdt = B.IC_E4M3 if kd == "e4m3" else B.IC_BF16
    apps = [B.DecodeAppend(pattern, layers, _new_rows(cfg, pattern, 300 + s), kdt) for s in range(steps)]
    fwds = [B.Forward(pattern, layers, k, q_pos0=pos0 + s, S=pos0 + s + 1) for s in range(steps)]
    st = torch.cuda.Stream()

    def reset():
        for L, S0 in zip(layers, start):
            for n in cached:
                if S0[n] is not None:
                    L[n].copy_(S0[n])
        torch.cuda.synchronize()

    def run():
        for s in range(steps):
            apps[s](pos0 + s, stream=st)
            fwds[s](stream=st)

    def results():
        return ([f.index_cache.clone() for f in fwds], [L["O"].clone() for L in layers],
                [L[n].clone() for L in layers for n in cached if L.get(n) is not None])

    reset()
    with torch.cuda.stream(st):
        run()
    st.synchronize()
    B.stream_status(st)
    eager = results()

    reset()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        run()
    reset()
    g.replay()
    torch.cuda.synchronize()
    B.stream_status(st)
    replay = results()

    for s, (a, b) in enumerate(zip(eager[0], replay[0])):
        assert torch.equal(a, b), ("index cache", s)
        assert (a >= 0).all() and (a <= pos0 + s).all()
    for l, (a, b) in enumerate(zip(eager[1], replay[1])):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), ("O", l)
    for i, (a, b) in enumerate(zip(eager[2], replay[2])):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), ("cache", i)
