"""ic_decode_append: the new token's indexer key (Full layers only), its scale
and its K/V rows land at row `pos` of every sequence in every layer, nothing
else changes, and the decode query that follows sees them (a decode step
against the oracle)."""

import math

import numpy as np
import pytest
import torch

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


@pytest.mark.parametrize("kd", ["bf16", "e4m3"])
def test_append_then_decode_step(kd):
    pattern = "FSSF"
    Bn, S_cap, pos, k = 3, 600, 513, 64
    cfg = synth.StackConfig("append", 4, pattern, Bn, 1, S_cap, 64, 128, k, 32, 128, kd, "int", q_pos0=pos)
    layers = synth.make_stack(cfg, 91, DEV, T=1, S=S_cap)
    new = []
    for l in range(len(pattern)):
        R = {}
        src = synth.make_indexer_inputs(cfg, l, 191, DEV, T=1, S=1)
        R["kI"] = src[1][:, 0].contiguous() if pattern[l] == "F" else None
        R["kscale"] = src[2][:, 0].contiguous() if (pattern[l] == "F" and src[2] is not None) else None
        kv = synth.make_attn_inputs(cfg, l, 191, DEV, T=1, S=1)
        R["K"], R["V"] = kv[1][:, 0].contiguous(), kv[2][:, 0].contiguous()
        new.append(R)
    before = [{n: (t.clone() if t is not None else None) for n, t in L.items()} for L in layers]
    app = B.DecodeAppend(pattern, layers, new, B.IC_E4M3 if kd == "e4m3" else B.IC_BF16)
    app(pos)
    torch.cuda.synchronize()
    for l, (L, P, R) in enumerate(zip(layers, before, new)):
        for name in ("K", "V"):
            want = P[name].clone()
            want[:, pos] = R[name]
            assert torch.equal(L[name], want), (l, name)
        if pattern[l] == "F":
            want = P["kI"].clone()
            want[:, pos] = R["kI"]
            assert torch.equal(L["kI"].view(torch.uint8), want.view(torch.uint8)), l
            if kd == "e4m3":
                ws = P["kscale"].clone()
                ws[:, pos] = R["kscale"]
                assert torch.equal(L["kscale"], ws)
        for name in ("q", "w", "Q"):
            if L.get(name) is not None:
                assert torch.equal(L[name], P[name])
    # the decode step that follows: the query at `pos` sees its own key
    cache, calls = B.forward_pattern(pattern, layers, k, q_pos0=pos, S=pos + 1)
    torch.cuda.synchronize()
    assert calls == 2
    L3 = layers[3]
    for b in range(Bn):
        ks = None if L3["kscale"] is None else L3["kscale"][b, : pos + 1]
        pu.check_topk(cache[b].cpu().numpy().astype(np.int64), pu.to_f64(L3["q"][b]),
                      pu.keys_f64(L3["kI"][b, : pos + 1], ks), pu.to_f64(L3["w"][b]), k, pos, [0],
                      exact=(kd == "bf16"))   # e4m3: scaled keys round in fp32, the tolerance rule applies
        pu.check_attention(L3["O"][b], L3["Q"][b], L3["K"][b, : pos + 1], L3["V"][b, : pos + 1], cache[b],
                           1.0 / math.sqrt(128))


def test_append_refusals():
    lib = B.load()
    K = torch.zeros((2, 16, 128), dtype=torch.bfloat16, device=DEV)
    kI = torch.zeros((2, 16, 128), dtype=torch.bfloat16, device=DEV)
    L = {"kI": kI, "kscale": None, "Q": K, "K": K, "V": K, "O": K}
    R = {"kI": kI[:, 0].contiguous(), "K": K[:, 0].contiguous(), "V": K[:, 0].contiguous()}
    app = B.DecodeAppend("FS", [L, L], [R, R], B.IC_BF16)
    with pytest.raises(ValueError):
        app(16)          # pos == S_cap
    with pytest.raises(ValueError):
        app(-1)
    bad = B.DecodeAppend("FS", [dict(L, kI=None), L], [R, R], B.IC_BF16)
    with pytest.raises(ValueError):
        bad(3)           # a Full layer without its indexer cache
    ok_s = B.DecodeAppend("FS", [L, dict(L, kI=None)], [R, dict(R, kI=None)], B.IC_BF16)
    ok_s(3)              # a Shared layer needs none
    torch.cuda.synchronize()
    with pytest.raises(B.PatternError):
        B.DecodeAppend("SF", [L, L], [R, R], B.IC_BF16)(3)
