"""One hot-path call on a seeded synthetic case, repeated: a small, bounded
target for a profiler (a few GB on the device at most).

    python -m cross_layer_top_indexer_b300.profile_case CASE [--reps N]

Cases (shapes of the workloads, sizes kept small enough to capture):
  indexer_prefill       L = 8192, H_I = 64, d_I = 128, bf16 keys, k = 2048
  indexer_prefill_e4m3  the same with e4m3 keys and per-key scales
  sparse_attn           L = 8192 query rows, 32 heads / 1 K/V head, dim 128, k = 2048
  decode_indexer        32 sequences, context 131073, e4m3 keys, k = 2048
  decode_attn           32 sequences, context 131073, one query row each, k = 2048
  indexer_prefill_32k   one Full layer of the L = 32768 stack (bf16 keys)
  sparse_attn_32k       one layer's attention of the L = 32768 stack

Each call is launched `--reps` times after two warm-up calls (so a
profiler skips the first launches with `-s`), and the run ends with a
stream synchronisation and the library's device status check.
"""

from __future__ import annotations

import argparse
import os
import sys

import torch

if __package__ in (None, ""):
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

from cross_layer_top_indexer_b300 import binding as B, synth  # noqa: E402

CASES = ("indexer_prefill", "indexer_prefill_e4m3", "sparse_attn", "decode_indexer", "decode_attn",
         "indexer_prefill_32k", "sparse_attn_32k")


def make_call(case: str, dev):
    k = 2048
    if case in ("indexer_prefill", "indexer_prefill_e4m3", "indexer_prefill_32k"):
        cfg = synth.PREFILL_32K if case.endswith("32k") else synth.SHORT
        cfg = cfg.with_(k_dtype="e4m3" if case.endswith("e4m3") else "bf16")
        q, kI, ks, w = synth.make_indexer_inputs(cfg, 0, 11, dev)
        out = torch.empty((cfg.B, cfg.T, k), dtype=torch.int32, device=dev)
        return lambda: B.indexer_topk(q, kI, w, k, kscale=ks, idx_out=out)
    if case in ("sparse_attn", "sparse_attn_32k"):
        cfg = synth.PREFILL_32K if case.endswith("32k") else synth.SHORT
        q, kI, _, w = synth.make_indexer_inputs(cfg, 0, 12, dev)
        idx = B.indexer_topk(q, kI, w, k)
        del q, kI, w
        Q, K, V = synth.make_attn_inputs(cfg, 0, 12, dev)
        O = torch.empty_like(Q)
        return lambda: B.sparse_attn(Q, K, V, idx, O=O)
    dc = synth.DECODE
    if case == "decode_indexer":
        q, kI, ks, w = synth.make_indexer_inputs(dc, 0, 13, dev, T=1, S=dc.S)
        out = torch.empty((dc.B, 1, k), dtype=torch.int32, device=dev)
        return lambda: B.indexer_topk(q, kI, w, k, dc.q_pos0, kscale=ks, S=dc.S, idx_out=out)
    if case == "decode_attn":
        q, kI, ks, w = synth.make_indexer_inputs(dc, 0, 14, dev, T=1, S=dc.S)
        idx = B.indexer_topk(q, kI, w, k, dc.q_pos0, kscale=ks, S=dc.S)
        del q, kI, ks, w
        Q, K, V = synth.make_attn_inputs(dc, 0, 14, dev, T=1, S=dc.S)
        O = torch.empty_like(Q)
        return lambda: B.sparse_attn(Q, K, V, idx, S=dc.S, O=O)
    raise ValueError("unknown case %r (one of %s)" % (case, ", ".join(CASES)))


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("case", choices=CASES)
    ap.add_argument("--reps", type=int, default=3)
    args = ap.parse_args(argv)
    B.load()
    dev = torch.device("cuda", 0)
    f = make_call(args.case, dev)
    torch.cuda.synchronize()
    for _ in range(2 + args.reps):
        f()
    torch.cuda.synchronize()
    B.stream_status()
    print("%s: %d calls done" % (args.case, 2 + args.reps))


if __name__ == "__main__":
    main()
