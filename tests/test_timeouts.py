"""Bounded device waits: a wait that runs out winds the kernel down cleanly.

The tensor-core prefill indexer bounds every wait on another part of the
kernel.  A debug limit of 1 ns (ic_debug_set_wait_limit_ns) makes its first
waits run out on purpose, without any fault, trap or endless loop: the call
must return, ic_stream_status must then report IC_ERR_DEVICE_TIMEOUT (and
clear it), and the next ordinary call on the same stream must be exact
against the oracle.
"""

import time

import numpy as np
import pytest
import torch

from tests import parity_util as pu
from cross_layer_top_indexer_b300 import binding as B
from cross_layer_top_indexer_b300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.load()


def test_prefill_indexer_wait_runs_out_then_recovers():
    lib = B.load()
    # integer inputs: exact scores, ties to the lower position (bit-exact parity)
    cfg = synth.StackConfig("timeout", 1, "F", 1, 1024, 1024, 64, 128, 64, 32, 128, "bf16", "int")
    q, kI, _, w = synth.make_indexer_inputs(cfg, 0, 77, DEV)
    out = torch.full((1, cfg.T, cfg.k), -7, dtype=torch.int32, device=DEV)
    stream = torch.cuda.current_stream()
    assert lib.ic_stream_status(stream.cuda_stream) == B.IC_OK
    assert lib.ic_debug_set_wait_limit_ns(1) == B.IC_OK
    try:
        t0 = time.perf_counter()
        B.indexer_topk(q, kI, w, cfg.k, idx_out=out, stream=stream)
        torch.cuda.synchronize()
        elapsed = time.perf_counter() - t0
        code = lib.ic_stream_status(stream.cuda_stream)
        msg = lib.ic_last_error()
    finally:
        assert lib.ic_debug_set_wait_limit_ns(0) == B.IC_OK
    assert code == B.IC_ERR_DEVICE_TIMEOUT, msg
    assert b"gave up" in msg
    assert elapsed < 30.0
    # the status word was cleared by the read above
    assert lib.ic_stream_status(stream.cuda_stream) == B.IC_OK
    # the same call again, default limits, same stream: exact against the oracle
    out.fill_(-7)
    B.indexer_topk(q, kI, w, cfg.k, idx_out=out, stream=stream)
    torch.cuda.synchronize()
    assert lib.ic_stream_status(stream.cuda_stream) == B.IC_OK
    rows = sorted(set([0, 1, 62, 63, 64, 65, 300, 511, 512, 1000, 1022, 1023]
                      + np.random.default_rng(3).integers(0, cfg.T, 40).tolist()))
    pu.check_topk(out[0].cpu().numpy().astype(np.int64), pu.to_f64(q[0]), pu.keys_f64(kI[0], None),
                  pu.to_f64(w[0]), cfg.k, 0, rows, exact=True)
