"""Query-row sharding on CPU: the zig-zag row split and the key-side
all-gather, the latter as two gloo ranks on 127.0.0.1 (no GPU)."""

import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

from cross_layer_top_indexer_b300 import sharding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("L,world", [(8, 2), (8192, 2), (32768, 4), (204800, 8), (1001, 3), (204800, 2)])
def test_zigzag_split_covers_every_row_once(L, world):
    seen = torch.zeros(L, dtype=torch.int32)
    for r in range(world):
        rr = sharding.rank_rows(L, world, r)
        assert len(rr) == 2 and rr[0][0] < rr[1][0]
        for q0, T in rr:
            assert T >= 1
            seen[q0:q0 + T] += 1
    assert torch.all(seen == 1)
    chunks = sharding.zigzag_chunks(L, world)
    assert chunks[0][0] == 0 and sum(T for _, T in chunks) == L
    assert all(a[0] + a[1] == b[0] for a, b in zip(chunks, chunks[1:]))


@pytest.mark.parametrize("L,world", [(32768, 2), (32768, 8), (204800, 8)])
def test_zigzag_split_balances_causal_work(L, world):
    work = [sharding.causal_pairs(sharding.rank_rows(L, world, r)) for r in range(world)]
    assert sum(work) == L * (L + 1) // 2
    # contiguous blocks would differ by a factor of about 2*world - 1
    assert max(work) / min(work) < 1.01


def test_split_refuses_too_few_rows():
    with pytest.raises(ValueError):
        sharding.zigzag_chunks(3, 2)
    with pytest.raises(ValueError):
        sharding.rank_rows(100, 2, 2)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _full(B, L, D, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    if dtype == torch.uint8:
        return torch.randint(0, 256, (B, L, D), generator=g, dtype=torch.int32).to(torch.uint8)
    return torch.randn(B, L, D, generator=g).to(dtype)


def _rank_main(rank, world, port, out_dir):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "MASTER_ADDR": "127.0.0.1",
                       "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    from cross_layer_top_indexer_b300 import sharding as sh
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ok = []
    for L, B, D, dtype in ((1001, 2, 128, torch.bfloat16), (4096, 1, 128, torch.uint8), (64, 3, 1, torch.float32)):
        full = _full(B, L, D, dtype, 7 + L)              # every rank can build the expected result
        mine = sh.rank_rows(L, world, rank)
        local = sh.take_rows(full, mine)                 # the key rows this rank produced
        got = sh.all_gather_rows(local, L, world, rank)
        ok.append(bool(torch.equal(got, full)))
    dist.barrier()
    dist.destroy_process_group()
    with open(os.path.join(out_dir, "rank%d.txt" % rank), "w") as f:
        f.write(",".join(str(x) for x in ok))


def test_all_gather_two_gloo_ranks(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    for r in range(world):
        assert open(tmp_path / ("rank%d.txt" % r)).read() == "True,True,True"
