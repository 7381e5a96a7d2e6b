"""The N > 1 path of bench.py on CPU: two gloo ranks on 127.0.0.1.

bench.py runs N independent replicas (the path shards by sequence with no
data-path exchange); what the ranks share is the rendezvous, the barriers
around the timed region and the max over ranks of the timed milliseconds.
These run here as two spawned processes, without a GPU.
"""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    w, r, local = bench.dist_setup()
    res = {"world": w, "rank": r, "local": local, "backend": dist.get_backend()}
    bench.barrier(w)
    # the timed milliseconds differ per rank; every rank must see the maximum
    res["max_ms"] = bench.reduce_max(10.0 + 5.0 * r, w)
    bench.barrier(w)
    # the reference arm prints from rank 0 only; other ranks return at once
    if r != 0:
        bench.reference_arm(None, w, r)
        res["reference_silent"] = True
    dist.destroy_process_group()
    with open(os.path.join(out_dir, "rank%d.json" % r), "w") as f:
        json.dump(res, f)


def test_two_gloo_ranks(tmp_path):
    world = 2
    port = _free_port()
    mp.start_processes(_rank_main, args=(world, port, str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    res = [json.load(open(tmp_path / ("rank%d.json" % r))) for r in range(world)]
    for r, d in enumerate(res):
        assert d["world"] == world and d["rank"] == r and d["local"] == r
        assert d["backend"] == "gloo"
        assert d["max_ms"] == pytest.approx(15.0)       # max over ranks, on every rank
    assert res[1].get("reference_silent")


def test_cli_reference_arm_rank1_prints_nothing():
    # under torchrun only rank 0 prints the reference arm's line; rank 1 of a
    # two-rank launch exits 0 without work (simulated with the rank's env
    # and WORLD_SIZE=1 so that no rendezvous is needed)
    env = dict(os.environ, RANK="1", WORLD_SIZE="1", LOCAL_RANK="1", CUDA_VISIBLE_DEVICES="")
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], env=env, capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stderr[-2000:]
    assert p.stdout.strip() == ""
