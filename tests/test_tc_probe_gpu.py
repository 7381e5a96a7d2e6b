"""One bf16 tile through the tensor-core plumbing (TMA with 128-byte swizzle,
UMMA shared-memory descriptors, tcgen05.mma into tensor memory, tcgen05.ld),
compared exactly with a matmul of integer-valued operands."""

import ctypes
import os
import subprocess

import pytest
import torch

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


@pytest.fixture(scope="module")
def probe(tmp_path_factory):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    out = str(tmp_path_factory.mktemp("probe") / "libtcprobe.so")
    cmd = ["/usr/local/cuda/bin/nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17",
           "-shared", "-Xcompiler", "-fPIC", "-I", os.path.join(ROOT, "include"),
           os.path.join(HERE, "cuda", "tc_tile_probe.cu"),
           os.path.join(ROOT, "cross_layer_top_indexer_b300", "csrc", "tmap.cu"), "-o", out]
    subprocess.run(cmd, check=True, capture_output=True)
    lib = ctypes.CDLL(out)
    lib.tc_tile_probe.argtypes = [ctypes.c_void_p] * 4
    lib.tc_tile_probe.restype = ctypes.c_int
    return lib


def test_single_tile_matches_matmul(probe):
    g = torch.Generator(device="cuda").manual_seed(0)
    A = torch.randint(-3, 4, (128, 128), device="cuda", generator=g).to(torch.bfloat16)
    Bm = torch.randint(-3, 4, (256, 128), device="cuda", generator=g).to(torch.bfloat16)
    D = torch.full((128, 256), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = probe.tc_tile_probe(A.data_ptr(), Bm.data_ptr(), D.data_ptr(), st.data_ptr())
    assert rc == 0 and int(st.item()) == 0, (rc, int(st.item()))
    want = A.float() @ Bm.float().T
    assert torch.equal(D, want), (D - want).abs().max()


@pytest.fixture(scope="module")
def attn_probe(tmp_path_factory):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    out = str(tmp_path_factory.mktemp("aprobe") / "libtcattnprobe.so")
    cmd = ["/usr/local/cuda/bin/nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17",
           "-shared", "-Xcompiler", "-fPIC", "-I", os.path.join(ROOT, "include"),
           os.path.join(HERE, "cuda", "tc_attn_probe.cu"),
           os.path.join(ROOT, "cross_layer_top_indexer_b300", "csrc", "tmap.cu"), "-o", out]
    subprocess.run(cmd, check=True, capture_output=True)
    lib = ctypes.CDLL(out)
    lib.tc_attn_probe.argtypes = [ctypes.c_void_p, ctypes.c_int] + [ctypes.c_void_p] * 6
    lib.tc_attn_probe.restype = ctypes.c_int
    return lib


def test_gather4_and_mn_major_operands(attn_probe):
    # the operand layouts of the sparse-attention kernel's P.V product
    g = torch.Generator(device="cuda").manual_seed(1)
    rows = 1000
    Kmat = torch.randint(-3, 4, (rows, 128), device="cuda", generator=g).to(torch.bfloat16)
    Q = torch.randint(-3, 4, (32, 128), device="cuda", generator=g).to(torch.bfloat16)
    P = torch.randint(-3, 4, (128, 32), device="cuda", generator=g).to(torch.bfloat16)
    idx = torch.randperm(rows, device="cuda", generator=g)[:128].to(torch.int32)
    S = torch.full((128, 32), float("nan"), device="cuda")
    Dv = torch.full((128, 32), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = attn_probe.tc_attn_probe(Kmat.data_ptr(), rows, Q.data_ptr(), idx.data_ptr(), P.data_ptr(),
                                  S.data_ptr(), Dv.data_ptr(), st.data_ptr())
    assert rc == 0 and int(st.item()) == 0, (rc, int(st.item()))
    Kg = Kmat[idx.long()].float()
    assert torch.equal(S, Kg @ Q.float().T), "gather4 + K-major product"
    assert torch.equal(Dv, Kg.T @ P.float()), "MN-major product"
