"""Host-only checks of the C ABI: the library loads, exports every declared
symbol, and refuses bad patterns / arguments before launching anything.
No GPU is needed: every call here returns before any CUDA call."""

import ctypes
import os
import re

import pytest

from cross_layer_top_indexer_b300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names.update(re.findall(r"\b(ic_[a-z_0-9]+)\s*\(", text))
    return names


@pytest.fixture(scope="module")
def lib():
    from cross_layer_top_indexer_b300 import build
    build.build()
    return B.load()


def test_exports_every_declared_symbol(lib):
    declared = _declared_functions()
    assert {"ic_indexer_topk", "ic_sparse_attn", "ic_forward_pattern"} <= declared
    for name in declared:
        assert hasattr(lib, name), name
    assert set(B.EXPORTED) >= declared
    assert lib.ic_abi_version() == 1


def _call_forward(lib, pattern, n_layers, dims=None, layers=True, cache=1):
    d = dims or B.make_dims(1, 256, 256, 4, 32, 16, 4, 64)
    arr = (B.ICLayer * max(n_layers, 1))() if layers else None
    calls = ctypes.c_int(-5)
    code = lib.ic_forward_pattern(pattern, n_layers, arr, ctypes.byref(d), cache, ctypes.byref(calls), None, 0,
                                  None)
    return code, lib.ic_last_error().decode(), calls.value


@pytest.mark.parametrize("pattern,n", [
    (b"", 1), (b"FSS", 4), (b"FSSFS", 4), (b"SFFF", 4), (b"FSXF", 4), (b"1001", 4), (b"fssf", 4), (b"F SF", 4),
    (b"FSSF", 0),
])
def test_bad_pattern_refused_before_launch(lib, pattern, n):
    code, msg, calls = _call_forward(lib, pattern, n)
    assert code == B.IC_ERR_PATTERN, msg
    assert calls == 0 and msg


def test_null_pattern(lib):
    code, msg, _ = _call_forward(lib, None, 4)
    assert code == B.IC_ERR_PATTERN


def test_valid_pattern_then_argument_checks(lib):
    # a valid pattern passes the pattern stage and stops at the pointer checks
    code, msg, calls = _call_forward(lib, b"FSSF", 4)
    assert code == B.IC_ERR_ARG and calls == 0
    code, msg, _ = _call_forward(lib, b"FSSF", 4, cache=None)
    assert code == B.IC_ERR_ARG


def _fake(n=64):
    # fake, 16-byte aligned, never-dereferenced addresses: argument checks
    # reject the call before anything touches them
    return 0x100000 + 256 * n


@pytest.mark.parametrize("kw,code", [
    (dict(T=0), B.IC_ERR_ARG),
    (dict(q_pos0=-1), B.IC_ERR_ARG),
    (dict(q_pos0=10, T=256, S=256), B.IC_ERR_ARG),        # q_pos0 + T > S
    (dict(S_cap=100), B.IC_ERR_ARG),                     # S_cap < S
    (dict(H=65), B.IC_ERR_UNSUPPORTED),
    (dict(D=48), B.IC_ERR_UNSUPPORTED),
    (dict(k=4096), B.IC_ERR_UNSUPPORTED),
    (dict(misalign=True), B.IC_ERR_ARG),
    (dict(kdtype=B.IC_E4M3), B.IC_ERR_ARG),              # e4m3 without a scale
    (dict(kdtype=7), B.IC_ERR_ARG),
])
def test_indexer_argument_checks(lib, kw, code):
    a = dict(B=1, T=256, S=256, S_cap=256, H=4, D=32, k=16, q_pos0=0, kdtype=B.IC_BF16, misalign=False)
    a.update(kw)
    q = _fake(1) + (8 if a["misalign"] else 0)
    r = lib.ic_indexer_topk(a["B"], a["T"], a["S"], a["S_cap"], a["H"], a["D"], a["k"], a["q_pos0"], q, _fake(2),
                            a["kdtype"], None, _fake(3), _fake(4), None, 0, None)
    assert r == code, lib.ic_last_error()


@pytest.mark.parametrize("kw,code", [
    (dict(Hq=33), B.IC_ERR_UNSUPPORTED),
    (dict(Dh=96), B.IC_ERR_UNSUPPORTED),
    (dict(k=0), B.IC_ERR_ARG),
    (dict(scale=-1.0), B.IC_ERR_ARG),
    (dict(nullO=True), B.IC_ERR_ARG),
])
def test_attention_argument_checks(lib, kw, code):
    a = dict(B=1, T=256, S=256, Hq=4, Dh=64, k=16, scale=0.0, nullO=False)
    a.update(kw)
    r = lib.ic_sparse_attn(a["B"], a["T"], a["S"], a["S"], a["Hq"], a["Dh"], a["k"], _fake(1), _fake(2), _fake(3),
                           _fake(4), a["scale"], None if a["nullO"] else _fake(5), None, 0, None)
    assert r == code, lib.ic_last_error()


def test_workspace_sizes(lib):
    # prefill needs no workspace; decode stages one fp32 score row per query
    assert B.workspace_size(B.make_dims(1, 8192, 8192, 64, 128, 2048, 32, 128)) == 0
    ws = B.workspace_size(B.make_dims(32, 1, 131073, 64, 128, 2048, 32, 128, q_pos0=131072))
    pitch = (131073 + 3) // 4 * 4
    # score rows, plus the clustered select's key histogram (2048 bins per row)
    assert ws >= 32 * pitch * 4 + 32 * 2048 * 4
    # and the split decode attention's partial states (32 rows x 16 splits)
    assert ws >= 32 * 16 * (2 * 32 + 32 * 128) * 4
    with pytest.raises(ValueError):
        B.workspace_size(B.make_dims(0, 1, 1, 1, 32, 1, 1, 64))


def test_forward_workspace_too_small_is_refused(lib):
    d = B.make_dims(32, 1, 1000, 4, 32, 16, 4, 64, q_pos0=999)
    arr = (B.ICLayer * 1)()
    arr[0] = B.ICLayer(_fake(1), _fake(2), None, _fake(3), _fake(4), _fake(5), _fake(6), _fake(7))
    calls = ctypes.c_int(0)
    r = lib.ic_forward_pattern(b"F", 1, arr, ctypes.byref(d), _fake(8), ctypes.byref(calls), None, 0, None)
    assert r == B.IC_ERR_ARG and "workspace" in lib.ic_last_error().decode()


def test_overlap_argument_checks(lib):
    f = _fake
    assert lib.ic_overlap(0, 16, f(1), f(2), f(3), None, None) == B.IC_ERR_ARG
    assert lib.ic_overlap(4, 0, f(1), f(2), f(3), None, None) == B.IC_ERR_ARG
    assert lib.ic_overlap(4, 16, None, f(2), f(3), None, None) == B.IC_ERR_ARG
    assert lib.ic_overlap(4, 16, f(1), f(2), None, None, None) == B.IC_ERR_ARG
    assert lib.ic_overlap(4, 16, f(1) + 4, f(2), f(3), None, None) == B.IC_ERR_ARG
    assert lib.ic_overlap(4, 4096, f(1), f(2), f(3), None, None) == B.IC_ERR_UNSUPPORTED


def test_debug_wait_limit_setter(lib):
    assert lib.ic_debug_set_wait_limit_ns(5) == B.IC_OK
    assert lib.ic_debug_set_wait_limit_ns(0) == B.IC_OK


@pytest.mark.parametrize("kw,code,text", [
    (dict(T=9), B.IC_ERR_UNSUPPORTED, "query rows"),
    (dict(B=32, S=300000, S_cap=300000, q_pos0=299999), B.IC_ERR_UNSUPPORTED, "scratch"),
    (dict(kdtype=B.IC_E4M3), B.IC_ERR_ARG, "k_scale"),
    (dict(scale=True), B.IC_ERR_ARG, "k_scale"),            # a scale given for bf16 keys
    (dict(nullq=True), B.IC_ERR_ARG, "null"),
    (dict(H=65), B.IC_ERR_UNSUPPORTED, "heads"),
    (dict(S_cap=1 << 30, B=2048), B.IC_ERR_UNSUPPORTED, "too large"),
])
def test_noalloc_argument_checks(lib, kw, code, text):
    # the allocation-free entry point refuses before touching any pointer
    a = dict(B=2, T=1, S=1000, S_cap=1000, H=64, D=128, k=64, q_pos0=999, kdtype=B.IC_BF16, scale=False,
             nullq=False)
    a.update(kw)
    r = lib.ic_indexer_topk_noalloc(a["B"], a["T"], a["S"], a["S_cap"], a["H"], a["D"], a["k"],
                                    a["S"] - a["T"] if "q_pos0" not in kw else a["q_pos0"],
                                    None if a["nullq"] else _fake(1), _fake(2), a["kdtype"],
                                    _fake(5) if a["scale"] else None, _fake(3), _fake(4), None)
    assert r == code, lib.ic_last_error()
    assert text.encode() in lib.ic_last_error()
