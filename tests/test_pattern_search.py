"""The library's greedy layer-selection driver, ic_greedy_full_layers (host
code, no GPU): the deep-read page's toy ("Training-free：直接用语言模型损失
选择 Full 层", importance [99, 3, 0.2, 2, 0.1], two removals -> "FFSFS"),
its forward count K(N-1) - K(K-1)/2, and agreement with the oracle's search
on random and tie-heavy losses."""

import ctypes

import numpy as np
import pytest

import oracle
from cross_layer_top_indexer_b300 import binding as B


@pytest.fixture(scope="module")
def lib():
    from cross_layer_top_indexer_b300 import build
    build.build()
    return B.load()


def _toy(pattern):
    importance = [99.0, 3.0, 0.2, 2.0, 0.1]
    return sum(s for r, s in zip(pattern, importance) if r == "S")


def test_toy_example(lib):
    pat, forwards = B.greedy_full_layers(5, 2, _toy)
    assert pat == "FFSFS"
    assert pat[0] == "F" and pat.count("F") == 3
    assert forwards == 2 * 4 - 2 * 1 // 2


@pytest.mark.parametrize("n,K", [(1, 0), (2, 1), (5, 0), (5, 4), (8, 3), (47, 35), (47, 46)])
def test_forward_count_formula(lib, n, K):
    seen = []

    def loss(p):
        seen.append(p)
        assert len(p) == n and p[0] == "F" and set(p) <= {"F", "S"}
        return float(p.count("S"))

    pat, forwards = B.greedy_full_layers(n, K, loss)
    assert forwards == K * (n - 1) - K * (K - 1) // 2 == len(seen)
    assert pat.count("S") == K and pat[0] == "F"


@pytest.mark.parametrize("seed", range(6))
def test_agrees_with_oracle_on_random_losses(lib, seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(3, 14))
    K = int(rng.integers(0, n))
    if seed % 2:
        # tie-heavy: a few integer weights, so many trials tie and the lower layer must win
        wts = rng.integers(0, 3, size=n).astype(float)
    else:
        wts = rng.standard_normal(n)
    pair = rng.standard_normal((n, n)) * (0 if seed % 2 else 0.3)

    def loss(p):
        s = np.array([c == "S" for c in p], dtype=float)
        return float(wts @ s + s @ pair @ s)

    want = oracle.greedy_full_layers(n, K, loss)
    got, forwards = B.greedy_full_layers(n, K, loss)
    assert got == want
    assert forwards == K * (n - 1) - K * (K - 1) // 2


def test_refusals(lib):
    cb = B.LOSS_FN(lambda p, u: 0.0)
    out = ctypes.create_string_buffer(8)
    fw = ctypes.c_longlong(-1)
    assert lib.ic_greedy_full_layers(0, 0, cb, None, out, ctypes.byref(fw)) == B.IC_ERR_ARG
    assert lib.ic_greedy_full_layers(4, 4, cb, None, out, ctypes.byref(fw)) == B.IC_ERR_ARG
    assert lib.ic_greedy_full_layers(4, -1, cb, None, out, ctypes.byref(fw)) == B.IC_ERR_ARG
    assert lib.ic_greedy_full_layers(4, 1, cb, None, None, ctypes.byref(fw)) == B.IC_ERR_ARG
    assert lib.ic_greedy_full_layers(4, 1, B.LOSS_FN(), None, out, ctypes.byref(fw)) == B.IC_ERR_ARG


def test_nan_loss_stops_with_error(lib):
    calls = []

    def loss(p):
        calls.append(p)
        return float("nan") if len(calls) == 3 else 1.0

    with pytest.raises(ValueError, match="NaN"):
        B.greedy_full_layers(6, 2, loss)
    assert len(calls) == 3


def test_exception_in_loss_is_reraised(lib):
    def loss(p):
        raise KeyError("model failed")

    with pytest.raises(KeyError):
        B.greedy_full_layers(4, 1, loss)
