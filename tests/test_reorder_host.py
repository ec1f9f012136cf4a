"""The library's offline row reordering (host code, no GPU) against the oracle's
grouped subset DP: the same canonical permutation for every tile, and the
error codes of the shapes it refuses."""
import ctypes

import numpy as np
import pytest

F16, I4 = 0, 1


@pytest.fixture(scope="module")
def lib():
    from bitmap_encoded_unstructured_ie_gb300 import build, binding
    build.build()
    binding.load()
    return binding


@pytest.mark.parametrize("cfg", [(16, 64, 2, 2), (16, 64, 4, 1), (16, 64, 2, 1), (16, 128, 1, 2), (16, 32, 4, 1)])
@pytest.mark.parametrize("elem", [F16, I4])
def test_reorder_matches_oracle(lib, orc, cfg, elem):
    TM, TK, RA, CA = cfg
    rng = np.random.default_rng(TM + TK * 3 + RA * 7 + CA + elem)
    M, K = TM * 3, TK * 2
    keep = rng.random((M, K)) < rng.uniform(0.15, 0.6)
    if elem == F16:
        W = np.where(keep, rng.standard_normal((M, K)), 0).astype(np.float16)
    else:
        W = np.where(keep, rng.integers(1, 8, (M, K)), 0).astype(np.int8)
    perm = lib.us_reorder_rows(W, TM, TK, RA, CA, elem, nthreads=3)
    assert np.array_equal(perm, orc.reorder_matrix(W, TM, TK, RA, CA))


def test_reorder_refuses_what_it_cannot_search(lib):
    L = lib.load()
    W = np.zeros((64, 64), np.int8)
    perm = np.zeros(64 * 4, np.uint8)
    P = ctypes.c_void_p
    # 64-row tiles: 2^64 row subsets
    assert L.us_reorder_rows(P(W.ctypes.data), 64, 64, 64, 64, 64, 2, 2, I4, P(perm.ctypes.data), 1) == 2
    # RA must divide TM, CA must divide TK; null pointers
    assert L.us_reorder_rows(P(W.ctypes.data), 64, 64, 64, 16, 64, 3, 1, I4, P(perm.ctypes.data), 1) == 1
    assert L.us_reorder_rows(None, 64, 64, 64, 16, 64, 2, 2, I4, P(perm.ctypes.data), 1) == 1
