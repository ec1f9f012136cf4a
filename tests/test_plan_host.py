"""Launch plans of the fp16 SpMM, on the host (no GPU): which kernel family a
call takes, its K split and its workspace size, through the C ABI's
us_pick_split_k and us_workspace_bytes.  Without a device the library sizes
plans for 148 SMs.

Row-scan 64 x 64 tiles with 1-63 tokens take the mma.sync decode kernel:
blocks of 8 / 16 / 32 tokens, slices of about 16 K tiles (more only when the
bands alone would leave SMs idle), and a workspace of the band counters plus
one fp32 partial per (slice, token block, band, token, row) when split > 1.
Column-scan tiles below 64 tokens stay on the generic kernel (32-token
blocks), and 64 tokens or more take the tensor-core kernel.
"""
import ctypes

import pytest

SMS = 148


@pytest.fixture(scope="module")
def lib():
    from bitmap_encoded_unstructured_ie_gb300 import build, binding
    build.build()
    return binding.load()


def desc(M, K, order, TM=64, TK=64):
    from bitmap_encoded_unstructured_ie_gb300 import binding as b
    return b.us_bitmap(M, K, TM, TK, b.US_F16, order, None, None, None, 0, 0, 0)


def pick(lib, d, N):
    from bitmap_encoded_unstructured_ie_gb300 import binding as b
    s = ctypes.c_int()
    assert lib.us_pick_split_k(b.US_OP_SPMM_F16, ctypes.byref(d), N, ctypes.byref(s)) == b.US_OK
    return s.value


def ws(lib, d, N, split=0):
    from bitmap_encoded_unstructured_ie_gb300 import binding as b
    n = ctypes.c_size_t()
    assert lib.us_workspace_bytes(b.US_OP_SPMM_F16, ctypes.byref(d), N, split, ctypes.byref(n)) == b.US_OK
    return n.value


def counters(nTM, ntb):
    return (nTM * ntb * 4 + 255) // 256 * 256


def dec_tok_block(N):
    return 8 if N <= 8 else (16 if N <= 16 else 32)


@pytest.mark.parametrize("M,K,N,split", [
    (4096, 4096, 1, 4),       # 64 K tiles: slices of 16
    (4096, 4096, 8, 4),
    (4096, 4096, 33, 4),      # two 32-token blocks
    (11008, 4096, 16, 4),
    (4096, 11008, 1, 8),      # 172 K tiles: slices of 21-22
    (256, 512, 1, 2),         # 4 bands only: sliced further, down to 4 tiles a slice
    (128, 128, 63, 1),        # 2 K tiles: no split
])
def test_row_tiles_below_64_tokens_take_the_decode_plan(lib, M, K, N, split):
    d = desc(M, K, 0)
    assert pick(lib, d, N) == split
    nTM = M // 64
    tb = dec_tok_block(N)
    ntb = (N + tb - 1) // tb
    want = counters(nTM, ntb) + (split * ntb * nTM * tb * 64 * 4 if split > 1 else 0)
    assert ws(lib, d, N) == want
    # an explicit split sizes the same way
    assert ws(lib, d, N, 2) == counters(nTM, ntb) + 2 * ntb * nTM * tb * 64 * 4


def test_col_tiles_below_64_tokens_stay_on_the_generic_plan(lib):
    d = desc(4096, 4096, 1)
    split = pick(lib, d, 1)
    # candidate splits 1, 2, 4, ... until 64 bands x split covers the SMs
    assert split == 4
    assert ws(lib, d, 1) == counters(64, 1) + split * 1 * 64 * 32 * 64 * 4


def test_64_tokens_take_the_tensor_plan(lib):
    d = desc(4096, 4096, 0)
    # tensor path: 128-row blocks, 256-token tiles; split doubles while the
    # grid stays within the SM count and slices keep >= 8 K tiles
    assert pick(lib, d, 64) == 4
    assert pick(lib, desc(4096, 4096, 0), 63) == 4
    assert ws(lib, d, 64) != ws(lib, d, 63)
