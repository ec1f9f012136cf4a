"""The C-ABI library without a GPU: it loads, exports every entry point that
include/us.h declares, sizes buffers, validates encoded matrices on the host and
rejects bad arguments before enqueuing anything.  Encoded matrices here come
from the CPU oracle (which is also what the validator is checked against)."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "us.h")


@pytest.fixture(scope="module")
def lib():
    from bitmap_encoded_unstructured_ie_gb300 import build, binding
    build.build()
    return binding.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(us_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_four_ops():
    names = declared_functions()
    for n in ("us_encode", "us_spmm_w4a4", "us_spmm_f16", "us_spmspv_f16"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from bitmap_encoded_unstructured_ie_gb300 import binding
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in us.h but not exported"
    assert set(binding.EXPORTED) <= set(declared_functions())
    assert lib.us_version() >= 100


def test_status_strings(lib):
    from bitmap_encoded_unstructured_ie_gb300 import binding as b
    for code in range(8):
        assert b.status_string(code) and b.status_string(code) != "unknown status"


def test_encode_sizes(lib):
    from bitmap_encoded_unstructured_ie_gb300 import binding as b
    bb, ob, vcap, ws = b.encode_sizes(4096, 4096, 64, 64, b.US_I4)
    assert bb == 4096 * 4096 // 8 and ob == (64 * 64 + 1) * 4 and vcap == 4096 * 4096 // 2 and ws >= 64 * 64 * 4
    for bad in [(4096, 4096, 48, 64), (4096, 4096, 64, 24), (4000, 4096, 64, 64), (65536, 65536, 64, 64)]:
        with pytest.raises(b.UsError):
            b.encode_sizes(*bad, b.US_F16)


def _oracle_encoded(seed=0, elem=1, order=0, M=256, K=256, TM=64, TK=64):
    from oracle import oracle as o
    rng = np.random.default_rng(seed)
    if elem == 1:
        W = rng.integers(-8, 8, size=(M, K)).astype(np.int8)
        W[rng.random((M, K)) < 0.5] = 0
    elif elem == 2:
        W = rng.integers(-2, 2, size=(M, K)).astype(np.int8)
        W[rng.random((M, K)) < 0.5] = 0
    else:
        W = (rng.standard_normal((M, K)) * 0.02).astype(np.float16)
        W[rng.random((M, K)) < 0.5] = 0
    return o.encode(W, TM, TK, elem, order)


@pytest.mark.parametrize("elem,order", [(0, 0), (0, 1), (1, 0), (1, 1), (2, 0), (2, 1)])
def test_validate_accepts_oracle_encoding(lib, elem, order):
    from bitmap_encoded_unstructured_ie_gb300 import binding as b
    bm, off, vals = _oracle_encoded(1, elem, order)
    assert b.us_validate_host(bm, off, vals, 256, 256, 64, 64, elem, order) == b.US_OK


def test_validate_rejects_corruption(lib):
    from bitmap_encoded_unstructured_ie_gb300 import binding as b
    bm, off, vals = _oracle_encoded(2)
    args = (256, 256, 64, 64, 1, 0)
    bad = off.copy(); bad[3] = bad[4] + 32
    assert b.us_validate_host(bm, bad, vals, *args) == b.US_ERR_CORRUPT          # not monotone
    bad = off.copy(); bad[5:] += 32
    assert b.us_validate_host(bm, bad, np.concatenate([vals, np.zeros(16, np.uint8)]), *args) == b.US_ERR_CORRUPT
    bad = off.copy(); bad[1] += 1
    assert b.us_validate_host(bm, bad, vals, *args) == b.US_ERR_CORRUPT          # not a 16-byte run
    assert b.us_validate_host(bm, off, vals[:-16], *args) == b.US_ERR_CORRUPT    # buffer too short
    bm2 = bm.copy(); bm2[0] |= np.uint64(0xFFFF)
    P0 = bin(int(bm2[0])).count("1")
    assert b.us_validate_host(bm2, off, vals, *args) in (b.US_OK, b.US_ERR_CORRUPT)
    bm3 = bm.copy(); bm3[:64] = np.uint64(0xFFFFFFFFFFFFFFFF)                   # popcount > run
    assert b.us_validate_host(bm3, off, vals, *args) == b.US_ERR_CORRUPT
    # nonzero padding
    t0_len = int(off[1])
    P = sum(bin(int(w)).count("1") for w in bm[:64])
    if P < t0_len:
        v2 = vals.copy(); v2[(t0_len - 1) // 2] |= 0xF0
        assert b.us_validate_host(bm, off, v2, *args) == b.US_ERR_CORRUPT
    assert P0 >= 0


def test_bad_arguments_rejected_without_launch(lib):
    """Every check below fails on the host, before any CUDA call."""
    from bitmap_encoded_unstructured_ie_gb300 import binding as b
    L = b.load()
    good = b.us_bitmap(256, 256, 64, 64, b.US_I4, b.US_ORDER_ROW, 0x1000, 0x2000, 0x3000, 4096)
    P = ctypes.c_void_p
    ws, X, Y = P(0x10000), P(0x20000), P(0x30000)
    assert L.us_spmm_w4a4(ctypes.byref(good), X, P(0x40000), P(0x50000), 0, Y, None, ws, 1 << 20, 0, None) == 1
    assert L.us_spmm_w4a4(ctypes.byref(good), X, P(0x40000), P(0x50000), 4096, Y, None, ws, 1 << 20, 0, None) == 1
    assert L.us_spmm_w4a4(None, X, None, None, 1, Y, None, ws, 1 << 20, 0, None) == 1
    mis = b.us_bitmap(256, 256, 64, 64, b.US_I4, b.US_ORDER_ROW, 0x1004, 0x2000, 0x3000, 4096)
    assert L.us_spmm_w4a4(ctypes.byref(mis), X, None, None, 1, Y, None, ws, 1 << 20, 0, None) == 1
    col = b.us_bitmap(256, 256, 64, 64, b.US_I4, b.US_ORDER_COL, 0x1000, 0x2000, 0x3000, 4096)
    assert L.us_spmm_w4a4(ctypes.byref(col), X, None, None, 1, Y, None, ws, 1 << 20, 0, None) == 2
    f16 = b.us_bitmap(256, 256, 64, 64, b.US_F16, b.US_ORDER_ROW, 0x1000, 0x2000, 0x3000, 4096)
    assert L.us_spmm_w4a4(ctypes.byref(f16), X, None, None, 1, Y, None, ws, 1 << 20, 0, None) == 1
    assert L.us_spmspv_f16(ctypes.byref(f16), X, ctypes.c_float(0.0), Y, ws, 1 << 20, None) == 2
    fcol = b.us_bitmap(256, 256, 64, 64, b.US_F16, b.US_ORDER_COL, 0x1000, 0x2000, 0x3000, 4096)
    assert L.us_spmspv_f16(ctypes.byref(fcol), X, ctypes.c_float(-1.0), Y, ws, 1 << 20, None) == 1
    assert L.us_spmspv_f16(ctypes.byref(fcol), X, ctypes.c_float(float("nan")), Y, ws, 1 << 20, None) == 1
    odd = b.us_bitmap(256, 272, 64, 16, b.US_I4, b.US_ORDER_ROW, 0x1000, 0x2000, 0x3000, 4096)
    assert L.us_spmm_w4a4(ctypes.byref(odd), X, None, None, 1, Y, None, ws, 1 << 20, 0, None) == 1  # K % 32
    assert L.us_encode(None, 64, 64, 64, 64, 64, 0, 0, P(16), P(32), P(48), 100, P(64), 1 << 20, None) == 1
    assert L.us_encode(P(16), 64, 64, 64, 64, 64, 0, 0, P(16), P(32), P(48), 100, P(64), 4, None) == 4
    # activation quantisation: K % 32, N >= 1, null and misaligned pointers
    assert L.us_quantize_x(X, 4, 48, Y, P(0x40000), None) == 1
    assert L.us_quantize_x(X, 0, 64, Y, P(0x40000), None) == 1
    assert L.us_quantize_x(None, 4, 64, Y, P(0x40000), None) == 1
    assert L.us_quantize_x(P(0x20008), 4, 64, Y, P(0x40000), None) == 1
    assert L.us_quantize_x(X, 4, 64, Y, P(0x40001), None) == 1
    # ColInfo and batched spMspV: COL order only, N >= 1, tau >= 0, aligned pointers
    CI = P(0x60000)
    assert L.us_colinfo(ctypes.byref(f16), CI, None) == 2                          # ROW order
    assert L.us_colinfo(ctypes.byref(fcol), None, None) == 1
    assert L.us_colinfo(ctypes.byref(fcol), P(0x60004), None) == 1
    assert L.us_colinfo(None, CI, None) == 1
    assert L.us_spmspv_f16_ci(ctypes.byref(f16), CI, X, 1, ctypes.c_float(0.0), Y, None, 0, None) == 2
    assert L.us_spmspv_f16_ci(ctypes.byref(good), CI, X, 1, ctypes.c_float(0.0), Y, None, 0, None) == 1  # I4
    assert L.us_spmspv_f16_ci(ctypes.byref(fcol), CI, X, 0, ctypes.c_float(0.0), Y, None, 0, None) == 1
    assert L.us_spmspv_f16_ci(ctypes.byref(fcol), CI, X, 2, ctypes.c_float(-1.0), Y, None, 0, None) == 1
    assert L.us_spmspv_f16_ci(ctypes.byref(fcol), None, X, 2, ctypes.c_float(0.0), Y, None, 0, None) == 1
    assert L.us_spmspv_f16_ci(ctypes.byref(fcol), CI, P(0x20002), 2, ctypes.c_float(0.0), Y, None, 0, None) == 1


def test_validate_int2_padding(lib):
    """int2 runs are padded to 64 elements; a nonzero crumb in the padding is corrupt."""
    from bitmap_encoded_unstructured_ie_gb300 import binding as b
    bm, off, vals = _oracle_encoded(3, 2, 0)
    assert b.us_validate_host(bm, off, vals, 256, 256, 64, 64, 2, 0) == b.US_OK
    P = bin(int(bm[0])).count("1")
    assert int(off[1]) % 64 == 0 and int(off[1]) > P
    bad = vals.copy()
    bad[(int(off[1]) - 1) // 4] |= 0x40                  # the last padding element of tile 0
    assert b.us_validate_host(bm, off, bad, 256, 256, 64, 64, 2, 0) == b.US_ERR_CORRUPT
