"""CPU oracle for bitmap-encoded unstructured-sparse SpMM (test infrastructure).

This module is test infrastructure: only the test-suite, the smoke check and the
CPU-baseline leg of the benchmark may import it.  It wraps ``us_oracle.c`` (plain
scalar C, built with gcc) through ctypes and takes numpy arrays.  It shares no
code with the CUDA library and never imports it.

What each call restates:

* ``encode`` / ``decode``: the IE-BME layout of "UnionSparse: An Index-Efficient
  Sparsity Framework for Low-Bit Sparse LLM Inference on Edge", section V-A
  (Union Bitmaps, Union Value Offsets o_t = sum of earlier payload lengths,
  Compressed Values CV[o_t + rho]) with one area (Q = 1), in the row-major scan
  of that section or the column-major tile scan of "Unified Static-Dynamic
  Pruning for Efficient LLM Inference" section 4.1 (Tiled-CBC), with the
  16-byte value padding of its section 4.2.3.
* ``spmm_w4a4``: UnionSparse Fig. 2 - INT4 weights times INT4 activations,
  INT32 result, dequantised to FP16 with per-output-channel and per-token
  scales.
* ``spmm_f16`` / ``spmspv_f16``: Y = W.X in fp64, rounded once to fp16; the
  spMspV form skips columns whose activation fails |x_k| > tau (SPDP section 2,
  dynamic pruning W (.) M(x)); ``spmspv_f16_batched`` applies it per token.
* ``encode_ie`` / ``decode_ie`` / ``reorder_rows``: IE-BME with Q = RA*CA
  areas (UnionSparse V-A, Fig. 7: one union mask, Q aligned value streams
  CV[o_t + q P_t + rho]) and the bitmap-aware row reordering of V-B (exact
  grouped subset DP, canonical permutation).
* ``colinfo``: the ColInfo array of SPDP section 4.1 (per tile column: its
  offset in the tile's value run and its nonzero count).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

F16, I4, I2 = 0, 1, 2
ROW, COL = 0, 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "us_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

_ERRORS = {1: "bad argument", 3: "too large", 4: "values capacity exceeded", 7: "corrupt format"}


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile us_oracle.c into _build/liboracle.so (gcc, scalar, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-fPIC", "-shared",
           "-std=gnu11", "-Wall", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        # US_ORACLE_LIB lets the mutation tests load a deliberately broken build
        path = os.environ.get("US_ORACLE_LIB") or build()
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i32, i64, u64 = ctypes.c_int, ctypes.c_int64, ctypes.c_uint64
        lib.or_half_to_float.argtypes = [ctypes.c_uint16]
        lib.or_half_to_float.restype = ctypes.c_float
        lib.or_float_to_half.argtypes = [ctypes.c_float]
        lib.or_float_to_half.restype = ctypes.c_uint16
        lib.or_double_to_half.argtypes = [ctypes.c_double]
        lib.or_double_to_half.restype = ctypes.c_uint16
        lib.or_num_tiles.argtypes = [i32, i32, i32, i32, ctypes.POINTER(i64)]
        lib.or_encode.argtypes = [P, i64, i32, i32, i32, i32, i32, i32, P, P, P, u64,
                                  ctypes.POINTER(u64)]
        lib.or_decode.argtypes = [P, P, P, u64, i32, i32, i32, i32, i32, i32, P, i64]
        lib.or_unpack_int4.argtypes = [P, i64, P]
        lib.or_unpack_int4.restype = None
        lib.or_spmm_w4a4.argtypes = [P, P, P, P, i32, i32, i32, P, P, i32]
        lib.or_spmm_w4a4_at.argtypes = [P, P, P, P, i32, i32, i32, P, P, i64, P, P]
        lib.or_spmm_f16.argtypes = [P, P, i32, i32, i32, P, i32]
        lib.or_spmm_f16_at.argtypes = [P, P, i32, i32, i32, P, P, i64, P, P]
        lib.or_spmspv_f16.argtypes = [P, P, ctypes.c_float, i32, i32, P, P, i32]
        lib.or_quantize_x.argtypes = [P, i32, i32, P, P]
        lib.or_colinfo.argtypes = [P, i32, i32, i32, i32, P]
        lib.or_encode_ie.argtypes = [P, i64, i32, i32, i32, i32, i32, i32, i32, P, P, P, P, u64,
                                     ctypes.POINTER(u64)]
        lib.or_decode_ie.argtypes = [P, P, P, u64, i32, i32, i32, i32, i32, i32, i32, P, P, i64]
        lib.or_reorder_rows.argtypes = [P, i32, i32, i32, i32, P, ctypes.POINTER(ctypes.c_int)]
        lib.or_max_threads.argtypes = []
        for name in ("or_num_tiles", "or_encode", "or_decode", "or_spmm_w4a4", "or_spmm_w4a4_at",
                     "or_spmm_f16", "or_spmm_f16_at", "or_spmspv_f16", "or_colinfo", "or_encode_ie",
                     "or_decode_ie", "or_reorder_rows", "or_max_threads"):
            getattr(lib, name).restype = ctypes.c_int
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str):
    if rc != 0:
        raise OracleError(f"{what}: {_ERRORS.get(rc, rc)}")


def max_threads() -> int:
    return int(_load().or_max_threads())


# ------------------------------------------------------------------ fp16 ----
def half_to_float(bits: int) -> float:
    return float(_load().or_half_to_float(int(bits)))


def float_to_half(x: float) -> int:
    return int(_load().or_float_to_half(float(x)))


def double_to_half(x: float) -> int:
    return int(_load().or_double_to_half(float(x)))


# ---------------------------------------------------------------- format ----
def num_tiles(M: int, K: int, TM: int, TK: int) -> int:
    n = ctypes.c_int64(0)
    _check(_load().or_num_tiles(M, K, TM, TK, ctypes.byref(n)), "num_tiles")
    return n.value


def _dense_view(W: np.ndarray, elem: int) -> np.ndarray:
    if elem == F16:
        if W.dtype == np.float16:
            W = W.view(np.uint16)
        assert W.dtype == np.uint16, "fp16 weights are passed as float16 or uint16 bit patterns"
    else:
        assert W.dtype == np.int8, "int4 / int2 weights are passed as int8 codes in [-8, 7] / [-2, 1]"
    return np.ascontiguousarray(W)


def encode(W: np.ndarray, TM: int, TK: int, elem: int, order: int):
    """Dense M x K -> (bitmap uint64[nT*TM*TK/64], tile_off uint32[nT+1], values uint8[used])."""
    W = _dense_view(W, elem)
    M, K = W.shape
    nT = num_tiles(M, K, TM, TK)
    bitmap = np.zeros(nT * TM * TK // 64, dtype=np.uint64)
    tile_off = np.zeros(nT + 1, dtype=np.uint32)
    cap = M * K * (2 if elem == F16 else 1) // (1 if elem == F16 else 2) + 16
    values = np.zeros(cap, dtype=np.uint8)
    used = ctypes.c_uint64(0)
    _check(_load().or_encode(_ptr(W), K, M, K, TM, TK, elem, order, _ptr(bitmap), _ptr(tile_off),
                             _ptr(values), cap, ctypes.byref(used)), "encode")
    return bitmap, tile_off, values[: used.value].copy()


def decode(bitmap, tile_off, values, M, K, TM, TK, elem, order) -> np.ndarray:
    """Inverse of ``encode``: returns uint16 fp16 bit patterns (F16) or int8 codes (I4)."""
    bitmap = np.ascontiguousarray(bitmap, dtype=np.uint64)
    tile_off = np.ascontiguousarray(tile_off, dtype=np.uint32)
    values = np.ascontiguousarray(values, dtype=np.uint8)
    out = np.zeros((M, K), dtype=np.uint16 if elem == F16 else np.int8)
    vb = values if values.size else np.zeros(1, dtype=np.uint8)
    _check(_load().or_decode(_ptr(bitmap), _ptr(tile_off), _ptr(vb), values.size, M, K, TM, TK,
                             elem, order, _ptr(out), K), "decode")
    return out


def unpack_int4(packed: np.ndarray, n: int) -> np.ndarray:
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    out = np.zeros(n, dtype=np.int8)
    _load().or_unpack_int4(_ptr(packed), n, _ptr(out))
    return out


# -------------------------------------------------------------- multiply ----
def spmm_w4a4(Wd: np.ndarray, Xd: np.ndarray, s_w: np.ndarray, s_x: np.ndarray, nthreads: int = 1):
    """Wd: M x K int8 codes, Xd: N x K int8 codes, s_w: M fp16, s_x: N fp16.
    Returns (Yacc int32 N x M, Y fp16 N x M)."""
    Wd = np.ascontiguousarray(Wd, dtype=np.int8)
    Xd = np.ascontiguousarray(Xd, dtype=np.int8)
    s_w = np.ascontiguousarray(s_w, dtype=np.float16).view(np.uint16)
    s_x = np.ascontiguousarray(s_x, dtype=np.float16).view(np.uint16)
    M, K = Wd.shape
    N = Xd.shape[0]
    assert Xd.shape[1] == K and s_w.size == M and s_x.size == N
    acc = np.zeros((N, M), dtype=np.int32)
    y = np.zeros((N, M), dtype=np.uint16)
    _check(_load().or_spmm_w4a4(_ptr(Wd), _ptr(Xd), _ptr(s_w), _ptr(s_x), M, N, K, _ptr(acc),
                                _ptr(y), nthreads), "spmm_w4a4")
    return acc, y.view(np.float16)


def spmm_w4a4_at(Wd, Xd, s_w, s_x, n_idx, m_idx):
    Wd = np.ascontiguousarray(Wd, dtype=np.int8)
    Xd = np.ascontiguousarray(Xd, dtype=np.int8)
    s_w = np.ascontiguousarray(s_w, dtype=np.float16).view(np.uint16)
    s_x = np.ascontiguousarray(s_x, dtype=np.float16).view(np.uint16)
    n_idx = np.ascontiguousarray(n_idx, dtype=np.int32)
    m_idx = np.ascontiguousarray(m_idx, dtype=np.int32)
    M, K = Wd.shape
    N = Xd.shape[0]
    acc = np.zeros(n_idx.size, dtype=np.int32)
    y = np.zeros(n_idx.size, dtype=np.uint16)
    _check(_load().or_spmm_w4a4_at(_ptr(Wd), _ptr(Xd), _ptr(s_w), _ptr(s_x), M, N, K, _ptr(n_idx),
                                   _ptr(m_idx), n_idx.size, _ptr(acc), _ptr(y)), "spmm_w4a4_at")
    return acc, y.view(np.float16)


def _f16bits(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        return a.view(np.uint16)
    assert a.dtype == np.uint16
    return a


def spmm_f16(Wd: np.ndarray, X: np.ndarray, nthreads: int = 1) -> np.ndarray:
    """Wd: M x K fp16, X: N x K fp16 (token-major).  Returns Y: N x M fp16."""
    Wd, X = _f16bits(Wd), _f16bits(X)
    M, K = Wd.shape
    N = X.shape[0]
    assert X.shape[1] == K
    y = np.zeros((N, M), dtype=np.uint16)
    _check(_load().or_spmm_f16(_ptr(Wd), _ptr(X), M, N, K, _ptr(y), nthreads), "spmm_f16")
    return y.view(np.float16)


def spmm_f16_at(Wd, X, n_idx, m_idx):
    """Selected outputs.  Returns (fp16 values, exact fp64 sums)."""
    Wd, X = _f16bits(Wd), _f16bits(X)
    n_idx = np.ascontiguousarray(n_idx, dtype=np.int32)
    m_idx = np.ascontiguousarray(m_idx, dtype=np.int32)
    M, K = Wd.shape
    N = X.shape[0]
    y = np.zeros(n_idx.size, dtype=np.uint16)
    ex = np.zeros(n_idx.size, dtype=np.float64)
    _check(_load().or_spmm_f16_at(_ptr(Wd), _ptr(X), M, N, K, _ptr(n_idx), _ptr(m_idx), n_idx.size,
                                  _ptr(y), _ptr(ex)), "spmm_f16_at")
    return y.view(np.float16), ex


def spmspv_f16(Wd: np.ndarray, x: np.ndarray, tau: float = 0.0, nthreads: int = 1):
    """Wd: M x K fp16, x: K fp16.  Returns (y fp16 M, exact fp64 sums M)."""
    Wd, x = _f16bits(Wd), _f16bits(x)
    M, K = Wd.shape
    assert x.size == K
    y = np.zeros(M, dtype=np.uint16)
    ex = np.zeros(M, dtype=np.float64)
    _check(_load().or_spmspv_f16(_ptr(Wd), _ptr(x), float(tau), M, K, _ptr(y), _ptr(ex), nthreads),
           "spmspv_f16")
    return y.view(np.float16), ex


def spmspv_f16_batched(Wd: np.ndarray, X: np.ndarray, tau: float = 0.0, nthreads: int = 1):
    """Batched dynamic pruning: token n keeps X[n][k] iff |X[n][k]| > tau, so
    each token's row of the result is its own spMspV.  Wd: M x K fp16, X: N x K
    fp16.  Returns (Y fp16 N x M, exact fp64 sums N x M)."""
    X = np.atleast_2d(X)
    ys, exs = zip(*(spmspv_f16(Wd, X[n], tau, nthreads) for n in range(X.shape[0])))
    return np.stack(ys), np.stack(exs)


def colinfo(bitmap: np.ndarray, M: int, K: int, TM: int, TK: int) -> np.ndarray:
    """ColInfo of a COL-order bitmap (SPDP section 4.1): uint32 per column of
    every tile, tile-major, (offset within the tile's run << 16) | nnz."""
    bitmap = np.ascontiguousarray(bitmap, dtype=np.uint64)
    nT = num_tiles(M, K, TM, TK)
    out = np.zeros(nT * TK, np.uint32)
    _check(_load().or_colinfo(_ptr(bitmap), M, K, TM, TK, _ptr(out)), "colinfo")
    return out


def encode_ie(W: np.ndarray, TM: int, TK: int, RA: int, CA: int, elem: int, perm: np.ndarray | None = None):
    """IE-BME with Q = RA*CA areas (UnionSparse V-A, Fig. 7): one union mask
    per tile over (TM/RA) x (TK/CA) logical positions, Q aligned value streams.
    perm: uint8, TM per tile (tile-major), row p of the reordered tile is
    original row perm[t*TM + p]; None = identity.  Returns (bitmap, tile_off,
    values)."""
    W = np.ascontiguousarray(_dense_view(W, elem))
    M, K = W.shape
    nT = (M // TM) * (K // TK)
    bitmap = np.zeros(max(nT * TM * TK // (64 * RA * CA), 1), dtype=np.uint64)
    tile_off = np.zeros(nT + 1, dtype=np.uint32)
    bits = 16 if elem == F16 else 4
    cap = (M * K + nT * 32) * bits // 8 + 16
    values = np.zeros(cap, dtype=np.uint8)
    used = ctypes.c_uint64(0)
    pp = None if perm is None else np.ascontiguousarray(perm, dtype=np.uint8)
    _check(_load().or_encode_ie(_ptr(W), K, M, K, TM, TK, RA, CA, elem, None if pp is None else _ptr(pp),
                                _ptr(bitmap), _ptr(tile_off), _ptr(values), cap, ctypes.byref(used)), "encode_ie")
    return bitmap[: nT * TM * TK // (64 * RA * CA)], tile_off, values[: used.value]


def decode_ie(bitmap, tile_off, values, M, K, TM, TK, RA, CA, elem, perm=None) -> np.ndarray:
    bitmap = np.ascontiguousarray(bitmap, dtype=np.uint64)
    tile_off = np.ascontiguousarray(tile_off, dtype=np.uint32)
    values = np.ascontiguousarray(values, dtype=np.uint8)
    out = np.zeros((M, K), dtype=np.uint16 if elem == F16 else np.int8)
    pp = None if perm is None else np.ascontiguousarray(perm, dtype=np.uint8)
    vp = _ptr(values) if values.size else None
    _check(_load().or_decode_ie(_ptr(bitmap), _ptr(tile_off), vp, values.size, M, K, TM, TK, RA, CA, elem,
                                None if pp is None else _ptr(pp), _ptr(out), K), "decode_ie")
    return out.view(np.float16) if elem == F16 else out


def reorder_rows(mask: np.ndarray, RA: int, CA: int):
    """Bitmap-aware row reordering of one local tile (UnionSparse V-B,
    Algorithm 1): exact grouped subset DP.  mask: HL x KL (nonzero = kept).
    Returns (perm uint8 HL, minimum union-mask cost)."""
    m = np.ascontiguousarray(mask != 0, dtype=np.uint8)
    HL, KL = m.shape
    perm = np.zeros(HL, np.uint8)
    cost = ctypes.c_int(0)
    _check(_load().or_reorder_rows(_ptr(m), HL, KL, RA, CA, _ptr(perm), ctypes.byref(cost)), "reorder_rows")
    return perm, cost.value


def reorder_matrix(W: np.ndarray, TM: int, TK: int, RA: int, CA: int) -> np.ndarray:
    """Per-tile row permutations of a whole matrix (tile-major, TM bytes each)."""
    Wv = np.asarray(W)
    nz = (Wv.view(np.uint16) & 0x7FFF) != 0 if Wv.dtype == np.float16 else Wv != 0
    M, K = Wv.shape
    out = []
    for tm in range(M // TM):
        for tk in range(K // TK):
            out.append(reorder_rows(nz[tm * TM:(tm + 1) * TM, tk * TK:(tk + 1) * TK], RA, CA)[0])
    return np.concatenate(out)


def quantize_x(X: np.ndarray):
    """Per-token int4 quantisation of fp16 activations (UnionSparse Fig. 2,
    "Quant"): codes int8 in [-8, 7] (N x K) and s_x fp16 (N)."""
    Xh = np.ascontiguousarray(_f16bits(np.atleast_2d(X)))
    N, K = Xh.shape
    codes = np.zeros((N, K), np.int8)
    s = np.zeros(N, np.uint16)
    _check(_load().or_quantize_x(_ptr(Xh), N, K, _ptr(codes), _ptr(s)), "or_quantize_x")
    return codes, s.view(np.float16)
