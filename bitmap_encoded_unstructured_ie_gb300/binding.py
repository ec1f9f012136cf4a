"""Thin ctypes binding of libus (include/us.h) over torch tensors.

Argument marshalling only: every step of encode / SpMM / spMspV runs in the
CUDA library.  Torch supplies device memory and the current stream.  If the
library has not been built, the first call raises ``LibraryMissing``: there is
no CPU fallback.

Function names follow the C ABI: ``us_encode``, ``us_spmm_w4a4``,
``us_spmm_f16``, ``us_spmspv_f16``, ``us_colinfo``, ``us_spmspv_f16_ci``, ``us_quantize_x``,
``us_workspace_bytes``, ``us_pick_split_k``,
``us_validate``, ``us_get_last_device_status``.
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libus.so")

US_OK, US_ERR_INVALID_ARG, US_ERR_UNSUPPORTED, US_ERR_TOO_LARGE = 0, 1, 2, 3
US_ERR_WORKSPACE, US_ERR_CUDA, US_ERR_TIMEOUT, US_ERR_CORRUPT = 4, 5, 6, 7
US_F16, US_I4, US_I2 = 0, 1, 2
US_ORDER_ROW, US_ORDER_COL = 0, 1
US_OP_ENCODE, US_OP_SPMM_W4A4, US_OP_SPMM_F16, US_OP_SPMSPV_F16 = 0, 1, 2, 3
US_BITMAP_STATIC = 1

EXPORTED = ("us_encode_sizes", "us_encode", "us_spmm_w4a4", "us_spmm_f16", "us_spmm_f16_noalloc", "us_spmspv_f16",
            "us_colinfo", "us_spmspv_f16_ci", "us_quantize_x",
            "us_encode_ie_sizes", "us_encode_ie", "us_reorder_rows", "us_spmm_w4a4_ie", "us_workspace_bytes_ie",
            "us_pick_split_k_ie",
            "us_workspace_bytes", "us_pick_split_k", "us_validate", "us_get_last_device_status",
            "us_selftest_wait_timeout", "us_status_string", "us_version")


class LibraryMissing(RuntimeError):
    pass


class UsError(RuntimeError):
    def __init__(self, fn: str, code: int, text: str):
        super().__init__(f"{fn}: {text} ({code})")
        self.code = code


class us_bitmap(ctypes.Structure):
    _fields_ = [("M", ctypes.c_int32), ("K", ctypes.c_int32), ("TM", ctypes.c_int32), ("TK", ctypes.c_int32),
                ("elem", ctypes.c_int32), ("order", ctypes.c_int32),
                ("bitmap", ctypes.c_void_p), ("tile_off", ctypes.c_void_p), ("values", ctypes.c_void_p),
                ("values_bytes", ctypes.c_uint64), ("flags", ctypes.c_uint32), ("reserved", ctypes.c_uint32)]


class us_bitmap_ie(ctypes.Structure):
    _fields_ = [("W", us_bitmap), ("RA", ctypes.c_int32), ("CA", ctypes.c_int32), ("perm", ctypes.c_void_p)]


_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH):
    """Load libus.so (once).  Raises LibraryMissing if it was not built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise LibraryMissing(f"{path} not found: build it with __graft_entry__.build() "
                                 f"or python -m bitmap_encoded_unstructured_ie_gb300.build")
        lib = ctypes.CDLL(path)
        P, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
        psz = ctypes.POINTER(ctypes.c_size_t)
        pbm = ctypes.POINTER(us_bitmap)
        lib.us_encode_sizes.argtypes = [i32, i32, i32, i32, i32, psz, psz, psz, psz]
        lib.us_encode.argtypes = [P, i64, i32, i32, i32, i32, i32, i32, P, P, P, sz, P, sz, P]
        lib.us_spmm_w4a4.argtypes = [pbm, P, P, P, i32, P, P, P, sz, i32, P]
        lib.us_spmm_f16.argtypes = [pbm, P, i32, P, P, sz, i32, P]
        lib.us_spmm_f16_noalloc.argtypes = [pbm, P, i32, P, i32, P]
        lib.us_spmspv_f16.argtypes = [pbm, P, ctypes.c_float, P, P, sz, P]
        lib.us_colinfo.argtypes = [pbm, P, P]
        pie = ctypes.POINTER(us_bitmap_ie)
        lib.us_encode_ie_sizes.argtypes = [i32, i32, i32, i32, i32, i32, i32, psz, psz, psz, psz]
        lib.us_encode_ie.argtypes = [P, i64, i32, i32, i32, i32, i32, i32, i32, P, P, P, P, sz, P, sz, P]
        lib.us_reorder_rows.argtypes = [P, i64, i32, i32, i32, i32, i32, i32, i32, P, i32]
        lib.us_spmm_w4a4_ie.argtypes = [pie, P, P, P, i32, P, P, P, sz, i32, P]
        lib.us_workspace_bytes_ie.argtypes = [pie, i32, i32, psz]
        lib.us_pick_split_k_ie.argtypes = [pie, i32, ctypes.POINTER(ctypes.c_int)]
        lib.us_spmspv_f16_ci.argtypes = [pbm, P, P, i32, ctypes.c_float, P, P, sz, P]
        lib.us_quantize_x.argtypes = [P, i32, i32, P, P, P]
        lib.us_workspace_bytes.argtypes = [i32, pbm, i32, i32, psz]
        lib.us_pick_split_k.argtypes = [i32, pbm, i32, ctypes.POINTER(ctypes.c_int)]
        lib.us_validate.argtypes = [pbm]
        lib.us_get_last_device_status.argtypes = [P]
        lib.us_selftest_wait_timeout.argtypes = [ctypes.c_uint64, P, P]
        lib.us_status_string.argtypes = [i32]
        lib.us_status_string.restype = ctypes.c_char_p
        lib.us_version.argtypes = []
        for name in EXPORTED:
            if name != "us_status_string":
                getattr(lib, name).restype = ctypes.c_int
        _lib = lib
        return lib


def status_string(code: int) -> str:
    return load().us_status_string(int(code)).decode()


def _check(fn: str, code: int):
    if code != US_OK:
        raise UsError(fn, code, status_string(code))


def _dptr(t: torch.Tensor | None):
    if t is None:
        return None
    assert t.is_cuda and t.is_contiguous(), "device tensors must be contiguous CUDA tensors"
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


@dataclass
class Encoded:
    """An encoded matrix: three device tensors plus its parameters."""
    M: int
    K: int
    TM: int
    TK: int
    elem: int
    order: int
    bitmap: torch.Tensor      # uint64 words (int64 storage)
    tile_off: torch.Tensor    # uint32 (int32 storage), nT + 1
    values: torch.Tensor      # uint8
    values_bytes: int
    flags: int = 0            # US_BITMAP_STATIC: not written by earlier work on the stream

    def desc(self) -> us_bitmap:
        return us_bitmap(self.M, self.K, self.TM, self.TK, self.elem, self.order,
                         self.bitmap.data_ptr(), self.tile_off.data_ptr(), self.values.data_ptr(),
                         self.values_bytes, self.flags, 0)

    def nbytes(self) -> int:
        return self.bitmap.numel() * 8 + self.tile_off.numel() * 4 + self.values_bytes


def encode_sizes(M, K, TM, TK, elem):
    b, o, v, w = (ctypes.c_size_t() for _ in range(4))
    _check("us_encode_sizes", load().us_encode_sizes(M, K, TM, TK, elem, ctypes.byref(b), ctypes.byref(o),
                                                     ctypes.byref(v), ctypes.byref(w)))
    return b.value, o.value, v.value, w.value


def us_encode(W: torch.Tensor, TM: int, TK: int, elem: int, order: int, stream=None, shrink: bool = True) -> Encoded:
    """Encode a dense CUDA matrix (fp16 for US_F16, int8 codes for US_I4)."""
    lib = load()
    M, K = W.shape
    dev = W.device
    assert W.is_cuda and W.stride(1) == 1, "W must be a CUDA matrix with unit column stride"
    bb, ob, vcap, wsb = encode_sizes(M, K, TM, TK, elem)
    bitmap = torch.empty(bb // 8, dtype=torch.int64, device=dev)
    tile_off = torch.empty(ob // 4, dtype=torch.int32, device=dev)
    values = torch.zeros(max(vcap, 16), dtype=torch.uint8, device=dev)
    ws = torch.zeros(max(wsb, 16), dtype=torch.uint8, device=dev)
    _check("us_encode", lib.us_encode(ctypes.c_void_p(W.data_ptr()), W.stride(0), M, K, TM, TK, elem, order, _dptr(bitmap),
                                      _dptr(tile_off), _dptr(values), values.numel(), _dptr(ws), ws.numel(),
                                      _stream(stream)))
    used_elems = int(tile_off[-1].item()) & 0xFFFFFFFF
    used = used_elems * {US_F16: 16, US_I4: 4, US_I2: 2}[elem] // 8
    if shrink:
        values = values[: max(used, 16)].clone()
    return Encoded(M, K, TM, TK, elem, order, bitmap, tile_off, values, used)


def us_encode_into(W: torch.Tensor, E: Encoded, ws: torch.Tensor, stream=None):
    """Re-encode W into E's existing buffers (no readback, no synchronisation).
    E.values must have the worst-case capacity (shrink=False)."""
    M, K = W.shape
    assert W.is_cuda and W.stride(1) == 1
    _check("us_encode", load().us_encode(ctypes.c_void_p(W.data_ptr()), W.stride(0), M, K, E.TM, E.TK, E.elem,
                                         E.order, _dptr(E.bitmap), _dptr(E.tile_off), _dptr(E.values),
                                         E.values.numel(), _dptr(ws), ws.numel(), _stream(stream)))


@dataclass
class EncodedIE:
    """IE-BME with RA x CA areas: an Encoded (ROW scan, union-mask bitmap) plus
    the area counts and the per-tile row permutation (device uint8, or None)."""
    E: Encoded
    RA: int
    CA: int
    perm: torch.Tensor | None = None

    def desc(self) -> us_bitmap_ie:
        return us_bitmap_ie(self.E.desc(), self.RA, self.CA, self.perm.data_ptr() if self.perm is not None else None)


def encode_ie_sizes(M, K, TM, TK, RA, CA, elem):
    b, o, v, w = (ctypes.c_size_t() for _ in range(4))
    _check("us_encode_ie_sizes", load().us_encode_ie_sizes(M, K, TM, TK, RA, CA, elem, ctypes.byref(b),
                                                           ctypes.byref(o), ctypes.byref(v), ctypes.byref(w)))
    return b.value, o.value, v.value, w.value


def us_encode_ie(W: torch.Tensor, TM: int, TK: int, RA: int, CA: int, elem: int, perm: torch.Tensor | None = None,
                 stream=None) -> EncodedIE:
    """Encode a dense CUDA matrix as IE-BME with RA x CA areas; perm: device
    uint8 tensor of TM bytes per tile (tile-major) or None."""
    lib = load()
    M, K = W.shape
    dev = W.device
    assert W.is_cuda and W.stride(1) == 1, "W must be a CUDA matrix with unit column stride"
    bb, ob, vcap, wsb = encode_ie_sizes(M, K, TM, TK, RA, CA, elem)
    bitmap = torch.empty(max(bb // 8, 2), dtype=torch.int64, device=dev)
    tile_off = torch.empty(ob // 4, dtype=torch.int32, device=dev)
    values = torch.zeros(max(vcap, 16), dtype=torch.uint8, device=dev)
    ws = torch.zeros(max(wsb, 16), dtype=torch.uint8, device=dev)
    _check("us_encode_ie", lib.us_encode_ie(ctypes.c_void_p(W.data_ptr()), W.stride(0), M, K, TM, TK, RA, CA, elem,
                                            _dptr(perm), _dptr(bitmap), _dptr(tile_off), _dptr(values),
                                            values.numel(), _dptr(ws), ws.numel(), _stream(stream)))
    used_elems = int(tile_off[-1].item()) & 0xFFFFFFFF
    used = used_elems * {US_F16: 16, US_I4: 4, US_I2: 2}[elem] // 8
    values = values[: max(used, 16)].clone()
    return EncodedIE(Encoded(M, K, TM, TK, elem, US_ORDER_ROW, bitmap, tile_off, values, used), RA, CA, perm)


def us_reorder_rows(W, TM: int, TK: int, RA: int, CA: int, elem: int, nthreads: int = 0):
    """Bitmap-aware row reordering on the host (offline): numpy W (fp16 or int8
    codes) -> numpy uint8 permutation, TM bytes per tile, tile-major."""
    import numpy as np
    Wh = np.ascontiguousarray(W)
    M, K = Wh.shape
    perm = np.zeros((M // TM) * (K // TK) * TM, np.uint8)
    n = nthreads or max(1, min(32, os.cpu_count() or 1))
    _check("us_reorder_rows", load().us_reorder_rows(Wh.ctypes.data, K, M, K, TM, TK, RA, CA, elem,
                                                     perm.ctypes.data, n))
    return perm


def us_workspace_bytes_ie(E: EncodedIE, N: int, split_k: int = 0) -> int:
    n = ctypes.c_size_t()
    d = E.desc()
    _check("us_workspace_bytes_ie", load().us_workspace_bytes_ie(ctypes.byref(d), N, split_k, ctypes.byref(n)))
    return n.value


def us_pick_split_k_ie(E: EncodedIE, N: int = 1) -> int:
    """0 when the balanced kernel serves us_spmm_w4a4_ie on E with N tokens."""
    s = ctypes.c_int()
    d = E.desc()
    _check("us_pick_split_k_ie", load().us_pick_split_k_ie(ctypes.byref(d), N, ctypes.byref(s)))
    return s.value


def workspace_ie(E: EncodedIE, N: int, split_k: int = 0) -> torch.Tensor:
    return torch.zeros(max(us_workspace_bytes_ie(E, N, split_k), 16), dtype=torch.uint8, device=E.E.bitmap.device)


def us_spmm_w4a4_ie(E: EncodedIE, Xq: torch.Tensor, s_w, s_x, N: int, Yacc: torch.Tensor, Y, ws: torch.Tensor,
                    split_k: int = 0, stream=None):
    d = E.desc()
    _check("us_spmm_w4a4_ie", load().us_spmm_w4a4_ie(ctypes.byref(d), _dptr(Xq), _dptr(s_w), _dptr(s_x), N,
                                                     _dptr(Yacc), _dptr(Y), _dptr(ws), ws.numel(), split_k,
                                                     _stream(stream)))


def from_host(bitmap, tile_off, values, M, K, TM, TK, elem, order, device="cuda") -> Encoded:
    """Wrap host numpy arrays of an encoded matrix as device tensors."""
    import numpy as np
    bm = torch.from_numpy(np.ascontiguousarray(bitmap).view(np.int64)).to(device)
    off = torch.from_numpy(np.ascontiguousarray(tile_off).view(np.int32)).to(device)
    v = np.ascontiguousarray(values, dtype=np.uint8)
    vb = v.size
    v = np.concatenate([v, np.zeros((-v.size) % 16 + (16 if v.size == 0 else 0), np.uint8)])
    return Encoded(M, K, TM, TK, elem, order, bm, off, torch.from_numpy(v).to(device), vb)


def us_workspace_bytes(op: int, E: Encoded, N: int = 1, split_k: int = 0) -> int:
    n = ctypes.c_size_t()
    d = E.desc()
    _check("us_workspace_bytes", load().us_workspace_bytes(op, ctypes.byref(d), N, split_k, ctypes.byref(n)))
    return n.value


def us_pick_split_k(op: int, E: Encoded, N: int = 1) -> int:
    s = ctypes.c_int()
    d = E.desc()
    _check("us_pick_split_k", load().us_pick_split_k(op, ctypes.byref(d), N, ctypes.byref(s)))
    return s.value


def workspace(op: int, E: Encoded, N: int = 1, split_k: int = 0) -> torch.Tensor:
    """A zero-filled workspace of the size the call needs."""
    return torch.zeros(max(us_workspace_bytes(op, E, N, split_k), 16), dtype=torch.uint8, device=E.bitmap.device)


def us_spmm_w4a4(E: Encoded, Xq: torch.Tensor, s_w: torch.Tensor, s_x: torch.Tensor, N: int,
                 Yacc: torch.Tensor, Y: torch.Tensor | None, ws: torch.Tensor, split_k: int = 0, stream=None):
    d = E.desc()
    _check("us_spmm_w4a4", load().us_spmm_w4a4(ctypes.byref(d), _dptr(Xq), _dptr(s_w), _dptr(s_x), N, _dptr(Yacc),
                                               _dptr(Y), _dptr(ws), ws.numel(), split_k, _stream(stream)))


def us_spmm_f16(E: Encoded, X: torch.Tensor, N: int, Y: torch.Tensor, ws: torch.Tensor, split_k: int = 0,
                stream=None):
    d = E.desc()
    _check("us_spmm_f16", load().us_spmm_f16(ctypes.byref(d), _dptr(X), N, _dptr(Y), _dptr(ws), ws.numel(),
                                             split_k, _stream(stream)))


def us_spmm_f16_noalloc(E: Encoded, X: torch.Tensor, N: int, Y: torch.Tensor, split_k: int = 0, stream=None):
    """fp16 SpMM whose split-K scratch lives inside the library (no workspace)."""
    d = E.desc()
    _check("us_spmm_f16_noalloc", load().us_spmm_f16_noalloc(ctypes.byref(d), _dptr(X), N, _dptr(Y), split_k,
                                                             _stream(stream)))


def us_spmspv_f16(E: Encoded, x: torch.Tensor, tau: float, y: torch.Tensor, ws: torch.Tensor, stream=None):
    d = E.desc()
    _check("us_spmspv_f16", load().us_spmspv_f16(ctypes.byref(d), _dptr(x), float(tau), _dptr(y), _dptr(ws),
                                                 ws.numel(), _stream(stream)))


def colinfo_words(E: Encoded) -> int:
    """Number of uint32 ColInfo words of a COL-order matrix (one per tile column)."""
    return (E.M // E.TM) * E.K


def us_colinfo(E: Encoded, colinfo: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """ColInfo of a COL-order matrix: int32 tensor (bit pattern of uint32) of
    (M / TM) * K words, tile-major, (offset << 16) | nnz per tile column."""
    if colinfo is None:
        colinfo = torch.empty(colinfo_words(E), dtype=torch.int32, device=E.bitmap.device)
    d = E.desc()
    _check("us_colinfo", load().us_colinfo(ctypes.byref(d), _dptr(colinfo), _stream(stream)))
    return colinfo


def us_spmspv_f16_ci(E: Encoded, colinfo: torch.Tensor, X: torch.Tensor, N: int, tau: float, Y: torch.Tensor,
                     ws: torch.Tensor | None = None, stream=None):
    """Batched spMspV through ColInfo: X N x K fp16 (bit pattern), Y N x M."""
    d = E.desc()
    _check("us_spmspv_f16_ci", load().us_spmspv_f16_ci(ctypes.byref(d), _dptr(colinfo), _dptr(X), N, float(tau),
                                                       _dptr(Y), _dptr(ws), ws.numel() if ws is not None else 0,
                                                       _stream(stream)))


def us_quantize_x(X: torch.Tensor, N: int, K: int, Xq: torch.Tensor, s_x: torch.Tensor, stream=None):
    """fp16 activations (N x K, token-major) -> packed int4 codes (N x K/2 bytes)
    and one fp16 scale per token."""
    _check("us_quantize_x", load().us_quantize_x(_dptr(X), N, K, _dptr(Xq), _dptr(s_x), _stream(stream)))


def us_validate_host(bitmap, tile_off, values, M, K, TM, TK, elem, order) -> int:
    """us_validate on host numpy arrays; returns the status code."""
    import numpy as np
    bm = np.ascontiguousarray(bitmap, dtype=np.uint64)
    off = np.ascontiguousarray(tile_off, dtype=np.uint32)
    v = np.ascontiguousarray(values, dtype=np.uint8)
    d = us_bitmap(M, K, TM, TK, elem, order, bm.ctypes.data, off.ctypes.data,
                  v.ctypes.data if v.size else None, v.size, 0, 0)
    return int(load().us_validate(ctypes.byref(d)))


def us_selftest_wait_timeout(limit_ns: int, elapsed: torch.Tensor | None = None, stream=None):
    """Run the bounded-wait self-test: one device wait that nothing completes,
    given up after limit_ns (elapsed: optional int64 device tensor of one element)."""
    _check("us_selftest_wait_timeout", load().us_selftest_wait_timeout(int(limit_ns), _dptr(elapsed),
                                                                       _stream(stream)))


def us_get_last_device_status(stream=None) -> int:
    return int(load().us_get_last_device_status(_stream(stream)))
