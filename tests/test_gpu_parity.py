"""Parity of the CUDA path (called through the C ABI) with the CPU oracle.

Bars: encoder bytes, int32 accumulators and the W4A4 fp16 epilogue bit-exact;
fp16 outputs (fp32 accumulation) within relative L2 <= 1e-3 and max-abs <= 2e-2
of the fp64 oracle.  Shapes span several tiles, uneven split-K slices and ragged
token blocks; edge cases cover empty and full tiles, single nonzeros, all-zero
matrices and offsets that a kernel must refuse to follow.
"""
import numpy as np
import pytest
import torch

from bitmap_encoded_unstructured_ie_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

F16, I4, ROW, COL = 0, 1, 0, 1
REL_L2, MAX_ABS = 1e-3, 2e-2


@pytest.fixture(scope="module")
def us():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from bitmap_encoded_unstructured_ie_gb300 import build, binding
    build.build()
    binding.load()
    return binding


@pytest.fixture(scope="module")
def orc():
    from oracle import oracle as o
    o._load()
    return o


def rand_i4(rng, M, K, density):
    q = rng.integers(-8, 8, size=(M, K)).astype(np.int8)
    q[rng.random((M, K)) >= density] = 0
    return q


def rand_f16(rng, M, K, density):
    w = (rng.standard_normal((M, K)) * 0.02).astype(np.float16)
    w[rng.random((M, K)) >= density] = 0
    return w


def check_f16(y_gpu: np.ndarray, exact: np.ndarray, what=""):
    y = y_gpu.astype(np.float64)
    err = y - exact
    denom = max(np.linalg.norm(exact), 1e-30)
    rel = np.linalg.norm(err) / denom
    mx = np.abs(err).max() if err.size else 0.0
    assert rel <= REL_L2 and mx <= MAX_ABS, f"{what}: rel L2 {rel:.3e}, max abs {mx:.3e}"


def encode_gpu(us, W: np.ndarray, TM, TK, elem, order):
    Wt = torch.from_numpy(W.view(np.int16) if elem == F16 else W).cuda()
    E = us.us_encode(Wt, TM, TK, elem, order)
    torch.cuda.synchronize()
    assert us.us_get_last_device_status() == us.US_OK
    return E


def gpu_arrays(E):
    bm = E.bitmap.cpu().numpy().view(np.uint64)
    off = E.tile_off.cpu().numpy().view(np.uint32)
    vals = E.values.cpu().numpy()[: E.values_bytes]
    return bm, off, vals


# ------------------------------------------------------------------ encode --
ENC_SHAPES = [(256, 512, 64, 64), (192, 320, 64, 16), (512, 256, 128, 32), (256, 256, 256, 128),
              (128, 384, 64, 128), (256, 64, 256, 16)]


@pytest.mark.parametrize("shape", ENC_SHAPES)
@pytest.mark.parametrize("elem", [F16, I4])
@pytest.mark.parametrize("order", [ROW, COL])
def test_encode_bytes_match_oracle(us, orc, shape, elem, order):
    M, K, TM, TK = shape
    rng = np.random.default_rng(M + K + TM + TK + 10 * elem + order)
    for density in (0.0, 0.004, 0.5, 1.0):
        W = rand_f16(rng, M, K, density) if elem == F16 else rand_i4(rng, M, K, density)
        E = encode_gpu(us, W, TM, TK, elem, order)
        bm, off, vals = gpu_arrays(E)
        obm, ooff, ovals = orc.encode(W, TM, TK, elem, order)
        assert np.array_equal(bm, obm)
        assert np.array_equal(off, ooff)
        assert np.array_equal(vals, ovals)


def test_encode_strided_input_and_signed_zero(us, orc):
    rng = np.random.default_rng(3)
    big = rand_f16(rng, 128, 512, 0.5)
    big[5, 9] = np.float16(-0.0)
    Wt = torch.from_numpy(big.view(np.int16)).cuda()[:, 64:320]
    E = us.us_encode(Wt, 64, 64, F16, ROW)
    bm, off, vals = gpu_arrays(E)
    obm, ooff, ovals = orc.encode(np.ascontiguousarray(big[:, 64:320]), 64, 64, F16, ROW)
    assert np.array_equal(bm, obm) and np.array_equal(off, ooff) and np.array_equal(vals, ovals)


@pytest.mark.parametrize("elem", [F16, I4, 2])
@pytest.mark.parametrize("TM", [64, 128, 256])
def test_encode_row64_tiles_match_oracle(us, orc, TM, elem):
    """Row-scan tiles 64 columns wide take the 16-byte-load count and pack
    kernels (fp16 up to 128-row tiles): every tile height, element type and
    density, a strided input whose rows stay 16-byte aligned (same kernels) and
    one shifted by an element (the one-element-per-lane kernels), all equal to
    the oracle byte for byte."""
    M, K = 512, 448
    rng = np.random.default_rng(TM + 7 * elem)
    for density in (0.0, 0.004, 0.5, 1.0):
        if elem == F16:
            W = rand_f16(rng, M, K, density)
        else:
            lo, hi = (-8, 8) if elem == I4 else (-2, 2)
            W = rng.integers(lo, hi, size=(M, K)).astype(np.int8)
            W[rng.random((M, K)) >= density] = 0
        E = encode_gpu(us, W, TM, 64, elem, ROW)
        bm, off, vals = gpu_arrays(E)
        obm, ooff, ovals = orc.encode(W, TM, 64, elem, ROW)
        assert np.array_equal(bm, obm) and np.array_equal(off, ooff) and np.array_equal(vals, ovals), density
    for shift in (64, 1):
        view = W.view(np.int16) if elem == F16 else W
        big = np.zeros((M, K + 128), view.dtype)
        big[:, shift:shift + K] = view
        Wt = torch.from_numpy(big).cuda()[:, shift:shift + K]
        E = us.us_encode(Wt, TM, 64, elem, ROW)
        torch.cuda.synchronize()
        assert us.us_get_last_device_status() == us.US_OK
        bm, off, vals = gpu_arrays(E)
        assert np.array_equal(bm, obm) and np.array_equal(off, ooff) and np.array_equal(vals, ovals), shift


def test_encode_reports_out_of_range_codes(us):
    W = torch.zeros(64, 64, dtype=torch.int8, device="cuda")
    W[3, 4] = 9
    us.us_encode(W, 64, 64, I4, ROW)
    assert us.us_get_last_device_status() == us.US_ERR_INVALID_ARG
    assert us.us_get_last_device_status() == us.US_OK        # cleared by the read
    for v in (2, -3):                                         # int2 codes lie in [-2, 1]
        W2 = torch.zeros(128, 128, dtype=torch.int8, device="cuda")
        W2[70, 100] = v
        us.us_encode(W2, 64, 64, 2, ROW)
        assert us.us_get_last_device_status() == us.US_ERR_INVALID_ARG
    W8 = torch.full((64, 64), -8, dtype=torch.int8, device="cuda")   # the int4 range's ends pass
    W8[:, 1::2] = 7
    us.us_encode(W8, 64, 64, I4, ROW)
    assert us.us_get_last_device_status() == us.US_OK


# -------------------------------------------------------------------- W4A4 --
def run_w4a4(us, E, Xq_packed, s_w, s_x, N, split_k=0, want_y=True, static=False):
    dev = "cuda"
    X = torch.from_numpy(Xq_packed).to(dev)
    sw = torch.from_numpy(s_w.view(np.int16)).to(dev)
    sx = torch.from_numpy(s_x.view(np.int16)).to(dev)
    Yacc = torch.empty(N, E.M, dtype=torch.int32, device=dev)
    Y = torch.empty(N, E.M, dtype=torch.int16, device=dev) if want_y else None
    ws = us.workspace(us.US_OP_SPMM_W4A4, E, N, split_k)
    E.flags = us.US_BITMAP_STATIC if static else 0
    us.us_spmm_w4a4(E, X, sw, sx, N, Yacc, Y, ws, split_k)
    E.flags = 0
    torch.cuda.synchronize()
    assert us.us_get_last_device_status() == us.US_OK
    y = Y.cpu().numpy().view(np.float16) if want_y else None
    return Yacc.cpu().numpy(), y


W4A4_CASES = [
    # M, K, TM, TK, N, density, split_k
    (256, 512, 64, 64, 1, 0.5, 0),
    (256, 512, 64, 64, 8, 0.5, 0),
    (256, 512, 64, 64, 16, 0.3, 0),
    (320, 640, 64, 64, 3, 0.7, 3),
    (256, 512, 64, 64, 33, 0.5, 2),
    (512, 384, 128, 32, 5, 0.5, 0),
    (256, 256, 256, 128, 2, 0.5, 0),
    (192, 320, 64, 16, 7, 0.5, 4),
    (128, 1024, 64, 64, 1, 1.0, 16),
    (128, 512, 64, 64, 64, 0.05, 0),
    (256, 512, 64, 64, 13, 0.5, 0),      # tensor path: 13 tokens padded to 16
    (256, 1024, 64, 64, 32, 0.5, 4),
    (192, 768, 64, 64, 24, 0.3, 0),      # M % 128 != 0: CUDA-core path, token blocks 8+8+8
    (384, 2048, 64, 64, 17, 0.5, 0),     # tensor path, BN = 32
    (128, 4096, 64, 64, 8, 1.0, 8),      # tensor path, full tiles, 8-slice cluster
    (256, 640, 64, 64, 9, 0.05, 3),      # tensor path, nearly empty tiles, uneven slices
    (320, 640, 64, 64, 4, 0.7, 3),       # cluster of 3: 256 outputs do not divide by 3
    (256, 640, 64, 64, 16, 0.3, 3),      # tensor path, cluster of 3 over 2048 outputs
    (128, 16384, 64, 64, 32, 0.2, 1),    # one slice: packed activations too large for the tensor path
]


@pytest.mark.parametrize("case", W4A4_CASES)
def test_w4a4_matches_oracle(us, orc, case):
    M, K, TM, TK, N, dens, split = case
    rng = np.random.default_rng(sum(case[:5]))
    W = rand_i4(rng, M, K, dens)
    Xq = rng.integers(-8, 8, size=(N, K)).astype(np.int8)
    s_w = (rng.random(M) * 0.01 + 1e-3).astype(np.float16)
    s_x = (rng.random(N) * 0.5 + 0.05).astype(np.float16)
    E = encode_gpu(us, W, TM, TK, I4, ROW)
    acc, y = run_w4a4(us, E, wl.pack_int4(Xq), s_w, s_x, N, split)
    oacc, oy = orc.spmm_w4a4(W, Xq, s_w, s_x)
    assert np.array_equal(acc, oacc)
    assert np.array_equal(y.view(np.uint16), oy.view(np.uint16))


# Shapes for the balanced W4A4 kernel (automatic choice, 64 x 64 tiles, N <= 8):
# bands shared by two or three CTAs, one CTA spanning several bands (K of one
# tile), fewer tiles than SMs, K wider than a CTA's range, ragged everything.
SK_SHAPES = [
    # M, K, N, density
    (64 * 200, 64, 3, 0.5),        # nTK = 1: every CTA covers whole bands
    (128, 64 * 300, 1, 0.4),       # two bands, 300 K tiles: each band split over ~76 CTAs
    (192, 64 * 7, 8, 0.6),         # 21 tiles: fewer tiles than SMs, one tile per CTA
    (64 * 37, 64 * 13, 5, 0.3),    # 481 tiles: ranges of 3-4 tiles crossing band edges
    (64 * 9, 64 * 61, 2, 0.9),     # dense runs: the value ring wraps many times
    (64 * 3, 64 * 5, 7, 0.0),      # all tiles empty
    (64 * 40, 64 * 200, 1, 0.5),   # 53 tiles per CTA: more than the dense slots hold
    (64 * 40, 64 * 200, 6, 0.5),
]


@pytest.mark.parametrize("static", [0, 1])
@pytest.mark.parametrize("M,K,N,dens", SK_SHAPES)
def test_w4a4_balanced_partition(us, orc, M, K, N, dens, static):
    """Automatic W4A4 path for few tokens against the oracle, three times in a
    row (the posted partial sums of shared bands must be cleared for the next
    call), and against an explicit K split, which takes the cluster kernel.
    Static weights are decoded before the dependency wait (as many tiles as the
    dense slots hold, the rest after it); others after it."""
    rng = np.random.default_rng(M + K + N)
    W = rand_i4(rng, M, K, dens)
    Xq = rng.integers(-8, 8, size=(N, K)).astype(np.int8)
    s_w = (rng.random(M) * 0.01 + 1e-3).astype(np.float16)
    s_x = (rng.random(N) * 0.5 + 0.05).astype(np.float16)
    E = encode_gpu(us, W, 64, 64, I4, ROW)
    E.flags = us.US_BITMAP_STATIC if static else 0
    assert us.us_pick_split_k(us.US_OP_SPMM_W4A4, E, N) == 0
    Xp = wl.pack_int4(Xq)
    dev = "cuda"
    X = torch.from_numpy(Xp).to(dev)
    sw = torch.from_numpy(s_w.view(np.int16)).to(dev)
    sx = torch.from_numpy(s_x.view(np.int16)).to(dev)
    ws = us.workspace(us.US_OP_SPMM_W4A4, E, N, 0)
    oacc, oy = orc.spmm_w4a4(W, Xq, s_w, s_x)
    for _ in range(3):
        Yacc = torch.full((N, M), 12345, dtype=torch.int32, device=dev)
        Y = torch.empty(N, M, dtype=torch.int16, device=dev)
        us.us_spmm_w4a4(E, X, sw, sx, N, Yacc, Y, ws, 0)
        torch.cuda.synchronize()
        assert us.us_get_last_device_status() == us.US_OK
        assert np.array_equal(Yacc.cpu().numpy(), oacc)
        assert np.array_equal(Y.cpu().numpy().view(np.uint16), oy.view(np.uint16))
    assert torch.count_nonzero(ws).item() == 0                    # every posted partial cleared
    acc2, _ = run_w4a4(us, E, Xp, s_w, s_x, N, split_k=min(2, K // 64))
    assert np.array_equal(acc2, oacc)


# Shapes for the balanced kernel's tensor-core consumer (automatic choice, 64 x
# 64 tiles, 8..32 tokens: decoded tiles feed mma.sync in 8-token blocks; fewer
# tokens use dp4a).
TC_SHAPES = [
    # M, K, N, density
    (128 * 100, 64, 8, 0.5),       # nTK = 1: 200 tiles over 152 CTAs, bands whole or split in two
    (256, 64 * 300, 16, 0.4),      # four bands of 300 tiles: owners add ~38 posts each
    (128 * 9, 64 * 61, 12, 0.9),   # dense runs, 1098 tiles: ranges cross band edges
    (128 * 3, 64 * 5, 20, 0.3),    # 30 tiles, 20 tokens padded to 32
    (128 * 7, 64 * 33, 32, 0.6),   # 462 tiles, 32 tokens
    (192, 64 * 6, 9, 0.0),         # all tiles empty, 9 tokens padded to 16
    (64 * 64, 64 * 64, 16, 0.5),   # 27 tiles per CTA, 26 dense slots when static
    (64 * 40, 64 * 200, 32, 0.5),  # 53 tiles per CTA, one CTA per SM
]


@pytest.mark.parametrize("static", [0, 1])
@pytest.mark.parametrize("M,K,N,dens", TC_SHAPES)
def test_w4a4_tensor_cores_balanced(us, orc, M, K, N, dens, static):
    """Automatic W4A4 path with the mma.sync consumer against the oracle, three
    calls in a row on one workspace (posted partials must be cleared each time),
    with and without the static-weights flag."""
    rng = np.random.default_rng(M * 7 + K + N)
    W = rand_i4(rng, M, K, dens)
    Xq = rng.integers(-8, 8, size=(N, K)).astype(np.int8)
    s_w = (rng.random(M) * 0.01 + 1e-3).astype(np.float16)
    s_x = (rng.random(N) * 0.5 + 0.05).astype(np.float16)
    E = encode_gpu(us, W, 64, 64, I4, ROW)
    E.flags = us.US_BITMAP_STATIC if static else 0
    dev = "cuda"
    X = torch.from_numpy(wl.pack_int4(Xq)).to(dev)
    sw = torch.from_numpy(s_w.view(np.int16)).to(dev)
    sx = torch.from_numpy(s_x.view(np.int16)).to(dev)
    ws = us.workspace(us.US_OP_SPMM_W4A4, E, N, 0)
    oacc, oy = orc.spmm_w4a4(W, Xq, s_w, s_x)
    for _ in range(3):
        Yacc = torch.full((N, M), -777, dtype=torch.int32, device=dev)
        Y = torch.empty(N, M, dtype=torch.int16, device=dev)
        us.us_spmm_w4a4(E, X, sw, sx, N, Yacc, Y, ws, 0)
        torch.cuda.synchronize()
        assert us.us_get_last_device_status() == us.US_OK
        assert np.array_equal(Yacc.cpu().numpy(), oacc)
        assert np.array_equal(Y.cpu().numpy().view(np.uint16), oy.view(np.uint16))
    assert torch.count_nonzero(ws).item() == 0


@pytest.mark.parametrize("N", [4, 16, 32])
def test_w4a4_extreme_values_exact(us, orc, N):
    """All weights and activations -8: the largest accumulators (64*K); both the
    CUDA-core (N = 4) and the tensor-core (N = 16, 32) paths must stay exact."""
    M, K = 128, 8192
    W = np.full((M, K), -8, np.int8)
    W[::3, ::5] = 7
    X = np.full((N, K), -8, np.int8)
    X[1::2, ::7] = 7
    one = np.ones(M, np.float16)
    E = encode_gpu(us, W, 64, 64, I4, ROW)
    acc, _ = run_w4a4(us, E, wl.pack_int4(X), one, np.ones(N, np.float16), N, want_y=False)
    oacc, _ = orc.spmm_w4a4(W, X, one, np.ones(N, np.float16))
    assert np.array_equal(acc, oacc)


def test_w4a4_edge_matrices(us, orc):
    M, K, N = 128, 256, 3
    rng = np.random.default_rng(0)
    X = rng.integers(-8, 8, size=(N, K)).astype(np.int8)
    s = np.ones(M, np.float16)
    for W in (np.zeros((M, K), np.int8), np.eye(M, K, dtype=np.int8) * 3):
        W = W.copy()
        E = encode_gpu(us, W, 64, 64, I4, ROW)
        acc, _ = run_w4a4(us, E, wl.pack_int4(X), s, np.ones(N, np.float16), N)
        oacc, _ = orc.spmm_w4a4(W, X, s, np.ones(N, np.float16))
        assert np.array_equal(acc, oacc)
    W = np.zeros((M, K), np.int8)
    W[77, 200] = -3                                     # one nonzero, everything else empty
    E = encode_gpu(us, W, 64, 64, I4, ROW)
    acc, _ = run_w4a4(us, E, wl.pack_int4(X), s, np.ones(N, np.float16), N)
    assert np.array_equal(acc[:, 77], -3 * X[:, 200].astype(np.int32)) and np.count_nonzero(acc[:, :77]) == 0


def test_corrupt_offsets_are_refused_on_device(us, orc):
    """Offsets that point outside the run are caught by the kernel's own checks:
    the tile is treated as empty and US_ERR_CORRUPT is reported."""
    rng = np.random.default_rng(1)
    W = rand_i4(rng, 128, 256, 0.5)
    bm, off, vals = orc.encode(W, 64, 64, I4, ROW)
    bad = off.copy()
    bad[2] = bad[1] + 16                                # misaligned, shorter than the popcount
    E = us.from_host(bm, bad, vals, 128, 256, 64, 64, I4, ROW)
    X = rng.integers(-8, 8, size=(1, 256)).astype(np.int8)
    Xt = torch.from_numpy(wl.pack_int4(X)).cuda()
    Yacc = torch.empty(1, 128, dtype=torch.int32, device="cuda")
    ws = us.workspace(us.US_OP_SPMM_W4A4, E, 1, 1)
    us.us_spmm_w4a4(E, Xt, None, None, 1, Yacc, None, ws, 1)
    assert us.us_get_last_device_status() == us.US_ERR_CORRUPT


def test_workspace_too_small_is_a_host_error(us, orc):
    rng = np.random.default_rng(2)
    W = rand_f16(rng, 256, 512, 0.5)
    E = encode_gpu(us, W, 64, 64, F16, ROW)
    X = torch.zeros(1, 512, dtype=torch.int16, device="cuda")
    Y = torch.empty(1, 256, dtype=torch.int16, device="cuda")
    need = us.us_workspace_bytes(us.US_OP_SPMM_F16, E, 1, 4)
    ws = torch.zeros(max(need - 16, 16), dtype=torch.uint8, device="cuda")
    with pytest.raises(us.UsError) as ei:
        us.us_spmm_f16(E, X, 1, Y, ws, 4)
    assert ei.value.code == us.US_ERR_WORKSPACE
    # the W4A4 decode path reduces split-K inside a cluster: no workspace at all
    Ei = encode_gpu(us, rand_i4(rng, 256, 512, 0.5), 64, 64, I4, ROW)
    assert us.us_workspace_bytes(us.US_OP_SPMM_W4A4, Ei, 1, 4) == 0


# -------------------------------------------------------------------- fp16 --
def run_f16(us, E, X: np.ndarray, split_k=0):
    N = X.shape[0]
    Xt = torch.from_numpy(X.view(np.int16)).cuda()
    Y = torch.empty(N, E.M, dtype=torch.int16, device="cuda")
    ws = us.workspace(us.US_OP_SPMM_F16, E, N, split_k)
    us.us_spmm_f16(E, Xt, N, Y, ws, split_k)
    torch.cuda.synchronize()
    assert us.us_get_last_device_status() == us.US_OK
    return Y.cpu().numpy().view(np.float16)


F16_CASES = [
    # tensor-core path (64x64 tiles, N >= 64): two M tiles, ragged token tiles, split-K
    (256, 512, 64, 64, 64, 0.5, 0),
    (256, 512, 64, 64, 100, 0.4, 0),
    (256, 1024, 64, 64, 300, 0.5, 2),
    (384, 768, 64, 64, 257, 0.6, 3),
    (128, 512, 64, 64, 512, 1.0, 0),
    # 512-token tiles: a second tile holding one token half, and one whose
    # second half holds 9 tokens, under split-K
    (256, 512, 64, 64, 600, 0.5, 0),
    (128, 1024, 64, 64, 777, 0.5, 3),
    # two row blocks under split-K, and a last tile whose second token half
    # holds no tokens
    (256, 1024, 64, 64, 600, 0.5, 2),
    # CUDA-core paths
    (256, 512, 64, 64, 1, 0.5, 0),
    (256, 512, 64, 64, 5, 0.5, 3),
    (512, 256, 128, 32, 32, 0.4, 0),
    (256, 512, 256, 16, 70, 0.5, 2),
    (128, 256, 128, 128, 2, 1.0, 0),
]


@pytest.mark.parametrize("case", F16_CASES)
def test_f16_matches_oracle(us, orc, case):
    M, K, TM, TK, N, dens, split = case
    rng = np.random.default_rng(sum(case[:5]) + 1)
    W = rand_f16(rng, M, K, dens)
    X = rng.standard_normal((N, K)).astype(np.float16)
    E = encode_gpu(us, W, TM, TK, F16, ROW)
    y = run_f16(us, E, X, split)
    n_idx, m_idx = np.meshgrid(np.arange(N), np.arange(M), indexing="ij")
    _, exact = orc.spmm_f16_at(W, X, n_idx.reshape(-1), m_idx.reshape(-1))
    check_f16(y.reshape(-1), exact, f"fp16 {case}")


def test_f16_split_k_is_deterministic(us):
    rng = np.random.default_rng(4)
    W = rand_f16(rng, 256, 1024, 0.5)
    X = rng.standard_normal((3, 1024)).astype(np.float16)
    E = encode_gpu(us, W, 64, 64, F16, ROW)
    for split in (1, 2, 5, 16):
        a = run_f16(us, E, X, split)
        b = run_f16(us, E, X, split)
        assert np.array_equal(a.view(np.uint16), b.view(np.uint16))


# ------------------------------------------------------------------ spMspV --
def run_spmspv(us, E, x: np.ndarray, tau: float):
    xt = torch.from_numpy(x.view(np.int16)).cuda()
    y = torch.empty(E.M, dtype=torch.int16, device="cuda")
    ws = us.workspace(us.US_OP_SPMSPV_F16, E, 1)
    us.us_spmspv_f16(E, xt, tau, y, ws)
    torch.cuda.synchronize()
    assert us.us_get_last_device_status() == us.US_OK
    return y.cpu().numpy().view(np.float16)


@pytest.mark.parametrize("TM,TK", [(64, 64), (256, 16), (128, 32), (64, 128), (256, 64), (256, 128)])
@pytest.mark.parametrize("zero_frac,tau", [(0.5, 0.0), (0.9, 0.0), (0.0, 0.7)])
def test_spmspv_matches_oracle(us, orc, TM, TK, zero_frac, tau):
    M, K = 512, 1024
    d = wl.spmspv(M, K, 0.5, zero_frac, seed=TM + TK)
    W, x = d["W"], d["x"]
    if zero_frac == 0.0:
        x = np.random.default_rng(9).standard_normal(K).astype(np.float16)   # both signs
    E = encode_gpu(us, W, TM, TK, F16, COL)
    y = run_spmspv(us, E, x, tau)
    _, exact = orc.spmspv_f16(W, x, tau)
    check_f16(y, exact, f"spmspv TM={TM} TK={TK} tau={tau}")


@pytest.mark.parametrize("M,K,TM,TK", [(64 * 400, 128, 64, 64), (512, 64 * 97, 64, 64), (1024, 1024, 128, 32)])
def test_spmspv_repeat(us, orc, M, K, TM, TK):
    """spMspV on tall, wide and mid-sized shapes (bands with one or several K
    slices): three calls on one workspace give bitwise identical results
    (fixed-order sums) and leave the workspace zero."""
    d = wl.spmspv(M, K, 0.5, 0.6, seed=M + K)
    E = encode_gpu(us, d["W"], TM, TK, F16, COL)
    xt = torch.from_numpy(d["x"].view(np.int16)).cuda()
    ws = us.workspace(us.US_OP_SPMSPV_F16, E, 1)
    outs = []
    for _ in range(3):
        y = torch.full((M,), 0x7E00, dtype=torch.int16, device="cuda")   # NaN until written
        us.us_spmspv_f16(E, xt, 0.0, y, ws)
        torch.cuda.synchronize()
        assert us.us_get_last_device_status() == us.US_OK
        outs.append(y.cpu().numpy())
    assert all(np.array_equal(outs[0], o) for o in outs[1:])
    assert torch.count_nonzero(ws).item() == 0
    _, exact = orc.spmspv_f16(d["W"], d["x"], 0.0)
    check_f16(outs[0].view(np.float16), exact, f"spmspv repeat {M}x{K}")


# --------------------------------------------------------- full-size shapes --
@pytest.mark.parametrize("static", [False, True])
@pytest.mark.parametrize("s", [0.3, 0.5, 0.7])
def test_w4a4_4096_full(us, orc, s, static):
    d = wl.w4a4(4096, 4096, 16, s, seed=0)
    E = encode_gpu(us, d["Wq"], 64, 64, I4, ROW)
    for N in (1, 8, 16):
        acc, y = run_w4a4(us, E, wl.pack_int4(d["Xq"][:N]), d["s_w"], d["s_x"][:N], N, static=static)
        oacc, oy = orc.spmm_w4a4(d["Wq"], d["Xq"][:N], d["s_w"], d["s_x"][:N], nthreads=orc.max_threads())
        assert np.array_equal(acc, oacc)
        assert np.array_equal(y.view(np.uint16), oy.view(np.uint16))


@pytest.mark.parametrize("static", [False, True])
@pytest.mark.parametrize("M,K", [(11008, 4096), (4096, 11008)])
def test_w4a4_ffn_full(us, orc, M, K, static):
    """The FFN shapes: with static weights a CTA's 73 tiles exceed its dense
    slots, so some are decoded before the dependency wait and the rest after."""
    d = wl.w4a4(M, K, 32, 0.5, seed=0, rows="beta")
    E = encode_gpu(us, d["Wq"], 64, 64, I4, ROW)
    for N in (1, 3, 4, 16, 32):
        acc, y = run_w4a4(us, E, wl.pack_int4(d["Xq"][:N]), d["s_w"], d["s_x"][:N], N, static=static)
        rng = np.random.default_rng(N)
        n_idx = rng.integers(0, N, 3000)
        m_idx = rng.integers(0, M, 3000)
        oacc, oy = orc.spmm_w4a4_at(d["Wq"], d["Xq"][:N], d["s_w"], d["s_x"][:N], n_idx, m_idx)
        assert np.array_equal(acc[n_idx, m_idx], oacc)
        assert np.array_equal(y[n_idx, m_idx].view(np.uint16), oy.view(np.uint16))


@pytest.mark.parametrize("static", [False, True])
def test_w4a4_balanced_wide_activation_block(us, orc, static):
    """153 x 257 tiles of 64 x 64: 259 tiles per CTA, so a CTA spans whole band
    widths and stages all 257 K tiles of every token (16 KB a token row at
    N = 16, one CTA per SM).  N = 2 (dp4a) and 16 (mma.sync); sampled outputs
    exact."""
    M, K = 64 * 153, 64 * 257
    rng = np.random.default_rng(257)
    W = rand_i4(rng, M, K, 0.3)
    Xq = rng.integers(-8, 8, size=(16, K)).astype(np.int8)
    s_w = (rng.random(M) * 0.01 + 1e-3).astype(np.float16)
    s_x = (rng.random(16) * 0.5 + 0.05).astype(np.float16)
    E = encode_gpu(us, W, 64, 64, I4, ROW)
    for N in (2, 16):
        assert us.us_pick_split_k(us.US_OP_SPMM_W4A4, E, N) == 0
        acc, y = run_w4a4(us, E, wl.pack_int4(Xq[:N]), s_w, s_x[:N], N, static=static)
        n_idx, m_idx = rng.integers(0, N, 3000), rng.integers(0, M, 3000)
        oacc, oy = orc.spmm_w4a4_at(W, Xq[:N], s_w, s_x[:N], n_idx, m_idx)
        assert np.array_equal(acc[n_idx, m_idx], oacc), N
        assert np.array_equal(y[n_idx, m_idx].view(np.uint16), oy.view(np.uint16)), N


@pytest.mark.parametrize("N", [256, 2048])
def test_f16_prefill_sampled(us, orc, N):
    d = wl.f16_spmm(4096, 4096, N, 0.6, seed=0)
    E = encode_gpu(us, d["W"], 64, 64, F16, ROW)
    y = run_f16(us, E, d["X"])
    rng = np.random.default_rng(N)
    n_idx = rng.integers(0, N, 4000)
    m_idx = rng.integers(0, 4096, 4000)
    _, exact = orc.spmm_f16_at(d["W"], d["X"], n_idx, m_idx)
    check_f16(y[n_idx, m_idx], exact, f"prefill N={N}")


@pytest.mark.parametrize("zero_frac", [0.5, 0.7, 0.9])
def test_spmspv_14336_full(us, orc, zero_frac):
    d = wl.spmspv(14336, 4096, 0.5, zero_frac, seed=0)
    E = encode_gpu(us, d["W"], 64, 64, F16, COL)
    y = run_spmspv(us, E, d["x"], 0.0)
    _, exact = orc.spmspv_f16(d["W"], d["x"], 0.0, nthreads=orc.max_threads())
    check_f16(y, exact, f"spmspv 14336 zeros={zero_frac}")


def test_one_workspace_shared_across_calls(us, orc):
    """Calls with different kernels, splits and token counts share one zero-filled
    workspace; each must leave behind the zeros the next one needs."""
    rng = np.random.default_rng(17)
    W = rand_i4(rng, 256, 1024, 0.5)
    E = encode_gpu(us, W, 64, 64, I4, ROW)
    Wf = rand_f16(rng, 256, 1024, 0.5)
    Ef = encode_gpu(us, Wf, 64, 64, F16, ROW)
    need = max(us.us_workspace_bytes(us.US_OP_SPMM_W4A4, E, n, s) for n in (1, 5, 13, 40) for s in (0, 2, 4))
    need = max(need, us.us_workspace_bytes(us.US_OP_SPMM_F16, Ef, 40, 4))
    need = max(need, us.us_workspace_bytes(us.US_OP_SPMM_F16, Ef, 100, 2))
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    one = np.ones(256, np.float16)
    for N, split in [(5, 4), (40, 2), (1, 0), (13, 4), (5, 2), (40, 4), (1, 4)]:
        Xq = rng.integers(-8, 8, size=(N, 1024)).astype(np.int8)
        Yacc = torch.empty(N, 256, dtype=torch.int32, device="cuda")
        us.us_spmm_w4a4(E, torch.from_numpy(wl.pack_int4(Xq)).cuda(), None, None, N, Yacc, None, ws, split)
        oacc, _ = orc.spmm_w4a4(W, Xq, one, np.ones(N, np.float16))
        assert np.array_equal(Yacc.cpu().numpy(), oacc), (N, split)
        X = rng.standard_normal((N, 1024)).astype(np.float16)
        Y = torch.empty(N, 256, dtype=torch.int16, device="cuda")
        us.us_spmm_f16(Ef, torch.from_numpy(X.view(np.int16)).cuda(), N, Y, ws, split)
        n_idx, m_idx = np.meshgrid(np.arange(N), np.arange(256), indexing="ij")
        _, exact = orc.spmm_f16_at(Wf, X, n_idx.reshape(-1), m_idx.reshape(-1))
        check_f16(Y.cpu().numpy().view(np.float16).reshape(-1), exact, f"shared ws N={N}")
    # tensor-core fp16 path with split-K and a ragged token tile: partials cleared too
    X = rng.standard_normal((100, 1024)).astype(np.float16)
    Y = torch.empty(100, 256, dtype=torch.int16, device="cuda")
    us.us_spmm_f16(Ef, torch.from_numpy(X.view(np.int16)).cuda(), 100, Y, ws, 2)
    n_idx, m_idx = np.meshgrid(np.arange(100), np.arange(256), indexing="ij")
    _, exact = orc.spmm_f16_at(Wf, X, n_idx.reshape(-1), m_idx.reshape(-1))
    check_f16(Y.cpu().numpy().view(np.float16).reshape(-1), exact, "shared ws tensor path")
    assert not ws.any().item(), "workspace not left zeroed"


def test_static_flag_same_results_back_to_back(us, orc):
    """Weights flagged US_BITMAP_STATIC may be fetched before the previous kernel
    ends; activations still are not.  Back-to-back calls where each call's
    activations are written by the kernel just before it must stay exact."""
    rng = np.random.default_rng(23)
    W = rand_i4(rng, 512, 2048, 0.5)
    E = encode_gpu(us, W, 64, 64, I4, ROW)
    E.flags = us.US_BITMAP_STATIC
    N = 4
    ws = us.workspace(us.US_OP_SPMM_W4A4, E, N)
    Xs = [rng.integers(-8, 8, size=(N, 2048)).astype(np.int8) for _ in range(6)]
    packed = [torch.from_numpy(wl.pack_int4(x)).cuda() for x in Xs]
    Xbuf = torch.empty_like(packed[0])
    outs = []
    for i in range(6):
        Xbuf.copy_(packed[i])                          # written right before the call
        Yacc = torch.empty(N, 512, dtype=torch.int32, device="cuda")
        us.us_spmm_w4a4(E, Xbuf, None, None, N, Yacc, None, ws)
        outs.append(Yacc)
    torch.cuda.synchronize()
    one = np.ones(512, np.float16)
    for i in range(6):
        oacc, _ = orc.spmm_w4a4(W, Xs[i], one, np.ones(N, np.float16))
        assert np.array_equal(outs[i].cpu().numpy(), oacc)
