"""Pins of the CPU oracle against what the pages and the mathematics fix.

No GPU.  Every check here compares the oracle with something other than itself:
worked examples printed on the pages (tests/golden), the Tiled-CBC storage
formula, a pure-Python brute force on tiny inputs (tests/brute.py), closed
forms (sparsity 0 -> dense GEMM via numpy, sparsity 100 % -> zero, one nonzero
-> one scaled activation), numpy's own fp16 conversions, and invariants
(round trip, per-tile popcount, offsets).
"""
import json
import os

import numpy as np
import pytest

from bitmap_encoded_unstructured_ie_gb300 import workloads as wl
from tests import brute

GOLD = os.path.join(os.path.dirname(__file__), "golden")
F16, I4, ROW, COL = 0, 1, 0, 1
I2 = 2


def _popcount64(a: np.ndarray) -> np.ndarray:
    a = a.astype(np.uint64)
    return np.array([bin(int(v)).count("1") for v in a.reshape(-1)], dtype=np.int64).reshape(a.shape)


def _rand_i4(rng, M, K, density):
    q = rng.integers(-8, 8, size=(M, K)).astype(np.int8)
    q[rng.random((M, K)) >= density] = 0
    return q


def _rand_i2(rng, M, K, density):
    q = rng.integers(-2, 2, size=(M, K)).astype(np.int8)
    q[rng.random((M, K)) >= density] = 0
    return q


def _rand_f16(rng, M, K, density):
    w = (rng.standard_normal((M, K)) * 0.02).astype(np.float16)
    w[rng.random((M, K)) >= density] = 0
    return w


# --------------------------------------------------------------- page pins --
def test_fig7_union_bitmap_words(orc):
    """UnionSparse Fig. 7: the four printed mask rows pack (leftmost = LSB)."""
    g = json.load(open(os.path.join(GOLD, "fig7_union_bitmap.json")))
    rows = [int(w, 16) for w in g["row_words"]]
    width = g["row_width"]
    W = np.zeros((4, width), dtype=np.int8)
    for i, word in enumerate(rows):
        for j in range(width):
            if (word >> j) & 1:
                W[i, j] = 1 + (i + j) % 7          # any nonzero payload
    # one 4 x 16 tile in row-major scan -> one 64-bit word, row i in bits 16i..16i+15
    bm, off, vals = orc.encode(W, 4, 16, I4, ROW)
    assert bm.size == 1
    expect = rows[0] | rows[1] << 16 | rows[2] << 32 | rows[3] << 48
    assert int(bm[0]) == expect
    for i in range(4):
        assert bin(rows[i]).count("1") == g["active_per_row"]
    assert int(_popcount64(bm).sum()) == g["P_t"]
    # Q = 1 here: the next offset is P_t rounded up to the 16-byte quantum
    assert int(off[1]) == (g["P_t"] + 31) // 32 * 32
    bmf, offf, _ = orc.encode(W.astype(np.float16), 4, 16, F16, ROW)
    assert int(bmf[0]) == expect and int(offf[1]) == g["P_t"]    # 40 is a multiple of 8
    # the Q-area offset of the figure is Q * P_t
    assert g["Q"] * g["P_t"] == g["next_offset_with_Q"]


def test_fig9c_segment_ranks(orc):
    """UnionSparse Fig. 9(c): segment 10110100 -> payload indices b..b+3."""
    g = json.load(open(os.path.join(GOLD, "fig9c_segment.json")))
    seg = [int(c) for c in g["segment_bits_position0_first"]]
    assert [p for p, b in enumerate(seg) if b] == g["active_positions"]
    # a 1 x 64 tile: 5 set positions before the segment give base b = 5
    W = np.zeros((1, 64), dtype=np.int8)
    W[0, 1:6] = [1, 2, 3, 4, 5]
    start = 16
    payload = [-8, 7, -1, 6]
    for v, p in zip(payload, g["active_positions"]):
        W[0, start + p] = v
    bm, off, vals = orc.encode(W, 1, 64, I4, ROW)
    assert (int(bm[0]) >> start) & 0xFF == 0b00101101 == 0x2D
    stream = orc.unpack_int4(vals, int(off[1]))
    b = 5
    for v, r in zip(payload, g["payload_index_minus_base"]):
        assert stream[b + r] == v
    dec = orc.decode(bm, off, vals, 1, 64, 1, 64, I4, ROW)
    assert np.array_equal(dec, W)


def test_tiled_cbc_storage_formula(orc):
    """SPDP 4.1: Stor = 4(N_GT+1) + 4 N_GT TILE_K + 8 N_BM + 2 NNZ.  Ours drops the
    ColInfo term and adds the 16-byte padding of each tile's run."""
    rng = np.random.default_rng(3)
    for (M, K, TM, TK) in [(256, 64, 256, 16), (128, 128, 64, 64), (512, 96, 256, 32)]:
        W = _rand_f16(rng, M, K, 0.45)
        bm, off, vals = orc.encode(W, TM, TK, F16, COL)
        NGT = (M // TM) * (K // TK)
        NBM = M * K // 64
        nz = (W.view(np.uint16) & 0x7FFF) != 0
        NNZ = int(nz.sum())
        per_tile = nz.reshape(M // TM, TM, K // TK, TK).sum(axis=(1, 3)).reshape(-1)
        pad_bytes = int(((-per_tile) % 8).sum()) * 2
        formula = 4 * (NGT + 1) + 4 * NGT * TK + 8 * NBM + 2 * NNZ
        ours = off.nbytes + bm.nbytes + vals.nbytes
        assert ours == formula - 4 * NGT * TK + pad_bytes


# ------------------------------------------------------------ brute force --
@pytest.mark.parametrize("elem", [F16, I4, I2])
@pytest.mark.parametrize("order", [ROW, COL])
@pytest.mark.parametrize("shape", [(8, 16, 8, 8), (16, 24, 8, 8), (4, 32, 4, 16), (64, 8, 64, 1)])
def test_encode_matches_brute_force(orc, elem, order, shape):
    M, K, TM, TK = shape
    rng = np.random.default_rng(M * 31 + K + elem * 7 + order)
    for density in (0.0, 0.3, 0.7, 1.0):
        if elem == F16:
            W = _rand_f16(rng, M, K, density).view(np.uint16)
        elif elem == I4:
            W = _rand_i4(rng, M, K, density)
        else:
            W = _rand_i2(rng, M, K, density)
        bm, off, vals = orc.encode(W, TM, TK, elem, order)
        words, offsets, data = brute.encode(brute.to_lists(W), TM, TK, elem, order)
        assert [int(v) for v in bm] == words
        assert [int(v) for v in off] == offsets
        assert bytes(vals.tobytes()) == data


def test_decode_matches_brute_force_values(orc):
    rng = np.random.default_rng(11)
    W = _rand_i4(rng, 8, 16, 0.5)
    words, offsets, data = brute.encode(brute.to_lists(W), 8, 8, I4, COL)
    dec = orc.decode(np.array(words, np.uint64), np.array(offsets, np.uint32),
                     np.frombuffer(data, np.uint8), 8, 16, 8, 8, I4, COL)
    assert np.array_equal(dec, W)


# ------------------------------------------------------------- invariants --
@pytest.mark.parametrize("elem", [F16, I4])
@pytest.mark.parametrize("order", [ROW, COL])
def test_round_trip_and_offsets(orc, elem, order):
    rng = np.random.default_rng(5 + elem + 2 * order)
    M, K, TM, TK = 256, 192, 64, 64
    for density in (0.0, 0.01, 0.5, 0.93, 1.0):
        W = _rand_f16(rng, M, K, density) if elem == F16 else _rand_i4(rng, M, K, density)
        bm, off, vals = orc.encode(W, TM, TK, elem, order)
        dec = orc.decode(bm, off, vals, M, K, TM, TK, elem, order)
        Wv = W.view(np.uint16) if elem == F16 else W
        assert np.array_equal(dec, Wv)
        wpt = TM * TK // 64
        P = _popcount64(bm).reshape(-1, wpt).sum(axis=1)
        E = 8 if elem == F16 else 32
        assert np.array_equal(np.diff(off.astype(np.int64)), (P + E - 1) // E * E)
        assert vals.nbytes == int(off[-1]) * (2 if elem == F16 else 1) // (1 if elem == F16 else 2)
        nz = (Wv & 0x7FFF) != 0 if elem == F16 else Wv != 0
        assert int(P.sum()) == int(nz.sum())


def test_row_and_col_orders_differ_but_decode_alike(orc):
    rng = np.random.default_rng(9)
    W = _rand_i4(rng, 128, 128, 0.5)
    a = orc.encode(W, 64, 64, I4, ROW)
    b = orc.encode(W, 64, 64, I4, COL)
    assert not np.array_equal(a[0], b[0])
    assert np.array_equal(orc.decode(*a, 128, 128, 64, 64, I4, ROW), orc.decode(*b, 128, 128, 64, 64, I4, COL))
    # same popcount per tile in both orders, so the offsets agree
    assert np.array_equal(a[1], b[1])


def test_f16_signed_zero_and_nan_presence(orc):
    W = np.zeros((64, 64), dtype=np.uint16)
    W[0, 0] = 0x8000          # -0.0: not stored
    W[0, 1] = 0x7E00          # NaN: stored
    W[5, 7] = 0x3C00          # 1.0
    bm, off, vals = orc.encode(W, 64, 64, F16, ROW)
    assert int(bm[0]) == 0b10 and int(off[1]) == 8
    dec = orc.decode(bm, off, vals, 64, 64, 64, 64, F16, ROW)
    assert dec[0, 0] == 0 and dec[0, 1] == 0x7E00 and dec[5, 7] == 0x3C00


def test_decode_rejects_corrupt_offsets(orc):
    rng = np.random.default_rng(2)
    W = _rand_i4(rng, 64, 128, 0.5)
    bm, off, vals = orc.encode(W, 64, 64, I4, ROW)
    bad = off.copy(); bad[1] = bad[2] + 32                     # not monotone
    with pytest.raises(orc.OracleError):
        orc.decode(bm, bad, vals, 64, 128, 64, 64, I4, ROW)
    bad = off.copy(); bad[1] -= 32                              # run shorter than popcount
    with pytest.raises(orc.OracleError):
        orc.decode(bm, bad, vals, 64, 128, 64, 64, I4, ROW)
    with pytest.raises(orc.OracleError):                        # values buffer too short
        orc.decode(bm, off, vals[:-16], 64, 128, 64, 64, I4, ROW)


def test_encode_rejects_bad_shapes_and_codes(orc):
    with pytest.raises(orc.OracleError):
        orc.encode(np.zeros((60, 64), np.int8), 64, 64, I4, ROW)
    with pytest.raises(orc.OracleError):
        orc.encode(np.full((64, 64), 9, np.int8), 64, 64, I4, ROW)


# ---------------------------------------------------------------- fp16 ----
def test_half_conversions_match_numpy(orc):
    for bits in list(range(0, 65536, 97)) + [0x7BFF, 0xFBFF, 0x0001, 0x8001, 0x3C00]:
        f = orc.half_to_float(bits)
        ref = float(np.array([bits], np.uint16).view(np.float16)[0])
        assert (f == ref) or (np.isnan(f) and np.isnan(ref))
    rng = np.random.default_rng(0)
    for x in np.concatenate([rng.standard_normal(2000) * 10.0 ** rng.integers(-8, 5, 2000),
                             [65519.99, 65520.0, 1e-8, 2.0 ** -25, 3 * 2.0 ** -26]]):
        assert orc.double_to_half(float(x)) == int(np.array([x], np.float64).astype(np.float16).view(np.uint16)[0])
        xf = np.float32(x)
        assert orc.float_to_half(float(xf)) == int(np.array([xf]).astype(np.float16).view(np.uint16)[0])


def test_int4_unpack_matches_independent_packer(orc):
    rng = np.random.default_rng(4)
    codes = rng.integers(-8, 8, size=1001).astype(np.int8)
    packed = wl.pack_int4(codes)
    assert np.array_equal(orc.unpack_int4(packed, codes.size), codes)
    assert packed[0] == ((int(codes[0]) & 15) | ((int(codes[1]) & 15) << 4))


# -------------------------------------------------------------- multiply ----
def test_w4a4_dense_equals_numpy_gemm(orc):
    """Sparsity 0: the product is the plain integer GEMM (numpy int64)."""
    rng = np.random.default_rng(7)
    M, K, N = 96, 160, 5
    W = rng.integers(-8, 8, size=(M, K)).astype(np.int8)
    X = rng.integers(-8, 8, size=(N, K)).astype(np.int8)
    s_w = (rng.random(M) * 0.01 + 1e-3).astype(np.float16)
    s_x = (rng.random(N) * 0.5 + 0.1).astype(np.float16)
    acc, y = orc.spmm_w4a4(W, X, s_w, s_x)
    ref = X.astype(np.int64) @ W.astype(np.int64).T
    assert np.array_equal(acc.astype(np.int64), ref)
    # dequantisation: two fp32 products, one fp16 rounding (numpy's own ops)
    yref = ((ref.astype(np.float32) * s_w.astype(np.float32)[None, :]) * s_x.astype(np.float32)[:, None]).astype(np.float16)
    assert np.array_equal(y.view(np.uint16), yref.view(np.uint16))


def test_w4a4_extremes_and_threads(orc):
    M, K, N = 64, 4096, 2
    W = np.full((M, K), -8, np.int8)
    X = np.full((N, K), -8, np.int8)
    one = np.ones(M, np.float16)
    acc, _ = orc.spmm_w4a4(W, X, one, np.ones(N, np.float16))
    assert (acc == 64 * K).all()
    W[:, 1::2] = 7
    acc4, _ = orc.spmm_w4a4(W, X, one, np.ones(N, np.float16), nthreads=4)
    assert (acc4 == (64 - 56) * K // 2).all()


def test_sparse_special_cases(orc):
    rng = np.random.default_rng(12)
    M, K, N = 128, 128, 3
    X = rng.integers(-8, 8, size=(N, K)).astype(np.int8)
    s = np.ones(M, np.float16)
    W = np.zeros((M, K), np.int8)                                    # sparsity 100 %
    bm, off, vals = orc.encode(W, 64, 64, I4, ROW)
    assert vals.size == 0 and int(off[-1]) == 0
    Wd = orc.decode(bm, off, vals, M, K, 64, 64, I4, ROW)
    acc, y = orc.spmm_w4a4(Wd, X, s, np.ones(N, np.float16))
    assert not acc.any() and not y.view(np.uint16).any()
    W[37, 99] = -5                                                   # one nonzero
    Wd = orc.decode(*orc.encode(W, 64, 64, I4, ROW), M, K, 64, 64, I4, ROW)
    acc, _ = orc.spmm_w4a4(Wd, X, s, np.ones(N, np.float16))
    expect = np.zeros((N, M), np.int64)
    expect[:, 37] = -5 * X[:, 99].astype(np.int64)
    assert np.array_equal(acc.astype(np.int64), expect)


def test_tiny_products_match_brute_force(orc):
    rng = np.random.default_rng(21)
    M, K, N = 8, 24, 3
    W = _rand_i4(rng, M, K, 0.5)
    X = rng.integers(-8, 8, size=(N, K)).astype(np.int8)
    acc, _ = orc.spmm_w4a4(W, X, np.ones(M, np.float16), np.ones(N, np.float16))
    for n in range(N):
        for m in range(M):
            assert acc[n, m] == brute.dot_w4a4(W[m], X[n])
    Wf = _rand_f16(rng, M, K, 0.6)
    Xf = rng.standard_normal((N, K)).astype(np.float16)
    y = orc.spmm_f16(Wf, Xf)
    for n in range(N):
        for m in range(M):
            exact = brute.dot_f16_exact(Wf[m], Xf[n])
            assert y[n, m] == np.float16(float(exact))


def test_f16_dense_equals_fp64_gemm(orc):
    """Sparsity 0: fp16 output = fp16(fp64 GEMM); the fp64 sum agrees with numpy."""
    rng = np.random.default_rng(8)
    M, K, N = 64, 512, 4
    W = (rng.standard_normal((M, K)) * 0.02).astype(np.float16)
    X = rng.standard_normal((N, K)).astype(np.float16)
    y = orc.spmm_f16(W, X)
    ref = X.astype(np.float64) @ W.astype(np.float64).T
    n_idx, m_idx = np.meshgrid(np.arange(N), np.arange(M), indexing="ij")
    y_at, exact = orc.spmm_f16_at(W, X, n_idx.reshape(-1), m_idx.reshape(-1))
    assert np.allclose(exact, ref.reshape(-1), rtol=1e-12, atol=1e-15)
    assert np.array_equal(y_at.view(np.uint16), exact.astype(np.float16).view(np.uint16))
    assert np.array_equal(y.reshape(-1).view(np.uint16), y_at.view(np.uint16))


def test_sampled_w4a4_equals_full(orc):
    d = wl.w4a4(128, 256, 3, 0.5, seed=1)
    acc, y = orc.spmm_w4a4(d["Wq"], d["Xq"], d["s_w"], d["s_x"])
    n = np.array([0, 2, 1, 2]); m = np.array([0, 127, 64, 5])
    a2, y2 = orc.spmm_w4a4_at(d["Wq"], d["Xq"], d["s_w"], d["s_x"], n, m)
    assert np.array_equal(a2, acc[n, m]) and np.array_equal(y2.view(np.uint16), y[n, m].view(np.uint16))


def test_spmspv_tau0_equals_spmv_and_threshold_is_mask(orc):
    """SPDP section 2: W.(x (.) M(x)); with tau = 0 skipping zeros changes nothing,
    and a COL-order encoding decodes to the same W as the ROW-order one."""
    d = wl.spmspv(256, 512, 0.5, 0.7, seed=3)
    W, x = d["W"], d["x"]
    col = orc.encode(W, 64, 64, F16, COL)
    row = orc.encode(W, 64, 64, F16, ROW)
    Wc = orc.decode(*col, 256, 512, 64, 64, F16, COL)
    Wr = orc.decode(*row, 256, 512, 64, 64, F16, ROW)
    assert np.array_equal(Wc, Wr)
    y, ex = orc.spmspv_f16(Wc, x, 0.0)
    y2 = orc.spmm_f16(Wr, x.reshape(1, -1))
    assert np.array_equal(y.view(np.uint16), y2.reshape(-1).view(np.uint16))
    tau = 0.6
    x = np.random.default_rng(5).standard_normal(512).astype(np.float16)   # both signs
    y3, ex3 = orc.spmspv_f16(Wc, x, tau)
    xm = np.where(np.abs(x.astype(np.float64)) > tau, x.astype(np.float64), 0.0)
    ref = Wc.view(np.float16).astype(np.float64) @ xm
    assert np.allclose(ex3, ref, rtol=1e-12, atol=1e-15)
    assert np.array_equal(y3.view(np.uint16), ex3.astype(np.float16).view(np.uint16))


# ----------------------------------------------------------- workloads -----
def test_workload_statistics():
    d = wl.w4a4(256, 1024, 2, 0.7, seed=0)
    dens = (d["Wq"] != 0).mean()
    assert 0.25 < dens < 0.31
    kept_rows = (d["Wq"] != 0).sum(axis=1)
    assert kept_rows.max() <= round(0.3 * 1024)
    b = wl.w4a4(512, 1024, 1, 0.5, seed=0, rows="beta")
    rd = (b["Wq"] != 0).mean(axis=1)
    assert rd.min() > 0.25 and rd.max() < 0.71 and abs(rd.mean() - 0.5) < 0.05
    x = wl.spmspv(64, 4096, 0.5, 0.9, seed=0)["x"]
    assert abs((x == 0).mean() - 0.9) < 1e-3


def test_clustered_workload_shares_patterns(orc):
    """Rows in groups of four share column scales before magnitude pruning,
    then are shuffled within each 16-row block: the density stays near the
    target, the recipe is seeded, and the row reordering finds groups whose
    4 x 1 area union is much sparser than that of the plain random workload."""
    c = wl.w4a4(64, 256, 1, 0.7, seed=0, rows="clustered")
    assert np.array_equal(c["Wq"], wl.w4a4(64, 256, 1, 0.7, seed=0, rows="clustered")["Wq"])
    assert 0.25 < (c["Wq"] != 0).mean() < 0.31
    r = wl.w4a4(64, 256, 1, 0.7, seed=0)
    cost = {}
    for name, W in (("clustered", c["Wq"]), ("random", r["Wq"])):
        cost[name] = sum(orc.reorder_rows(W[b:b + 16, k:k + 64] != 0, 4, 1)[1]
                         for b in range(0, 64, 16) for k in range(0, 256, 64))
    # union cost in set positions over 16 tiles of 4 x 64 logical positions
    assert cost["clustered"] < 0.8 * cost["random"], cost


# ------------------------------------------------- activation quantisation --
# UnionSparse Fig. 2 "Quant" (FP16 X -> INT4 X, per-token scale): s = fp16(amax / 7),
# codes = clamp(rint(x / s), -8, 7) with ties to even, s = 1 for an all-zero token.

def test_quantize_worked_examples(orc):
    """Hand-worked tokens: amax 7 gives s = 1 exactly, so codes are rint(x)."""
    X = np.array([[1, -2, 3.5, 7],          # 3.5 -> 4 (tie to even)
                  [0.5, 1.5, 2.5, -7],       # ties: 0.5 -> 0, 1.5 -> 2, 2.5 -> 2
                  [-7, 3, 0, 6.5],           # the maximum magnitude may be negative; 6.5 -> 6
                  [0, 0, 0, 0]], np.float16)  # all zero: scale 1, codes 0
    codes, s = orc.quantize_x(X)
    assert codes.tolist() == [[1, -2, 4, 7], [0, 2, 2, -7], [-7, 3, 0, 6], [0, 0, 0, 0]]
    assert s.tolist() == [1.0, 1.0, 1.0, 1.0]
    # amax 14 -> s = 2: every code halves
    c2, s2 = orc.quantize_x(X[:1] * 2)
    assert s2.tolist() == [2.0] and c2.tolist() == [[1, -2, 4, 7]]
    # amax 3.5: s = fp16(0.5) exactly; x = 1.25 -> 2.5 -> 2 (tie to even), 1.75 -> 3.5 -> 4
    c3, s3 = orc.quantize_x(np.array([[1.25, 1.75, -3.5, 0.25]], np.float16))
    assert s3.tolist() == [0.5] and c3.tolist() == [[2, 4, -7, 0]]


def test_quantize_invariants(orc):
    """On random tokens: the largest magnitude lands on +-7, every other value
    is within half a step, and scaling a token by a power of two scales s only."""
    rng = np.random.default_rng(5)
    X = (rng.standard_normal((64, 256)) * rng.uniform(0.01, 50, (64, 1))).astype(np.float16)
    codes, s = orc.quantize_x(X)
    xf, sf = X.astype(np.float64), s.astype(np.float64)
    assert codes.min() >= -8 and codes.max() <= 7
    big = np.argmax(np.abs(xf), axis=1)
    assert np.all(np.abs(codes[np.arange(64), big]) == 7)
    err = np.abs(xf - codes * sf[:, None])
    assert np.all(err <= sf[:, None] * (0.5 + 1e-3))
    c4, s4 = orc.quantize_x((X.astype(np.float32) * 4).astype(np.float16))
    assert np.array_equal(c4, codes) and np.array_equal(s4.astype(np.float32), s.astype(np.float32) * 4)


# ------------------------------------------------------------------ ColInfo --
def _colinfo_from_dense(W: np.ndarray, TM: int, TK: int) -> np.ndarray:
    """ColInfo counted on the dense matrix itself (no bitmap): per tile, per
    column, its nonzeros and the nonzeros of the columns before it."""
    M, K = W.shape
    out = []
    for tm in range(M // TM):
        for tk in range(K // TK):
            blk = W[tm * TM:(tm + 1) * TM, tk * TK:(tk + 1) * TK]
            nnz = np.count_nonzero(blk.astype(np.float32) != 0, axis=0)
            off = np.concatenate([[0], np.cumsum(nnz)[:-1]])
            out.append((off.astype(np.uint32) << 16) | nnz.astype(np.uint32))
    return np.concatenate(out)


def test_colinfo_worked_example(orc):
    """Column j of the only tile holds j nonzeros (rows 0..j-1): NNZ_Column = j
    and TileOffset_Col = 0 + 1 + ... + (j - 1) = j (j - 1) / 2."""
    TM, TK = 64, 16
    W = np.zeros((TM, TK), np.float16)
    for j in range(TK):
        W[:j, j] = 1.0 + j
    bm, off, vals = orc.encode(W, TM, TK, F16, COL)
    ci = orc.colinfo(bm, TM, TK, TM, TK)
    assert [int(v) & 0xFFFF for v in ci] == list(range(TK))
    assert [int(v) >> 16 for v in ci] == [j * (j - 1) // 2 for j in range(TK)]


@pytest.mark.parametrize("shape", [(128, 256, 64, 64), (256, 64, 256, 16), (192, 384, 64, 128), (128, 96, 128, 32)])
def test_colinfo_matches_dense_counts(orc, shape):
    M, K, TM, TK = shape
    rng = np.random.default_rng(M + K)
    W = _rand_f16(rng, M, K, 0.45)
    W[:, 5] = 0                                     # an empty column
    W[: TM, K - 1] = 1.0                            # a full column
    bm, off, vals = orc.encode(W, TM, TK, F16, COL)
    ci = orc.colinfo(bm, M, K, TM, TK)
    assert np.array_equal(ci, _colinfo_from_dense(W, TM, TK))


def test_colinfo_addresses_each_column_run(orc):
    """TileOffset_Col points at the column's first value in the tile's run and
    NNZ_Column values follow: they are that column's nonzeros in row order."""
    M, K, TM, TK = 128, 128, 64, 32
    rng = np.random.default_rng(3)
    W = _rand_f16(rng, M, K, 0.5)
    bm, off, vals = orc.encode(W, TM, TK, F16, COL)
    ci = orc.colinfo(bm, M, K, TM, TK)
    v16 = vals.view(np.float16)
    nTK = K // TK
    for t in range((M // TM) * nTK):
        tm, tk = divmod(t, nTK)
        for j in range(TK):
            o, n = int(ci[t * TK + j]) >> 16, int(ci[t * TK + j]) & 0xFFFF
            col = W[tm * TM:(tm + 1) * TM, tk * TK + j]
            want = col[col.astype(np.float32) != 0]
            got = v16[int(off[t]) + o: int(off[t]) + o + n]
            assert np.array_equal(got.view(np.uint16), want.view(np.uint16)), (t, j)


def test_batched_spmspv_pins(orc):
    """Per-token dynamic pruning: with tau = 0 and no zero activations the
    batched spMspV is the dense fp16 product; a token whose activations all
    fail the test gives zeros; every row equals that token's own spMspV."""
    rng = np.random.default_rng(8)
    M, K, N = 96, 128, 4
    W = _rand_f16(rng, M, K, 0.5)
    X = rng.standard_normal((N, K)).astype(np.float16)
    X[X == 0] = np.float16(0.5)
    Y0, ex0 = orc.spmspv_f16_batched(W, X, 0.0)
    Yd = orc.spmm_f16(W, X)
    assert np.array_equal(Y0.view(np.uint16), Yd.view(np.uint16))
    X[2] = np.clip(X[2], -0.25, 0.25)
    Y1, ex1 = orc.spmspv_f16_batched(W, X, 0.25)
    assert not Y1[2].view(np.uint16).any()
    for n in range(N):
        y, e = orc.spmspv_f16(W, X[n], 0.25)
        assert np.array_equal(Y1[n].view(np.uint16), y.view(np.uint16))
    # the pruned product equals the dense product of the pruned activations
    Xp = np.where(np.abs(X.astype(np.float32)) > 0.25, X, np.float16(0))
    assert np.allclose(ex1, Xp.astype(np.float64) @ W.astype(np.float64).T, rtol=0, atol=1e-9)


# ------------------------------------------------- IE-BME with Q = RA*CA areas --
def test_fig7_areas_union_mask_and_offset(orc):
    """UnionSparse Fig. 7 with its four areas: the printed logical rows are the
    union of the areas' masks, P_t = 40 active positions, and the LT's payload
    of Q * P_t = 160 int4 values puts the next offset at 160."""
    g = json.load(open(os.path.join(GOLD, "fig7_union_bitmap.json")))
    rows = [int(w, 16) for w in g["row_words"]]
    LM, LK, RA, CA = 4, g["row_width"], 2, 2
    W = np.zeros((LM * RA, LK * CA), np.int8)
    for i, word in enumerate(rows):
        for j in range(LK):
            if (word >> j) & 1:
                q = (i + j) % 4                              # the nonzero sits in any one area
                a, c = divmod(q, CA)
                W[a * LM + i, c * LK + j] = 1 + (i + 3 * j) % 7
    bm, off, vals = orc.encode_ie(W, LM * RA, LK * CA, RA, CA, I4)
    assert bm.size == 1
    assert int(bm[0]) == rows[0] | rows[1] << 16 | rows[2] << 32 | rows[3] << 48
    assert int(_popcount64(bm).sum()) == g["P_t"] == 40
    assert int(off[1]) == g["next_offset_with_Q"] == 160
    assert np.array_equal(orc.decode_ie(bm, off, vals, *W.shape, LM * RA, LK * CA, RA, CA, I4), W)


def test_fig7_aligned_values_include_zeros(orc):
    """A set logical position emits one value per area even when some are zero
    (the red-framed [1, 30, 59, 0] of Fig. 7): CV[o_t + q P_t + rho]."""
    RA, CA, LM, LK = 2, 2, 4, 16
    W = np.zeros((LM * RA, LK * CA), np.float16)
    i, j = 2, 5                                              # one logical position ...
    for q, v in enumerate([1.0, 30.0, 59.0, 0.0]):           # ... its four area values
        a, c = divmod(q, CA)
        W[a * LM + i, c * LK + j] = v
    W[0, 0] = 7.0                                           # an earlier position: rho = 1
    bm, off, vals = orc.encode_ie(W, LM * RA, LK * CA, RA, CA, F16)
    P = int(_popcount64(bm).sum())
    assert P == 2
    v16 = vals.view(np.float16)
    assert [float(v16[q * P + 1]) for q in range(4)] == [1.0, 30.0, 59.0, 0.0]
    assert [float(v16[q * P + 0]) for q in range(4)] == [7.0, 0.0, 0.0, 0.0]


@pytest.mark.parametrize("cfg", [(16, 64, 2, 2), (16, 64, 4, 1), (16, 64, 1, 4), (64, 64, 2, 1), (64, 128, 1, 2),
                                 (8, 32, 2, 2)])
@pytest.mark.parametrize("elem", [F16, I4])
def test_ie_round_trip_with_row_permutations(orc, cfg, elem):
    TM, TK, RA, CA = cfg
    rng = np.random.default_rng(TM * 7 + TK + RA + 10 * CA + elem)
    M, K = TM * 3, TK * 2
    W = _rand_f16(rng, M, K, 0.35) if elem == F16 else _rand_i4(rng, M, K, 0.35)
    nT = (M // TM) * (K // TK)
    perm = np.concatenate([rng.permutation(TM) for _ in range(nT)]).astype(np.uint8)
    for pm in (None, perm):
        bm, off, vals = orc.encode_ie(W, TM, TK, RA, CA, elem, pm)
        D = orc.decode_ie(bm, off, vals, M, K, TM, TK, RA, CA, elem, pm)
        assert np.array_equal(D.view(np.uint8), W.view(np.uint8))
        # the run of each tile is Q * P_t padded to 16 bytes
        Q, E = RA * CA, (8 if elem == F16 else 32)
        wpt = TM * TK // (64 * Q)
        P = _popcount64(bm).reshape(nT, wpt).sum(axis=1)
        assert np.array_equal(np.diff(off.astype(np.int64)), (Q * P + E - 1) // E * E)


def test_ie_single_area_is_the_plain_format(orc):
    """Q = 1 with the identity permutation is the plain row-scan encoding."""
    rng = np.random.default_rng(1)
    W = _rand_i4(rng, 128, 128, 0.5)
    a = orc.encode_ie(W, 64, 64, 1, 1, I4)
    b = orc.encode(W, 64, 64, I4, ROW)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def _brute_min_cost(mask, RA, CA):
    """Every partition of the rows into groups of RA, by plain recursion."""
    HL, KL = mask.shape
    LK = KL // CA

    def cost(g):
        return sum(any(mask[r, c * LK + j] for r in g for c in range(CA)) for j in range(LK))

    def rec(rest):
        if not rest:
            return 0
        first, others = rest[0], rest[1:]
        best = None
        from itertools import combinations
        for mates in combinations(others, RA - 1):
            g = (first,) + mates
            v = cost(g) + rec([r for r in others if r not in mates])
            best = v if best is None or v < best else best
        return best

    return rec(list(range(HL)))


@pytest.mark.parametrize("shape", [(4, 8, 2, 1), (6, 8, 2, 2), (8, 16, 2, 2), (8, 8, 4, 1), (8, 16, 4, 2),
                                   (8, 12, 2, 3)])
def test_reorder_dp_matches_brute_force(orc, shape):
    HL, KL, RA, CA = shape
    rng = np.random.default_rng(HL * 31 + KL + RA + CA)
    for trial in range(6):
        mask = rng.random((HL, KL)) < rng.uniform(0.1, 0.6)
        perm, cost = orc.reorder_rows(mask, RA, CA)
        assert cost == _brute_min_cost(mask, RA, CA)
        assert sorted(perm.tolist()) == list(range(HL))
        # the permutation realises that cost: union bits of the reordered tile
        G = HL // RA
        groups = [[int(perm[p * G + g]) for p in range(RA)] for g in range(G)]
        LK = KL // CA
        realised = sum(any(mask[r, c * LK + j] for r in grp for c in range(CA)) for grp in groups for j in range(LK))
        assert realised == cost
        # canonical: ascending inside a group, groups in lexicographic order
        assert all(grp == sorted(grp) for grp in groups) and groups == sorted(groups)


def test_reordering_never_grows_the_union_mask(orc):
    rng = np.random.default_rng(6)
    W = _rand_i4(rng, 64, 128, 0.4)
    base = orc.encode_ie(W, 16, 64, 2, 2, I4)
    perm = orc.reorder_matrix(W, 16, 64, 2, 2)
    re = orc.encode_ie(W, 16, 64, 2, 2, I4, perm)
    nT = 4 * 2
    pb = _popcount64(base[0]).reshape(nT, -1).sum(axis=1)
    pr = _popcount64(re[0]).reshape(nT, -1).sum(axis=1)
    assert np.all(pr <= pb) and pr.sum() < pb.sum()


# ---------------------------------------------------------------- W2A4 --
def test_int2_packing_worked_example(orc):
    """The int2 reading: four values per byte, the earlier element in the lower
    bits, two's complement.  Row [1, -1, -2, 0, 1, 1, -2, -1]: the seven
    nonzeros pack to 0b01_10_11_01 = 0x6D and 0b00_11_10_01 = 0x39, then zero
    padding to 64 elements (16 bytes)."""
    W = np.zeros((1, 64), np.int8)
    W[0, :8] = [1, -1, -2, 0, 1, 1, -2, -1]
    bm, off, vals = orc.encode(W, 1, 64, I2, ROW)
    assert int(bm[0]) == 0b11110111
    assert int(off[1]) == 64 and vals.size == 16
    assert vals[0] == 0x6D and vals[1] == 0x39 and not vals[2:].any()
    assert np.array_equal(orc.decode(bm, off, vals, 1, 64, 1, 64, I2, ROW), W)


def test_w2a4_dense_equals_numpy_gemm_and_refuses_range(orc):
    rng = np.random.default_rng(12)
    M, K, N = 64, 192, 5
    W = rng.integers(-2, 2, size=(M, K)).astype(np.int8)      # every code, zeros included
    X = rng.integers(-8, 8, size=(N, K)).astype(np.int8)
    bm, off, vals = orc.encode(W, 64, 64, I2, ROW)
    Wd = orc.decode(bm, off, vals, M, K, 64, 64, I2, ROW)
    assert np.array_equal(Wd, W)
    one = np.ones(M, np.float16)
    acc, _ = orc.spmm_w4a4(Wd, X, one, np.ones(N, np.float16))
    assert np.array_equal(acc.astype(np.int64), X.astype(np.int64) @ W.T.astype(np.int64))
    for bad in (2, -3, 7):
        Wb = W.copy()
        Wb[3, 5] = bad
        with pytest.raises(Exception):
            orc.encode(Wb, 64, 64, I2, ROW)
