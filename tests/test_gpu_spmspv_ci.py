"""ColInfo and the batched spMspV that reads it, through the C ABI, against the
CPU oracle.  Bars: ColInfo words bit-exact; fp16 outputs (fp32 accumulation)
within relative L2 <= 1e-3 and max-abs <= 2e-2 of the oracle's fp64 sums.
Shapes cover every tile height and width, K slices that do not divide the
tile count, token counts that leave a ragged token block, tokens whose every
activation is pruned, and ColInfo that contradicts the bitmap.
"""
import numpy as np
import pytest
import torch

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


def rand_f16(rng, M, K, density, scale=0.02):
    w = (rng.standard_normal((M, K)) * scale).astype(np.float16)
    w[rng.random((M, K)) >= density] = 0
    return w


def relu_acts(rng, N, K, zeros):
    """ReLU-thresholded N(0,1) activations with about `zeros` of them zero."""
    x = rng.standard_normal((N, K))
    thr = np.quantile(x, zeros) if zeros > 0 else -np.inf
    return np.where(x > thr, x, 0.0).astype(np.float16)


def check_f16(y_gpu, exact, what=""):
    y = y_gpu.astype(np.float64)
    err = y - exact
    rel = np.linalg.norm(err) / max(np.linalg.norm(exact), 1e-30)
    mx = np.abs(err).max() if err.size else 0.0
    assert rel <= REL_L2 and mx <= MAX_ABS, f"{what}: rel L2 {rel:.3e}, max abs {mx:.3e}"


def upload(us, orc_arrays, M, K, TM, TK, elem, order):
    bm, off, vals = orc_arrays
    dev = "cuda"
    return us.Encoded(M, K, TM, TK, elem, order,
                      torch.from_numpy(np.ascontiguousarray(bm).view(np.int64)).to(dev),
                      torch.from_numpy(np.ascontiguousarray(off).view(np.int32)).to(dev),
                      torch.from_numpy(np.concatenate([vals, np.zeros(16, np.uint8)])).to(dev),
                      int(vals.size))


CI_SHAPES = [
    # M, K, TM, TK
    (256, 512, 64, 64),
    (192, 320, 64, 16),
    (512, 256, 128, 32),
    (256, 256, 256, 128),
    (128, 384, 64, 128),
    (256, 64, 256, 16),
]


@pytest.mark.parametrize("shape", CI_SHAPES)
@pytest.mark.parametrize("elem", [F16, I4])
def test_colinfo_bit_exact(us, orc, shape, elem):
    M, K, TM, TK = shape
    rng = np.random.default_rng(M + 3 * K + TM + TK + elem)
    for density in (0.0, 0.3, 1.0):
        if elem == F16:
            W = rand_f16(rng, M, K, density)
        else:
            W = rng.integers(-8, 8, size=(M, K)).astype(np.int8)
            W[rng.random((M, K)) >= density] = 0
        arrs = orc.encode(W, TM, TK, elem, COL)
        E = upload(us, arrs, M, K, TM, TK, elem, COL)
        ci = us.us_colinfo(E)
        torch.cuda.synchronize()
        got = ci.cpu().numpy().view(np.uint32)
        assert np.array_equal(got, orc.colinfo(arrs[0], M, K, TM, TK)), density


SPV_CASES = [
    # M, K, TM, TK, N, density, activation zeros, tau
    (256, 1024, 64, 64, 1, 0.5, 0.5, 0.0),
    (256, 1024, 64, 64, 3, 0.5, 0.9, 0.0),
    (192, 1600, 64, 16, 8, 0.4, 0.7, 0.25),      # 100 K tiles: uneven K slices
    (512, 512, 128, 32, 5, 0.5, 0.5, 0.5),       # NB = 4: a ragged second block
    (256, 2048, 256, 128, 3, 0.6, 0.9, 0.0),     # NB = 2 at TM = 256
    (128, 640, 64, 128, 11, 0.5, 0.3, 1.0),      # two blocks of 8, the second ragged
    (64, 4096, 64, 64, 2, 0.5, 0.99, 0.0),       # one band, nearly every column skipped
]


@pytest.mark.parametrize("case", SPV_CASES)
def test_spmspv_ci_matches_oracle(us, orc, case):
    M, K, TM, TK, N, dens, zeros, tau = case
    rng = np.random.default_rng(M * 7 + K + N)
    W = rand_f16(rng, M, K, dens)
    X = relu_acts(rng, N, K, zeros)
    arrs = orc.encode(W, TM, TK, F16, COL)
    E = upload(us, arrs, M, K, TM, TK, F16, COL)
    ci = us.us_colinfo(E)
    Xt = torch.from_numpy(X.view(np.int16)).cuda()
    for rep in range(2):                               # the clusters leave nothing behind
        Y = torch.full((N, M), 0x7E00, dtype=torch.int16, device="cuda")
        us.us_spmspv_f16_ci(E, ci, Xt, N, tau, Y)
        torch.cuda.synchronize()
        assert us.us_get_last_device_status() == us.US_OK
        _, exact = orc.spmspv_f16_batched(W, X, tau)
        check_f16(Y.cpu().numpy().view(np.float16).reshape(-1), exact.reshape(-1), f"{case} rep {rep}")


def test_spmspv_ci_pruned_token_and_empty_matrix(us, orc):
    M, K, TM, TK, N = 256, 512, 64, 64, 4
    rng = np.random.default_rng(11)
    W = rand_f16(rng, M, K, 0.5)
    X = relu_acts(rng, N, K, 0.5)
    X[1] = np.clip(X[1], -0.1, 0.1)                    # every activation of token 1 fails |x| > 0.1
    arrs = orc.encode(W, TM, TK, F16, COL)
    E = upload(us, arrs, M, K, TM, TK, F16, COL)
    ci = us.us_colinfo(E)
    Y = torch.empty(N, M, dtype=torch.int16, device="cuda")
    us.us_spmspv_f16_ci(E, ci, torch.from_numpy(X.view(np.int16)).cuda(), N, 0.1, Y)
    torch.cuda.synchronize()
    y = Y.cpu().numpy().view(np.float16)
    assert not y[1].view(np.uint16).any()
    _, exact = orc.spmspv_f16_batched(W, X, 0.1)
    check_f16(y.reshape(-1), exact.reshape(-1), "pruned token")
    # an all-zero matrix: every column empty, so nothing is fetched
    Z = np.zeros((M, K), np.float16)
    arrs0 = orc.encode(Z, TM, TK, F16, COL)
    E0 = upload(us, arrs0, M, K, TM, TK, F16, COL)
    ci0 = us.us_colinfo(E0)
    assert not ci0.any().item()
    Y0 = torch.full((N, M), 0x3C00, dtype=torch.int16, device="cuda")
    us.us_spmspv_f16_ci(E0, ci0, torch.from_numpy(X.view(np.int16)).cuda(), N, 0.0, Y0)
    torch.cuda.synchronize()
    assert not Y0.any().item()


def test_spmspv_ci_agrees_with_bitmap_scan_kernel(us, orc):
    """N = 1: the ColInfo kernel and the bitmap-scanning spMspV compute the same
    masked product (both within the bar of the oracle, and close to each other)."""
    M, K, TM, TK = 512, 2048, 64, 64
    rng = np.random.default_rng(5)
    W = rand_f16(rng, M, K, 0.5)
    x = relu_acts(rng, 1, K, 0.7)
    arrs = orc.encode(W, TM, TK, F16, COL)
    E = upload(us, arrs, M, K, TM, TK, F16, COL)
    ci = us.us_colinfo(E)
    xt = torch.from_numpy(x.view(np.int16)).cuda()
    y1 = torch.empty(1, M, dtype=torch.int16, device="cuda")
    y2 = torch.empty(M, dtype=torch.int16, device="cuda")
    us.us_spmspv_f16_ci(E, ci, xt, 1, 0.0, y1)
    ws = us.workspace(us.US_OP_SPMSPV_F16, E, 1)
    us.us_spmspv_f16(E, xt.reshape(-1), 0.0, y2, ws)
    torch.cuda.synchronize()
    a = y1.cpu().numpy().view(np.float16).astype(np.float64).reshape(-1)
    b = y2.cpu().numpy().view(np.float16).astype(np.float64)
    _, exact = orc.spmspv_f16(W, x[0], 0.0)
    check_f16(a, exact, "ColInfo kernel")
    check_f16(b, exact, "bitmap-scan kernel")
    assert np.abs(a - b).max() <= 2 * MAX_ABS


def test_spmspv_ci_reports_contradicting_colinfo(us, orc):
    """ColInfo whose counts disagree with the bitmap is refused as corrupt; no
    read leaves the tile's run (the bounds are checked before each load)."""
    M, K, TM, TK = 128, 256, 64, 64
    rng = np.random.default_rng(9)
    W = rand_f16(rng, M, K, 0.5)
    arrs = orc.encode(W, TM, TK, F16, COL)
    E = upload(us, arrs, M, K, TM, TK, F16, COL)
    good = orc.colinfo(arrs[0], M, K, TM, TK)
    x = relu_acts(rng, 1, K, 0.0)
    xt = torch.from_numpy(x.view(np.int16)).cuda()
    for bad_kind in ("count_low", "offset_past_run"):
        bad = good.copy()
        if bad_kind == "count_low":
            j = int(np.flatnonzero(bad & 0xFFFF)[3])
            bad[j] -= 1                                # one fewer nonzero than the bitmap holds
        else:
            bad[5] = (0xFFF0 << 16) | (int(bad[5]) & 0xFFFF)
        ci = torch.from_numpy(bad.view(np.int32)).cuda()
        Y = torch.empty(1, M, dtype=torch.int16, device="cuda")
        us.us_spmspv_f16_ci(E, ci, xt, 1, 0.0, Y)
        torch.cuda.synchronize()
        assert us.us_get_last_device_status() == us.US_ERR_CORRUPT, bad_kind


def test_spmspv_ci_full_size_sampled(us, orc):
    """14336 x 4096, 64 x 64 COL tiles, 50 % static sparsity, ReLU activations
    with 90 % zeros, N = 1 and a batch of 8: every output row of the first and
    last tokens against the oracle, in the launch configuration the benchmark
    times."""
    M, K, TM, TK = 14336, 4096, 64, 64
    rng = np.random.default_rng(2024)
    W = rand_f16(rng, M, K, 0.5)
    X = relu_acts(rng, 8, K, 0.9)
    Wt = torch.from_numpy(W.view(np.int16)).cuda()
    E = us.us_encode(Wt, TM, TK, F16, COL)
    ci = us.us_colinfo(E)
    Xt = torch.from_numpy(X.view(np.int16)).cuda()
    for N in (1, 8):
        Y = torch.empty(N, M, dtype=torch.int16, device="cuda")
        us.us_spmspv_f16_ci(E, ci, Xt[:N].contiguous(), N, 0.0, Y)
        torch.cuda.synchronize()
        assert us.us_get_last_device_status() == us.US_OK
        y = Y.cpu().numpy().view(np.float16)
        for n in sorted({0, N - 1}):
            _, exact = orc.spmspv_f16(W, X[n], 0.0, nthreads=orc.max_threads())
            check_f16(y[n], exact, f"N={N} token {n}")
