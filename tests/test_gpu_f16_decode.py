"""fp16 SpMM for decode-sized token counts (1-63) on 64 x 64 row-scan tiles:
the mma.sync decode kernel, through the C ABI, against the oracle.

Covers one token block of 8, 16 and 32 tokens and two blocks, slices whose
tile count leaves some of the four warps idle or with one tile fewer,
split-K (even and uneven slices), fully dense tiles (the longest runs), a
matrix with no nonzero, an FFN-sized shape on sampled outputs, the
no-allocation entry point, offsets that the kernel must refuse, and the
launch captured in a CUDA graph and replayed.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

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


def rand_f16(rng, M, K, density):
    w = (rng.standard_normal((M, K)) * 0.02).astype(np.float16)
    w[rng.random((M, K)) >= density] = 0
    return w


def check(y, exact, what):
    err = y.astype(np.float64).reshape(-1) - exact.reshape(-1)
    rel = np.linalg.norm(err) / max(np.linalg.norm(exact), 1e-30)
    mx = np.abs(err).max() if err.size else 0.0
    assert rel <= REL_L2 and mx <= MAX_ABS, f"{what}: rel L2 {rel:.3e}, max abs {mx:.3e}"


def encode(us, W):
    E = us.us_encode(torch.from_numpy(W.view(np.int16)).cuda(), 64, 64, us.US_F16, us.US_ORDER_ROW)
    torch.cuda.synchronize()
    assert us.us_get_last_device_status() == us.US_OK
    return E


def run(us, E, X, split_k=0):
    N = X.shape[0]
    Y = torch.empty(N, E.M, dtype=torch.int16, device="cuda")
    ws = us.workspace(us.US_OP_SPMM_F16, E, N, split_k)
    us.us_spmm_f16(E, torch.from_numpy(X.view(np.int16)).cuda(), N, Y, ws, split_k)
    torch.cuda.synchronize()
    assert us.us_get_last_device_status() == us.US_OK
    assert not ws.any().item(), "split-K partials or counters not cleared"
    return Y.cpu().numpy().view(np.float16)


def exact_all(orc, W, X):
    N, M = X.shape[0], W.shape[0]
    n, m = np.meshgrid(np.arange(N), np.arange(M), indexing="ij")
    return orc.spmm_f16_at(W, X, n.reshape(-1), m.reshape(-1))[1].reshape(N, M)


CASES = [
    # M, K, N, density, split_k
    (256, 512, 1, 0.5, 0),
    (256, 512, 8, 0.5, 0),
    (320, 1152, 7, 0.5, 0),      # 18 K tiles: warps with one tile fewer
    (192, 640, 9, 0.3, 0),       # 16-token block, one token in the second n8 block
    (256, 1024, 16, 0.5, 4),
    (128, 768, 17, 0.5, 0),      # 32-token block, 17 tokens
    (256, 512, 33, 0.5, 2),      # two token blocks, the second holding one token
    (128, 512, 63, 1.0, 0),      # fully dense tiles: runs of 4096 values
    (192, 192, 3, 0.5, 0),       # 3 K tiles: one warp idle
    (64, 4096, 2, 0.02, 1),      # one slice of 64 tiles, nearly empty tiles
    (128, 1280, 5, 0.5, 3),      # uneven slices (6, 7, 7 tiles)
    (256, 1024, 24, 0.6, 16),    # slices of one tile
]


@pytest.mark.parametrize("case", CASES)
def test_f16_decode_matches_oracle(us, orc, case):
    M, K, N, dens, split = case
    rng = np.random.default_rng(sum(case[:3]) + int(dens * 10))
    W = rand_f16(rng, M, K, dens)
    X = rng.standard_normal((N, K)).astype(np.float16)
    E = encode(us, W)
    check(run(us, E, X, split), exact_all(orc, W, X), f"fp16 decode {case}")


def test_f16_decode_empty_matrix(us):
    W = np.zeros((128, 512), np.float16)
    X = np.random.default_rng(0).standard_normal((4, 512)).astype(np.float16)
    y = run(us, encode(us, W), X)
    assert not np.any(y.view(np.uint16))


@pytest.mark.parametrize("N", [8, 12])
def test_f16_decode_ffn_shape_sampled(us, orc, N):
    """11008 x 4096, 50 % sparse, 8 and 12 tokens (8- and 16-token blocks), in
    the launch shape the library picks: 688 CTAs, more than one wave at two an
    SM, so three an SM with two stages a group.  20000 sampled outputs against
    the oracle."""
    rng = np.random.default_rng(7)
    W = rand_f16(rng, 11008, 4096, 0.5)
    X = rng.standard_normal((N, 4096)).astype(np.float16)
    y = run(us, encode(us, W), X)
    n = rng.integers(0, N, 20000)
    m = rng.integers(0, 11008, 20000)
    _, exact = orc.spmm_f16_at(W, X, n.astype(np.int32), m.astype(np.int32))
    check(y[n, m], exact, "fp16 decode 11008 x 4096")


def test_f16_decode_noalloc(us, orc):
    rng = np.random.default_rng(3)
    W = rand_f16(rng, 256, 1024, 0.5)
    X = rng.standard_normal((4, 1024)).astype(np.float16)
    E = encode(us, W)
    Y = torch.empty(4, 256, dtype=torch.int16, device="cuda")
    for split in (0, 4):
        us.us_spmm_f16_noalloc(E, torch.from_numpy(X.view(np.int16)).cuda(), 4, Y, split)
        torch.cuda.synchronize()
        assert us.us_get_last_device_status() == us.US_OK
        check(Y.cpu().numpy().view(np.float16), exact_all(orc, W, X), f"noalloc split {split}")


def test_f16_decode_refuses_corrupt_offsets(us, orc):
    """An offset that is not a 16-byte run boundary, and a run shorter than its
    bitmap's popcount: the kernel skips those tiles and reports US_ERR_CORRUPT."""
    rng = np.random.default_rng(1)
    W = rand_f16(rng, 128, 256, 0.5)
    bm, off, vals = orc.encode(W, 64, 64, orc.F16, orc.ROW)
    X = torch.from_numpy(rng.standard_normal((2, 256)).astype(np.float16).view(np.int16)).cuda()
    for k in ("misaligned", "short"):
        bad = off.copy()
        if k == "misaligned":
            bad[2] = bad[1] + 4
        else:
            bad[2] = bad[1] + 8                     # aligned, far shorter than the tile's nonzeros
        us.us_get_last_device_status()          # returns and clears the word
        E = us.from_host(bm, bad, vals, 128, 256, 64, 64, us.US_F16, us.US_ORDER_ROW)
        Y = torch.empty(2, 128, dtype=torch.int16, device="cuda")
        us.us_spmm_f16(E, X, 2, Y, us.workspace(us.US_OP_SPMM_F16, E, 2))
        torch.cuda.synchronize()
        assert us.us_get_last_device_status() == us.US_ERR_CORRUPT, k


def test_f16_decode_in_cuda_graph(us, orc):
    rng = np.random.default_rng(5)
    W = rand_f16(rng, 512, 2048, 0.5)
    X = rng.standard_normal((3, 2048)).astype(np.float16)
    E = encode(us, W)
    Xt = torch.from_numpy(X.view(np.int16)).cuda()
    Y = torch.zeros(3, 512, dtype=torch.int16, device="cuda")
    ws = us.workspace(us.US_OP_SPMM_F16, E, 3)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        us.us_spmm_f16(E, Xt, 3, Y, ws, 0, stream)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        us.us_spmm_f16(E, Xt, 3, Y, ws, 0, stream)
    Y.zero_()
    with torch.cuda.stream(stream):
        for _ in range(4):
            g.replay()
    stream.synchronize()
    assert us.us_get_last_device_status(stream) == us.US_OK
    check(Y.cpu().numpy().view(np.float16), exact_all(orc, W, X), "graph replay")
