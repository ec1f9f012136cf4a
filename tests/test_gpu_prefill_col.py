"""One format for prefill and decode: us_spmm_f16 on COL-order tiles (the
Tiled-CBC layout that spMspV reads), through the C ABI, against the oracle.

Where both scan orders run the same kernel (the tensor-core path: 64 x 64
tiles, N >= 64; the generic CUDA-core path: other tile shapes) they decode to
the same dense operand and sum it in the same order, so a matrix encoded ROW
and COL must give bit-identical outputs. For 64 x 64 tiles and N < 64, ROW
tiles take the mma.sync decode kernel and COL tiles the generic one, whose
fp32 sums run in another order: there each is held to the oracle on its own.
Every output must be within the fp16 bar of the fp64 oracle: relative
L2 <= 1e-3, max-abs <= 2e-2.

Cases cover the tensor-core path (64 x 64 tiles, N >= 64, with and without
split-K, ragged token tiles) and the CUDA-core paths (any tile, any N).
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

F16, ROW, COL = 0, 0, 1
REL_L2, MAX_ABS = 1e-3, 2e-2


@pytest.fixture(scope="module")
def us():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from bitmap_encoded_unstructured_ie_gb300 import build, binding
    build.build()
    binding.load()
    return binding


def rand_f16(rng, M, K, density):
    w = (rng.standard_normal((M, K)) * 0.02).astype(np.float16)
    w[rng.random((M, K)) >= density] = 0
    return w


def check_f16(y_gpu, exact, what=""):
    y = y_gpu.astype(np.float64)
    err = y - exact
    rel = np.linalg.norm(err) / max(np.linalg.norm(exact), 1e-30)
    mx = np.abs(err).max() if err.size else 0.0
    assert rel <= REL_L2 and mx <= MAX_ABS, f"{what}: rel L2 {rel:.3e}, max abs {mx:.3e}"


def run(us, W, X, TM, TK, order, split_k=0):
    M, K = W.shape
    N = X.shape[0]
    E = us.us_encode(torch.from_numpy(W.view(np.int16)).cuda(), TM, TK, F16, order)
    ws = us.workspace(us.US_OP_SPMM_F16, E, N, split_k)
    Y = torch.full((N, M), 0x7E00, dtype=torch.int16, device="cuda")
    us.us_spmm_f16(E, torch.from_numpy(X.view(np.int16)).cuda(), N, Y, ws, split_k)
    torch.cuda.synchronize()
    assert us.us_get_last_device_status() == us.US_OK
    assert not ws.any().item(), "workspace not left zeroed"
    return Y.cpu().numpy().view(np.float16)


CASES = [
    # M, K, TM, TK, N, density, split_k
    (256, 1024, 64, 64, 64, 0.4, 0),      # tensor cores, one token tile
    (384, 512, 64, 64, 300, 0.6, 0),      # tensor cores, a ragged second token tile
    (256, 2048, 64, 64, 128, 0.5, 4),     # tensor cores, split-K
    (256, 512, 64, 64, 700, 0.5, 2),      # tensor cores, 512-token tiles, split-K, ragged
    (128, 768, 64, 64, 1, 0.5, 0),        # CUDA cores (ROW: mma.sync decode kernel), one token
    (256, 512, 64, 64, 33, 0.3, 2),       # the same, split-K, ragged token block
    (256, 512, 128, 32, 40, 0.5, 0),      # other tile shapes: CUDA cores
    (512, 256, 256, 16, 7, 0.5, 0),
    (128, 384, 64, 128, 65, 0.5, 0),      # TK = 128: CUDA cores even at N >= 64
]


@pytest.mark.parametrize("case", CASES)
def test_col_tiles_match_row_tiles_and_oracle(us, orc, case):
    M, K, TM, TK, N, dens, split = case
    rng = np.random.default_rng(M + K + N + TM)
    W = rand_f16(rng, M, K, dens)
    X = rng.standard_normal((N, K)).astype(np.float16)
    y_col = run(us, W, X, TM, TK, COL, split)
    y_row = run(us, W, X, TM, TK, ROW, split)
    same_kernel = not (TM == 64 and TK == 64 and N < 64)
    if same_kernel:
        assert np.array_equal(y_col.view(np.uint16), y_row.view(np.uint16)), "ROW and COL tiles disagree"
    n_idx, m_idx = np.meshgrid(np.arange(N), np.arange(M), indexing="ij")
    sel = rng.choice(N * M, size=min(N * M, 4096), replace=False)
    _, exact = orc.spmm_f16_at(W, X, n_idx.reshape(-1)[sel], m_idx.reshape(-1)[sel])
    check_f16(y_col.reshape(-1)[sel], exact, f"{case} COL")
    if not same_kernel:
        check_f16(y_row.reshape(-1)[sel], exact, f"{case} ROW")


def test_col_prefill_edge_tiles(us, orc):
    """Empty, full and single-nonzero tiles, with columns whose run crosses the
    32-row halves that the decoder threads split."""
    M, K, N = 128, 256, 96
    W = np.zeros((M, K), np.float16)
    W[:64, 64:128] = 0.5                            # one full tile
    W[64:, :64] = np.float16(-0.25)                 # another full tile
    W[31:33, 130] = 2.0                             # a column run across the row halves
    W[127, 255] = -3.0                              # a single nonzero in the last position
    rng = np.random.default_rng(4)
    X = rng.standard_normal((N, K)).astype(np.float16)
    y = run(us, W, X, 64, 64, COL)
    assert np.array_equal(y.view(np.uint16), run(us, W, X, 64, 64, ROW).view(np.uint16))
    n_idx, m_idx = np.meshgrid(np.arange(N), np.arange(M), indexing="ij")
    _, exact = orc.spmm_f16_at(W, X, n_idx.reshape(-1), m_idx.reshape(-1))
    check_f16(y.reshape(-1), exact, "edge tiles")


def test_col_prefill_full_size_sampled(us, orc):
    """4096 x 4096 at 60 % sparsity, N = 1024, COL tiles, the tensor-core launch
    configuration the benchmark times: sampled outputs against the oracle and
    bit-identical to ROW tiles."""
    M = K = 4096
    N = 1024
    rng = np.random.default_rng(77)
    W = rand_f16(rng, M, K, 0.4)
    X = rng.standard_normal((N, K)).astype(np.float16)
    y_col = run(us, W, X, 64, 64, COL)
    y_row = run(us, W, X, 64, 64, ROW)
    assert np.array_equal(y_col.view(np.uint16), y_row.view(np.uint16))
    n_idx = rng.integers(0, N, 3000)
    m_idx = rng.integers(0, M, 3000)
    _, exact = orc.spmm_f16_at(W, X, n_idx, m_idx)
    check_f16(y_col[n_idx, m_idx], exact, "4096^2 COL N=1024")
