"""The streamed spMspV kernel (64 x 64 column-scan tiles, the us_spmspv_f16 path
for that tile shape) against the oracle, on the cases its design has to get
right: a tile whose 64 columns are all active (two groups of 32 compacted
columns), fully dense tiles (the largest value runs in the byte ring), empty
matrices and empty tiles, activations that are all pruned, K slices reduced in
a cluster, static weights, bitwise repeatability and corrupt offsets."""
import numpy as np
import pytest
import torch

from bitmap_encoded_unstructured_ie_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

F16, COL = 0, 1
REL_L2, MAX_ABS = 1e-3, 2e-2


@pytest.fixture(scope="module")
def us():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from bitmap_encoded_unstructured_ie_gb300 import build, binding
    build.build()
    binding.load()
    return binding


def check(y, exact, what):
    err = y.astype(np.float64).reshape(-1) - exact.reshape(-1)
    rel = np.linalg.norm(err) / max(np.linalg.norm(exact), 1e-30)
    mx = np.abs(err).max() if err.size else 0.0
    assert rel <= REL_L2 and mx <= MAX_ABS, f"{what}: rel L2 {rel:.3e}, max abs {mx:.3e}"


def rand_w(rng, M, K, density):
    w = (rng.standard_normal((M, K)) * 0.02).astype(np.float16)
    w[rng.random((M, K)) >= density] = 0
    return w


def run(us, W, x, tau=0.0, static=False, E=None):
    M, K = W.shape
    if E is None:
        E = us.us_encode(torch.from_numpy(W.view(np.int16)).cuda(), 64, 64, us.US_F16, us.US_ORDER_COL)
    E.flags = us.US_BITMAP_STATIC if static else 0
    xt = torch.from_numpy(x.view(np.int16)).cuda()
    y = torch.full((M,), 0x7E00, dtype=torch.int16, device="cuda")      # NaN until written
    us.us_spmspv_f16(E, xt, tau, y, us.workspace(us.US_OP_SPMSPV_F16, E, 1))
    torch.cuda.synchronize()
    return y.cpu().numpy().view(np.float16), E


@pytest.mark.parametrize("M,K,density,zero_frac", [
    (1024, 1024, 1.0, 0.0),          # every column of every tile active: two groups of 32
    (640, 512, 1.0, 0.5),            # fully dense tiles, the longest runs
    (9728, 256, 0.5, 0.3),           # many bands, one slice each
    (192, 4096, 0.5, 0.5),           # few bands: K sliced, slices reduced in a cluster
    (256, 64 * 33, 0.3, 0.8),        # uneven slices
])
def test_stream_matches_oracle(us, orc, M, K, density, zero_frac):
    rng = np.random.default_rng(M + K)
    W = rand_w(rng, M, K, density)
    x = rng.standard_normal(K).astype(np.float32)
    x = wl.relu_threshold(x, zero_frac).astype(np.float16) if zero_frac else x.astype(np.float16)
    y, E = run(us, W, x)
    assert us.us_get_last_device_status() == us.US_OK
    _, exact = orc.spmspv_f16(W, x, 0.0)
    check(y, exact, f"{M}x{K} density {density} zeros {zero_frac}")
    # static weights: the weights stream before the dependency wait, same result
    y2, _ = run(us, W, x, static=True, E=E)
    assert np.array_equal(y.view(np.uint16), y2.view(np.uint16))


def test_stream_threshold_and_column_counts(us, orc):
    """tau > 0 on both signs; columns with 1..64 nonzeros, so the compacted
    groups hold 1..32 columns and 16-column blocks are padded."""
    rng = np.random.default_rng(3)
    M, K = 512, 2048
    W = np.zeros((M, K), np.float16)
    for j in range(K):
        rows = rng.choice(M, size=1 + (j % 64) * (M // 64) // 8, replace=False)
        W[rows, j] = (rng.standard_normal(rows.size) * 0.05).astype(np.float16)
    x = rng.standard_normal(K).astype(np.float16)
    for tau in (0.0, 0.3, 1.5, 10.0):
        y, _ = run(us, W, x, tau)
        assert us.us_get_last_device_status() == us.US_OK
        _, exact = orc.spmspv_f16(W, x, tau)
        if tau == 10.0:
            assert not np.any(y.view(np.uint16) & 0x7FFF), "every column pruned: y must be zero"
        else:
            check(y, exact, f"tau {tau}")


def test_stream_empty_matrix_and_zero_activations(us, orc):
    M, K = 256, 1024
    y, _ = run(us, np.zeros((M, K), np.float16), np.ones(K, np.float16))
    assert not np.any(y.view(np.uint16) & 0x7FFF)
    rng = np.random.default_rng(4)
    y, _ = run(us, rand_w(rng, M, K, 0.5), np.zeros(K, np.float16))
    assert not np.any(y.view(np.uint16) & 0x7FFF)
    assert us.us_get_last_device_status() == us.US_OK


def test_stream_repeat_is_bitwise(us, orc):
    d = wl.spmspv(14336, 4096, 0.5, 0.7, seed=5)
    E = us.us_encode(torch.from_numpy(d["W"].view(np.int16)).cuda(), 64, 64, us.US_F16, us.US_ORDER_COL)
    outs = [run(us, d["W"], d["x"], E=E)[0].view(np.uint16).copy() for _ in range(3)]
    assert all(np.array_equal(outs[0], o) for o in outs[1:])
    _, exact = orc.spmspv_f16(d["W"], d["x"], 0.0, nthreads=orc.max_threads())
    check(outs[0].view(np.float16), exact, "14336 x 4096 repeat")


def test_stream_corrupt_offsets_are_refused(us, orc):
    rng = np.random.default_rng(6)
    M, K = 256, 512
    W = rand_w(rng, M, K, 0.5)
    bm, off, vals = orc.encode(W, 64, 64, F16, COL)
    bad = off.copy()
    bad[3] = bad[2] + 8                               # shorter than the tile's popcount
    E = us.from_host(bm, bad, vals, M, K, 64, 64, F16, COL)
    x = rng.standard_normal(K).astype(np.float16)
    xt = torch.from_numpy(x.view(np.int16)).cuda()
    y = torch.empty(M, dtype=torch.int16, device="cuda")
    us.us_spmspv_f16(E, xt, 0.0, y, us.workspace(us.US_OP_SPMSPV_F16, E, 1))
    assert us.us_get_last_device_status() == us.US_ERR_CORRUPT
    # bands that no corrupt tile touches are still exact
    _, exact = orc.spmspv_f16(W, x, 0.0)
    check(y.cpu().numpy().view(np.float16)[128:], exact[128:], "bands after the corrupt one")
