# Per-token activation quantisation on the GPU against the oracle: codes and
# scales bit-exact.
import numpy as np
import pytest
import torch

from bitmap_encoded_unstructured_ie_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def us():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from bitmap_encoded_unstructured_ie_gb300 import build, binding
    build.build()
    binding.load()
    return binding


def run_quant(us, X: np.ndarray):
    N, K = X.shape
    Xt = torch.from_numpy(np.ascontiguousarray(X).view(np.int16)).cuda()
    Xq = torch.full((N, K // 2), 0x5A, dtype=torch.uint8, device="cuda")
    s = torch.zeros(N, dtype=torch.int16, device="cuda")
    us.us_quantize_x(Xt, N, K, Xq, s)
    torch.cuda.synchronize()
    assert us.us_get_last_device_status() == us.US_OK
    return Xq.cpu().numpy(), s.cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("N,K,scale", [(1, 32, 1.0), (7, 4096, 3.0), (16, 11008, 0.01), (33, 96, 200.0), (2048, 4096, 1.0)])
def test_quantize_matches_oracle(us, orc, N, K, scale):
    rng = np.random.default_rng(N * 31 + K)
    X = (rng.standard_normal((N, K)) * scale * rng.uniform(0.1, 2.0, (N, 1))).astype(np.float16)
    q, s = run_quant(us, X)
    oc, os_ = orc.quantize_x(X)
    assert np.array_equal(s, os_.view(np.uint16))
    assert np.array_equal(q.reshape(-1), wl.pack_int4(oc))


def test_quantize_edge_tokens(us, orc):
    """All-zero token (scale 1), exact ties, a NaN and an infinity, negative
    maximum, subnormals, and the largest fp16 magnitudes."""
    K = 64
    X = np.zeros((8, K), np.float16)
    X[1, :8] = [0.5, 1.5, 2.5, -7, 3.5, -0.5, 6.5, 7]              # s = 1: ties to even
    X[2, :4] = [np.nan, 1, -2, 3]
    X[3, :3] = [np.inf, 1, -1]
    X[4, :3] = [-7, 3, 1]
    X[5, :] = np.float16(6e-8) * np.arange(K)                     # subnormal inputs
    X[6, :2] = [65504, -65504]
    X[7, :] = np.float16(-1e-3)
    q, s = run_quant(us, X)
    oc, os_ = orc.quantize_x(X)
    assert np.array_equal(s, os_.view(np.uint16))
    assert np.array_equal(q.reshape(-1), wl.pack_int4(oc))
    assert os_[0] == 1.0 and not oc[0].any()


def test_quantize_feeds_spmm(us, orc):
    """us_quantize_x output drives us_spmm_w4a4 as the oracle's codes do."""
    rng = np.random.default_rng(3)
    M, K, N = 256, 1024, 9
    W = rng.integers(-8, 8, size=(M, K)).astype(np.int8)
    W[rng.random((M, K)) >= 0.5] = 0
    X = rng.standard_normal((N, K)).astype(np.float16)
    s_w = (rng.random(M) * 0.01 + 1e-3).astype(np.float16)
    q, s = run_quant(us, X)
    E = us.us_encode(torch.from_numpy(W).cuda(), 64, 64, us.US_I4, us.US_ORDER_ROW)
    Yacc = torch.empty(N, M, dtype=torch.int32, device="cuda")
    Y = torch.empty(N, M, dtype=torch.int16, device="cuda")
    ws = us.workspace(us.US_OP_SPMM_W4A4, E, N, 0)
    us.us_spmm_w4a4(E, torch.from_numpy(q.reshape(-1)).cuda(), torch.from_numpy(s_w.view(np.int16)).cuda(),
                    torch.from_numpy(s.view(np.int16)).cuda(), N, Yacc, Y, ws, 0)
    torch.cuda.synchronize()
    assert us.us_get_last_device_status() == us.US_OK
    oc, os_ = orc.quantize_x(X)
    oacc, oy = orc.spmm_w4a4(W, oc, s_w, os_)
    assert np.array_equal(Yacc.cpu().numpy(), oacc)
    assert np.array_equal(Y.cpu().numpy().view(np.uint16), oy.view(np.uint16))
