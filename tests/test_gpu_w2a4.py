"""W2A4: int2 weights (two's complement in [-2, 1], four per byte) times int4
activations, through the C ABI, against the CPU oracle.

Bars, all bit-exact:
- the encoder's bytes;
- the int32 accumulators;
- the fp16 epilogue.

Cases cover the balanced kernel's dp4a (1-7 tokens) and mma.sync (8-32
tokens) consumers with and without the static-weights flag. They also cover
the CUDA-core kernel (explicit K splits, other tile shapes) and a sampled
4096 x 4096 launch.
"""
import numpy as np
import pytest
import torch

from bitmap_encoded_unstructured_ie_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

I2, ROW, COL = 2, 0, 1


@pytest.fixture(scope="module")
def us():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from bitmap_encoded_unstructured_ie_gb300 import build, binding
    build.build()
    binding.load()
    return binding


def rand_i2(rng, M, K, density):
    q = rng.integers(-2, 2, size=(M, K)).astype(np.int8)
    q[rng.random((M, K)) >= density] = 0
    return q


@pytest.mark.parametrize("shape", [(256, 512, 64, 64), (192, 320, 64, 16), (512, 256, 128, 32), (256, 256, 256, 128)])
@pytest.mark.parametrize("order", [ROW, COL])
def test_encode_int2_bytes_match_oracle(us, orc, shape, order):
    M, K, TM, TK = shape
    rng = np.random.default_rng(M + K + TM + order)
    for density in (0.0, 0.004, 0.5, 1.0):
        W = rand_i2(rng, M, K, density)
        E = us.us_encode(torch.from_numpy(W).cuda(), TM, TK, I2, order)
        torch.cuda.synchronize()
        assert us.us_get_last_device_status() == us.US_OK
        obm, ooff, ovals = orc.encode(W, TM, TK, I2, order)
        assert np.array_equal(E.bitmap.cpu().numpy().view(np.uint64), obm)
        assert np.array_equal(E.tile_off.cpu().numpy().view(np.uint32), ooff)
        assert np.array_equal(E.values.cpu().numpy()[: E.values_bytes], ovals)


def test_encode_int2_reports_out_of_range_codes(us):
    W = np.zeros((64, 64), np.int8)
    W[3, 4] = 2                                          # not an int2 code
    us.us_encode(torch.from_numpy(W).cuda(), 64, 64, I2, ROW)
    torch.cuda.synchronize()
    assert us.us_get_last_device_status() == us.US_ERR_INVALID_ARG


CASES = [
    # M, K, TM, TK, N, density, split_k
    (128, 64 * 300, 64, 64, 1, 0.5, 0),       # balanced kernel, dp4a, bands split over many CTAs
    (64 * 37, 64 * 13, 64, 64, 5, 0.3, 0),
    (64 * 9, 64 * 61, 64, 64, 7, 0.9, 0),     # dense runs: the ring wraps
    (128 * 7, 64 * 33, 64, 64, 8, 0.6, 0),    # mma.sync consumer
    (256, 64 * 300, 64, 64, 16, 0.4, 0),
    (128 * 3, 64 * 5, 64, 64, 20, 0.3, 0),    # 20 tokens padded to 32
    (64 * 40, 64 * 200, 64, 64, 32, 0.5, 0),  # more tiles per CTA than dense slots
    (256, 512, 64, 64, 3, 0.5, 4),            # explicit split: CUDA-core kernel
    (512, 256, 128, 32, 40, 0.5, 0),          # other tile shape: CUDA-core kernel
]


@pytest.mark.parametrize("static", [0, 1])
@pytest.mark.parametrize("case", CASES)
def test_w2a4_exact(us, orc, case, static):
    M, K, TM, TK, N, dens, split = case
    rng = np.random.default_rng(M * 3 + K + N + split)
    W = rand_i2(rng, M, K, dens)
    Xq = rng.integers(-8, 8, size=(N, K)).astype(np.int8)
    s_w = (rng.random(M) * 0.01 + 1e-3).astype(np.float16)
    s_x = (rng.random(N) * 0.5 + 0.05).astype(np.float16)
    E = us.us_encode(torch.from_numpy(W).cuda(), TM, TK, I2, ROW)
    E.flags = us.US_BITMAP_STATIC if static else 0
    X = torch.from_numpy(wl.pack_int4(Xq)).cuda()
    sw = torch.from_numpy(s_w.view(np.int16)).cuda()
    sx = torch.from_numpy(s_x.view(np.int16)).cuda()
    ws = us.workspace(us.US_OP_SPMM_W4A4, E, N, split)
    oacc, oy = orc.spmm_w4a4(W, Xq, s_w, s_x)
    for _ in range(2):
        Yacc = torch.full((N, M), -5, dtype=torch.int32, device="cuda")
        Y = torch.empty(N, M, dtype=torch.int16, device="cuda")
        us.us_spmm_w4a4(E, X, sw, sx, N, Yacc, Y, ws, split)
        torch.cuda.synchronize()
        assert us.us_get_last_device_status() == us.US_OK
        assert np.array_equal(Yacc.cpu().numpy(), oacc)
        assert np.array_equal(Y.cpu().numpy().view(np.uint16), oy.view(np.uint16))
    assert not ws.any().item(), "workspace not left zeroed"


def test_w2a4_full_size_sampled(us, orc):
    """W2A4 4096 x 4096, 50 % magnitude-pruned, static weights, N = 1 and 16,
    the launch configuration the benchmark times: sampled outputs exact."""
    d = wl.w2a4(4096, 4096, 16, 0.5, seed=0)
    E = us.us_encode(torch.from_numpy(d["Wq"]).cuda(), 64, 64, I2, ROW)
    E.flags = us.US_BITMAP_STATIC
    sw = torch.from_numpy(d["s_w"].view(np.int16)).cuda()
    rng = np.random.default_rng(3)
    for N in (1, 16):
        X = torch.from_numpy(wl.pack_int4(d["Xq"][:N])).cuda()
        sx = torch.from_numpy(d["s_x"][:N].view(np.int16)).cuda()
        ws = us.workspace(us.US_OP_SPMM_W4A4, E, N)
        Yacc = torch.empty(N, 4096, dtype=torch.int32, device="cuda")
        Y = torch.empty(N, 4096, dtype=torch.int16, device="cuda")
        us.us_spmm_w4a4(E, X, sw, sx, N, Yacc, Y, ws)
        torch.cuda.synchronize()
        assert us.us_get_last_device_status() == us.US_OK
        n_idx, m_idx = rng.integers(0, N, 3000), rng.integers(0, 4096, 3000)
        oacc, oy = orc.spmm_w4a4_at(d["Wq"], d["Xq"][:N], d["s_w"], d["s_x"][:N], n_idx, m_idx)
        assert np.array_equal(Yacc.cpu().numpy()[n_idx, m_idx], oacc)
        assert np.array_equal(Y.cpu().numpy().view(np.uint16)[n_idx, m_idx], oy.view(np.uint16))
