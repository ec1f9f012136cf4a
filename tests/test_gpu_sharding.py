"""Row-band shards run through the C ABI on one GPU.

A rank of a multi-GPU product holds a range of tile-row bands (bitmap and
value pieces of the whole matrix, tile_off rebased) and the whole X.  Here
every shard of one matrix runs on the same GPU, one call each, and the output
rows concatenate to the whole matrix's call: bit for bit for W4A4 (int32 and
fp16) and for fp16 on the same kernel, and within tolerance of the oracle.
"""
import numpy as np
import pytest
import torch

from bitmap_encoded_unstructured_ie_gb300 import sharding
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


@pytest.mark.parametrize("M,K,N,world,static", [(4096, 4096, 1, 3, True), (4096, 4096, 16, 2, True),
                                                (1024, 11008, 8, 5, False), (704, 512, 32, 4, True)])
def test_w4a4_shards_concatenate_bitwise(us, M, K, N, world, static):
    d = wl.w4a4(M, K, N, 0.5, seed=M + N)
    E = us.us_encode(torch.from_numpy(d["Wq"]).cuda(), 64, 64, us.US_I4, us.US_ORDER_ROW)
    E.flags = us.US_BITMAP_STATIC if static else 0
    X = torch.from_numpy(wl.pack_int4(d["Xq"][:N])).cuda()
    sw = torch.from_numpy(d["s_w"].view(np.int16)).cuda()
    sx = torch.from_numpy(d["s_x"][:N].view(np.int16)).cuda()
    ya = torch.empty(N, M, dtype=torch.int32, device="cuda")
    yh = torch.empty(N, M, dtype=torch.int16, device="cuda")
    us.us_spmm_w4a4(E, X, sw, sx, N, ya, yh, us.workspace(us.US_OP_SPMM_W4A4, E, N))
    parts_a, parts_h = [], []
    for b0, b1 in sharding.band_ranges(M // 64, world):
        S = sharding.shard_encoded(E, b0, b1)
        sa = torch.empty(N, S.M, dtype=torch.int32, device="cuda")
        sh = torch.empty(N, S.M, dtype=torch.int16, device="cuda")
        us.us_spmm_w4a4(S, X, sw[b0 * 64: b1 * 64].contiguous(), sx, N, sa, sh, us.workspace(us.US_OP_SPMM_W4A4, S, N))
        parts_a.append(sa)
        parts_h.append(sh)
    torch.cuda.synchronize()
    assert us.us_get_last_device_status() == us.US_OK
    assert torch.equal(torch.cat(parts_a, dim=1), ya)
    assert torch.equal(torch.cat(parts_h, dim=1), yh)


@pytest.mark.parametrize("N,order", [(1, 0), (256, 0), (512, 1)])
def test_f16_shards_match_the_whole_call(us, orc, N, order):
    M, K = 1024, 1024
    f = wl.f16_spmm(M, K, N, 0.5, seed=N)
    E = us.us_encode(torch.from_numpy(f["W"].view(np.int16)).cuda(), 64, 64, us.US_F16, order)
    X = torch.from_numpy(f["X"].view(np.int16)).cuda()
    Y = torch.empty(N, M, dtype=torch.int16, device="cuda")
    us.us_spmm_f16(E, X, N, Y, us.workspace(us.US_OP_SPMM_F16, E, N), 1)
    parts = []
    for b0, b1 in sharding.band_ranges(M // 64, 2):    # 8 bands each: 128-row blocks stay whole
        S = sharding.shard_encoded(E, b0, b1)
        Ys = torch.empty(N, S.M, dtype=torch.int16, device="cuda")
        us.us_spmm_f16(S, X, N, Ys, us.workspace(us.US_OP_SPMM_F16, S, N), 1)
        parts.append(Ys)
    torch.cuda.synchronize()
    assert us.us_get_last_device_status() == us.US_OK
    Yc = torch.cat(parts, dim=1)
    assert torch.equal(Yc, Y)                         # same kernel, one K slice: same sums
    s = np.random.default_rng(1)
    n_idx = s.integers(0, N, 3000).astype(np.int32)
    m_idx = s.integers(0, M, 3000).astype(np.int32)
    _, exact = orc.spmm_f16_at(f["W"], f["X"], n_idx, m_idx)
    got = Yc.cpu().numpy().view(np.float16)[n_idx, m_idx].astype(np.float64)
    rel = np.linalg.norm(got - exact) / np.linalg.norm(exact)
    assert rel <= 1e-3 and np.abs(got - exact).max() <= 2e-2
