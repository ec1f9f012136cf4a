"""IE-BME with areas (Q = RA*CA union mask, Q aligned value streams) and the
bitmap-aware row reordering, through the C ABI, against the CPU oracle.

Bars, all bit-exact:
- the encoder's bitmap, offsets and value bytes;
- the W4A4 int32 accumulators;
- the fp16 epilogue.

Cases cover every area split, 16-row local tiles (the DP-sized ones) and
64-row tiles, identity, random and DP-optimal row permutations, ragged
token blocks, split-K, and permutations that are not permutations.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

F16, I4, ROW = 0, 1, 0


@pytest.fixture(scope="module")
def us():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from bitmap_encoded_unstructured_ie_gb300 import build, binding
    build.build()
    binding.load()
    return binding


def rand_w(rng, M, K, density, elem):
    if elem == F16:
        w = (rng.standard_normal((M, K)) * 0.02).astype(np.float16)
    else:
        w = rng.integers(-8, 8, size=(M, K)).astype(np.int8)
    w[rng.random((M, K)) >= density] = 0
    return w


def dev_w(W, elem):
    return torch.from_numpy(W.view(np.int16) if elem == F16 else W).cuda()


CFGS = [
    # TM, TK, RA, CA
    (16, 64, 2, 2),
    (16, 64, 4, 1),
    (16, 64, 1, 4),
    (16, 128, 2, 1),
    (64, 64, 2, 2),
    (64, 64, 1, 1),
    (128, 32, 4, 1),
]


@pytest.mark.parametrize("cfg", CFGS)
@pytest.mark.parametrize("elem", [F16, I4])
def test_encode_ie_bytes_match_oracle(us, orc, cfg, elem):
    TM, TK, RA, CA = cfg
    rng = np.random.default_rng(TM * 3 + TK + 11 * RA + CA + elem)
    M, K = TM * 4, TK * 3
    nT = (M // TM) * (K // TK)
    for density in (0.0, 0.3, 1.0):
        W = rand_w(rng, M, K, density, elem)
        perms = [None, np.concatenate([rng.permutation(TM) for _ in range(nT)]).astype(np.uint8)]
        if TM <= 20:
            perms.append(us.us_reorder_rows(W, TM, TK, RA, CA, elem))
        for pm in perms:
            pt = None if pm is None else torch.from_numpy(pm).cuda()
            E = us.us_encode_ie(dev_w(W, elem), TM, TK, RA, CA, elem, pt)
            torch.cuda.synchronize()
            assert us.us_get_last_device_status() == us.US_OK
            obm, ooff, ovals = orc.encode_ie(W, TM, TK, RA, CA, elem, pm)
            assert np.array_equal(E.E.bitmap.cpu().numpy().view(np.uint64)[: obm.size], obm)
            assert np.array_equal(E.E.tile_off.cpu().numpy().view(np.uint32), ooff)
            assert np.array_equal(E.E.values.cpu().numpy()[: E.E.values_bytes], ovals)


def test_encode_ie_refuses_non_permutations(us):
    TM, TK, M, K = 16, 64, 32, 128
    W = rand_w(np.random.default_rng(0), M, K, 0.5, I4)
    nT = (M // TM) * (K // TK)
    for bad_kind in ("repeat", "range"):
        pm = np.tile(np.arange(TM, dtype=np.uint8), nT)
        if bad_kind == "repeat":
            pm[TM + 3] = pm[TM + 4]                    # tile 1 names one row twice
        else:
            pm[2 * TM + 5] = 200                       # tile 2 names a row outside the tile
        us.us_encode_ie(dev_w(W, I4), TM, TK, 2, 2, I4, torch.from_numpy(pm).cuda())
        torch.cuda.synchronize()
        assert us.us_get_last_device_status() == us.US_ERR_INVALID_ARG, bad_kind


SPMM_CASES = [
    # M, K, TM, TK, RA, CA, N, density, split_k, permutation
    (64, 512, 16, 64, 2, 2, 1, 0.5, 0, "dp"),
    (128, 1024, 16, 64, 2, 2, 5, 0.3, 0, "dp"),
    (96, 640, 16, 64, 4, 1, 33, 0.5, 2, "random"),
    (64, 1024, 16, 128, 2, 1, 8, 0.7, 0, "dp"),
    (256, 512, 64, 64, 2, 2, 3, 0.5, 0, None),
    (256, 256, 128, 32, 4, 1, 40, 0.4, 2, "random"),
]


@pytest.mark.parametrize("case", SPMM_CASES)
def test_spmm_w4a4_ie_exact(us, orc, case):
    M, K, TM, TK, RA, CA, N, dens, split, pkind = case
    rng = np.random.default_rng(M + K + N + RA)
    W = rand_w(rng, M, K, dens, I4)
    Xq = rng.integers(-8, 8, size=(N, K)).astype(np.int8)
    s_w = (rng.random(M) * 0.01 + 1e-3).astype(np.float16)
    s_x = (rng.random(N) * 0.5 + 0.05).astype(np.float16)
    nT = (M // TM) * (K // TK)
    pm = None
    if pkind == "dp":
        pm = us.us_reorder_rows(W, TM, TK, RA, CA, I4)
    elif pkind == "random":
        pm = np.concatenate([rng.permutation(TM) for _ in range(nT)]).astype(np.uint8)
    E = us.us_encode_ie(dev_w(W, I4), TM, TK, RA, CA, I4, None if pm is None else torch.from_numpy(pm).cuda())
    from bitmap_encoded_unstructured_ie_gb300 import workloads as wl
    X = torch.from_numpy(wl.pack_int4(Xq)).cuda()
    sw = torch.from_numpy(s_w.view(np.int16)).cuda()
    sx = torch.from_numpy(s_x.view(np.int16)).cuda()
    ws = us.workspace_ie(E, N, split)
    oacc, oy = orc.spmm_w4a4(W, Xq, s_w, s_x)
    for _ in range(2):
        Yacc = torch.full((N, M), 777, dtype=torch.int32, device="cuda")
        Y = torch.empty(N, M, dtype=torch.int16, device="cuda")
        us.us_spmm_w4a4_ie(E, X, sw, sx, N, Yacc, Y, ws, split)
        torch.cuda.synchronize()
        assert us.us_get_last_device_status() == us.US_OK
        assert np.array_equal(Yacc.cpu().numpy(), oacc)
        assert np.array_equal(Y.cpu().numpy().view(np.uint16), oy.view(np.uint16))
    assert not ws.any().item(), "workspace not left zeroed"


def test_spmm_w4a4_ie_full_size_sampled(us, orc):
    """W4A4 4096 x 4096 at 50 % (magnitude-pruned rows), 16 x 64 local tiles,
    2 x 2 areas, DP-reordered rows, N = 8: sampled accumulators exact."""
    from bitmap_encoded_unstructured_ie_gb300 import workloads as wl
    d = wl.w4a4(4096, 4096, 8, 0.5, seed=0)
    W = d["Wq"]
    pm = us.us_reorder_rows(W, 16, 64, 2, 2, I4)
    E = us.us_encode_ie(torch.from_numpy(W).cuda(), 16, 64, 2, 2, I4, torch.from_numpy(pm).cuda())
    N = 8
    ws = us.workspace_ie(E, N, 0)
    Yacc = torch.empty(N, 4096, dtype=torch.int32, device="cuda")
    us.us_spmm_w4a4_ie(E, torch.from_numpy(wl.pack_int4(d["Xq"][:N])).cuda(), None, None, N, Yacc, None, ws, 0)
    torch.cuda.synchronize()
    assert us.us_get_last_device_status() == us.US_OK
    rng = np.random.default_rng(1)
    n_idx, m_idx = rng.integers(0, N, 4000), rng.integers(0, 4096, 4000)
    one = np.ones(4096, np.float16)
    oacc, _ = orc.spmm_w4a4_at(W, d["Xq"][:N], one, np.ones(N, np.float16), n_idx, m_idx)
    assert np.array_equal(Yacc.cpu().numpy()[n_idx, m_idx], oacc)
