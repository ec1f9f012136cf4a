"""The balanced W4A4 kernel on IE-BME with areas (16 x 64 local tiles, four of
them stacked along M per 64 x 64 super-tile) against the CPU oracle, bit-exact
on the int32 accumulators and the fp16 epilogue.

Cases: every area split it takes (RA x CA = 1x1, 2x1, 4x1, 1x2, 2x2); one
super-tile per CTA, a ragged partition, and chunks that run across band
boundaries (two K tiles per band); 1..32 tokens (dp4a and mma.sync
consumers); identity, random and DP-optimal row permutations; static and
non-static weights; permutation entries outside the tile and corrupt offsets.
"""
import numpy as np
import pytest
import torch

from bitmap_encoded_unstructured_ie_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

I4 = 1
GEOMS = [(1, 1), (2, 1), (4, 1), (1, 2), (2, 2)]
SHAPES = [
    (128, 512),          # 16 super-tiles: one per CTA
    (2048, 1024),        # 512 super-tiles over the SMs: ragged ranges, chunks of four
    (64 * 160, 128),     # two K tiles per band: chunks run across band boundaries
]


@pytest.fixture(scope="module")
def us():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from bitmap_encoded_unstructured_ie_gb300 import build, binding
    build.build()
    binding.load()
    return binding


def problem(seed, M, K, N, density=0.5):
    rng = np.random.default_rng(seed)
    W = rng.integers(-8, 8, size=(M, K)).astype(np.int8)
    W[rng.random((M, K)) >= density] = 0
    Xq = rng.integers(-8, 8, size=(N, K)).astype(np.int8)
    s_w = (rng.random(M) * 0.01 + 1e-3).astype(np.float16)
    s_x = (rng.random(N) * 0.5 + 0.05).astype(np.float16)
    return rng, W, Xq, s_w, s_x


def call(us, E, Xq, s_w, s_x, N, static=False, reps=2):
    E.E.flags = us.US_BITMAP_STATIC if static else 0
    X = torch.from_numpy(wl.pack_int4(Xq)).cuda()
    sw = torch.from_numpy(s_w.view(np.int16)).cuda()
    sx = torch.from_numpy(s_x.view(np.int16)).cuda()
    ws = us.workspace_ie(E, N, 0)
    outs = []
    for _ in range(reps):
        Yacc = torch.full((N, E.E.M), 777, dtype=torch.int32, device="cuda")
        Y = torch.full((N, E.E.M), 0x7E00, dtype=torch.int16, device="cuda")
        us.us_spmm_w4a4_ie(E, X, sw, sx, N, Yacc, Y, ws, 0)
        torch.cuda.synchronize()
        outs.append((Yacc.cpu().numpy(), Y.cpu().numpy().view(np.uint16)))
    assert not ws.any().item(), "workspace not left zeroed"
    return outs


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("geom", GEOMS)
def test_balanced_ie_exact(us, orc, geom, shape):
    RA, CA = geom
    M, K = shape
    Nmax = 32
    rng, W, Xq, s_w, s_x = problem(M + K + 7 * RA + CA, M, K, Nmax)
    nT = (M // 16) * (K // 64)
    perms = [None, np.concatenate([rng.permutation(16) for _ in range(nT)]).astype(np.uint8)]
    for pi, pm in enumerate(perms):
        E = us.us_encode_ie(torch.from_numpy(W).cuda(), 16, 64, RA, CA, I4,
                            None if pm is None else torch.from_numpy(pm).cuda())
        torch.cuda.synchronize()
        assert us.us_get_last_device_status() == us.US_OK
        for N in (1, 3, 8, 16, 32):
            assert us.us_pick_split_k_ie(E, N) == 0, "the balanced kernel should serve this call"
            oacc, oy = orc.spmm_w4a4(W, Xq[:N], s_w, s_x[:N])
            for static in (False, True):
                for acc, y in call(us, E, Xq[:N], s_w, s_x[:N], N, static):
                    assert us.us_get_last_device_status() == us.US_OK
                    assert np.array_equal(acc, oacc), f"{geom} {shape} perm {pi} N {N} static {static}"
                    assert np.array_equal(y, oy.view(np.uint16)), f"{geom} {shape} perm {pi} N {N} static {static}"


def test_balanced_ie_dp_reordered(us, orc):
    """DP-optimal permutations (bitmap-aware row reordering), 2 x 2 areas."""
    M, K, N = 512, 1024, 8
    _, W, Xq, s_w, s_x = problem(11, M, K, N, density=0.3)
    pm = us.us_reorder_rows(W, 16, 64, 2, 2, I4)
    E = us.us_encode_ie(torch.from_numpy(W).cuda(), 16, 64, 2, 2, I4, torch.from_numpy(pm).cuda())
    assert us.us_pick_split_k_ie(E, N) == 0
    oacc, oy = orc.spmm_w4a4(W, Xq, s_w, s_x)
    for acc, y in call(us, E, Xq, s_w, s_x, N, static=True):
        assert us.us_get_last_device_status() == us.US_OK
        assert np.array_equal(acc, oacc)
        assert np.array_equal(y, oy.view(np.uint16))


def test_balanced_ie_empty_and_dense(us, orc):
    M, K, N = 256, 512, 4
    for density in (0.0, 1.0):
        _, W, Xq, s_w, s_x = problem(3, M, K, N, density)
        E = us.us_encode_ie(torch.from_numpy(W).cuda(), 16, 64, 2, 2, I4, None)
        oacc, oy = orc.spmm_w4a4(W, Xq, s_w, s_x)
        for acc, y in call(us, E, Xq, s_w, s_x, N):
            assert us.us_get_last_device_status() == us.US_OK
            assert np.array_equal(acc, oacc), density
            assert np.array_equal(y, oy.view(np.uint16)), density


def test_balanced_ie_bad_permutation_entry(us, orc):
    """A permutation entry that names no row of the tile records
    US_ERR_CORRUPT; every access stays in bounds."""
    M, K, N = 128, 256, 2
    rng, W, Xq, s_w, s_x = problem(5, M, K, N)
    nT = (M // 16) * (K // 64)
    pm = np.tile(np.arange(16, dtype=np.uint8), nT)
    E = us.us_encode_ie(torch.from_numpy(W).cuda(), 16, 64, 2, 2, I4, torch.from_numpy(pm).cuda())
    torch.cuda.synchronize()
    assert us.us_get_last_device_status() == us.US_OK
    E.perm[3 * 16 + 5] = 200                           # after encoding: tile 3 names a row outside the tile
    call(us, E, Xq, s_w, s_x, N, reps=1)
    assert us.us_get_last_device_status() == us.US_ERR_CORRUPT


def test_balanced_ie_corrupt_offsets(us, orc):
    M, K, N = 256, 512, 1
    _, W, Xq, s_w, s_x = problem(9, M, K, N)
    E = us.us_encode_ie(torch.from_numpy(W).cuda(), 16, 64, 2, 2, I4, None)
    torch.cuda.synchronize()
    off = E.E.tile_off.view(torch.int32)
    off[5] = off[4] + 16                               # 16-element run: shorter than Q * P_t
    call(us, E, Xq, s_w, s_x, N, reps=1)
    assert us.us_get_last_device_status() == us.US_ERR_CORRUPT


def test_balanced_ie_full_size(us, orc):
    """W4A4 4096 x 4096 at 50 % (magnitude-pruned), 2 x 2 areas, DP-reordered
    rows, N = 1 and 16, static weights as the benchmark runs them: sampled
    accumulators exact; repeated calls bitwise equal."""
    d = wl.w4a4(4096, 4096, 16, 0.5, seed=0)
    W = d["Wq"]
    pm = us.us_reorder_rows(W, 16, 64, 2, 2, I4)
    E = us.us_encode_ie(torch.from_numpy(W).cuda(), 16, 64, 2, 2, I4, torch.from_numpy(pm).cuda())
    rng = np.random.default_rng(1)
    one = np.ones(4096, np.float16)
    for N in (1, 16):
        assert us.us_pick_split_k_ie(E, N) == 0
        outs = call(us, E, d["Xq"][:N], d["s_w"], d["s_x"][:N], N, static=True, reps=3)
        assert us.us_get_last_device_status() == us.US_OK
        assert all(np.array_equal(outs[0][0], o[0]) for o in outs[1:])
        n_idx, m_idx = rng.integers(0, N, 3000), rng.integers(0, 4096, 3000)
        oacc, _ = orc.spmm_w4a4_at(W, d["Xq"][:N], one, np.ones(N, np.float16), n_idx, m_idx)
        assert np.array_equal(outs[0][0][n_idx, m_idx], oacc)


def test_balanced_ie_ffn_shape_ring_recycles(us, orc):
    """11008 x 4096 as 16 x 64 local tiles with 2 x 1 areas: 73 super-tiles a
    CTA, more chunks than the byte ring holds at once (the producer waits for
    the consumers to free it, before and after the dependency wait), with
    random row permutations; N = 1 (dp4a) and 32 (four mma token blocks),
    sampled outputs exact."""
    M, K = 11008, 4096
    rng, W, Xq, s_w, s_x = problem(21, M, K, 32)
    nT = (M // 16) * (K // 64)
    pm = np.concatenate([rng.permutation(16) for _ in range(nT)]).astype(np.uint8)
    E = us.us_encode_ie(torch.from_numpy(W).cuda(), 16, 64, 2, 1, I4, torch.from_numpy(pm).cuda())
    torch.cuda.synchronize()
    assert us.us_get_last_device_status() == us.US_OK
    for N in (1, 32):
        assert us.us_pick_split_k_ie(E, N) == 0
        for static in (False, True):
            acc, y = call(us, E, Xq[:N], s_w, s_x[:N], N, static, reps=1)[0]
            assert us.us_get_last_device_status() == us.US_OK
            n_idx, m_idx = rng.integers(0, N, 3000), rng.integers(0, M, 3000)
            oacc, oy = orc.spmm_w4a4_at(W, Xq[:N], s_w, s_x[:N], n_idx, m_idx)
            assert np.array_equal(acc[n_idx, m_idx], oacc), f"N {N} static {static}"
            assert np.array_equal(y[n_idx, m_idx], oy.view(np.uint16)), f"N {N} static {static}"
