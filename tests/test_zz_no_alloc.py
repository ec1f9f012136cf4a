"""us_spmm_f16_noalloc: the fp16 SpMM entry point for callers that cannot
allocate device memory where they multiply (behind a fixed-arena allocator, in
embedders that own every allocation).  Its split-K scratch is a device array
inside the library.  With the same split it runs the same kernel as the
workspace-taking us_spmm_f16, whose fp32 partials are reduced in fixed slice
order, so the two must agree bit for bit; both are also held to the oracle.
Checked on two calls in a row, the second one reusing whatever the first left
in that shared array.

Named to be collected last: it must pass alone in a fresh process and after
every other test."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

REL_L2, MAX_ABS = 1e-3, 2e-2
SCRATCH = 8 << 20                               # US_NOALLOC_SCRATCH_BYTES


def _check_oracle(orc, W, X, y, n_idx, m_idx, what):
    _, exact = orc.spmm_f16_at(W, X, n_idx, m_idx)
    got = y.astype(np.float64).reshape(-1)
    err = got - exact
    rel = np.linalg.norm(err) / max(np.linalg.norm(exact), 1e-30)
    assert rel <= REL_L2 and np.abs(err).max() <= MAX_ABS, f"{what}: rel L2 {rel:.3e}, max abs {np.abs(err).max():.3e}"


@pytest.fixture(scope="module")
def us():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from bitmap_encoded_unstructured_ie_gb300 import build, binding
    build.build()
    binding.load()
    return binding


@pytest.mark.parametrize("N,split", [(5, 4), (40, 3), (300, 2), (1, 0)])
def test_noalloc_matches_workspace_entry_point_twice(us, orc, N, split):
    rng = np.random.default_rng(N + split)
    M, K = 512, 1024
    W = (rng.standard_normal((M, K)) * 0.02).astype(np.float16)
    W[rng.random((M, K)) < 0.5] = 0
    E = us.us_encode(torch.from_numpy(W.view(np.int16)).cuda(), 64, 64, us.US_F16, us.US_ORDER_ROW)
    ws = us.workspace(us.US_OP_SPMM_F16, E, N, split)
    # the scratch fits, so both entry points plan the same kernel and split
    assert us.us_workspace_bytes(us.US_OP_SPMM_F16, E, N, split) <= SCRATCH
    n_idx, m_idx = np.meshgrid(np.arange(N), np.arange(M), indexing="ij")
    for call in range(2):                      # two calls in a row on the shared scratch array
        X = rng.standard_normal((N, K)).astype(np.float16)
        Xt = torch.from_numpy(X.view(np.int16)).cuda()
        Y_ref = torch.empty(N, M, dtype=torch.int16, device="cuda")
        Y_na = torch.empty(N, M, dtype=torch.int16, device="cuda")
        us.us_spmm_f16(E, Xt, N, Y_ref, ws, split)
        us.us_spmm_f16_noalloc(E, Xt, N, Y_na, split)
        torch.cuda.synchronize()
        assert us.us_get_last_device_status() == us.US_OK
        assert torch.equal(Y_na, Y_ref), f"call {call}: no-allocation result is not bitwise equal to us_spmm_f16"
        a = Y_na.cpu().numpy().view(np.float16)
        _check_oracle(orc, W, X, a, n_idx.reshape(-1), m_idx.reshape(-1), f"call {call}")


def test_noalloc_rejects_scratch_beyond_its_limit(us, orc):
    """256-row tiles run on the generic kernel, whose split-K partials live in
    the scratch array: an explicit split whose partials exceed it is refused,
    and an automatic split that would exceed it falls back to one slice.  (The
    tensor-core path reduces its slices in a cluster and needs no scratch.)"""
    rng = np.random.default_rng(3)
    M = K = 4096
    W = (rng.standard_normal((M, K)) * 0.02).astype(np.float16)
    W[rng.random((M, K)) < 0.5] = 0
    E = us.us_encode(torch.from_numpy(W.view(np.int16)).cuda(), 256, 64, us.US_F16, us.US_ORDER_ROW)
    N = 40
    X = rng.standard_normal((N, K)).astype(np.float16)
    Xt = torch.from_numpy(X.view(np.int16)).cuda()
    Y = torch.empty(N, M, dtype=torch.int16, device="cuda")
    # an explicit split whose partials exceed the 8 MiB array is refused on the host
    assert us.us_workspace_bytes(us.US_OP_SPMM_F16, E, N, 16) > SCRATCH
    with pytest.raises(us.UsError) as ei:
        us.us_spmm_f16_noalloc(E, Xt, N, Y, 16)
    assert ei.value.code == us.US_ERR_TOO_LARGE
    # the automatic choice would not fit either, so it falls back to one slice:
    # the same result, bit for bit, as an explicit split of 1 with a workspace
    assert us.us_workspace_bytes(us.US_OP_SPMM_F16, E, N, 0) > SCRATCH
    for call in range(2):
        us.us_spmm_f16_noalloc(E, Xt, N, Y, 0)
        Y1 = torch.empty_like(Y)
        us.us_spmm_f16(E, Xt, N, Y1, us.workspace(us.US_OP_SPMM_F16, E, N, 1), 1)
        torch.cuda.synchronize()
        assert us.us_get_last_device_status() == us.US_OK
        assert torch.equal(Y, Y1), f"call {call}: fallback result differs from split_k = 1"
    s = np.random.default_rng(5)
    n_idx = s.integers(0, N, 4000).astype(np.int32)
    m_idx = s.integers(0, M, 4000).astype(np.int32)
    y = Y.cpu().numpy().view(np.float16)[n_idx, m_idx]
    _check_oracle(orc, W, X, y, n_idx, m_idx, "fallback, sampled outputs")


def test_noalloc_tensor_core_path_needs_no_scratch(us, orc):
    """The tensor-core path with the largest split (8 slices in one cluster)
    through the no-allocation entry point: bitwise equal to us_spmm_f16."""
    rng = np.random.default_rng(4)
    M = K = 4096
    W = (rng.standard_normal((M, K)) * 0.02).astype(np.float16)
    W[rng.random((M, K)) < 0.6] = 0
    E = us.us_encode(torch.from_numpy(W.view(np.int16)).cuda(), 64, 64, us.US_F16, us.US_ORDER_ROW)
    N = 256
    Xt = torch.from_numpy(rng.standard_normal((N, K)).astype(np.float16).view(np.int16)).cuda()
    assert us.us_workspace_bytes(us.US_OP_SPMM_F16, E, N, 8) <= 16
    Y = torch.empty(N, M, dtype=torch.int16, device="cuda")
    Y1 = torch.empty_like(Y)
    us.us_spmm_f16_noalloc(E, Xt, N, Y, 8)
    us.us_spmm_f16(E, Xt, N, Y1, us.workspace(us.US_OP_SPMM_F16, E, N, 8), 8)
    torch.cuda.synchronize()
    assert us.us_get_last_device_status() == us.US_OK
    assert torch.equal(Y, Y1)
