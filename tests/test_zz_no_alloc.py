"""us_spmm_f16_noalloc: the fp16 SpMM entry point for callers that cannot
allocate device memory where they multiply (inside CUDA graph capture, behind a
fixed-arena allocator, in embedders that own every allocation).  Its split-K
scratch is a device array inside the library, so the results must match the
workspace-taking us_spmm_f16 on the same inputs - checked on two calls in a row,
the second one reusing whatever the first left in that shared array.

Named to be collected last: it must pass alone in a fresh process and after
every other test."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

REL_L2, MAX_ABS = 1e-3, 2e-2


def _close(a: np.ndarray, b: np.ndarray):
    a = a.astype(np.float64).reshape(-1)
    b = b.astype(np.float64).reshape(-1)
    rel = np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30)
    return rel <= REL_L2 and np.abs(a - b).max() <= MAX_ABS


@pytest.fixture(scope="module")
def us():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from bitmap_encoded_unstructured_ie_gb300 import build, binding
    build.build()
    binding.load()
    return binding


@pytest.mark.parametrize("N,split", [(5, 4), (40, 3), (300, 2), (1, 0)])
def test_noalloc_matches_workspace_entry_point_twice(us, N, split):
    rng = np.random.default_rng(N + split)
    M, K = 512, 1024
    W = (rng.standard_normal((M, K)) * 0.02).astype(np.float16)
    W[rng.random((M, K)) < 0.5] = 0
    E = us.us_encode(torch.from_numpy(W.view(np.int16)).cuda(), 64, 64, us.US_F16, us.US_ORDER_ROW)
    ws = us.workspace(us.US_OP_SPMM_F16, E, N, split)
    for call in range(2):                      # two calls in a row on the shared scratch array
        X = rng.standard_normal((N, K)).astype(np.float16)
        Xt = torch.from_numpy(X.view(np.int16)).cuda()
        Y_ref = torch.empty(N, M, dtype=torch.int16, device="cuda")
        Y_na = torch.empty(N, M, dtype=torch.int16, device="cuda")
        us.us_spmm_f16(E, Xt, N, Y_ref, ws, split)
        us.us_spmm_f16_noalloc(E, Xt, N, Y_na, split)
        torch.cuda.synchronize()
        assert us.us_get_last_device_status() == us.US_OK
        a = Y_na.cpu().numpy().view(np.float16)
        b = Y_ref.cpu().numpy().view(np.float16)
        assert _close(a, b), f"call {call}: no-allocation result differs from us_spmm_f16"


def test_noalloc_rejects_scratch_beyond_its_limit(us):
    rng = np.random.default_rng(3)
    W = (rng.standard_normal((4096, 4096)) * 0.02).astype(np.float16)
    E = us.us_encode(torch.from_numpy(W.view(np.int16)).cuda(), 64, 64, us.US_F16, us.US_ORDER_ROW)
    N = 256
    X = torch.zeros(N, 4096, dtype=torch.int16, device="cuda")
    Y = torch.empty(N, 4096, dtype=torch.int16, device="cuda")
    # an explicit split whose partials exceed the 8 MiB array is refused on the host
    assert us.us_workspace_bytes(us.US_OP_SPMM_F16, E, N, 8) > 8 << 20
    with pytest.raises(us.UsError) as ei:
        us.us_spmm_f16_noalloc(E, X, N, Y, 8)
    assert ei.value.code == us.US_ERR_TOO_LARGE
    # the automatic choice falls back to a split that fits
    us.us_spmm_f16_noalloc(E, X, N, Y, 0)
    torch.cuda.synchronize()
    assert us.us_get_last_device_status() == us.US_OK
