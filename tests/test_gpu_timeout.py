"""The device-side timeout path, made to run out without a fault or a hang.

Every wait in the kernels (mbarrier phases, posted partials) is bounded by the
GPU's global timer; a wait that runs out records US_ERR_TIMEOUT in the device
status word and the kernel returns.  us_selftest_wait_timeout runs that same
bounded mbarrier wait on a barrier that nothing completes, with no copy in
flight and a short limit.  The tests check that the status comes back as
US_ERR_TIMEOUT once and is then cleared, that the wait lasted at least its
limit, and that the context is still usable: a normal SpMM afterwards is still
bit-exact against the oracle.
"""
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


def test_wait_runs_out_and_reports_timeout(us, orc):
    assert us.us_get_last_device_status() == us.US_OK          # nothing pending from earlier tests
    elapsed = torch.zeros(1, dtype=torch.int64, device="cuda")
    limit = 1_000_000                                            # 1 ms
    us.us_selftest_wait_timeout(limit, elapsed)
    assert us.us_get_last_device_status() == us.US_ERR_TIMEOUT
    assert us.us_get_last_device_status() == us.US_OK          # read and cleared
    ns = int(elapsed.item())
    assert limit <= ns < 200 * limit, f"wait gave up after {ns} ns"

    # the context survives: a W4A4 call right after is still bit-exact
    d = wl.w4a4(256, 1024, 8, 0.5, seed=11)
    E = us.us_encode(torch.from_numpy(d["Wq"]).cuda(), 64, 64, us.US_I4, us.US_ORDER_ROW)
    N = 8
    ya = torch.empty(N, 256, dtype=torch.int32, device="cuda")
    yh = torch.empty(N, 256, dtype=torch.int16, device="cuda")
    us.us_spmm_w4a4(E, torch.from_numpy(wl.pack_int4(d["Xq"][:N])).cuda(),
                    torch.from_numpy(d["s_w"].view(np.int16)).cuda(),
                    torch.from_numpy(d["s_x"][:N].view(np.int16)).cuda(), N, ya, yh,
                    us.workspace(us.US_OP_SPMM_W4A4, E, N))
    assert us.us_get_last_device_status() == us.US_OK
    oa, oh = orc.spmm_w4a4(d["Wq"], d["Xq"][:N], d["s_w"], d["s_x"][:N])
    assert np.array_equal(ya.cpu().numpy(), oa)
    assert np.array_equal(yh.cpu().numpy().view(np.uint16), oh.view(np.uint16))


def test_timeout_twice_in_a_row(us):
    for _ in range(2):
        us.us_selftest_wait_timeout(20_000)                     # 20 us, no elapsed output
        assert us.us_get_last_device_status() == us.US_ERR_TIMEOUT
    assert us.us_get_last_device_status() == us.US_OK


def test_limit_is_checked_on_the_host(us):
    for bad in (0, 999, 1_000_000_001):
        with pytest.raises(us.UsError) as ei:
            us.us_selftest_wait_timeout(bad)
        assert ei.value.code == us.US_ERR_INVALID_ARG
