"""Back-to-back W4A4 launches captured in a CUDA graph on a side stream, as a
decode loop runs them: static weights (a launch may fetch and decode its
weights while the previous one still runs), one shared workspace and one
output buffer, several graph replays in a row with no host sync in between.

Every launch's int32 accumulators must equal the oracle's, the posted-partial
workspace must be left all zero, and the device status word must stay clean.
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


@pytest.fixture(scope="module")
def orc():
    from oracle import oracle as o
    o._load()
    return o


@pytest.mark.parametrize("M,K,N,bits", [(1024, 2048, 1, 4), (1024, 2048, 8, 4), (1024, 2048, 16, 4), (704, 1536, 5, 4),
                                        (11008, 4096, 1, 4), (11008, 4096, 3, 4), (1024, 2048, 3, 2),
                                        (1024, 2048, 16, 2)])
def test_w4a4_graph_of_static_launches(us, orc, M, K, N, bits):
    dev = "cuda"
    # four distinct weight matrices (int4, or int2 for W2A4), launched in turn,
    # each writing its own output
    gen = wl.w4a4 if bits == 4 else wl.w2a4
    mats = [gen(M, K, N, 0.5, seed=10 + i) for i in range(4)]
    Es = []
    for d in mats:
        E = us.us_encode(torch.from_numpy(d["Wq"]).to(dev), 64, 64, us.US_I4 if bits == 4 else us.US_I2,
                         us.US_ORDER_ROW)
        E.flags = us.US_BITMAP_STATIC
        Es.append(E)
    X = torch.from_numpy(mats[0]["Xq_packed"]).to(dev)
    sx = torch.from_numpy(mats[0]["s_x"].view(np.int16)).to(dev)
    sws = [torch.from_numpy(d["s_w"].view(np.int16)).to(dev) for d in mats]
    Ya = [torch.zeros(N, M, dtype=torch.int32, device=dev) for _ in mats]
    Yh = [torch.zeros(N, M, dtype=torch.int16, device=dev) for _ in mats]
    ws = us.workspace(us.US_OP_SPMM_W4A4, Es[0], N)
    stream = torch.cuda.Stream()

    def run():
        for i, E in enumerate(Es):
            us.us_spmm_w4a4(E, X, sws[i], sx, N, Ya[i], Yh[i], ws, 0, stream)

    with torch.cuda.stream(stream):
        run()
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        run()
    for y in Ya:
        y.zero_()
    with torch.cuda.stream(stream):
        for _ in range(5):
            g.replay()
    assert us.us_get_last_device_status(stream) == us.US_OK
    assert not ws.any().item(), "posted partials not cleared"
    for i, d in enumerate(mats):
        oacc, oy = orc.spmm_w4a4(d["Wq"], mats[0]["Xq"], d["s_w"], mats[0]["s_x"])
        assert np.array_equal(Ya[i].cpu().numpy(), oacc), f"launch {i}: accumulators differ"
        assert np.array_equal(Yh[i].cpu().numpy().view(np.uint16), oy.view(np.uint16)), f"launch {i}: fp16 differs"


@pytest.mark.parametrize("M,K,N", [(640, 4096, 1), (704, 1024, 5), (640, 1536, 3), (1088, 4096, 16)])
def test_w4a4_static_ranges_of_unequal_length(us, orc, M, K, N):
    """Where the SM count does not divide the tile count, the balanced ranges
    differ by one tile: with static weights every CTA decodes before the wait
    only the tiles of its own range (e.g. 640 x 4096 on 152 SMs: ranges of 4
    and 5 tiles, all of them decoded early). The status word must stay clean."""
    d = wl.w4a4(M, K, N, 0.5, seed=3)
    E = us.us_encode(torch.from_numpy(d["Wq"]).cuda(), 64, 64, us.US_I4, us.US_ORDER_ROW)
    assert us.us_get_last_device_status() == us.US_OK
    E.flags = us.US_BITMAP_STATIC
    Ya = torch.empty(N, M, dtype=torch.int32, device="cuda")
    Yh = torch.empty(N, M, dtype=torch.int16, device="cuda")
    ws = us.workspace(us.US_OP_SPMM_W4A4, E, N)
    for _ in range(3):
        us.us_spmm_w4a4(E, torch.from_numpy(d["Xq_packed"]).cuda(), torch.from_numpy(d["s_w"].view(np.int16)).cuda(),
                        torch.from_numpy(d["s_x"].view(np.int16)).cuda(), N, Ya, Yh, ws)
        assert us.us_get_last_device_status() == us.US_OK
    oacc, oy = orc.spmm_w4a4(d["Wq"], d["Xq"], d["s_w"], d["s_x"])
    assert np.array_equal(Ya.cpu().numpy(), oacc)
    assert np.array_equal(Yh.cpu().numpy().view(np.uint16), oy.view(np.uint16))
