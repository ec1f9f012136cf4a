"""Row-band sharding of an encoded matrix, checked on the CPU.

Two ranks over gloo: each takes its tile-row bands of the encoded matrix
(bitmap and value pieces of the whole arrays, tile_off rebased), decodes and
multiplies them with the oracle, and the ranks all-gather their output rows.
The concatenation must equal the whole matrix's oracle result (int32 and
fp16 bits for W4A4, fp16 bits for fp16), and each shard must decode to
exactly its rows of W.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from bitmap_encoded_unstructured_ie_gb300 import sharding
from bitmap_encoded_unstructured_ie_gb300 import workloads as wl


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _gather_rows(dist, y: np.ndarray, world: int) -> np.ndarray:
    """All-gather N x M_r blocks (one per rank, sizes may differ) along M."""
    t = torch.from_numpy(np.ascontiguousarray(y).view(np.uint8).reshape(y.shape[0], -1).copy())
    sizes = [torch.zeros(1, dtype=torch.int64) for _ in range(world)]
    dist.all_gather(sizes, torch.tensor([t.shape[1]], dtype=torch.int64))
    mx = int(max(s.item() for s in sizes))
    pad = torch.zeros(t.shape[0], mx, dtype=torch.uint8)
    pad[:, : t.shape[1]] = t
    parts = [torch.zeros_like(pad) for _ in range(world)]
    dist.all_gather(parts, pad)
    cols = [p[:, : int(s.item())] for p, s in zip(parts, sizes)]
    return torch.cat(cols, dim=1).numpy().copy().view(y.dtype)


def _worker(rank, world, port, outdir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    from oracle import oracle as orc
    dist.init_process_group("gloo")
    try:
        M, K, TM, TK, N = 448, 256, 64, 64, 3          # 7 bands: 3 + 4
        d = wl.w4a4(M, K, N, 0.5, seed=21)
        bm, off, vals = orc.encode(d["Wq"], TM, TK, orc.I4, orc.ROW)
        b0, b1 = sharding.band_ranges(M // TM, world)[rank]
        sbm, soff, svals, Ms = sharding.shard_arrays(bm, off, vals, M, K, TM, TK, orc.I4, b0, b1)
        assert soff[0] == 0 and Ms == (b1 - b0) * TM
        Wd = orc.decode(sbm, soff, svals, Ms, K, TM, TK, orc.I4, orc.ROW)
        assert np.array_equal(Wd, d["Wq"][b0 * TM: b1 * TM]), "shard does not decode to its rows"
        acc, y = orc.spmm_w4a4(Wd, d["Xq"], d["s_w"][b0 * TM: b1 * TM], d["s_x"])
        acc_all = _gather_rows(dist, acc, world)
        y_all = _gather_rows(dist, y.view(np.uint16), world)

        # fp16, COL order (the spMspV format), 5 bands: 2 + 3
        f = wl.f16_spmm(320, 192, 2, 0.5, seed=22)
        fb, fo, fv = orc.encode(f["W"], 64, 64, orc.F16, orc.COL)
        c0, c1 = sharding.band_ranges(5, world)[rank]
        gb, go, gv, Mf = sharding.shard_arrays(fb, fo, fv, 320, 192, 64, 64, orc.F16, c0, c1)
        Wf = orc.decode(gb, go, gv, Mf, 192, 64, 64, orc.F16, orc.COL)
        assert np.array_equal(Wf.view(np.uint16), f["W"][c0 * 64: c1 * 64].view(np.uint16))
        yf_all = _gather_rows(dist, orc.spmm_f16(Wf, f["X"]).view(np.uint16), world)
        if rank == 0:
            np.savez(os.path.join(outdir, "out.npz"), acc=acc_all, y=y_all, yf=yf_all)
    finally:
        dist.destroy_process_group()


def test_band_ranges_cover_every_band_once():
    for nTM in (0, 1, 7, 64, 224):
        for world in (1, 2, 3, 8):
            r = sharding.band_ranges(nTM, world)
            assert len(r) == world and r[0][0] == 0 and r[-1][1] == nTM
            assert all(a <= b for a, b in r) and all(r[i][1] == r[i + 1][0] for i in range(world - 1))
            sizes = [b - a for a, b in r]
            assert max(sizes) - min(sizes) <= 1


def test_shards_concatenate_to_the_whole_product(tmp_path, orc):
    mp.spawn(_worker, args=(2, _free_port(), str(tmp_path)), nprocs=2, join=True)
    out = np.load(tmp_path / "out.npz")
    d = wl.w4a4(448, 256, 3, 0.5, seed=21)
    acc, y = orc.spmm_w4a4(d["Wq"], d["Xq"], d["s_w"], d["s_x"])
    assert np.array_equal(out["acc"], acc)
    assert np.array_equal(out["y"], y.view(np.uint16))
    f = wl.f16_spmm(320, 192, 2, 0.5, seed=22)
    assert np.array_equal(out["yf"], orc.spmm_f16(f["W"], f["X"]).view(np.uint16))


def test_shard_offsets_stay_padded_and_valid(orc):
    """Every shard is a well-formed encoding of its own (host validator rules:
    monotone offsets, runs padded to 16 bytes, padding zero)."""
    from bitmap_encoded_unstructured_ie_gb300 import binding
    try:
        binding.load()
    except binding.LibraryMissing:
        pytest.skip("library not built")
    d = wl.w4a4(512, 320, 1, 0.3, seed=23)
    bm, off, vals = orc.encode(d["Wq"], 64, 64, orc.I4, orc.ROW)
    for world in (2, 3, 8):
        for b0, b1 in sharding.band_ranges(8, world):
            if b0 == b1:
                continue
            sbm, soff, svals, Ms = sharding.shard_arrays(bm, off, vals, 512, 320, 64, 64, orc.I4, b0, b1)
            assert binding.us_validate_host(sbm, soff, svals, Ms, 320, 64, 64, orc.I4, orc.ROW) == 0
