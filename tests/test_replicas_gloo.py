"""The multi-GPU host logic on the CPU: world size 2 over gloo.

Tile-row bands are independent, so a multi-GPU run is N independent replicas
with no collective on the data path. These tests check what the ranks do
share, on the same code the benchmark uses: the barriers, the maximum of the
ranks' times, the whole-job rate, the reference arm's other ranks exiting
without work, and a failing rank surfacing on the host.
"""
import argparse
import json
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, outdir, fail_rank):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    from bitmap_encoded_unstructured_ie_gb300 import replicas
    w, r, local = replicas.rank_env()
    dist = replicas.init(w, "gloo")
    try:
        replicas.barrier(dist)
        if r == fail_rank:
            raise RuntimeError("rank failed between steps")
        my_ms = 10.0 + 5.0 * r                           # the ranks' own timed regions
        mx = replicas.max_over_ranks(dist, my_ms)
        replicas.barrier(dist)
        rate = replicas.aggregate_rate(100.0, w, mx * 1e-3)
        with open(os.path.join(outdir, f"rank{r}.json"), "w") as f:
            json.dump({"world": w, "rank": r, "local": local, "max_ms": mx, "rate": rate}, f)
    finally:
        replicas.finish(dist)


def test_two_replicas_share_only_the_timing(tmp_path):
    mp.spawn(_worker, args=(2, _free_port(), str(tmp_path), -1), nprocs=2, join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    for r, d in enumerate(res):
        assert d["world"] == 2 and d["rank"] == r and d["local"] == r
        assert d["max_ms"] == 15.0                       # every rank sees the slowest rank's time
        assert d["rate"] == pytest.approx(100.0 * 2 / 15e-3)


def test_failing_rank_is_reported_on_the_host(tmp_path):
    """A rank that raises before the collective: the launcher sees the failure
    (no GPU is involved; the other rank's wait is ended by the process group)."""
    with pytest.raises(Exception):
        mp.spawn(_worker, args=(2, _free_port(), str(tmp_path), 1), nprocs=2, join=True)
    assert not (tmp_path / "rank1.json").exists()


def test_single_process_needs_no_process_group():
    from bitmap_encoded_unstructured_ie_gb300 import replicas
    assert replicas.init(1) is None
    assert replicas.max_over_ranks(None, 3.5) == 3.5
    assert replicas.aggregate_rate(10.0, 1, 2.0) == 5.0


def test_reference_arm_other_ranks_exit_without_work(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = argparse.Namespace(gpus=2, steps=1, warmup=3)
    assert bench.run_reference(args) == 0
    assert capsys.readouterr().out == ""
