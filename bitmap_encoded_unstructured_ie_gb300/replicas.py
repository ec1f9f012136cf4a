"""Host logic of a multi-GPU run: one process per GPU, each an independent
replica of the whole product on its own weight copies (tile-row bands are
independent, so nothing crosses GPUs inside a product; the benchmark shards
nothing and adds no collective to the data path).  The only cross-rank steps
are the timing ones: a barrier on each side of the timed region and the
maximum of the ranks' times, so that whole-job throughput is the units all
ranks processed over the slowest rank's time (weak scaling)."""
from __future__ import annotations

import os


def rank_env():
    """(world, rank, local_rank) from the launcher's environment."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def init(world: int, backend: str = "nccl"):
    """torch.distributed for world > 1 (None for a single process)."""
    if world <= 1:
        return None
    import torch.distributed as dist
    if not dist.is_initialized():
        dist.init_process_group(backend)
    return dist


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, value: float, device=None) -> float:
    """The largest of the ranks' values (every rank gets it)."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_rate(units_per_rank: float, world: int, seconds: float) -> float:
    """Whole-job rate: every rank processed units_per_rank in at most `seconds`."""
    return units_per_rank * world / seconds


def finish(dist):
    if dist is not None:
        dist.destroy_process_group()
