"""Host-side logic for running the layer on several GPUs of one node.

Channels (and batch rows) are independent in every step of the S4 forward
path, so ranks never exchange data: each rank runs its own shard of work on
its own GPU.  The only collectives are outside the data path -- a barrier
before and after a timed region and a max over ranks of its duration -- and
they live here so that they can be exercised with the gloo backend on CPU.
"""
from __future__ import annotations

import os


def dist_env():
    """(rank, local_rank, world_size) from the torchrun environment (1 process if unset)."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def channel_shard(H: int, rank: int, world: int):
    """Contiguous channel range [lo, hi) of `rank` when H channels are split
    over `world` ranks as evenly as possible (for strong scaling)."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad rank/world")
    base, extra = divmod(H, world)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


def max_over_ranks(ms: float, device=None) -> float:
    """Maximum of a per-rank duration over all ranks (the job's time); the
    value itself when torch.distributed is not initialised."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(ms)
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device or "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.barrier()


def job_throughput(units_per_rank_step: int, steps: int, world: int, ms_max: float) -> float:
    """Units per second of the whole job: every rank processed
    units_per_rank_step per step (weak scaling) and the job took ms_max."""
    return units_per_rank_step * world * steps / (ms_max / 1e3)
