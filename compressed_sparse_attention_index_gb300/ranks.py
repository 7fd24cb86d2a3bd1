"""Host logic of a multi-GPU run (bench.py under torchrun): one process per GPU.

Decode batches are independent sequences, so the ranks are replicas: each rank
decodes its own batch (same shapes, its own generator seed) with no collective
on the data path.  Only the timing crosses ranks: a barrier on both sides of
the timed region, the maximum elapsed time over ranks, and the units of all
ranks over that time (weak scaling).  The collectives are torch.distributed's
(NCCL on GPUs; the CPU tests run the same calls on gloo)."""
import dataclasses
import os


def rank_env():
    """(rank, world size, local rank) from the launcher's environment."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def rank_workload(wl, rank: int):
    """Rank r's batch: the configuration's shapes with a seed of its own (rank 0
    keeps the configuration's seed, so a one-GPU run is unchanged)."""
    if rank == 0:
        return wl
    return dataclasses.replace(wl, name=f"{wl.name}_rank{rank}", seed=wl.seed + 7919 * rank)


def _world():
    import torch.distributed as dist
    return dist.get_world_size() if dist.is_available() and dist.is_initialized() else 1


def barrier():
    """Every rank reaches this point (no-op on one rank)."""
    import torch.distributed as dist
    if _world() > 1:
        dist.barrier()


def max_over_ranks(x: float, device=None) -> float:
    """The largest value over ranks (the job's time is its slowest rank's)."""
    if _world() == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, max_ms: float) -> float:
    """Units of all ranks per second over the slowest rank's time."""
    return units_per_rank * world / (max_ms / 1e3)
