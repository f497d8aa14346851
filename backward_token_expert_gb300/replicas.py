"""Independent replicas of the recalibration path, one per rank.

Nothing in the path exchanges data inside one layer: route statistics, the
score, the per-expert selection, compaction and both grouped GEMMs all work on
the layer's own tokens and experts.  N GPUs therefore run N independent layer
batches, with no collective on the data path.  This module holds the host
logic around that:

* the seed each replica draws its synthetic batch with (rank 0 draws the
  single-GPU batch, so a one-rank run and rank 0 of a multi-rank run agree);
* the job-wide totals: retained pairs summed over ranks, elapsed time as the
  slowest rank's, so the throughput is the whole job's.

torch.distributed is used only when a process group is initialised with more
than one rank; the same code runs on gloo (CPU) and NCCL.
"""

from __future__ import annotations


def replica_seed(rank: int, base_seed: int = 0) -> int:
    """Seed of the synthetic layer batch of replica `rank`."""
    if rank < 0:
        raise ValueError("rank must be non-negative")
    return base_seed + rank


def _group_size() -> int:
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return 1
    return dist.get_world_size()


def job_totals(retained: int, elapsed_s: float, device=None) -> tuple[int, float]:
    """(retained pairs summed over ranks, elapsed seconds of the slowest rank),
    the same on every rank.  `device` is where the reduction tensors live: the
    rank's GPU under NCCL, the CPU under gloo (the default picks by backend)."""
    if retained < 0 or elapsed_s < 0:
        raise ValueError("retained pairs and elapsed time must be non-negative")
    if _group_size() == 1:
        return int(retained), float(elapsed_s)
    import torch
    import torch.distributed as dist

    if device is None:
        device = "cuda" if dist.get_backend() == "nccl" else "cpu"
    r = torch.tensor([float(retained)], dtype=torch.float64, device=device)
    t = torch.tensor([float(elapsed_s)], dtype=torch.float64, device=device)
    dist.all_reduce(r, op=dist.ReduceOp.SUM)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return int(round(r.item())), float(t.item())


def job_throughput(retained_per_step: int, steps: int, elapsed_s: float, device=None) -> float:
    """Whole-job retained pairs per second over `steps` steps of every rank."""
    if steps <= 0:
        raise ValueError("steps must be positive")
    total, slowest = job_totals(retained_per_step * steps, elapsed_s, device)
    if slowest <= 0:
        raise ValueError("elapsed time must be positive")
    return total / slowest
