"""Host-side logic of multi-GPU runs: the path shards by token with no
exchange step, so N GPUs run N independent replicas (one process per GPU).
Each rank draws its own seeded inputs; the timed region is bracketed by
barriers; the whole-job figure divides the bytes all ranks processed by the
slowest rank's time. Nothing here touches a GPU: the reductions run on the
process group's own device (CUDA tensors under NCCL, CPU under gloo)."""

from __future__ import annotations


def rank_seed(base: int, rank: int, index: int = 0) -> int:
    """Seed of input set ``index`` of ``rank``: distinct for every (rank, set)
    of a run with fewer than 101 sets per rank."""
    return base + 101 * rank + index


def reduce_over_ranks(dist, value: float, op: str, device="cpu") -> float:
    """All-reduces one float64 over the ranks (``op``: "max" or "sum"); the
    value itself without a process group."""
    if dist is None:
        return float(value)
    import torch

    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


def job_rate(dist, elapsed_ms: float, bytes_per_step: float, steps: int, device="cpu"):
    """(ms per step of the slowest rank, bytes per step summed over the ranks,
    whole-job GB/s)."""
    slowest = reduce_over_ranks(dist, elapsed_ms, "max", device)
    total = reduce_over_ranks(dist, bytes_per_step, "sum", device)
    ms = slowest / steps
    return ms, total, total / (ms * 1e-3) / 1e9
