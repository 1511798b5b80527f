"""Whole-job accounting for independent replicas of the verify step.

The verify pass does not shard (one GPU holds the whole W8A8 model and the
path has no exchange step), so N GPUs run N independent replicas, one
process per GPU. Each rank times its own steps between two barriers; the job
takes as long as its slowest rank, and its throughput counts every rank's
tokens over that time (weak scaling: the per-rank work is fixed).
"""
from __future__ import annotations

import torch
import torch.distributed as dist


def world_size() -> int:
    return dist.get_world_size() if dist.is_available() and dist.is_initialized() else 1


def barrier():
    if world_size() > 1:
        dist.barrier()


def job_step_time_and_rate(ms_per_step: float, tokens_per_step: int, device) -> tuple[float, float]:
    """(max over ranks of the per-step milliseconds, whole-job tokens/s =
    world size x tokens per step / that time). Collective over all ranks."""
    t = torch.tensor([float(ms_per_step)], dtype=torch.float64, device=device)
    w = world_size()
    if w > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    ms_max = float(t.item())
    return ms_max, w * tokens_per_step / (ms_max / 1e3)
