"""Process-group plumbing for running independent replicas of the workload, one
process per GPU (launched by torchrun). The attention path itself needs no
exchange between GPUs: every (batch, head) is independent, so each rank runs
its own copy of the workload and only the host-side timing is combined (a
barrier around the timed region and the maximum elapsed time over ranks)."""
from __future__ import annotations

import os

import torch
import torch.distributed as dist


def world() -> tuple[int, int, int]:
    """(rank, world_size, local_rank) from the torchrun environment (1 process if unset)."""
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def init(backend: str) -> bool:
    """Initialises the default process group when more than one rank runs."""
    _, ws, _ = world()
    if ws > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return ws > 1


def barrier():
    if dist.is_initialized():
        dist.barrier()


def max_over_ranks(x: float, device=None) -> float:
    """Maximum of a host float over all ranks (the slowest rank sets the time)."""
    if not dist.is_initialized():
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, device=None) -> float:
    if not dist.is_initialized():
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def aggregate_throughput(units_per_rank: float, elapsed_per_rank_s: float, device=None) -> dict:
    """Whole-job throughput: units processed by all ranks / slowest rank's time."""
    total_units = sum_over_ranks(units_per_rank, device)
    t_max = max_over_ranks(elapsed_per_rank_s, device)
    return {"total_units": total_units, "max_elapsed_s": t_max,
            "throughput": total_units / t_max if t_max > 0 else float("nan")}


def finalize():
    if dist.is_initialized():
        dist.destroy_process_group()
