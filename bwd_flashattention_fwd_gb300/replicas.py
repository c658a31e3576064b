"""One process per GPU, each running an independent replica of the workload.

The attention path has no exchange step between GPUs: every (batch, KV head)
group is independent, so more GPUs means more independent problems (weak
scaling) and the only cross-rank traffic is timing bookkeeping: a barrier
around the timed region and a max / sum over ranks of the measured numbers.
"""

from __future__ import annotations

import os

import torch
import torch.distributed as dist


def world() -> tuple[int, int, int]:
    """(rank, local_rank, world_size) from the torchrun environment."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def init(backend: str) -> None:
    """Join the process group when launched with more than one rank."""
    _, _, ws = world()
    if ws > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)


def barrier(device=None) -> None:
    if dist.is_available() and dist.is_initialized():
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[torch.device(device).index])
        else:
            dist.barrier()


def _reduce(x: float, op, device) -> float:
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=op)
    return float(t.item())


def max_over_ranks(x: float, device="cpu") -> float:
    return _reduce(x, dist.ReduceOp.MAX, device)


def sum_over_ranks(x: float, device="cpu") -> float:
    return _reduce(x, dist.ReduceOp.SUM, device)


def aggregate_throughput(units_local: float, seconds_local: float, device="cpu") -> tuple[float, float, float]:
    """Whole-job throughput: all ranks' units over the slowest rank's time.

    Returns (value, total_units, max_seconds)."""
    total = sum_over_ranks(units_local, device)
    tmax = max_over_ranks(seconds_local, device)
    return total / tmax, total, tmax


def shutdown() -> None:
    if dist.is_available() and dist.is_initialized():
        dist.destroy_process_group()
