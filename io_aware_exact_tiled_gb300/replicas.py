"""Host-side logic of replica runs: one process per GPU, each working on its
own (batch, head) problems, with no exchange of data between them.

Attention heads are independent, so the work shards across ranks without a
collective on the data path. The only communication is for timing: a barrier
on each side of the timed region, and the maximum over ranks of the timed
values. The whole-job throughput is the work all ranks did divided by the
slowest rank's time. Works with any torch.distributed backend: nccl between
GPUs, gloo on the host (which is how it is tested).
"""

from __future__ import annotations

import os
from typing import Iterable, List, Optional, Tuple

import torch
import torch.distributed as dist


def env() -> Tuple[int, int, int]:
    """(rank, world size, local rank) from the launcher's environment
    (torch.distributed.run sets RANK, WORLD_SIZE and LOCAL_RANK); (0, 1, 0)
    when run as a single process."""
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def active() -> bool:
    """True when a process group with more than one rank is initialised."""
    return dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1


def init(backend: str, world: int) -> None:
    """Join the process group (MASTER_ADDR / MASTER_PORT from the
    environment) when there is more than one rank."""
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend)


def barrier() -> None:
    if active():
        dist.barrier()


def max_over_ranks(values: Iterable[float], device: Optional[torch.device] = None) -> List[float]:
    """Element-wise maximum of `values` over all ranks. `device` must be one
    the backend can reduce on (a CUDA device for nccl, the CPU for gloo)."""
    vals = [float(v) for v in values]
    if not active():
        return vals
    t = torch.tensor(vals, dtype=torch.float64, device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def whole_job_rate(units_per_rank: float, seconds: float, world: int) -> float:
    """Units per second of the whole job: every rank processed
    `units_per_rank`, and the job took as long as its slowest rank."""
    if seconds <= 0:
        raise ValueError("the timed region must have a positive duration")
    return units_per_rank * world / seconds


def finish() -> None:
    if dist.is_available() and dist.is_initialized():
        dist.destroy_process_group()
