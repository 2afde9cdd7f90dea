"""Process-group helpers for running one independent replica of the path per
GPU (weak scaling: every GPU dispatches and combines its own batch of R
virtual ranks; no data crosses GPUs, so no collective is on the data path).

Only the benchmark's bookkeeping uses a collective: a barrier around the
timed region, the maximum of the per-rank step times and the sum of the
per-rank token counts.
"""
from __future__ import annotations

import os
from dataclasses import dataclass

import torch
import torch.distributed as dist


@dataclass
class RankInfo:
    rank: int
    world: int
    local_rank: int


def init_from_env(backend: str = "nccl") -> RankInfo:
    """Reads RANK / WORLD_SIZE / LOCAL_RANK (torchrun) and joins the group when
    WORLD_SIZE > 1.  With the nccl backend the process binds cuda:LOCAL_RANK."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if backend == "nccl":
        torch.cuda.set_device(local)
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        if backend == "nccl":
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group(backend)
    return RankInfo(rank, world, local)


def _device(backend_hint=None):
    if dist.is_initialized() and dist.get_backend() == "nccl":
        return torch.device("cuda", torch.cuda.current_device())
    return torch.device("cpu")


def barrier():
    if dist.is_initialized() and dist.get_world_size() > 1:
        dist.barrier()


def max_over_ranks(v: float) -> float:
    if not (dist.is_initialized() and dist.get_world_size() > 1):
        return float(v)
    t = torch.tensor([float(v)], dtype=torch.float64, device=_device())
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(v: float) -> float:
    if not (dist.is_initialized() and dist.get_world_size() > 1):
        return float(v)
    t = torch.tensor([float(v)], dtype=torch.float64, device=_device())
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def rank_seed(base: int, rank: int) -> int:
    """Seed of a rank's own batch: distinct per rank, fixed per (base, rank)."""
    return base + 1000 * rank


def shutdown():
    if dist.is_initialized():
        dist.destroy_process_group()
