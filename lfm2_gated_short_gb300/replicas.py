"""Independent replicas across GPUs: rank discovery, barrier, max-over-ranks.

The ShortConv path has no exchange between sequences, so N GPUs run N
independent replicas (weak scaling). The only collectives are the barrier
around the timed region and one max-reduction of the elapsed time; no data
moves between ranks.
"""
from __future__ import annotations

import os

import torch
import torch.distributed as td


def env_rank():
    """(rank, world_size, local_rank) from the torchrun environment (1 process if unset)."""
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


class Group:
    """Barrier and max-reduction over the replicas; a no-op for one process."""

    def __init__(self, world: int, backend: str = "nccl"):
        self.world = world
        self.backend = backend
        self.owns = False
        if world > 1 and not td.is_initialized():
            td.init_process_group(backend=backend)
            self.owns = True

    def _device(self):
        if self.backend == "nccl":
            return torch.device("cuda", torch.cuda.current_device())
        return torch.device("cpu")

    def barrier(self):
        if self.world > 1:
            td.barrier()

    def max(self, value: float) -> float:
        if self.world == 1:
            return float(value)
        t = torch.tensor([float(value)], dtype=torch.float64, device=self._device())
        td.all_reduce(t, op=td.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.owns and td.is_initialized():
            td.destroy_process_group()
            self.owns = False


def aggregate_gbs(bytes_per_step: int, steps: int, world: int, max_ms: float) -> float:
    """Whole-job GB/s: every rank moved bytes_per_step x steps within the slowest rank's time."""
    if max_ms <= 0:
        raise ValueError("elapsed time must be positive")
    return bytes_per_step * steps * world / (max_ms * 1e-3) / 1e9
