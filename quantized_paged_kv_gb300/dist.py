"""Host-side helpers for running the decode path on several GPUs of one node.

The path shards by sequence: a rank owns whole sequences (their pages, block
tables, queries and outputs), so decode attention needs no exchange between
GPUs.  The only collectives are a barrier around timed regions and a max over
ranks of the measured times.  Works with the ``nccl`` backend (CUDA tensors)
and the ``gloo`` backend (CPU tensors).
"""
from __future__ import annotations

import heapq

import numpy as np


def shard_sequences(seq_lens, world):
    """Assign sequences to ``world`` ranks: longest first, each to the rank with
    the fewest tokens so far (ties to the lower rank).  Returns a list of sorted
    int64 index arrays, one per rank; every sequence appears exactly once."""
    if world < 1:
        raise ValueError("world must be >= 1")
    lens = np.asarray(seq_lens, dtype=np.int64)
    order = sorted(range(len(lens)), key=lambda i: (-int(lens[i]), i))
    heap = [(0, r) for r in range(world)]
    owned = [[] for _ in range(world)]
    for i in order:
        load, r = heapq.heappop(heap)
        owned[r].append(i)
        heapq.heappush(heap, (load + int(lens[i]), r))
    return [np.asarray(sorted(o), dtype=np.int64) for o in owned]


def problem_seed(base_seed, index):
    """Seed of independent problem ``index`` of a job made of several copies of
    one workload (index 0 keeps the workload's own seed)."""
    return int(base_seed) + 7919 * int(index)


class RankGroup:
    """Barrier and max-over-ranks for the timing protocol (identity at world 1)."""

    def __init__(self, world, rank, device=None):
        self.world, self.rank, self.device = world, rank, device

    @classmethod
    def from_env(cls, backend):
        import os

        import torch.distributed as dist

        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        if world > 1 and not dist.is_initialized():
            dist.init_process_group(backend)
        return cls(world, rank, "cuda" if backend == "nccl" else "cpu")

    def barrier(self):
        if self.world > 1:
            import torch.distributed as dist

            dist.barrier()

    def allmax(self, x):
        if self.world == 1:
            return float(x)
        import torch
        import torch.distributed as dist

        t = torch.tensor([float(x)], dtype=torch.float64, device=self.device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.world > 1:
            import torch.distributed as dist

            if dist.is_initialized():
                dist.destroy_process_group()
