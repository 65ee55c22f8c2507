"""Host-side helpers for running the decode path on several GPUs of one node.

Two ways to split the work:
  * by sequence (shard_sequences): a rank owns whole sequences (their pages,
    block tables, queries and outputs), so decode attention needs no exchange
    between GPUs; the only collectives are a barrier around timed regions and a
    max over ranks of the measured times;
  * by context, for one very long sequence (context_slices, gather_partials,
    merged_offsets): each rank holds a contiguous run of the sequence's pages
    and decodes it alone, keeping the log-sum-exp of its partial result; the
    ranks then exchange their (o, lse) partials once (an all-gather of B x Hq x
    (D + 1) floats a rank), and every rank combines them with the same split
    merge the single-GPU path uses ("long-context-attention-and-lessons",
    section "Give more GPU workers a piece of the attention calculation": each
    worker returns its piece's weighted values with the terms needed to
    normalise them).
Works with the ``nccl`` backend (CUDA tensors) and the ``gloo`` backend (CPU
tensors).
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


def context_slices(seq_len, world, page_size=16):
    """Token ranges [t0, t1) of one sequence of ``seq_len`` tokens for ``world``
    ranks: contiguous runs of whole pages, as even as pages allow (a rank may get
    none when the sequence has fewer pages than ranks)."""
    if world < 1 or page_size < 1 or seq_len < 0:
        raise ValueError("world and page_size must be >= 1, seq_len >= 0")
    npages = -(-int(seq_len) // page_size)
    bounds = [r * npages // world for r in range(world + 1)]
    return [(min(b0 * page_size, seq_len), min(b1 * page_size, seq_len)) for b0, b1 in zip(bounds, bounds[1:])]


def gather_partials(o, lse, world):
    """All-gather of every rank's partial decode result: o [B, Hq, D] and lse
    [B, Hq] (any float dtype, the same on every rank) -> (o_all [world, B, Hq, D],
    lse_all [world, B, Hq]), rank r's partial at index r.  The one exchange of the
    context-parallel decode; the identity at world 1."""
    import torch

    if world == 1:
        return o.unsqueeze(0), lse.unsqueeze(0)
    import torch.distributed as dist

    o_all = [torch.empty_like(o) for _ in range(world)]
    l_all = [torch.empty_like(lse) for _ in range(world)]
    dist.all_gather(o_all, o.contiguous())
    dist.all_gather(l_all, lse.contiguous())
    return torch.stack(o_all), torch.stack(l_all)


def merged_offsets(batch, world):
    """Split offsets [B + 1] of gathered partials laid out sequence-major
    ([B, world, Hq, D], see split_major): sequence b's world splits are rows
    b * world .. b * world + world - 1."""
    return np.arange(batch + 1, dtype=np.int32) * int(world)


def split_major(o_all, lse_all):
    """[world, B, ...] gathered partials -> the split-merge layout [B * world, ...]
    (sequence-major: the splits of one sequence are consecutive rows)."""
    w, b = o_all.shape[0], o_all.shape[1]
    return (o_all.transpose(0, 1).reshape(b * w, *o_all.shape[2:]).contiguous(),
            lse_all.transpose(0, 1).reshape(b * w, *lse_all.shape[2:]).contiguous())


def context_parallel_decode(cache, plan, q, block_tables, seq_lens, out, sm_scale, world, lse_out=None,
                            stream=None):
    """One rank's part of a context-parallel decode (CUDA tensors, ``nccl``).

    ``cache`` holds this rank's slice of every sequence (context_slices), and
    ``block_tables`` / ``seq_lens`` / ``plan`` describe that slice (its own pages,
    its own token count; a rank whose slice is empty passes 0).  The rank decodes
    its slice with the log-sum-exp kept (fp32), the ranks all-gather the (o, lse)
    partials, and every rank merges them into ``out`` [B, Hq, D] with
    kvq_split_merge (a slice with no tokens has lse = -inf and weight 0)."""
    import torch

    from . import _binding as B
    from .cache import decode

    nb, hq, d = q.shape
    o = torch.empty((nb, hq, d), dtype=torch.float32, device=q.device)
    lse = torch.empty((nb, hq), dtype=torch.float32, device=q.device)
    decode(cache, plan, q, block_tables, seq_lens, o, sm_scale, lse_out=lse, stream=stream)
    o_all, l_all = gather_partials(o, lse, world)
    o_s, l_s = split_major(o_all, l_all)
    offs = torch.from_numpy(merged_offsets(nb, world)).to(q.device)
    B.kvq_split_merge(o_s.data_ptr(), l_s.data_ptr(), offs, nb, hq, d, out, lse_out, stream=stream)
    return out


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
