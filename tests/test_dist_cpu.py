"""The multi-rank host logic on the CPU: sequence sharding, and barrier +
max-over-ranks with two ``gloo`` ranks (127.0.0.1)."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

from quantized_paged_kv_gb300 import workloads as W
from quantized_paged_kv_gb300.dist import RankGroup, problem_seed, shard_sequences


def test_shard_sequences_is_a_balanced_partition():
    wl = W.make("serving_int8")
    for world in (1, 2, 3, 8):
        parts = shard_sequences(wl.seq_lens, world)
        assert len(parts) == world
        allidx = np.sort(np.concatenate(parts))
        assert np.array_equal(allidx, np.arange(wl.B))
        loads = [int(wl.seq_lens[p].sum()) for p in parts]
        # longest-first greedy: no rank exceeds the mean by more than the longest sequence
        assert max(loads) - sum(loads) / world <= int(wl.seq_lens.max())
    # equal problems go one per rank
    assert [p.tolist() for p in shard_sequences([32768] * 4, 4)] == [[0], [1], [2], [3]]
    assert [p.tolist() for p in shard_sequences([5, 0], 3)] == [[0], [1], []]
    with pytest.raises(ValueError):
        shard_sequences([1], 0)


def test_problem_seed_keeps_problem_zero():
    assert problem_seed(1, 0) == 1
    assert len({problem_seed(1, i) for i in range(16)}) == 16


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, seq_lens, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank))
    g = RankGroup.from_env("gloo")
    try:
        mine = shard_sequences(seq_lens, world)[rank]
        g.barrier()
        t = 1.0 + rank  # a per-rank "time"
        results[rank] = (mine.tolist(), g.allmax(t), g.allmax(-t))
        g.barrier()
    finally:
        g.close()


def test_two_gloo_ranks_shard_and_take_the_max():
    ctx = mp.get_context("spawn")
    port = _free_port()
    seq_lens = [300, 17, 1000, 64, 0, 2500, 1]
    with ctx.Manager() as m:
        results = m.dict()
        procs = [ctx.Process(target=_rank_main, args=(r, 2, port, seq_lens, results)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(results)
    assert sorted(res) == [0, 1]
    owned = sorted(res[0][0] + res[1][0])
    assert owned == list(range(len(seq_lens)))
    assert not set(res[0][0]) & set(res[1][0])
    for r in (0, 1):
        assert res[r][1] == 2.0 and res[r][2] == -1.0
