"""The multi-rank host logic on the CPU: sequence sharding, and barrier +
max-over-ranks with two ``gloo`` ranks (127.0.0.1); the context-parallel split
of one long sequence (contiguous page runs, one all-gather of the (o, lse)
partials, the split merge) with two ``gloo`` ranks whose slices the oracle
decodes."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

from quantized_paged_kv_gb300 import workloads as W
from oracle import attention as oatt
from oracle import layout as olay
from quantized_paged_kv_gb300.dist import (RankGroup, context_slices, gather_partials, merged_offsets, problem_seed,
                                           shard_sequences, split_major)


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


def test_context_slices_are_contiguous_whole_pages():
    for L in (0, 1, 15, 16, 17, 700, 32768, 32767):
        for world in (1, 2, 3, 4, 8):
            sl = context_slices(L, world)
            assert len(sl) == world
            assert sl[0][0] == 0 and sl[-1][1] == L
            for (a0, a1), (b0, b1) in zip(sl, sl[1:]):
                assert a1 == b0  # contiguous, in order
            for t0, t1 in sl:
                assert t0 <= t1 and t0 % 16 == 0  # every slice starts on a page boundary
            pages = [-(-(t1 - t0) // 16) for t0, t1 in sl]
            assert max(pages) - min(pages) <= 1  # as even as whole pages allow
    assert context_slices(40, 2) == [(0, 16), (16, 40)]  # 3 pages: 1 and 2
    with pytest.raises(ValueError):
        context_slices(10, 0)


def test_split_major_layout_matches_the_merged_offsets():
    import torch

    world, nb, hq, d = 3, 2, 4, 8
    o_all = torch.arange(world * nb * hq * d, dtype=torch.float64).reshape(world, nb, hq, d)
    l_all = torch.arange(world * nb * hq, dtype=torch.float64).reshape(world, nb, hq)
    o_s, l_s = split_major(o_all, l_all)
    offs = merged_offsets(nb, world)
    assert offs.tolist() == [0, 3, 6]
    for b in range(nb):
        for r in range(world):
            assert torch.equal(o_s[offs[b] + r], o_all[r, b]) and torch.equal(l_s[offs[b] + r], l_all[r, b])


def _slice_pools(wl, t0, t1):
    """The oracle's INT8 pool of tokens t0..t1-1 of sequence 0 (this rank's pages
    only, in the workload's own block-table order) and its local block table."""
    k, v = wl.kv(0)
    n = t1 - t0
    npages = -(-n // 16)
    pages = wl.block_tables[0, t0 // 16:t0 // 16 + npages]
    local = {int(p): i for i, p in enumerate(pages)}  # the rank's pool holds its pages only
    slots = np.array([local[int(wl.block_tables[0, t // 16])] * 16 + t % 16 for t in range(t0, t1)], np.int64)
    pools = {"k_codes": np.zeros((max(npages, 1), wl.Hkv, 16, wl.D), np.uint8),
             "v_codes": np.zeros((max(npages, 1), wl.Hkv, 16, wl.D), np.uint8),
             "k_scales": np.zeros((max(npages, 1), wl.Hkv, 16), np.float32),
             "v_scales": np.zeros((max(npages, 1), wl.Hkv, 16), np.float32)}
    for name, x in (("k", k), ("v", v)):
        for h in range(wl.Hkv):
            c, sc = oatt.quantize_rows("int8", x[t0:t1, h, :])
            olay.scatter_rows(pools[name + "_codes"], slots, h, c)
            olay.scatter_rows(pools[name + "_scales"], slots, h, sc)
    bt = np.arange(max(npages, 1), dtype=np.int32)[None]
    return pools, bt


def _cp_rank_main(rank, world, port, L, results):
    import torch

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank))
    g = RankGroup.from_env("gloo")
    try:
        wl = W.make("tiny_int8", lens=("list", [L]))
        t0, t1 = context_slices(L, world)[rank]
        pools, bt = _slice_pools(wl, t0, t1)
        o, lse = oatt.paged_decode("int8", pools, wl.q(), bt, np.array([t1 - t0]), wl.sm_scale)
        o_all, l_all = gather_partials(torch.from_numpy(o), torch.from_numpy(lse), world)
        o_s, l_s = split_major(o_all, l_all)
        offs = merged_offsets(1, world)
        merged, mlse = oatt.merge(o_s[offs[0]:offs[1]].numpy(), l_s[offs[0]:offs[1]].numpy())
        results[rank] = (merged, mlse, o_all.shape[0])
    finally:
        g.close()


def test_two_gloo_ranks_context_parallel_decode_equals_the_unsplit_oracle():
    """Each rank decodes its contiguous page run of one 700-token sequence (the
    oracle over that rank's own pool), the two (o, lse) partials are all-gathered
    over gloo, and the merge of the gathered partials equals the oracle's decode
    of the whole sequence on every rank."""
    L, world = 700, 2
    ctx = mp.get_context("spawn")
    port = _free_port()
    with ctx.Manager() as m:
        results = m.dict()
        procs = [ctx.Process(target=_cp_rank_main, args=(r, world, port, L, results)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(300)
            assert p.exitcode == 0
        res = dict(results)
    wl = W.make("tiny_int8", lens=("list", [L]))
    full, _ = _slice_pools(wl, 0, L)
    ref, ref_lse = oatt.paged_decode("int8", full, wl.q(), np.arange(full["k_codes"].shape[0], dtype=np.int32)[None],
                                     np.array([L]), wl.sm_scale)
    for r in range(world):
        merged, mlse, n = res[r]
        assert n == world
        assert np.abs(merged - ref[0]).max() < 1e-12
        assert np.abs(mlse - ref_lse[0]).max() < 1e-12
