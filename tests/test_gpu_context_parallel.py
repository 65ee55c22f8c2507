"""The context-parallel data path of one long sequence on one GPU: every "rank"
holds a contiguous run of the sequence's pages in a pool of its own and decodes
it with its log-sum-exp kept; the partials are stacked as the all-gather would
lay them out and merged by kvq_split_merge.  The result is compared with the
float64 oracle's decode of the whole sequence (max-abs 2e-3, fp32 output).
The ranks' decodes are independent launches that never wait on one another."""
import numpy as np
import pytest
import torch

from quantized_paged_kv_gb300 import workloads as W
from tests import harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    H.ensure_built()


def _rank_decode(wl, fmt, gs, t0, t1):
    """(o [1, Hq, D] fp32, lse [1, Hq]) of tokens t0..t1-1 of sequence 0, from a
    pool that holds that slice's pages only."""
    from quantized_paged_kv_gb300 import DecodePlan, KVCache, decode

    n = t1 - t0
    npages = max(1, -(-n // 16))
    cache = KVCache(fmt, npages, wl.Hkv, wl.D, k_global_scale=gs[0], v_global_scale=gs[1], fill=H.SENTINEL)
    if n > 0:
        k, v = wl.kv(0)
        slots = torch.arange(n, dtype=torch.int64, device="cuda")  # the slice's own pages, in order
        cache.append(torch.from_numpy(k[t0:t1]).to(torch.bfloat16).cuda(), torch.from_numpy(v[t0:t1]).to(torch.bfloat16).cuda(),
                     slots)
    bt = torch.arange(npages, dtype=torch.int32, device="cuda")[None]
    sl = torch.tensor([n], dtype=torch.int32, device="cuda")
    plan = DecodePlan(cache, np.array([n], np.int32), wl.Hq)
    q = torch.from_numpy(wl.q()).to(torch.bfloat16).cuda()
    o = torch.full((1, wl.Hq, wl.D), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((1, wl.Hq), float("nan"), dtype=torch.float32, device="cuda")
    decode(cache, plan, q, bt, sl, o, wl.sm_scale, lse_out=lse, checked=True)
    return o, lse


@pytest.mark.parametrize("fmt", ["int8", "nvfp4"])
@pytest.mark.parametrize("world", [2, 3, 5])
def test_slices_merged_equal_the_whole_sequence(fmt, world):
    from quantized_paged_kv_gb300 import kvq_split_merge
    from quantized_paged_kv_gb300.dist import context_slices, merged_offsets, split_major

    L = 3000  # 188 pages: uneven slices and a ragged last page
    wl = W.make("tiny_int8", lens=("list", [L]))
    gs = H.global_scales(wl, fmt)
    parts = [_rank_decode(wl, fmt, gs, t0, t1) for t0, t1 in context_slices(L, world)]
    o_all = torch.stack([p[0] for p in parts])
    l_all = torch.stack([p[1] for p in parts])
    o_s, l_s = split_major(o_all, l_all)
    offs = torch.from_numpy(merged_offsets(1, world)).cuda()
    out = torch.full((1, wl.Hq, wl.D), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((1, wl.Hq), float("nan"), dtype=torch.float32, device="cuda")
    kvq_split_merge(o_s.data_ptr(), l_s.data_ptr(), offs, 1, wl.Hq, wl.D, out, lse)
    torch.cuda.synchronize()
    ref, ref_lse = H.oracle_decode(wl, fmt, H.oracle_pools(wl, fmt, gs))
    assert np.abs(out.cpu().numpy() - ref).max() <= 2e-3
    assert np.abs(lse.cpu().numpy() - ref_lse).max() < 1e-3


def test_more_ranks_than_pages_leave_empty_slices():
    """A 40-token sequence (3 pages) over 5 ranks: two ranks decode nothing
    (lse = -inf, weight 0 in the merge)."""
    from quantized_paged_kv_gb300 import kvq_split_merge
    from quantized_paged_kv_gb300.dist import context_slices, merged_offsets, split_major

    L, world = 40, 5
    wl = W.make("tiny_int8", lens=("list", [L]))
    sl = context_slices(L, world)
    assert sum(1 for t0, t1 in sl if t1 == t0) == 2
    parts = [_rank_decode(wl, "int8", (1.0, 1.0), t0, t1) for t0, t1 in sl]
    o_s, l_s = split_major(torch.stack([p[0] for p in parts]), torch.stack([p[1] for p in parts]))
    out = torch.empty((1, wl.Hq, wl.D), dtype=torch.float32, device="cuda")
    kvq_split_merge(o_s.data_ptr(), l_s.data_ptr(), torch.from_numpy(merged_offsets(1, world)).cuda(), 1, wl.Hq,
                    wl.D, out)
    torch.cuda.synchronize()
    ref, _ = H.oracle_decode(wl, "int8", H.oracle_pools(wl, "int8"))
    assert np.abs(out.cpu().numpy() - ref).max() <= 2e-3
