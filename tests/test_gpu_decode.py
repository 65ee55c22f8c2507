"""paged_decode_attention + split_merge on the GPU against the float64 oracle.

The oracle attends over pools it built itself from the same seeded bf16 inputs
(codes equal the GPU's bit for bit, see test_gpu_append.py): the comparison
isolates the kernel's arithmetic and layout handling from quantization error.
Tolerance: max-abs 2e-3 (fp32 output) / 1e-2 (bf16 output).
"""
import math

import numpy as np
import pytest
import torch

from quantized_paged_kv_gb300 import workloads as W
from tests import harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    H.ensure_built()


def _check(wl, fmt, split=0, out_dtype=None, units=None, target_ctas=0, gs=None):
    od = out_dtype or wl.out_dtype
    gs = H.global_scales(wl, fmt) if gs is None else gs
    seqs = None if units is None else sorted({b for b, _ in units})
    cache = H.gpu_cache(wl, fmt, gs)  # every sequence, as the benchmark runs it
    out, lse, plan = H.run_decode(cache, wl, split=split, out_dtype=od, target_ctas=target_ctas)
    pools = H.oracle_pools(wl, fmt, gs, seqs=seqs)
    ref, ref_lse = H.oracle_decode(wl, fmt, pools, units=units)
    sel = np.isfinite(ref_lse) | (wl.seq_lens[:, None] == 0)
    if units is not None:
        mask = np.zeros_like(sel)
        for b, h in units:
            mask[b, h * wl.G:(h + 1) * wl.G] = True
        sel &= mask
    err = np.abs(out - ref)[sel]
    assert np.all(np.isfinite(out[sel]))
    assert np.all(err <= H.bound(od, ref[sel])), (fmt, split, od, err.max())
    fin = sel & np.isfinite(ref_lse)
    le = np.abs(lse[fin] - ref_lse[fin])
    assert le.size == 0 or le.max() < 1e-3, le.max()
    assert np.all(np.isneginf(lse[sel & ~np.isfinite(ref_lse)]))
    return plan, err.max()


@pytest.mark.parametrize("split", [1, 4, 0])
def test_tiny_int8(split):
    wl = W.make("tiny_int8")
    plan, _ = _check(wl, "int8", split)
    if split:
        assert plan.total_splits == split


@pytest.mark.parametrize("fmt", ["int8", "int8_g32", "nvfp4", "bf16"])
@pytest.mark.parametrize("D,Hq,Hkv", [(256, 24, 4), (128, 32, 8), (256, 8, 8), (128, 16, 2)])
@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
def test_ragged_batch(fmt, D, Hq, Hkv, out_dtype):
    wl = W.make("serving_int8", lens=("list", [1, 17, 300, 0, 64, 1000]), seed=7)
    wl.Hq, wl.Hkv, wl.D = Hq, Hkv, D
    if out_dtype == "f32":  # large values; the bf16-output cases keep N(0, 0.5^2) as the bf16 workloads do
        wl.outlier_channels, wl.outlier_gain = 4, 8.0
    for split in (1, 3, 0):
        _check(wl, fmt, split, out_dtype=out_dtype)


def test_bf16_output_with_large_values():
    wl = W.make("tiny_int8", lens=("list", [1, 40, 700]), seed=8)
    _check(wl, "int8", 2, out_dtype="bf16")


def test_group_sizes_1_to_8():
    for G in (1, 2, 3, 5, 7, 8):
        wl = W.make("tiny_int8", lens=("list", [203, 45]), seed=11)
        wl.Hkv = 2
        wl.Hq = 2 * G
        _check(wl, "int8", 2)


def test_empty_context_gives_zero_and_neg_inf():
    wl = W.make("tiny_int8", lens=("list", [0, 33]), seed=3)
    cache = H.gpu_cache(wl, "int8")
    for split in (1, 5):
        out, lse, _ = H.run_decode(cache, wl, split=split)
        assert np.all(out[0] == 0.0) and np.all(np.isneginf(lse[0]))


def test_single_token_returns_its_value_row():
    wl = W.make("tiny_int8", lens=("list", [1]), seed=4)
    pools = H.oracle_pools(wl, "int8")
    cache = H.gpu_cache(wl, "int8")
    out, _, _ = H.run_decode(cache, wl, split=1)
    from oracle import attention as oatt
    for h in range(wl.Hkv):
        v = oatt.cache_rows("int8", pools["v_codes"], pools["v_scales"], wl.slots(0), h)[0]
        assert np.max(np.abs(out[0, h * wl.G:(h + 1) * wl.G] - v[None, :])) < 1e-5


def test_block_table_permutation_is_bit_identical():
    wl = W.make("tiny_int8", lens=("list", [700, 77]), seed=5)
    a = H.run_decode(H.gpu_cache(wl, "int8"), wl, split=3)[0]
    wl2 = W.make("tiny_int8", lens=("list", [700, 77]), seed=5)
    perm = np.random.default_rng(1).permutation(wl2.num_pages).astype(np.int32)
    wl2.block_tables = perm[wl2.block_tables]
    b = H.run_decode(H.gpu_cache(wl2, "int8"), wl2, split=3)[0]
    assert np.array_equal(a, b)


def test_skip_merge_then_split_merge_matches():
    from quantized_paged_kv_gb300 import DecodePlan, decode, kvq_split_merge

    wl = W.make("tiny_int8", lens=("list", [900, 333, 16]), seed=9)
    cache = H.gpu_cache(wl, "int8")
    full, lse_full, _ = H.run_decode(cache, wl, split=4)
    q = torch.from_numpy(wl.q()).to(torch.bfloat16).cuda()
    out = torch.full((wl.B, wl.Hq, wl.D), float("nan"), device="cuda")
    lse = torch.full((wl.B, wl.Hq), float("nan"), device="cuda")
    plan = DecodePlan(cache, wl.seq_lens, wl.Hq, split_override=4)
    bt = torch.from_numpy(wl.block_tables).cuda()
    sl = torch.from_numpy(wl.seq_lens).cuda()
    decode(cache, plan, q, bt, sl, out, wl.sm_scale, lse_out=lse, skip_merge=True)
    o_ptr, l_ptr = plan.partials()
    kvq_split_merge(o_ptr, l_ptr, plan.plan, wl.B, wl.Hq, wl.D, out, lse)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), full)
    assert np.array_equal(lse.cpu().numpy(), lse_full)


def test_checked_mode_reports_bad_metadata():
    from quantized_paged_kv_gb300 import DecodePlan, KvqError, decode, kvq_read_status

    wl = W.make("tiny_int8", lens=("list", [64, 64]), seed=2)
    cache = H.gpu_cache(wl, "int8")
    q = torch.from_numpy(wl.q()).to(torch.bfloat16).cuda()
    out = torch.empty((wl.B, wl.Hq, wl.D), device="cuda")
    plan = DecodePlan(cache, wl.seq_lens, wl.Hq, split_override=2)
    sl = torch.from_numpy(wl.seq_lens).cuda()
    bt = torch.from_numpy(wl.block_tables).cuda()
    bad = bt.clone()
    bad[1, 2] = wl.num_pages + 5          # page id out of range: skipped, flagged
    with pytest.raises(KvqError) as e:
        decode(cache, plan, q, bad, sl, out, wl.sm_scale, checked=True)
    assert e.value.code == 5
    bad_len = sl.clone()
    bad_len[0] = 10**6                    # longer than the block table: the plan no longer matches
    with pytest.raises(KvqError) as e:
        decode(cache, plan, q, bt, bad_len, out, wl.sm_scale, checked=True)
    assert e.value.code == 1
    # raw mode: the kernel clamps the length to the block table and flags it
    decode(cache, plan, q, bt, bad_len, out, wl.sm_scale, checked=False)
    rc, bits = kvq_read_status(plan.workspace)
    assert rc == 5 and bits & 2  # KVQ_DEV_BAD_SEQLEN
    good_plan = plan.plan
    bad_plan = good_plan.clone()
    bad_plan[wl.B + 1] = 99               # CTA count differs from num_ctas
    plan.plan = bad_plan
    with pytest.raises(KvqError) as e:
        decode(cache, plan, q, bt, sl, out, wl.sm_scale, checked=True)
    assert e.value.code == 1
    bad_plan = good_plan.clone()
    A = (wl.B + 2 + 3) // 4 * 4
    bad_plan[A + 1] = plan.total_splits + 3  # first item of CTA 0 names a split that does not exist
    plan.plan = bad_plan
    with pytest.raises(KvqError) as e:
        decode(cache, plan, q, bt, sl, out, wl.sm_scale, checked=True)
    assert e.value.code == 1
    # after the errors the context is still usable and a good call is exact
    good = DecodePlan(cache, wl.seq_lens, wl.Hq, split_override=2)
    decode(cache, good, q, bt, sl, out, wl.sm_scale, checked=True)


@pytest.mark.parametrize("fmt", ["int8", "int8_g32", "nvfp4", "bf16"])
def test_raw_mode_bad_page_ids_contribute_nothing(fmt):
    """Raw mode: a block-table entry outside the pool is skipped and flagged, and
    its page's tokens are left out of the softmax (whatever the stage held before:
    the pool is sentinel-filled, so stale bytes would show as NaN or garbage).
    The result equals the oracle's attention over the sequence without those
    tokens; a sequence whose every page is bad gives 0 and -inf."""
    from oracle import attention as oatt
    from oracle import layout as olay
    from quantized_paged_kv_gb300 import DecodePlan, decode, kvq_read_status

    wl = W.make("tiny_int8", lens=("list", [700, 64, 20]), seed=14)
    gs = H.global_scales(wl, fmt)
    cache = H.gpu_cache(wl, fmt, gs)
    q = wl.q()
    bad = wl.block_tables.copy()
    drop = {0: [0, 5, 43], 1: [0, 1, 2, 3], 2: []}  # pages made bad (sequence 1: all of them)
    for b, js in drop.items():
        for j in js:
            bad[b, j] = wl.num_pages + 7 + j
    for split in (1, 3):
        plan = DecodePlan(cache, wl.seq_lens, wl.Hq, split_override=split)
        out = torch.full((wl.B, wl.Hq, wl.D), float("nan"), device="cuda")
        lse = torch.full((wl.B, wl.Hq), float("nan"), device="cuda")
        decode(cache, plan, torch.from_numpy(q).to(torch.bfloat16).cuda(), torch.from_numpy(bad).cuda(),
               torch.from_numpy(wl.seq_lens).cuda(), out, wl.sm_scale, lse_out=lse)
        rc, bits = kvq_read_status(plan.workspace)
        assert rc == 5 and bits == 1  # KVQ_DEV_BAD_PAGE only
        o, l = out.cpu().numpy(), lse.cpu().numpy()
        pools = H.oracle_pools(wl, fmt, gs)
        for b in range(wl.B):
            L = int(wl.seq_lens[b])
            keep = np.array([t for t in range(L) if t // 16 not in drop[b]], dtype=np.int64)
            slots = olay.token_slots(wl.block_tables[b], L, 16)[keep]
            for h in range(wl.Hkv):
                k = oatt.cache_rows(fmt, pools["k_codes"], pools.get("k_scales"), slots, h, gs[0])
                v = oatt.cache_rows(fmt, pools["v_codes"], pools.get("v_scales"), slots, h, gs[1])
                ro, rl = oatt.attend(q[b, h * wl.G:(h + 1) * wl.G], k, v, wl.sm_scale)
                rows = slice(h * wl.G, (h + 1) * wl.G)
                assert np.all(np.abs(o[b, rows] - ro) <= H.bound("f32", ro)), (fmt, split, b, h)
                if len(keep) == 0:
                    assert np.all(o[b, rows] == 0) and np.all(np.isneginf(l[b, rows]))
                else:
                    assert np.abs(l[b, rows] - rl).max() < 1e-3


def test_nan_sentinels_in_unwritten_tail_slots_do_not_leak():
    for fmt in ("int8", "int8_g32", "nvfp4", "bf16"):
        wl = W.make("tiny_int8", lens=("list", [33, 5, 47]), seed=6)
        _check(wl, fmt, 2)


# ---------------------------------------------------------------- full-size workloads
# (launch configuration of bench.py: automatic split plan, sampled (b, h) units)
def test_long_int8_full_size_sampled():
    wl = W.make("long_int8")
    for split in (0, 16, 64):
        _check(wl, "int8", split, units=[(0, 0), (0, 3)])


def test_long_int8_bf16_cache_full_size_sampled():
    wl = W.make("long_int8")
    _check(wl, "bf16", 0, units=[(0, 1)])


def test_serving_int8_full_size_sampled():
    wl = W.make("serving_int8")
    order = np.argsort(wl.seq_lens)
    units = [(int(order[0]), 0), (int(order[-1]), 7), (int(order[len(order) // 2]), 3)]
    _check(wl, "int8", 0, units=units)


def test_append_workload_decode_full_size_sampled():
    # the B = 8 decode over contexts of 4K..16K with 1% spikes x 20 (bf16 output)
    wl = W.make("append_int8")
    order = np.argsort(wl.seq_lens)
    _check(wl, "int8", 0, units=[(int(order[0]), 0), (int(order[-1]), 3)])


def test_long_int8_g32_full_size_sampled():
    wl = W.make("long_int8")
    _check(wl, "int8_g32", 0, units=[(0, 2)])


def test_serving_int8_g32_full_size_sampled():
    wl = W.make("serving_int8")
    order = np.argsort(wl.seq_lens)
    _check(wl, "int8_g32", 0, units=[(int(order[-1]), 5)])


def test_per_32_scales_bring_int8_closer_to_exact_attention():
    # outlier channels x8: one scale per 32 values keeps the groups without an
    # outlier fine-grained, so the output is closer (RMS over all elements) to
    # attention over the bf16 K/V.  The largest error stays in the outlier
    # channels, whose group scale equals the row scale.
    wl = W.make("tiny_int8", lens=("list", [700]), seed=23)
    exact, _ = H.oracle_decode(wl, "bf16", H.oracle_pools(wl, "bf16"))
    errs = {}
    for fmt in ("int8", "int8_g32"):
        out, _, _ = H.run_decode(H.gpu_cache(wl, fmt), wl, out_dtype="f32")
        errs[fmt] = np.sqrt(((out - exact) ** 2).mean())
    assert errs["int8_g32"] < 0.7 * errs["int8"], errs


def test_long_nvfp4_full_size_sampled():
    wl = W.make("long_nvfp4")
    order = np.argsort(wl.seq_lens)
    units = [(int(order[0]), 1), (int(order[-1]), 2)]
    _check(wl, "nvfp4", 0, units=units)


def test_serving_nvfp4_full_size_sampled():
    # the batch-64 serving mix (D = 128, G = 4) in NVFP4 with the tensor global
    # scales 448 * 6 / amax, bf16 output, the bench's automatic plan
    wl = W.make("serving_int8")
    order = np.argsort(wl.seq_lens)
    units = [(int(order[0]), 0), (int(order[-1]), 7), (int(order[len(order) // 2]), 4)]
    _check(wl, "nvfp4", 0, units=units)


def test_long_context_nvfp4_full_size_sampled():
    # the 32K batch-1 workload in NVFP4 (D = 256, G = 6) with tensor global scales, fp32 output
    wl = W.make("long_int8")
    _check(wl, "nvfp4", 0, units=[(0, 0), (0, 3)])


def test_nvfp4_d128_gqa_shapes_and_splits():
    # D = 128 with 1, 3, 5 and 8 query heads a KV head; page-crossing lengths
    for G in (1, 3, 5, 8):
        wl = W.make("serving_int8", lens=("list", [1, 15, 16, 17, 333, 2049]), seed=60 + G)
        wl.Hkv, wl.Hq = 2, 2 * G
        for split in (1, 4, 0):
            _check(wl, "nvfp4", split, out_dtype="f32")


def test_early_start_chain_in_a_graph_matches_plain_calls():
    """Calls launched as programmatic dependents of each other (early start): a
    CUDA graph of back-to-back calls on alternating queries and output buffers
    gives exactly the plain calls' results."""
    from quantized_paged_kv_gb300 import DecodePlan, decode

    wl = W.make("tiny_int8", lens=("list", [700, 33, 4096]), seed=13)
    cache = H.gpu_cache(wl, "int8")
    plan = DecodePlan(cache, wl.seq_lens, wl.Hq, split_override=5)
    bt = torch.from_numpy(wl.block_tables).cuda()
    sl = torch.from_numpy(wl.seq_lens).cuda()
    qs = [torch.from_numpy(wl.q()).to(torch.bfloat16).cuda()]
    qs.append((qs[0].float() * -0.5 + 0.25).to(torch.bfloat16))
    refs = []
    for q in qs:
        o = torch.empty((wl.B, wl.Hq, wl.D), device="cuda")
        decode(cache, plan, q, bt, sl, o, wl.sm_scale)
        refs.append(o)
    outs = [torch.full((wl.B, wl.Hq, wl.D), float("nan"), device="cuda") for _ in range(4)]
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):  # warm-up outside capture
        for i in range(4):
            decode(cache, plan, qs[i % 2], bt, sl, outs[i], wl.sm_scale, early_start=True)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(4):
            decode(cache, plan, qs[i % 2], bt, sl, outs[i], wl.sm_scale, early_start=True)
    for o in outs:
        o.fill_(float("nan"))
    torch.cuda.synchronize()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    for i in range(4):
        assert torch.equal(outs[i], refs[i % 2]), i


@pytest.mark.parametrize("split", [1, 4])
def test_pinned_host_buffers_give_the_device_result(split):
    """q, block table, sequence lengths, out and lse_out in pinned host memory
    (read and written by the kernels over the host link) give exactly the result
    of device buffers, for direct (one split) and merged outputs."""
    from quantized_paged_kv_gb300 import DecodePlan, decode

    wl = W.make("tiny_int8", lens=("list", [700, 33, 4096]), seed=17)
    cache = H.gpu_cache(wl, "int8")
    plan = DecodePlan(cache, wl.seq_lens, wl.Hq, split_override=split)
    q = torch.from_numpy(wl.q()).to(torch.bfloat16)
    bt = torch.from_numpy(wl.block_tables)
    sl = torch.from_numpy(wl.seq_lens)
    for od in (torch.float32, torch.bfloat16):
        o_d = torch.empty((wl.B, wl.Hq, wl.D), dtype=od, device="cuda")
        l_d = torch.empty((wl.B, wl.Hq), device="cuda")
        decode(cache, plan, q.cuda(), bt.cuda(), sl.cuda(), o_d, wl.sm_scale, lse_out=l_d, checked=True)
        o_h = torch.full((wl.B, wl.Hq, wl.D), float("nan"), dtype=od).pin_memory()
        l_h = torch.full((wl.B, wl.Hq), float("nan")).pin_memory()
        decode(cache, plan, q.pin_memory(), bt.pin_memory(), sl.pin_memory(), o_h, wl.sm_scale, lse_out=l_h,
               checked=True)
        torch.cuda.synchronize()
        assert torch.equal(o_h, o_d.cpu())
        assert torch.equal(l_h, l_d.cpu())


def test_pageable_host_output_is_refused():
    from quantized_paged_kv_gb300 import DecodePlan, KvqError, decode

    wl = W.make("tiny_int8", lens=("list", [64]), seed=18)
    cache = H.gpu_cache(wl, "int8")
    plan = DecodePlan(cache, wl.seq_lens, wl.Hq)
    q = torch.from_numpy(wl.q()).to(torch.bfloat16).cuda()
    out = torch.empty((wl.B, wl.Hq, wl.D))  # pageable
    from quantized_paged_kv_gb300 import _binding as Bd
    with pytest.raises(KvqError) as e:
        Bd.lib()  # loaded
        import ctypes
        rc = Bd.lib().kvq_paged_decode_attention(
            ctypes.byref(cache.struct), Bd._ptr(q), wl.B, wl.Hq, float(wl.sm_scale),
            Bd._ptr(torch.from_numpy(wl.block_tables).cuda()), wl.block_tables.shape[1],
            Bd._ptr(torch.from_numpy(wl.seq_lens).cuda()), Bd._ptr(plan.plan), plan.total_splits, plan.num_ctas,
            Bd._ptr(plan.workspace), plan.workspace.numel(), Bd._ptr(out), Bd.KVQ_OUT_F32, None, 0, None)
        Bd._check(rc, "kvq_paged_decode_attention")
    assert e.value.code == 1 and "pageable" in str(e.value)


def test_stalled_pipeline_times_out_and_the_context_survives():
    """Failure path without a fault: with KVQ_TEST_STALL the producers issue no
    page copies, every bounded wait gives up after 2 ms, and checked mode reports
    KVQ_ERR_DEVICE_TIMEOUT; the next call on the same plan and workspace (the
    status word was read and cleared) gives the oracle's result."""
    from quantized_paged_kv_gb300 import DecodePlan, KvqError, decode
    from quantized_paged_kv_gb300 import _binding as B

    wl = W.make("tiny_int8")
    cache = H.gpu_cache(wl, "int8")
    qt = torch.from_numpy(wl.q()).to(torch.bfloat16).cuda()
    bt = torch.from_numpy(wl.block_tables).cuda()
    sl = torch.from_numpy(wl.seq_lens).cuda()
    out = torch.full((wl.B, wl.Hq, wl.D), float("nan"), dtype=torch.float32, device="cuda")
    plan = DecodePlan(cache, wl.seq_lens, wl.Hq, split_override=4)
    with pytest.raises(KvqError) as e:
        B.kvq_paged_decode_attention(cache.struct, qt, wl.sm_scale, bt, sl, plan.plan, plan.total_splits,
                                     plan.num_ctas, plan.workspace, out, None, B.KVQ_CHECKED | B.KVQ_TEST_STALL)
    assert e.value.code == 6 and "timed out" in str(e.value)
    decode(cache, plan, qt, bt, sl, out, wl.sm_scale, checked=True)
    torch.cuda.synchronize()
    ref, _ = H.oracle_decode(wl, "int8", H.oracle_pools(wl, "int8"))
    assert np.abs(out.cpu().numpy() - ref).max() <= H.tol("f32")

