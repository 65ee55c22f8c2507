"""The C-ABI library on a machine without a GPU: it loads, exports every symbol
include/kvq.h declares, and its host-only helpers (byte accounting, split
planning, workspace layout, argument validation) behave as documented."""
import ctypes
import os
import re

import numpy as np
import pytest

from tests import harness as H
from oracle import accounting as acc
from tests import oracle_pins as pins

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def kvq():
    H.ensure_built()
    import quantized_paged_kv_gb300 as k
    return k


def header_symbols():
    text = open(os.path.join(ROOT, "include", "kvq.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvq_[a-z_]+)\s*\(", text)))


def test_library_exports_every_header_symbol(kvq):
    syms = header_symbols()
    assert len(syms) >= 10
    lib = ctypes.CDLL(kvq._binding.LIB_PATH)
    for s in syms:
        assert hasattr(lib, s), s
    assert sorted(kvq._binding.EXPORTS) == syms


def header_constants():
    """Every KVQ_* enumerator of include/kvq.h with its value."""
    text = open(os.path.join(ROOT, "include", "kvq.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    out = {}
    for body in re.findall(r"enum\s*\w*\s*\{(.*?)\}", text, flags=re.S):
        for name, expr in re.findall(r"\b(KVQ_[A-Z0-9_]+)\s*=\s*([^,]+)", body):
            m = re.fullmatch(r"(\d+)u?(?:\s*<<\s*(\d+))?", expr.strip())  # N, Nu or Nu << K
            assert m, (name, expr)
            out[name] = int(m.group(1)) << int(m.group(2) or 0)
    return out


def test_binding_constants_match_the_header(kvq):
    consts = header_constants()
    assert len(consts) >= 20
    shared = [n for n in consts if hasattr(kvq._binding, n)]
    for n in shared:
        assert getattr(kvq._binding, n) == consts[n], n
    # the flags and format codes a caller passes must all be there
    for n in ("KVQ_CHECKED", "KVQ_SKIP_MERGE", "KVQ_EARLY_START", "KVQ_ROTATE", "KVQ_TEST_STALL", "KVQ_FMT_BF16",
              "KVQ_FMT_INT8", "KVQ_FMT_NVFP4", "KVQ_FMT_INT8_G32", "KVQ_OUT_F32", "KVQ_OUT_BF16"):
        assert n in shared, n
    flags = [consts[n] for n in ("KVQ_CHECKED", "KVQ_SKIP_MERGE", "KVQ_EARLY_START", "KVQ_ROTATE", "KVQ_TEST_STALL")]
    assert all(f & (f - 1) == 0 for f in flags) and len(set(flags)) == len(flags)  # distinct single bits


def test_bytes_per_token_matches_the_pages(kvq):
    cf = pins.closed_forms()
    assert kvq.kvq_bytes_per_token("int8", 1, 256) == cf["int8_bytes_per_token_head_D256"]
    assert kvq.kvq_bytes_per_token("bf16", 1, 256) == cf["bf16_bytes_per_token_head_D256"]
    assert kvq.kvq_bytes_per_token("nvfp4", 2, 256) == cf["nvfp4_bytes_per_token_layer_2H_D256"]
    assert kvq.kvq_bytes_per_token("nvfp4", 1, 256) == cf["nvfp4_bytes_per_kv_head_D256"]
    assert 16 * kvq.kvq_bytes_per_token("bf16", 4, 256) == cf["bf16_bytes_per_token_16L_4H_D256"]
    assert kvq.kvq_bytes_per_token("int8", 8, 128) == 8 * 2 * (128 + 4)
    assert kvq.kvq_bytes_per_token(7, 1, 256) == -1
    cb, sb = kvq.kvq_cache_array_bytes("nvfp4", 10, 16, 2, 256)
    assert (cb, sb) == (10 * 2 * 16 * 128, 10 * 2 * 16 * 16)
    cb, sb = kvq.kvq_cache_array_bytes("int8", 3, 16, 4, 256)
    assert (cb, sb) == (3 * 4 * 16 * 256, 3 * 4 * 16 * 4)
    # one fp32 scale per 32 values
    assert kvq.kvq_bytes_per_token("int8_g32", 1, 256) == 2 * acc.record_bytes("int8_g32", 256)
    assert kvq.kvq_bytes_per_token("int8_g32", 8, 128) == 8 * 2 * acc.record_bytes("int8_g32", 128)
    cb, sb = kvq.kvq_cache_array_bytes("int8_g32", 3, 16, 4, 256)
    assert (cb, sb) == (3 * 4 * 16 * 256, 3 * 4 * 16 * 8 * 4)


def _struct(kvq, fmt="int8", pages=4096, Hkv=4, D=256):
    return kvq._binding.KvqCacheStruct(None, None, None, None, pages, 16, Hkv, D, kvq._binding.FORMATS[fmt], 1.0, 1.0)


def _descriptors(plan, B, C, n_items):
    """(first-item descriptors [C, 4], CTA offsets [C+1], rest descriptors) of a plan."""
    A = (B + 2 + 3) // 4 * 4
    R = (A + 5 * C + 1 + 3) // 4 * 4
    firsts = plan[A:A + 4 * C].reshape(C, 4)
    ro = plan[A + 4 * C:A + 5 * C + 1]
    rest = plan[R:R + 4 * (n_items - C)].reshape(-1, 4)
    return firsts, ro, rest


def _check_plan(plan, seq_lens, total, nctas, nhg, override=None):
    B = len(seq_lens)
    offs = plan[:B + 1]
    assert offs[0] == 0 and offs[-1] == total
    C = plan[B + 1]
    assert C == nctas and 1 <= C <= total * nhg
    n_items = total * nhg
    firsts, ro, rest = _descriptors(plan, B, C, n_items)
    assert ro[0] == 0 and ro[-1] == n_items - C and all(ro[i] <= ro[i + 1] for i in range(C))
    expect = {}  # (split, group) -> (b, first page, n, direct)
    for b, L in enumerate(seq_lens):
        n = -(-L // 16)
        S = offs[b + 1] - offs[b]
        assert S >= 1
        if override:
            assert S == max(1, min(override, max(n, 1)))
        bounds = [(s * n // S, (s + 1) * n // S) for s in range(S)]
        assert bounds[0][0] == 0 and bounds[-1][1] == n
        assert all(bounds[i][1] == bounds[i + 1][0] for i in range(S - 1))
        assert max(e - b_ for b_, e in bounds) - min(e - b_ for b_, e in bounds) <= 1
        for s, (b0, e0) in enumerate(bounds):
            for g in range(nhg):
                expect[(int(offs[b]) + s, g)] = (b, b0, e0 - b0, int(S == 1))
    seen = set()
    loads = []
    for c in range(C):
        descs = [firsts[c]] + [rest[i] for i in range(ro[c], ro[c + 1])]
        sz = []
        for d in descs:
            b, split, pb, w = (int(x) for x in d)
            n, direct, g = w & 0x7FFFFF, (w >> 23) & 1, w >> 24
            key = (split, g)
            assert key in expect and key not in seen
            seen.add(key)
            assert expect[key] == (b, pb, n, direct)
            sz.append(n)
        # longest-first packing: within a CTA the items come in decreasing size
        assert sz == sorted(sz, reverse=True)
        loads.append(sum(x + 8 for x in sz))
    assert len(seen) == n_items
    # and no CTA carries more than the average load plus one item (LPT bound)
    biggest = max(v[2] for v in expect.values()) + 8
    assert max(loads) <= sum(loads) / C + biggest


def test_planner_override_and_auto(kvq):
    s = _struct(kvq)  # Hkv = 4, D = 256: the 4 heads form one group (nhg = 1)
    rng = np.random.default_rng(0)
    for seq_lens in ([32768], [512], [0], [1, 17, 300, 0, 64], rng.integers(512, 8193, 64).tolist()):
        for ov in (1, 2, 4, 64):
            plan, total, nctas = kvq.kvq_plan_splits(s, seq_lens, ov, 152)
            _check_plan(plan.numpy(), seq_lens, total, nctas, 1, ov)
        plan, total, nctas = kvq.kvq_plan_splits(s, seq_lens, 0, 152)
        _check_plan(plan.numpy(), seq_lens, total, nctas, 1)
    plan, total, nctas = kvq.kvq_plan_splits(s, [32768], 0, 152)
    # 2048 page units over 152 CTAs: 152 splits of 13 or 14 pages, one per CTA
    assert total == 152 and nctas == 152
    # the per-32 format plans with the same head groups (its stage holds 4 pages)
    g = _struct(kvq, fmt="int8_g32")
    for seq_lens in ([32768], [1, 17, 300, 0, 64]):
        plan, total, nctas = kvq.kvq_plan_splits(g, seq_lens, 0, 152)
        _check_plan(plan.numpy(), seq_lens, total, nctas, 1)
    # uneven lengths: a split granularity whose packing fills every CTA evenly
    # wins over one split per CTA's worth of pages (which leaves some CTAs two items)
    lens = [4096 * 16, 3000 * 16, 900 * 16, 333 * 16, 4100 * 16]
    plan, total, nctas = kvq.kvq_plan_splits(s, lens, 0, 152)
    _check_plan(plan.numpy(), lens, total, nctas, 1)
    sizes = []
    off = plan.numpy()[:len(lens) + 1]
    for b, L in enumerate(lens):
        n, S = -(-L // 16), off[b + 1] - off[b]
        sizes += [(s_ + 1) * n // S - s_ * n // S for s_ in range(S)]
    loads = sorted(sizes, reverse=True)
    bins = [0] * nctas
    for x in loads:
        bins[bins.index(min(bins))] += x + 8
    assert max(bins) <= 1.25 * (sum(loads) + 8 * len(loads)) / nctas
    s8 = _struct(kvq, pages=4096, Hkv=8, D=128)  # 12 consumer warps at D = 128 -> groups of 4 heads
    lens = rng.integers(512, 8193, 64).tolist()
    plan, total, nctas = kvq.kvq_plan_splits(s8, lens, 0, 152)
    _check_plan(plan.numpy(), lens, total, nctas, 2)
    assert nctas == 152


def test_verify_plan_computes_the_causal_lengths(kvq):
    s = _struct(kvq)
    # query token i of a sequence of L tokens (q_len T) sees L - T + 1 + i tokens,
    # none when that is not positive; worked by hand:
    cases = [([5, 40], 3, [3, 4, 5, 38, 39, 40]),
             ([1], 3, [0, 0, 1]),
             ([2, 0, 17], 2, [1, 2, 0, 0, 16, 17]),
             ([33], 1, [33])]
    for lens, T, virtual in cases:
        for ov, tc in ((0, 152), (3, 152), (0, 7)):
            got, total, nctas = kvq.kvq_plan_verify_splits(s, lens, T, ov, tc)
            ref, rtotal, rctas = kvq.kvq_plan_splits(s, virtual, ov, tc)
            assert (total, nctas) == (rtotal, rctas)
            assert np.array_equal(got.numpy()[:ref.numel()], ref.numpy())
            _check_plan(got.numpy(), virtual, total, nctas, 1, ov or None)
    L = kvq.lib()
    total, nctas = ctypes.c_int32(), ctypes.c_int32()
    lens = (ctypes.c_int32 * 2)(5, 9)
    assert L.kvq_plan_verify_splits(ctypes.byref(s), lens, 2, 0, 0, 152, None, 0, ctypes.byref(total),
                                    ctypes.byref(nctas)) == 1 and "q_len" in kvq.kvq_last_error()
    bad = (ctypes.c_int32 * 2)(5, -1)
    assert L.kvq_plan_verify_splits(ctypes.byref(s), bad, 2, 2, 0, 152, None, 0, ctypes.byref(total),
                                    ctypes.byref(nctas)) == 1 and "seq_lens" in kvq.kvq_last_error()


def test_workspace_layout(kvq):
    n = kvq.kvq_decode_workspace_bytes(38, 24, 256)
    # status, lse partials (padded), o partials (padded), a bf16 copy of q
    assert n == 256 + ((38 * 24 * 4 + 255) // 256) * 256 + 38 * 24 * 256 * 4 + 38 * 24 * 256 * 2


def test_host_validation_errors(kvq):
    L = kvq.lib()
    s = _struct(kvq, pages=4)
    s.page_size = 32
    total, mx = ctypes.c_int32(), ctypes.c_int32()
    lens = (ctypes.c_int32 * 1)(10)
    rc = L.kvq_plan_splits(ctypes.byref(s), lens, 1, 1, 0, None, 0, ctypes.byref(total), ctypes.byref(mx))
    assert rc == 2 and "page_size" in kvq.kvq_last_error()
    s.page_size = 16
    s.format = 2
    s.head_dim = 64
    rc = L.kvq_plan_splits(ctypes.byref(s), lens, 1, 1, 0, None, 0, ctypes.byref(total), ctypes.byref(mx))
    assert rc == 2 and "head_dim" in kvq.kvq_last_error()
    s.head_dim = 128  # NVFP4 at head_dim 128 is planned like any other cache
    rc = L.kvq_plan_splits(ctypes.byref(s), lens, 1, 1, 152, None, 0, ctypes.byref(total), ctypes.byref(mx))
    assert rc == 3 and total.value == 1
    s.head_dim = 256
    s.k_global_scale = 0.0
    rc = L.kvq_plan_splits(ctypes.byref(s), lens, 1, 1, 0, None, 0, ctypes.byref(total), ctypes.byref(mx))
    assert rc == 1
    s.k_global_scale = 1.0
    rc = L.kvq_plan_splits(ctypes.byref(s), lens, 1, 1, 152, None, 0, ctypes.byref(total), ctypes.byref(mx))
    assert rc == 3 and total.value == 1 and mx.value == 1  # size query: 1 split, 1 CTA
    # device calls refuse NULL / misaligned arguments before touching the GPU
    rc = L.kvq_quant_append(ctypes.byref(s), None, None, None, 4, None, 0, None)
    assert rc == 1
    rc = L.kvq_paged_decode_attention(ctypes.byref(s), None, 1, 4, 0.1, None, 1, None, None, 1, 1, None, 0, None,
                                      0, None, 0, None)
    assert rc == 1
    assert L.kvq_split_merge(None, None, None, 1, 1, 256, None, 0, None, None) == 1


def test_prefill_split_choice_and_workspace(kvq):
    s = _struct(kvq)  # INT8, Hkv = 4, D = 256
    # 2048 tokens x 6 heads = 96 row blocks of 128 a KV head, 384 CTAs: 2.5 waves;
    # three splits make eight even waves of a third (measured 2,783 against 2,918 us)
    assert kvq.kvq_prefill_splits(s, 2048, 24, 32768, 152) == 3
    assert kvq.kvq_prefill_splits(s, 512, 24, 32768, 152) == 3  # 723 against 818 us at 4
    # 6 tokens: one row block a head, 4 CTAs a split -> one wave of ~37 splits
    # (measured 47.5 us at 38 splits, 83.2 at 16)
    assert kvq.kvq_prefill_splits(s, 6, 24, 32768, 152) == 37
    assert kvq.kvq_prefill_splits(s, 6, 24, 100, 152) == 1  # 7 pages: under two tiles
    for T, L in ((1, 700), (6, 8192), (2048, 32768), (100, 5000)):  # never past 64, at least a tile a split
        S = kvq.kvq_prefill_splits(s, T, 24, L, 152)
        assert 1 <= S <= min(64, max(1, -(-L // 16) // 4))
    assert kvq.kvq_prefill_workspace_bytes(6, 24, 256, 1) == 256
    n = kvq.kvq_prefill_workspace_bytes(6, 24, 256, 3)
    rows = 6 * 3 * 24
    assert n == 256 + (rows * 4 + 255) // 256 * 256 + rows * 256 * 4
    with pytest.raises(kvq.KvqError):
        kvq.kvq_prefill_splits(s, 10, 24, 5, 152)  # q_len > seq_len
    nv = _struct(kvq, fmt="nvfp4")
    assert kvq.kvq_prefill_splits(nv, 10, 24, 500, 152) == 8  # NVFP4 runs on the same prefill kernel
    g32 = _struct(kvq, fmt="int8_g32")
    with pytest.raises(kvq.KvqError, match="no prefill kernel"):  # per-32 scales: decode and verify only
        kvq.kvq_prefill_splits(g32, 10, 24, 500, 152)


def test_verify_workspace_covers_the_tensor_core_route(kvq):
    """A verify call with 4+ query tokens a sequence (3+ for NVFP4) may take the
    prefill kernel, one launch for the batch, with the key splits
    kvq_prefill_splits picks (at most 64; the workspace is sized for the longest
    context): its workspace covers both routes; any other call needs the decode
    workspace."""
    s = _struct(kvq)  # INT8, Hkv = 4, D = 256
    dec = kvq.kvq_decode_workspace_bytes
    pre = kvq.kvq_prefill_workspace_bytes
    vws = lambda st, b, T, hq, ts: kvq.kvq_verify_workspace_bytes(st, b, T, hq, ts, 152)
    # 6 tokens x 6 heads = 36 rows: one row block a KV head, 4 items -> 38 splits
    assert vws(s, 1, 6, 24, 40) == max(dec(40, 24, 256), pre(6, 24, 256, 38)) == pre(6, 24, 256, 38)
    assert vws(s, 1, 6, 24, 4000) == dec(4000, 24, 256)  # a wide decode plan needs more
    assert vws(s, 2, 6, 24, 40) == pre(12, 24, 256, 19)  # two sequences: one launch, 8 CTAs a split
    assert vws(s, 2, 5, 24, 40) == dec(40, 24, 256)  # a batch: 6 INT8 tokens a sequence at least
    assert vws(s, 1, 4, 24, 40) == pre(4, 24, 256, 38)  # 4 tokens: routed on a long context
    assert vws(s, 1, 3, 24, 40) == dec(40, 24, 256)  # 3 INT8 tokens: the decode kernel
    assert vws(s, 1, 43, 24, 43) == max(dec(43, 24, 256), pre(43, 24, 256, 38))  # 258 rows: 12 CTAs a split
    assert vws(s, 1, 8, 8, 8) == max(dec(8, 8, 256), pre(8, 8, 256, 38))  # G = 2: one row block a head
    assert kvq.kvq_verify_workspace_bytes(s, 1, 16, 8, 16, 1000) == max(dec(16, 8, 256), pre(16, 8, 256, 64))
    nv = _struct(kvq, fmt="nvfp4")
    assert vws(nv, 1, 3, 24, 40) == pre(3, 24, 256, 38)  # NVFP4 from 3 tokens
    assert vws(nv, 1, 2, 24, 40) == dec(40, 24, 256)
    assert vws(nv, 3, 3, 24, 40) == dec(40, 24, 256)  # a batch: 4 NVFP4 tokens a sequence at least
    assert vws(nv, 3, 4, 24, 40) > dec(40, 24, 256)
    g32 = _struct(kvq, fmt="int8_g32")  # no prefill kernel: the decode kernel
    assert vws(g32, 1, 6, 24, 40) == dec(40, 24, 256)
    with pytest.raises(kvq.KvqError):
        vws(s, 1, 0, 24, 40)


def test_binding_refuses_undersized_buffers(kvq):
    """The Python binding checks the buffers a device call writes against q's shape
    before anything reaches the library (host tensors stand in for device ones)."""
    import torch

    s = _struct(kvq)  # D = 256
    chk = kvq._binding._shapes
    q = torch.zeros(3, 6, 24, 256)
    bt, sl = torch.zeros(3, 10, dtype=torch.int32), torch.zeros(3, dtype=torch.int32)
    chk(q, torch.zeros(3, 6, 24, 256), torch.zeros(3, 6, 24), bt, sl, s)
    chk(q, torch.zeros(18, 24 * 256), None, bt, sl, s)  # a view of the same size is accepted
    for bad in (dict(out=torch.zeros(1, 6, 24, 256)), dict(lse=torch.zeros(1, 6, 24)),
                dict(bt=torch.zeros(2, 10, dtype=torch.int32)), dict(sl=torch.zeros(2, dtype=torch.int32)),
                dict(q=torch.zeros(3, 6, 24, 128), out=torch.zeros(3, 6, 24, 128))):
        args = dict(q=q, out=torch.zeros(3, 6, 24, 256), lse=None, bt=bt, sl=sl)
        args.update(bad)
        with pytest.raises(ValueError):
            chk(args["q"], args["out"], args["lse"], args["bt"], args["sl"], s)
