"""kvq_paged_decode_attention_static (library-owned scratch, no allocation)
against the CPU oracle and against kvq_paged_decode_attention (caller's
workspace), through the C ABI.

The file name makes pytest collect it last, so that it runs both after every
other test in one process and, alone, in a fresh one.  Calls come in a row with
different shapes: each finds the previous call's partials in the shared region.
Tolerance: the decode tests' max-abs 2e-3 (fp32 output) / 1e-2 (bf16 output).
"""
import numpy as np
import pytest
import torch

from quantized_paged_kv_gb300 import workloads as W
from tests import harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    H.ensure_built()


def _inputs(wl, fmt, split):
    from quantized_paged_kv_gb300 import DecodePlan

    cache = H.gpu_cache(wl, fmt, H.global_scales(wl, fmt))
    plan = DecodePlan(cache, wl.seq_lens, wl.Hq, split_override=split)
    q = torch.from_numpy(wl.q()).to(torch.bfloat16).cuda()
    bt = torch.from_numpy(wl.block_tables).cuda()
    sl = torch.from_numpy(wl.seq_lens).cuda()
    return cache, plan, q, bt, sl


def _both(wl, fmt, split, out_dtype, checked=True):
    """(static out, static lse, workspace out, workspace lse) on the same inputs."""
    from quantized_paged_kv_gb300 import KVQ_CHECKED, decode, kvq_paged_decode_attention_static

    cache, plan, q, bt, sl = _inputs(wl, fmt, split)
    od = {"f32": torch.float32, "bf16": torch.bfloat16}[out_dtype]
    o_s = torch.full((wl.B, wl.Hq, wl.D), float("nan"), dtype=od, device="cuda")
    l_s = torch.full((wl.B, wl.Hq), float("nan"), device="cuda")
    o_w, l_w = torch.full_like(o_s, float("nan")), torch.full_like(l_s, float("nan"))
    kvq_paged_decode_attention_static(cache.struct, q, wl.sm_scale, bt, sl, plan.plan, plan.total_splits,
                                      plan.num_ctas, o_s, l_s, KVQ_CHECKED if checked else 0)
    decode(cache, plan, q, bt, sl, o_w, wl.sm_scale, lse_out=l_w, checked=checked)
    torch.cuda.synchronize()
    return (o_s.float().cpu().numpy(), l_s.cpu().numpy(), o_w.float().cpu().numpy(), l_w.cpu().numpy(),
            plan.total_splits)


def _compare(wl, fmt, split, out_dtype):
    o_s, l_s, o_w, l_w, total = _both(wl, fmt, split, out_dtype)
    assert total > wl.B  # the merge reads partials out of the static region
    assert np.all(np.isfinite(o_s))
    # against the oracle (float64 attention over the oracle's own pools)
    ref, ref_lse = H.oracle_decode(wl, fmt, H.oracle_pools(wl, fmt, H.global_scales(wl, fmt)))
    assert np.all(np.abs(o_s - ref) <= H.bound(out_dtype, ref))
    fin_ref = np.isfinite(ref_lse)
    assert np.array_equal(fin_ref, np.isfinite(l_s))
    assert fin_ref.sum() == 0 or np.abs(l_s[fin_ref] - ref_lse[fin_ref]).max() < 1e-3
    # and against the workspace entry point on the same inputs
    assert np.abs(o_s - o_w).max() <= H.tol(out_dtype)
    fin = np.isfinite(l_w)
    assert np.array_equal(fin, np.isfinite(l_s))
    assert fin.sum() == 0 or np.abs(l_s[fin] - l_w[fin]).max() < 1e-3


def test_two_calls_in_a_row_match_the_workspace_entry_point():
    # call 1: a ragged D=128 serving batch; call 2: a D=256 6:1 GQA batch with
    # more splits per sequence and a different partial-row stride
    wl1 = W.make("serving_int8", lens=("list", [1, 17, 300, 0, 64, 1000, 2500]), seed=11)
    wl2 = W.make("tiny_int8", lens=("list", [700, 33, 4096]), seed=12)
    _compare(wl1, "int8", 3, "bf16")
    _compare(wl2, "int8", 5, "f32")
    # and back, now over the larger call's leftovers, in NVFP4 (tensor global scales)
    _compare(wl1, "nvfp4", 3, "bf16")


def test_status_block_is_cleared_between_calls():
    from quantized_paged_kv_gb300 import KVQ_CHECKED, kvq_paged_decode_attention_static

    wl = W.make("tiny_int8", lens=("list", [64, 64]), seed=2)
    cache, plan, q, bt, sl = _inputs(wl, "int8", 2)
    out = torch.empty((wl.B, wl.Hq, wl.D), device="cuda")
    bad = bt.clone()
    bad[1, 2] = wl.num_pages + 5  # out-of-range page id: the kernel skips it and flags the status block
    kvq_paged_decode_attention_static(cache.struct, q, wl.sm_scale, bad, sl, plan.plan, plan.total_splits,
                                      plan.num_ctas, out, None, 0)  # unchecked: the flag stays in the region
    torch.cuda.synchronize()
    # a valid checked call must not see the previous call's flag
    kvq_paged_decode_attention_static(cache.struct, q, wl.sm_scale, bt, sl, plan.plan, plan.total_splits,
                                      plan.num_ctas, out, None, KVQ_CHECKED)
    o_s, _, o_w, _, _ = _both(wl, "int8", 2, "f32")
    assert np.abs(o_s - o_w).max() <= H.tol("f32")


def test_oversized_request_is_rejected_before_any_work():
    from quantized_paged_kv_gb300 import KvqError, kvq_decode_workspace_bytes, kvq_paged_decode_attention_static
    from quantized_paged_kv_gb300._binding import KVQ_STATIC_SCRATCH_BYTES

    wl = W.make("tiny_int8", lens=("list", [64]), seed=3)
    cache, plan, q, bt, sl = _inputs(wl, "int8", 1)
    per_split = kvq_decode_workspace_bytes(2, wl.Hq, wl.D) - kvq_decode_workspace_bytes(1, wl.Hq, wl.D)
    too_many = KVQ_STATIC_SCRATCH_BYTES // per_split + 1
    assert kvq_decode_workspace_bytes(too_many, wl.Hq, wl.D) > KVQ_STATIC_SCRATCH_BYTES
    out = torch.full((wl.B, wl.Hq, wl.D), 7.0, device="cuda")
    with pytest.raises(KvqError) as e:
        kvq_paged_decode_attention_static(cache.struct, q, wl.sm_scale, bt, sl, plan.plan, too_many, plan.num_ctas,
                                          out, None, 0)
    assert e.value.code == 3 and "static region" in str(e.value)
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)
