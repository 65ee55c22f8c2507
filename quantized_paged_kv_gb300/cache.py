"""Device pools, split plans and workspaces around the C ABI (torch supplies the
device memory and the stream; every step of the path runs in libkvq's kernels).
"""
from __future__ import annotations

import torch

from . import _binding as B


class KVCache:
    """A paged K/V pool in one format, laid out as include/kvq.h documents:
    codes [num_pages][Hkv][16][row_bytes] and scales [num_pages][Hkv][16][...]
    for K and for V.  ``fill`` (a byte value) pre-fills every array, e.g. 0xFF
    so that unwritten slots hold NaN scales."""

    def __init__(self, fmt, num_pages, num_kv_heads, head_dim, page_size=16, device="cuda",
                 k_global_scale=1.0, v_global_scale=1.0, fill=None):
        self.fmt = fmt
        self.num_pages, self.num_kv_heads, self.head_dim, self.page_size = num_pages, num_kv_heads, head_dim, page_size
        cb, sb = B.kvq_cache_array_bytes(fmt, num_pages, page_size, num_kv_heads, head_dim)
        alloc = (lambda n: torch.empty(n, dtype=torch.uint8, device=device)) if fill is None else \
            (lambda n: torch.full((n,), fill, dtype=torch.uint8, device=device))
        self.k_codes, self.v_codes = alloc(cb), alloc(cb)
        self.k_scales, self.v_scales = (alloc(sb), alloc(sb)) if sb else (None, None)
        self.k_global_scale, self.v_global_scale = float(k_global_scale), float(v_global_scale)
        self.struct = B.KvqCacheStruct(
            self.k_codes.data_ptr(), self.v_codes.data_ptr(),
            self.k_scales.data_ptr() if sb else None, self.v_scales.data_ptr() if sb else None,
            num_pages, page_size, num_kv_heads, head_dim, B.FORMATS[fmt], self.k_global_scale, self.v_global_scale)

    @property
    def row_bytes(self):
        return {"bf16": 2 * self.head_dim, "int8": self.head_dim, "int8_g32": self.head_dim,
                "nvfp4": self.head_dim // 2}[self.fmt]

    def views(self):
        """(k_codes, v_codes, k_scales, v_scales) reshaped to [num_pages, Hkv, P, ...]."""
        shp = (self.num_pages, self.num_kv_heads, self.page_size)
        kc = self.k_codes.view(*shp, self.row_bytes)
        vc = self.v_codes.view(*shp, self.row_bytes)
        if self.k_scales is None:
            return kc, vc, None, None
        if self.fmt == "int8":
            return kc, vc, self.k_scales.view(torch.float32).view(*shp), self.v_scales.view(torch.float32).view(*shp)
        if self.fmt == "int8_g32":  # group-major: [num_pages, Hkv, D/32, P]
            gshp = (self.num_pages, self.num_kv_heads, self.head_dim // 32, self.page_size)
            return kc, vc, self.k_scales.view(torch.float32).view(*gshp), self.v_scales.view(torch.float32).view(*gshp)
        return kc, vc, self.k_scales.view(*shp, self.head_dim // 16), self.v_scales.view(*shp, self.head_dim // 16)

    def append(self, k_new, v_new, slot_mapping, dev_status=None, checked=False, rotate=False, stream=None):
        flags = (B.KVQ_CHECKED if checked else 0) | (B.KVQ_ROTATE if rotate else 0)
        B.kvq_quant_append(self.struct, k_new, v_new, slot_mapping, dev_status, flags, stream)


class DecodePlan:
    """Host split plan for one batch composition, copied to the device, plus the
    workspace it needs (status word zeroed once).  q_len > 1: the plan of a
    verify call over q_len query tokens a sequence."""

    def __init__(self, cache, seq_lens, num_q_heads, split_override=0, target_ctas=0, device="cuda", q_len=1):
        lens = [int(x) for x in seq_lens]
        if q_len == 1:
            plan, self.total_splits, self.num_ctas = B.kvq_plan_splits(cache.struct, lens, split_override, target_ctas)
        else:
            plan, self.total_splits, self.num_ctas = B.kvq_plan_verify_splits(cache.struct, lens, q_len,
                                                                              split_override, target_ctas)
        self.plan_host = plan
        self.plan = plan.to(device)
        self.q_len = q_len
        self.batch = len(seq_lens) * q_len
        self.num_q_heads = num_q_heads
        self.head_dim = cache.head_dim
        if q_len == 1:
            ws = B.kvq_decode_workspace_bytes(self.total_splits, num_q_heads, cache.head_dim)
        else:  # room for the tensor-core route of a one-sequence verify call as well
            ws = B.kvq_verify_workspace_bytes(cache.struct, len(seq_lens), q_len, num_q_heads, self.total_splits)
        self.workspace = torch.zeros(ws, dtype=torch.uint8, device=device)

    def partials(self):
        """(o_part pointer, lse_part pointer) inside the workspace."""
        return B.kvq_workspace_partials(self.workspace, self.total_splits, self.num_q_heads, self.head_dim)


def decode(cache, plan, q, block_tables, seq_lens, out, sm_scale, lse_out=None, checked=False, skip_merge=False,
           early_start=False, stream=None):
    """early_start: the plan and block tables are not written by the kernel just before this call on the stream
    (e.g. they were uploaded once for all layers of a step), so the decode may read them early."""
    flags = ((B.KVQ_CHECKED if checked else 0) | (B.KVQ_SKIP_MERGE if skip_merge else 0)
             | (B.KVQ_EARLY_START if early_start else 0))
    B.kvq_paged_decode_attention(cache.struct, q, sm_scale, block_tables, seq_lens, plan.plan, plan.total_splits,
                                 plan.num_ctas, plan.workspace, out, lse_out, flags, stream)


def verify(cache, plan, q, block_tables, seq_lens, out, sm_scale, lse_out=None, checked=False, skip_merge=False,
           early_start=False, stream=None):
    """Causal attention for q.shape[1] query tokens a sequence; plan: DecodePlan(..., q_len=q.shape[1])."""
    if plan.q_len != q.shape[1]:
        raise ValueError(f"the plan is for q_len {plan.q_len}, q has {q.shape[1]} query tokens")
    flags = ((B.KVQ_CHECKED if checked else 0) | (B.KVQ_SKIP_MERGE if skip_merge else 0)
             | (B.KVQ_EARLY_START if early_start else 0))
    B.kvq_paged_verify_attention(cache.struct, q, sm_scale, block_tables, seq_lens, plan.plan, plan.total_splits,
                                 plan.num_ctas, plan.workspace, out, lse_out, flags, stream)


def prefill(cache, q, block_table, seq_len, out, sm_scale, lse_out=None, splits=0, workspace=None, checked=False,
            stream=None):
    """Causal attention of a prompt chunk: q [T, Hq, D] holds the last T of the sequence's seq_len tokens (their
    K/V already appended); block_table [max_pages] int32.  splits 0 = kvq_prefill_splits' choice.  Returns the
    workspace used (reusable for the same T / splits)."""
    T, Hq, D = q.shape
    if splits == 0:
        splits = B.kvq_prefill_splits(cache.struct, T, Hq, int(seq_len))
    need = B.kvq_prefill_workspace_bytes(T, Hq, D, splits)
    if workspace is None or workspace.numel() < need:
        workspace = torch.zeros(need, dtype=torch.uint8, device=q.device)
    B.kvq_paged_prefill_attention(cache.struct, q, sm_scale, block_table, seq_len, splits, workspace, out, lse_out,
                                  B.KVQ_CHECKED if checked else 0, stream)
    return workspace
