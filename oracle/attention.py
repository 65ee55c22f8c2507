"""Float64 decode attention over a quantized paged cache — TEST INFRASTRUCTURE ONLY.

What is computed (the plain definition; the GPU path reaches the same result by
a different order of operations):

  For a sequence b and query head g, with KV head h = g // G (G = Hq / Hkv
  consecutive query heads share one KV head: grouped-query attention, 24 query
  and 4 KV heads = 6:1 on the "long-context-attention-and-lessons" page, section
  "Give more GPU workers a piece of the attention calculation"):

      z_t  = sm_scale * sum_d q[g, d] * k_hat[t, d]        t < L_b
      p_t  = exp(z_t - max z) / sum_u exp(z_u - max z)
      out  = sum_t p_t * v_hat[t]
      lse  = max z + log sum_t exp(z_t - max z)

  where k_hat / v_hat are the dequantized cache rows (formats.py) in the logical
  token order given by the block table (layout.py).  sm_scale = 1/sqrt(D) is
  passed in explicitly.

Split-KV (flash-decoding), same page and section: the context is cut into
segments, each segment yields a normalised partial output plus its log-sum-exp
("a weighted value sum and information needed to normalise it"), and the merge
uses those terms; averaging the partial outputs would be wrong.

  merge:  M = max_s lse_s;  w_s = exp(lse_s - M);  out = sum_s w_s o_s / sum_s w_s;
          lse = M + log sum_s w_s;  a segment with no tokens has lse = -inf, weight 0.

An empty context (L = 0) gives out = 0 and lse = -inf.

Verification of several proposed tokens ("half-the-memory-int8-kv-cache", section
"Read the compressed cache without copying it first": one program both generates
a token and checks several proposed ones, 6 query tokens x 6 heads at a verify
step): T query tokens of sequence b, whose K/V are already the last T entries of
its cache (L_b tokens in all).  Reading: causal, as in any autoregressive check —
query token i sits at position L_b - T + i and sees tokens 0 .. L_b - T + i, i.e.
the decode above over the first max(0, L_b - T + i + 1) tokens.
"""
from __future__ import annotations

import numpy as np

from . import formats, layout


def attend(q, k, v, sm_scale):
    """q [G, D], k/v [L, D] (float64 values) -> (out [G, D], lse [G])."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    G, D = q.shape
    if k.shape[0] == 0:
        return np.zeros((G, D)), np.full(G, -np.inf)
    z = np.float64(sm_scale) * (q @ k.T)  # [G, L]
    m = z.max(axis=1, keepdims=True)
    e = np.exp(z - m)
    l = e.sum(axis=1)
    out = (e @ v) / l[:, None]
    lse = m[:, 0] + np.log(l)
    return out, lse


def probabilities(q, k, sm_scale):
    """The softmax weights p [G, L] of ``attend`` (used by invariant tests)."""
    z = np.float64(sm_scale) * (np.asarray(q, np.float64) @ np.asarray(k, np.float64).T)
    m = z.max(axis=1, keepdims=True)
    e = np.exp(z - m)
    return e / e.sum(axis=1, keepdims=True)


def merge(outs, lses):
    """Log-sum-exp combine of split partials: outs [S, G, D], lses [S, G]."""
    outs = np.asarray(outs, dtype=np.float64)
    lses = np.asarray(lses, dtype=np.float64)
    M = lses.max(axis=0)  # [G]
    finite = np.isfinite(M)
    Ms = np.where(finite, M, 0.0)
    w = np.where(np.isfinite(lses), np.exp(lses - Ms[None, :]), 0.0)  # [S, G]
    wsum = w.sum(axis=0)
    safe = np.where(wsum > 0, wsum, 1.0)
    out = (w[:, :, None] * np.where(np.isfinite(lses)[:, :, None], outs, 0.0)).sum(axis=0) / safe[:, None]
    out = np.where(finite[:, None], out, 0.0)
    lse = np.where(finite, Ms + np.log(safe), -np.inf)
    return out, lse


def attend_split(q, k, v, sm_scale, token_bounds):
    """Split-then-merge: ``token_bounds`` is a list of (begin, end) token ranges
    that partition [0, L); each range is attended alone, then merged."""
    outs, lses = [], []
    for (b, e) in token_bounds:
        o, s = attend(q, k[b:e], v[b:e], sm_scale)
        outs.append(o)
        lses.append(s)
    return merge(np.stack(outs), np.stack(lses))


# ---------------------------------------------------------------------------
# Paged cache in a given storage format
# ---------------------------------------------------------------------------
def dequantize_rows(fmt, codes, scales, global_scale=1.0):
    """Rows of one format -> float64 values [n, D]."""
    if fmt == "int8":
        return formats.int8_dequantize(codes.view(np.int8), scales)
    if fmt == "int8_g32":
        return formats.int8_group_dequantize(codes.view(np.int8), scales)
    if fmt == "nvfp4":
        return formats.nvfp4_dequantize(codes, scales, global_scale)
    if fmt == "bf16":
        return formats.bf16_bits_to_f32(codes.view(np.uint16)).astype(np.float64)
    raise ValueError(fmt)


def cache_rows(fmt, codes_pool, scales_pool, slots, head, global_scale=1.0):
    c = layout.gather_rows(codes_pool, slots, head)
    s = None if scales_pool is None else layout.gather_rows(scales_pool, slots, head)
    return dequantize_rows(fmt, c, s, global_scale)


def paged_decode(fmt, pools, q, block_tables, seq_lens, sm_scale, heads=None, page_size=16):
    """Decode attention for a batch over a paged pool.

    pools: dict with 'k_codes', 'v_codes', 'k_scales', 'v_scales' (numpy, layout of
    layout.py; scales None for bf16) and 'k_global_scale', 'v_global_scale'
    (nvfp4 only).  q: [B, Hq, D] float (bf16 values).  heads: optional list of
    (b, kv_head) units to compute (others stay NaN) for sampled checks.

    Returns (out [B, Hq, D] float64, lse [B, Hq] float64).
    """
    q = np.asarray(q, dtype=np.float64)
    B, Hq, D = q.shape
    Hkv = pools["k_codes"].shape[1]
    G = Hq // Hkv
    out = np.full((B, Hq, D), np.nan)
    lse = np.full((B, Hq), np.nan)
    gk = pools.get("k_global_scale", 1.0)
    gv = pools.get("v_global_scale", 1.0)
    units = heads if heads is not None else [(b, h) for b in range(B) for h in range(Hkv)]
    for (b, h) in units:
        slots = layout.token_slots(block_tables[b], seq_lens[b], page_size)
        k = cache_rows(fmt, pools["k_codes"], pools.get("k_scales"), slots, h, gk)
        v = cache_rows(fmt, pools["v_codes"], pools.get("v_scales"), slots, h, gv)
        o, s = attend(q[b, h * G:(h + 1) * G], k, v, sm_scale)
        out[b, h * G:(h + 1) * G] = o
        lse[b, h * G:(h + 1) * G] = s
    return out, lse


def paged_verify(fmt, pools, q, block_tables, seq_lens, sm_scale, units=None, page_size=16):
    """Attention for T query tokens a sequence over a paged pool, causal (module
    docstring).  q: [B, T, Hq, D].  units: optional list of (b, i, kv_head) to
    compute (others stay NaN).  Returns (out [B, T, Hq, D], lse [B, T, Hq])."""
    q = np.asarray(q, dtype=np.float64)
    B, T, Hq, D = q.shape
    Hkv = pools["k_codes"].shape[1]
    G = Hq // Hkv
    out = np.full((B, T, Hq, D), np.nan)
    lse = np.full((B, T, Hq), np.nan)
    gk = pools.get("k_global_scale", 1.0)
    gv = pools.get("v_global_scale", 1.0)
    todo = units if units is not None else [(b, i, h) for b in range(B) for i in range(T) for h in range(Hkv)]
    for (b, i, h) in todo:
        visible = max(0, int(seq_lens[b]) - T + i + 1)
        slots = layout.token_slots(block_tables[b], visible, page_size)
        k = cache_rows(fmt, pools["k_codes"], pools.get("k_scales"), slots, h, gk)
        v = cache_rows(fmt, pools["v_codes"], pools.get("v_scales"), slots, h, gv)
        o, s = attend(q[b, i, h * G:(h + 1) * G], k, v, sm_scale)
        out[b, i, h * G:(h + 1) * G] = o
        lse[b, i, h * G:(h + 1) * G] = s
    return out, lse


def quantize_rows(fmt, x, global_scale=1.0):
    """bf16-valued rows x [n, D] -> (codes, scales) in the given format."""
    x = np.asarray(x, dtype=np.float32)
    if fmt == "int8":
        c, s = formats.int8_quantize(x)
        return c.view(np.uint8), s
    if fmt == "int8_g32":
        c, s = formats.int8_group_quantize(x)
        return c.view(np.uint8), s
    if fmt == "nvfp4":
        return formats.nvfp4_quantize(x, global_scale)
    if fmt == "bf16":
        bits = (x.view(np.uint32) >> 16).astype(np.uint16)  # x already holds bf16 values
        return bits.view(np.uint8).reshape(x.shape[:-1] + (2 * x.shape[-1],)), None
    raise ValueError(fmt)
