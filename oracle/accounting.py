"""Byte accounting of the KV formats — TEST INFRASTRUCTURE ONLY (oracle).

Closed forms the pages print and that the tests check:
  * BF16: 2 bytes per element, K and V ("half-the-memory-int8-kv-cache" page,
    opening section: 16 layers x 4 KV heads x D 256 -> 64 KiB per token).
  * INT8: D code bytes + one 4-byte scale per tensor ("An 8-bit cache was already
    available": 520 bytes per token per head at D = 256; "Read the compressed
    cache without copying it first": the next head starts at byte 260).
  * INT8 with one scale per 32 values: D code bytes + D/32 four-byte scales per
    tensor ("Is 8 bits enough?": one scale per 32 values instead of one per 256).
  * NVFP4: D/2 code bytes + D/16 E4M3 scale bytes per tensor ("Building an NVFP4
    KV cache for a hybrid Qwen model", section "How 2,048 bytes became 576").
  * FP8 (accounting only, one byte per element): the same section's 1,024-byte row.
"""
from __future__ import annotations


def record_bytes(fmt, head_dim):
    """Bytes of one K (or V) record for one token and one KV head."""
    D = int(head_dim)
    if fmt == "bf16":
        return 2 * D
    if fmt == "fp8":
        return D
    if fmt == "int8":
        return D + 4
    if fmt == "int8_g32":
        return D + 4 * (D // 32)
    if fmt == "nvfp4":
        return D // 2 + D // 16
    raise ValueError(fmt)


def bytes_per_token_head(fmt, head_dim):
    """K + V bytes for one token and one KV head."""
    return 2 * record_bytes(fmt, head_dim)


def bytes_per_token_layer(fmt, num_kv_heads, head_dim):
    return num_kv_heads * bytes_per_token_head(fmt, head_dim)


def bytes_per_token(fmt, num_layers, num_kv_heads, head_dim):
    return num_layers * bytes_per_token_layer(fmt, num_kv_heads, head_dim)


def token_slots(budget_bytes, per_token_bytes):
    """Whole tokens that fit in a byte budget."""
    return int(budget_bytes) // int(per_token_bytes)


def decode_kv_bytes(fmt, seq_lens, num_kv_heads, head_dim):
    """Bytes of cache one decode-attention call must read: every valid token of
    every sequence, K and V, all KV heads (page padding not counted)."""
    return sum(int(L) for L in seq_lens) * bytes_per_token_layer(fmt, num_kv_heads, head_dim)


def attention_flops(query_rows, context, head_dim, num_kv_heads):
    """Multiply-add flops of q.K and P.V for ``query_rows`` rows per KV head."""
    return 2 * 2 * int(query_rows) * int(context) * int(head_dim) * int(num_kv_heads)


def conversion_scratch_bytes(tokens, num_kv_heads, head_dim, elem_bytes=2):
    """Bytes of a K+V staging copy of ``tokens`` tokens at ``elem_bytes`` per element."""
    return 2 * int(tokens) * int(num_kv_heads) * int(head_dim) * int(elem_bytes)


def ceil_div(a, b):
    return -(-int(a) // int(b))

