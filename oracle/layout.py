"""Reader of the paged KV pool layout — TEST INFRASTRUCTURE ONLY (oracle).

The pool layout is the one the library documents in its C header; this module
re-derives token positions from that written description alone.

  * A pool holds ``num_pages`` pages of ``P`` token slots (PagedAttention's
    fixed-size blocks: "Smaller KV cache, faster first token" page, section "Why
    KV capacity drives TTFT under load").  Slot ``s`` lives in page ``s // P``,
    row ``s % P``.
  * Codes: array ``[num_pages, Hkv, P, row_bytes]`` (row_bytes = 2D for bf16, D
    for int8, D/2 for nvfp4), one contiguous row per (page, KV head, slot).
  * Scales: int8 ``[num_pages, Hkv, P]`` float32; nvfp4 ``[num_pages, Hkv, P,
    D/16]`` E4M3 bytes; bf16 has none.  int8 with one scale per 32 values stores
    its scales group-major inside each (page, KV head) block, ``[num_pages, Hkv,
    D/32, P]`` float32: ``group_major_scales`` turns that array into the
    ``[num_pages, Hkv, P, D/32]`` form the functions below index.
  * Token ``t`` of sequence ``b`` sits in slot ``block_table[b, t // P] * P + t % P``.

Pinned by hand-worked slot lists (tests/golden/page_mapping.txt), pools whose
cells hold their own coordinates, and decode / verify checks over pools that the
tests fill token by token without these functions.
"""
from __future__ import annotations

import numpy as np


def token_slots(block_table_row, seq_len, page_size):
    """Physical slot of each logical token 0..seq_len-1 of one sequence."""
    t = np.arange(int(seq_len), dtype=np.int64)
    pages = np.asarray(block_table_row, dtype=np.int64)[t // page_size]
    return pages * page_size + t % page_size


def gather_rows(pool, slots, head):
    """Rows of ``pool`` ([num_pages, Hkv, P, ...]) for the given slots and KV head."""
    pool = np.asarray(pool)
    P = pool.shape[2]
    slots = np.asarray(slots, dtype=np.int64)
    return pool[slots // P, head, slots % P]


def scatter_rows(pool, slots, head, rows):
    """Write ``rows`` into ``pool`` at the given slots of one KV head (in place)."""
    P = pool.shape[2]
    slots = np.asarray(slots, dtype=np.int64)
    pool[slots // P, head, slots % P] = rows


def group_major_scales(pool):
    """A ``[num_pages, Hkv, groups, P]`` scale array as ``[num_pages, Hkv, P, groups]``
    (slot-major: one row of group scales per slot)."""
    return np.ascontiguousarray(np.swapaxes(np.asarray(pool), 2, 3))


def to_group_major_scales(rows_pool):
    """Inverse of ``group_major_scales``: the device's storage order."""
    return np.ascontiguousarray(np.swapaxes(np.asarray(rows_pool), 2, 3))
