"""Planted mistakes in (copies of) the oracle must be caught by the pins.

Each mutant is a plausible slip — a wrong tie rule, a reciprocal instead of a
division, a wrong bias, a swapped nibble, an averaged merge, a dropped scale —
applied to the oracle on the CPU only.  A pin that lets a mutant pass would not
be pinning anything.
"""
import numpy as np
import pytest

from oracle import attention, formats, layout
from tests import oracle_pins as pins


def _fails(check, *args):
    with pytest.raises(AssertionError):
        check(*args)


def test_int8_mutants_are_caught():
    def half_away(x):
        x = np.asarray(x, np.float32)
        s = (np.max(np.abs(x), -1) / np.float32(127)).astype(np.float32)
        q = x / s[..., None]
        c = np.clip(np.sign(q) * np.floor(np.abs(q) + 0.5), -127, 127)
        return c.astype(np.int8), s

    def reciprocal(x):
        x = np.asarray(x, np.float32)
        s = (np.max(np.abs(x), -1) / np.float32(127)).astype(np.float32)
        q = (x * (np.float32(1) / s)[..., None]).astype(np.float32)
        return np.clip(np.rint(q), -127, 127).astype(np.int8), s

    def scale128(x):
        x = np.asarray(x, np.float32)
        s = (np.max(np.abs(x), -1) / np.float32(128)).astype(np.float32)
        return np.clip(np.rint(x / s[..., None]), -127, 127).astype(np.int8), s

    _fails(pins.check_int8_ties, half_away)
    _fails(pins.check_int8_exact, reciprocal, 0, 512, 64)
    _fails(pins.check_int8_exact, scale128)


def test_int8_group_mutants_are_caught():
    def strided(x, group=32):  # group = every (D/32)-th element
        x = np.asarray(x, np.float32)
        D = x.shape[-1]
        c, s = formats.int8_quantize(x.reshape(x.shape[:-1] + (group, D // group)).swapaxes(-1, -2))
        return c.swapaxes(-1, -2).reshape(x.shape), s

    def row_scale(x, group=32):  # one scale for the whole row, repeated
        c, s = formats.int8_quantize(x)
        return c, np.repeat(s[..., None], x.shape[-1] // group, axis=-1)

    def deq_wrong_group(codes, scales, group=32):  # group index off by one
        c = np.asarray(codes, np.float64)
        sc = np.roll(np.asarray(scales, np.float64), 1, axis=-1)
        return (c.reshape(c.shape[:-1] + (-1, group)) * sc[..., None]).reshape(c.shape)

    _fails(pins.check_int8_group_exact, strided)
    _fails(pins.check_int8_group_exact, row_scale)
    _fails(pins.check_int8_group_hand_example, formats.int8_group_quantize, deq_wrong_group)
    _fails(pins.check_int8_group_invariants, formats.int8_group_quantize, deq_wrong_group, formats.int8_quantize)


def test_fp8_fp4_mutants_are_caught():
    def bias8(b):
        return formats.e4m3_value(b) / 2.0

    def ties_up(t):
        t = np.asarray(t, np.float64)
        grid = formats._E4M3_POS
        idx = np.clip(np.searchsorted(grid, np.abs(t), side="right"), 1, len(grid) - 1)
        lo, hi = idx - 1, idx
        pick = np.abs(t) - grid[lo] >= grid[hi] - np.abs(t)
        return np.where(pick, hi, lo).astype(np.uint8)

    def swapped_grid(c):
        g = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 4.0, 3.0, 6.0])
        c = np.asarray(c, np.int64)
        return np.where(c & 8, -1.0, 1.0) * g[c & 7]

    def swapped_nibbles(c):
        c = np.asarray(c, np.uint8)
        return (c[..., 1::2] | (c[..., 0::2] << 4)).astype(np.uint8)

    def amax_over_4(x, gs):
        return formats.nvfp4_quantize(np.asarray(x, np.float32) * np.float32(1.5), gs)

    _fails(pins.check_e4m3_decode, bias8)
    _fails(pins.check_e4m3_encode, ties_up)
    _fails(pins.check_e2m1_grid, swapped_grid)
    _fails(pins.check_nibble_order, swapped_nibbles)
    _fails(pins.check_nvfp4_exact, amax_over_4, formats.unpack_nibbles)


def test_attention_mutants_are_caught():
    from oracle import brute

    def no_scale(q, k, v, sm):
        return attention.attend(q, k, v, 1.0)

    def transposed_v(q, k, v, sm):
        o, s = attention.attend(q, k, v, sm)
        return o[:, ::-1], s

    def averaged(outs, lses):
        return np.mean(outs, axis=0), np.max(lses, axis=0)

    def split_with_average(q, k, v, sm, bounds):
        outs, lses = zip(*[attention.attend(q, k[b:e], v[b:e], sm) for b, e in bounds])
        return averaged(np.stack(outs), np.stack(lses))

    def lse_without_log(q, k, v, sm):
        o, s = attention.attend(q, k, v, sm)
        p = attention.probabilities(q, k, sm)
        return o, s - np.log(1.0 / p.max(axis=1)) * 0 + 0.5

    def verify_off_by_one(fmt, pools, q, bt, lens, sm, page_size=16):
        # each query token sees one token too few
        return attention.paged_verify(fmt, pools, q, bt, np.asarray(lens) - 1, sm, page_size=page_size)

    def verify_tokens_swapped(fmt, pools, q, bt, lens, sm, page_size=16):
        # query token i paired with token T-1-i's visible prefix
        return attention.paged_verify(fmt, pools, q[:, ::-1], bt, lens, sm, page_size=page_size)

    def verify_sees_all(fmt, pools, q, bt, lens, sm, page_size=16):
        B, T = q.shape[:2]
        outs = [attention.paged_verify(fmt, pools, q[:, i:i + 1], bt, lens, sm, page_size=page_size) for i in range(T)]
        return np.concatenate([o for o, _ in outs], axis=1), np.concatenate([s for _, s in outs], axis=1)

    _fails(pins.check_verify, verify_off_by_one)
    _fails(pins.check_verify, verify_tokens_swapped)
    _fails(pins.check_verify, verify_sees_all)
    _fails(pins.check_attend_brute, no_scale, brute.attend_brute)
    _fails(pins.check_attend_brute, transposed_v, brute.attend_brute)
    _fails(pins.check_attend_brute, lse_without_log, brute.attend_brute)
    _fails(pins.check_split_merge, attention.attend, split_with_average)
    _fails(pins.check_merge_not_average, attention.attend, averaged)


def test_layout_mutants_are_caught(monkeypatch):
    def slots_page_row_swapped(bt, L, P):  # page from t % P, row from t // P (table index kept in range)
        t = np.arange(int(L), dtype=np.int64)
        bt = np.asarray(bt, np.int64)
        return bt[(t % P) % len(bt)] * P + t // P

    def slots_table_mod(bt, L, P):  # block_table[t % P] instead of block_table[t // P]
        t = np.arange(int(L), dtype=np.int64)
        bt = np.asarray(bt, np.int64)
        return bt[(t % P) % len(bt)] * P + t % P

    def slots_identity_pages(bt, L, P):  # block table ignored
        return np.arange(int(L), dtype=np.int64)

    def gather_page_row_swapped(pool, slots, head):
        pool = np.asarray(pool)
        P = pool.shape[2]
        slots = np.asarray(slots, np.int64)
        return pool[slots % P, head, slots // P]

    def gather_head_page_swapped(pool, slots, head):
        pool = np.asarray(pool)
        P = pool.shape[2]
        slots = np.asarray(slots, np.int64)
        return pool[head, slots // P, slots % P] if pool.shape[0] > head else pool[slots // P, head, slots % P]

    def scatter_page_row_swapped(pool, slots, head, rows):
        P = pool.shape[2]
        slots = np.asarray(slots, np.int64)
        pool[slots % P, head, slots // P] = rows

    def group_major_reshaped(a):  # reshape instead of a transpose
        a = np.asarray(a)
        return a.reshape(a.shape[0], a.shape[1], a.shape[3], a.shape[2])

    def group_major_wrong_axes(a):
        return np.ascontiguousarray(np.swapaxes(np.asarray(a), 1, 2))

    def fails_or_raises(check, *args):  # an out-of-range index is as much a catch as a wrong value
        with pytest.raises((AssertionError, IndexError)):
            check(*args)

    for m in (slots_page_row_swapped, slots_table_mod, slots_identity_pages):
        _fails(pins.check_token_slots, m)
    fails_or_raises(pins.check_gather_scatter, gather_page_row_swapped, layout.scatter_rows)
    fails_or_raises(pins.check_gather_scatter, gather_head_page_swapped, layout.scatter_rows)
    fails_or_raises(pins.check_gather_scatter, layout.gather_rows, scatter_page_row_swapped)
    _fails(pins.check_group_major, group_major_reshaped)
    with pytest.raises((AssertionError, ValueError)):
        pins.check_group_major(group_major_wrong_axes)
    # the same slips inside the oracle's decode and verify are caught by the
    # pins of those functions (hand-placed pools, brute force over logical rows)
    for m in (slots_page_row_swapped, slots_table_mod):
        with monkeypatch.context() as mp:
            mp.setattr(layout, "token_slots", m)
            _fails(pins.check_verify, attention.paged_verify)
            _fails(pins.check_paged_decode, attention.paged_decode)
    with monkeypatch.context() as mp:
        mp.setattr(layout, "gather_rows", gather_page_row_swapped)
        fails_or_raises(pins.check_paged_decode, attention.paged_decode)
