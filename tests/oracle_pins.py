"""Independent checks ("pins") of the CPU oracle.

Each ``check_*`` function takes the oracle function it checks as an argument and
raises AssertionError on a mismatch, so that the same check can run against the
real oracle (tests/test_oracle_*.py) and against deliberately broken copies of
it (tests/test_oracle_mutations.py), showing that a plausible mistake is caught.

The expected values never come from the oracle itself: they come from the
pages' printed values (tests/golden/), exact rational arithmetic
(``fractions.Fraction``), torch's float8_e4m3fn cast (a library routine that
shares nothing with the oracle), brute force, or invariants.
"""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------------------
# exact helpers
# ---------------------------------------------------------------------------
def rn_f32(r: Fraction) -> Fraction:
    """Round a rational to the nearest IEEE binary32 value, ties to even
    (finite range only).  Written from the IEEE definition: quantum 2^(e-23)
    for normal numbers, 2^-149 below 2^-126."""
    if r == 0:
        return Fraction(0)
    sign = -1 if r < 0 else 1
    a = abs(r)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    quantum = Fraction(2) ** (max(e, -126) - 23)
    n = a / quantum
    k = round(n)  # Fraction.__round__ rounds half to even
    return sign * k * quantum


def bf16_values(rng, shape, scale=1.0):
    """Random bf16-representable float32 values (rounded by torch)."""
    x = torch.from_numpy((rng.standard_normal(shape) * scale).astype(np.float32))
    return x.to(torch.bfloat16).to(torch.float32).numpy()


def read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line)
    return rows


def closed_forms():
    out = {}
    for row in read_golden("closed_forms.txt"):
        k, v = row.split("=")
        out[k.strip()] = int(v.strip())
    return out


# ---------------------------------------------------------------------------
# INT8
# ---------------------------------------------------------------------------
def int8_expected_exact(row):
    """Codes and scale of one row by exact rational arithmetic + IEEE rounding."""
    amax = max(abs(Fraction(float(v))) for v in row)
    s = rn_f32(amax / 127)
    if s == 0:
        return [0] * len(row), 0.0
    codes = []
    for v in row:
        q = rn_f32(Fraction(float(v)) / s)
        c = round(q)  # half to even
        codes.append(max(-127, min(127, c)))
    return codes, float(s)


def check_int8_exact(int8_quantize, seed=0, rows=64, D=16):
    rng = np.random.default_rng(seed)
    x = bf16_values(rng, (rows, D))
    x[::7, 3] *= 40.0  # outlier channel
    x = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    codes, scales = int8_quantize(x)
    for i in range(rows):
        ec, es = int8_expected_exact(x[i])
        assert float(scales[i]) == es, (i, float(scales[i]), es)
        assert [int(c) for c in codes[i]] == ec, (i, codes[i], ec)


def all_finite_bf16_upto(m):
    """Every finite bf16 value v with |v| <= m (both signs, both zeros), as float32."""
    v = (np.arange(1 << 16, dtype=np.uint32) << 16).view(np.float32)
    return v[np.isfinite(v) & (np.abs(v) <= m)]


def check_int8_exhaustive_bf16(int8_quantize, maxima=(1.0, 15.875, 29952.0, 1.0005e-30)):
    """Every finite bf16 value up to a row maximum m, at several m (so several fixed
    scales fp32(m/127), one of them near the bottom of the fp32 normal range): the
    oracle's code of each value against exact rational arithmetic."""
    for m in maxima:
        m = float(torch.tensor([m]).to(torch.bfloat16).to(torch.float32)[0])
        vals = all_finite_bf16_upto(m)
        D = 32
        n = -(-len(vals) // (D - 1))
        body = np.zeros(n * (D - 1), np.float32)
        body[:len(vals)] = vals
        rows = np.empty((n, D), np.float32)
        rows[:, 0] = m  # every row's maximum, so every row has the scale fp32(m / 127)
        rows[:, 1:] = body.reshape(n, D - 1)
        codes, scales = int8_quantize(rows)
        s = rn_f32(Fraction(m) / 127)
        assert np.all(scales.astype(np.float64) == float(s)), m
        expect = {}
        for v in np.unique(vals):
            q = rn_f32(Fraction(float(v)) / s)
            expect[float(v)] = max(-127, min(127, round(q)))
        got = np.asarray(codes).astype(np.int64)[:, 1:].reshape(-1)[:len(vals)]
        want = np.array([expect[float(v)] for v in vals], dtype=np.int64)
        bad = np.nonzero(got != want)[0]
        assert bad.size == 0, (m, vals[bad[:5]], got[bad[:5]], want[bad[:5]])


def check_nvfp4_exhaustive_bf16(nvfp4_quantize, unpack_nibbles, cases=((1.0, 1.0), (3.0, 0.37), (448.0, 13.5))):
    """Every finite bf16 value up to a group maximum m, under global scale gs: the
    oracle's E4M3 scale of the group and E2M1 code of each value against exact
    rational arithmetic (fp32 steps by rn_f32, the E4M3 step by torch's cast, the
    E2M1 step by the nearest grid value with ties to the even code)."""
    grid = [Fraction(0), Fraction(1, 2), Fraction(1), Fraction(3, 2), Fraction(2), Fraction(3), Fraction(4), Fraction(6)]
    for m, gs in cases:
        m = float(torch.tensor([m]).to(torch.bfloat16).to(torch.float32)[0])
        gsf = Fraction(float(np.float32(gs)))
        vals = all_finite_bf16_upto(m)
        n = -(-len(vals) // 15)
        body = np.zeros(n * 15, np.float32)
        body[:len(vals)] = vals
        rows = np.empty((n, 16), np.float32)
        rows[:, 0] = m  # every group's maximum
        rows[:, 1:] = body.reshape(n, 15)
        codes, scales = nvfp4_quantize(rows, gs)
        t2 = rn_f32(rn_f32(Fraction(m) / 6) * gsf)
        sf = int(torch.tensor([float(t2)], dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8)[0])
        if float(t2) > 448:
            sf = 0x7E
        sd = Fraction(float(torch.tensor([sf], dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float32)[0]))
        assert np.all(np.asarray(scales).reshape(-1) == sf), (m, gs)
        assert sd > 0
        expect = {}
        for v in np.unique(vals):
            y = rn_f32(rn_f32(Fraction(float(v)) * gsf) / sd)
            a = abs(y)
            best = min(range(8), key=lambda i: (abs(a - grid[i]), i % 2))
            expect[float(v)] = best
        c = np.asarray(unpack_nibbles(codes)).astype(np.int64)[:, 1:].reshape(-1)[:len(vals)]
        want = np.array([expect[float(v)] | (8 if np.signbit(v) else 0) for v in vals], dtype=np.int64)
        bad = np.nonzero(c != want)[0]
        assert bad.size == 0, (m, gs, vals[bad[:5]], c[bad[:5]], want[bad[:5]])


def check_int8_ties(int8_quantize):
    """Rows whose scale is exactly 1/8 (amax = 127/8), so x/s = k + 1/2 exactly."""
    s = 0.125
    amax = 127 * s
    halves = [0.5, 1.5, 2.5, 3.5, -0.5, -1.5, -2.5, 125.5, 126.5, -126.5]
    expect = [0, 2, 2, 4, 0, -2, -2, 126, 126, -126]  # round half to even
    row = np.array([amax] + [h * s for h in halves], dtype=np.float32)
    codes, scale = int8_quantize(row[None, :])
    assert float(scale[0]) == s
    assert int(codes[0, 0]) == 127
    assert [int(c) for c in codes[0, 1:]] == expect, codes


def check_int8_invariants(int8_quantize, int8_dequantize, seed=1):
    rng = np.random.default_rng(seed)
    x = bf16_values(rng, (200, 256))
    x[:, [3, 77, 140, 201]] *= 8.0
    x = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    codes, s = int8_quantize(x)
    assert codes.dtype == np.int8
    assert codes.min() >= -127 and codes.max() <= 127
    xh = int8_dequantize(codes, s)
    err = np.abs(x.astype(np.float64) - xh)
    bound = (0.5 + 127 * 2.0 ** -24) * s.astype(np.float64)[:, None]
    assert np.all(err <= bound)
    i = np.argmax(np.abs(x), axis=1)
    assert np.all(np.abs(codes[np.arange(len(x)), i]) == 127)
    c2, s2 = int8_quantize(-x)
    assert np.array_equal(c2, -codes) and np.array_equal(s2, s)
    cz, sz = int8_quantize(np.zeros((3, 256), np.float32))
    assert not cz.any() and not sz.any()


# ---------------------------------------------------------------------------
# INT8 with one scale per 32 values
# ---------------------------------------------------------------------------
def check_int8_group_exact(int8_group_quantize, seed=10, rows=24, D=128):
    """Each group of 32 consecutive elements against exact rational arithmetic:
    groups of a row get magnitudes 2^-6 .. 2^6 apart, so a wrong grouping (a
    stride, a transposed reshape, a shared scale) changes scales and codes."""
    rng = np.random.default_rng(seed)
    mags = 2.0 ** rng.integers(-6, 7, (rows, D // 32))
    x = bf16_values(rng, (rows, D)) * np.repeat(mags, 32, axis=1)
    x[::5, 9] *= 30.0  # an outlier in group 0
    x = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).to(torch.float32).numpy()
    codes, scales = int8_group_quantize(x)
    assert codes.shape == x.shape and scales.shape == (rows, D // 32)
    for i in range(rows):
        for g in range(D // 32):
            ec, es = int8_expected_exact(x[i, 32 * g:32 * g + 32])
            assert float(scales[i, g]) == es, (i, g, float(scales[i, g]), es)
            assert [int(c) for c in codes[i, 32 * g:32 * g + 32]] == ec, (i, g)


def check_int8_group_hand_example(int8_group_quantize, int8_group_dequantize):
    """A 64-element row worked by hand: group 0 holds 127/8 and halves of 1/8
    (scale exactly 1/8, ties to even), group 1 holds 254 and the integers
    -31 .. -1 times 2 (scale exactly 2, codes -31 .. -1)."""
    halves = [0.5, 1.5, 2.5, 3.5, -0.5, -1.5, -2.5, 125.5, 126.5, -126.5]
    g0 = [127 / 8] + [h / 8 for h in halves] + [0.0] * 21
    g1 = [254.0] + [2.0 * k for k in range(-31, 0)]
    codes, scales = int8_group_quantize(np.array([g0 + g1], dtype=np.float32))
    assert [float(v) for v in scales[0]] == [0.125, 2.0]
    assert [int(c) for c in codes[0, :11]] == [127, 0, 2, 2, 4, 0, -2, -2, 126, 126, -126]
    assert not codes[0, 11:32].any()
    assert [int(c) for c in codes[0, 32:]] == [127] + list(range(-31, 0))
    back = int8_group_dequantize(np.arange(64, dtype=np.int8).reshape(1, 64), np.array([[0.5, 4.0]]))
    assert np.array_equal(back[0], np.concatenate([np.arange(32) * 0.5, np.arange(32, 64) * 4.0]))


def check_int8_group_invariants(int8_group_quantize, int8_group_dequantize, int8_quantize, seed=11):
    """Per-group error bound and maxima; an outlier channel moves only its own
    group; a row of 32 is the per-token codec's row."""
    rng = np.random.default_rng(seed)
    x = bf16_values(rng, (100, 256))
    codes, s = int8_group_quantize(x)
    xh = int8_group_dequantize(codes, s)
    err = np.abs(x.astype(np.float64) - xh)
    bound = (0.5 + 127 * 2.0 ** -24) * np.repeat(s.astype(np.float64), 32, axis=1)
    assert np.all(err <= bound)
    g = np.abs(x).reshape(100, 8, 32).argmax(axis=2)
    assert np.all(np.abs(codes.reshape(100, 8, 32)[np.arange(100)[:, None], np.arange(8)[None, :], g]) == 127)
    y = x.copy()
    y[:, 77] *= 50.0  # channel 77 is in group 2
    cy, sy = int8_group_quantize(y)
    keep = [k for k in range(8) if k != 2]
    assert np.array_equal(sy[:, keep], s[:, keep])
    assert np.array_equal(cy.reshape(100, 8, 32)[:, keep], codes.reshape(100, 8, 32)[:, keep])
    c32, s32 = int8_quantize(x[:, :32])
    c1, s1 = int8_group_quantize(x[:, :32])
    assert np.array_equal(c1, c32) and np.array_equal(s1[:, 0], s32)


# ---------------------------------------------------------------------------
# E4M3 / E2M1 / NVFP4
# ---------------------------------------------------------------------------
def torch_e4m3_values():
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float32).numpy().astype(np.float64)


def check_e4m3_decode(e4m3_value):
    ours = e4m3_value(np.arange(256, dtype=np.uint8))
    ref = torch_e4m3_values()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def check_e4m3_encode(e4m3_encode_satfinite, seed=2):
    ref_vals = torch_e4m3_values()[:0x7F]
    mids = (ref_vals[:-1] + ref_vals[1:]) / 2
    rng = np.random.default_rng(seed)
    t = np.concatenate([ref_vals, mids, rng.uniform(0, 448, 20000), np.exp(rng.uniform(-12, 6, 20000)),
                        [2.0 ** -10, 2.0 ** -11, 3 * 2.0 ** -11]])
    t = t.astype(np.float32).astype(np.float64)
    ours = e4m3_encode_satfinite(t)
    ref = torch.from_numpy(t.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref), np.nonzero(ours != ref)
    big = e4m3_encode_satfinite(np.array([448.0, 449.0, 470.0, 1e6]))
    assert list(big) == [0x7E] * 4


def check_e2m1_grid(e2m1_value):
    golden = [float(v) for v in read_golden("e2m1_grid.txt")]
    assert list(e2m1_value(np.arange(8))) == golden
    assert list(e2m1_value(np.arange(8, 16))) == [-v for v in golden]


def check_e2m1_ties(e2m1_encode):
    # midpoints between neighbours go to the code with mantissa bit 0 (even code)
    y = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -5.0, 7.0, 100.0, 0.3, -0.1, -0.0, 0.0, 5.5])
    expect = [0, 2, 2, 4, 4, 6, 6, 8, 14, 7, 7, 1, 8, 8, 0, 7]
    assert [int(c) for c in e2m1_encode(y)] == expect


def check_nibble_order(pack_nibbles):
    for row in read_golden("nibble_order.txt"):
        lhs, rhs = row.split("->")
        codes = np.array([int(t, 16) for t in lhs.split()], dtype=np.uint8)
        packed = [int(t, 16) for t in rhs.split()]
        assert [int(b) for b in pack_nibbles(codes)] == packed


def nvfp4_expected_exact(row, gs):
    """One row by exact rationals: fp32 steps by rn_f32, the E4M3 step by torch's
    cast, the E2M1 step by brute-force nearest with ties to the even code."""
    gs = Fraction(float(np.float32(gs)))
    grid = [Fraction(0), Fraction(1, 2), Fraction(1), Fraction(3, 2), Fraction(2), Fraction(3), Fraction(4), Fraction(6)]
    codes, scales = [], []
    for g0 in range(0, len(row), 16):
        grp_f = [float(v) for v in row[g0:g0 + 16]]
        grp = [Fraction(v) for v in grp_f]
        amax = max(abs(v) for v in grp)
        t = rn_f32(amax / 6)
        t2 = rn_f32(t * gs)
        sf = int(torch.tensor([float(t2)], dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8)[0])
        if float(t2) > 448:
            sf = 0x7E
        sd = Fraction(float(torch.tensor([sf], dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float32)[0]))
        scales.append(sf)
        for v, vf in zip(grp, grp_f):
            if sd == 0:
                codes.append(0)
                continue
            y = rn_f32(rn_f32(v * gs) / sd)
            a = abs(y)
            best = min(range(8), key=lambda i: (abs(a - grid[i]), i % 2))
            neg = y < 0 or (y == 0 and math.copysign(1.0, vf) < 0)
            codes.append(best | (8 if neg else 0))
    return codes, scales


def check_nvfp4_exact(nvfp4_quantize, unpack_nibbles, seed=3, gs_list=(1.0, None)):
    rng = np.random.default_rng(seed)
    x = bf16_values(rng, (24, 64))
    x[0, :16] = 0.0
    x[1, 16:32] = 1e-4
    x[2, 5] = -0.0
    x[3, :] *= 30.0
    x = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    for gs in gs_list:
        if gs is None:
            gs = float(np.float32(448.0 * 6.0) / np.float32(np.max(np.abs(x))))
        codes, scales = nvfp4_quantize(x, gs)
        c = unpack_nibbles(codes)
        for i in range(x.shape[0]):
            ec, es = nvfp4_expected_exact(x[i], gs)
            assert [int(v) for v in scales[i]] == es, (gs, i)
            assert [int(v) for v in c[i]] == ec, (gs, i)


def check_nvfp4_invariants(nvfp4_quantize, nvfp4_dequantize, e4m3_value, seed=4):
    rng = np.random.default_rng(seed)
    x = bf16_values(rng, (100, 256))
    for gs in (1.0, float(np.float32(2688.0) / np.float32(np.max(np.abs(x))))):
        codes, scales = nvfp4_quantize(x, gs)
        xh = nvfp4_dequantize(codes, scales, gs)
        sd = e4m3_value(scales).repeat(16, axis=1) / np.float64(np.float32(gs))
        err = np.abs(x - xh)
        # largest gap of the E2M1 grid is 2 (between 4 and 6); within a group whose
        # scale was rounded, |y| <= 6 * (1 + 2^-4); so the error is at most one grid gap.
        assert np.all(err <= 2.0 * sd + 1e-12)
        small = np.abs(x) * np.float64(np.float32(gs)) / np.maximum(e4m3_value(scales).repeat(16, axis=1), 1e-30) <= 4.0
        assert np.all(err[small] <= 0.5 * sd[small] * (1 + 2.0 ** -18) + 1e-12)


# ---------------------------------------------------------------------------
# attention
# ---------------------------------------------------------------------------
def tiny_case(rng, G=3, L=17, D=8):
    q = rng.standard_normal((G, D))
    k = rng.standard_normal((L, D))
    v = rng.standard_normal((L, D))
    return q, k, v


def check_attend_brute(attend, attend_brute, seed=5):
    rng = np.random.default_rng(seed)
    for (G, L, D) in [(1, 1, 8), (3, 17, 8), (6, 40, 16), (4, 33, 16), (2, 5, 8)]:
        q, k, v = tiny_case(rng, G, L, D)
        sm = 1.0 / math.sqrt(D)
        o, s = attend(q, k, v, sm)
        ob, sb = attend_brute(q.tolist(), k.tolist(), v.tolist(), sm)
        assert np.max(np.abs(o - np.array(ob))) < 1e-12
        assert np.max(np.abs(s - np.array(sb))) < 1e-12


def check_split_merge(attend, attend_split, seed=6):
    rng = np.random.default_rng(seed)
    q, k, v = tiny_case(rng, 6, 96, 16)
    sm = 0.25
    o, s = attend(q, k, v, sm)
    for bounds in ([(0, 96)], [(0, 48), (48, 96)], [(0, 16), (16, 17), (17, 80), (80, 96)],
                   [(0, 0), (0, 96), (96, 96)], [(i, i + 16) for i in range(0, 96, 16)]):
        om, sm_ = attend_split(q, k, v, sm, bounds)
        assert np.max(np.abs(om - o)) < 1e-12
        assert np.max(np.abs(sm_ - s)) < 1e-12


def check_merge_not_average(attend, merge, seed=7):
    """The page's warning: averaging partial outputs is not the attention result."""
    rng = np.random.default_rng(seed)
    q, k, v = tiny_case(rng, 2, 64, 8)
    k[:32] *= 3.0
    o1, s1 = attend(q, k[:32], v[:32], 1.0)
    o2, s2 = attend(q, k[32:], v[32:], 1.0)
    o, _ = attend(q, k, v, 1.0)
    om, _ = merge(np.stack([o1, o2]), np.stack([s1, s2]))
    assert np.max(np.abs(om - o)) < 1e-12
    assert np.max(np.abs((o1 + o2) / 2 - o)) > 1e-3


def check_attention_invariants(attend, probabilities, seed=8):
    rng = np.random.default_rng(seed)
    q, k, v = tiny_case(rng, 6, 50, 16)
    p = probabilities(q, k, 0.3)
    assert np.max(np.abs(p.sum(axis=1) - 1.0)) < 1e-14
    # identical keys -> mean of V
    kk = np.repeat(k[:1], 50, axis=0)
    o, _ = attend(q, kk, v, 0.3)
    assert np.max(np.abs(o - v.mean(axis=0)[None, :])) < 1e-12
    # single token -> that V row, exactly
    o, s = attend(q, k[:1], v[:1], 0.3)
    assert np.array_equal(o, np.repeat(v[:1], 6, axis=0))
    assert np.allclose(s, 0.3 * (q @ k[0]), atol=1e-14)
    # empty context
    o, s = attend(q, k[:0], v[:0], 0.3)
    assert not o.any() and np.all(np.isneginf(s))
    # identical queries in a group -> identical outputs
    qq = np.repeat(q[:1], 6, axis=0)
    o, _ = attend(qq, k, v, 0.3)
    assert np.max(np.abs(o - o[:1])) == 0.0
    # one dominant logit -> that row of V
    kd = k.copy()
    kd[17] = q[0] * 1e3
    o, _ = attend(q[:1], kd, v, 1.0)
    assert np.max(np.abs(o[0] - v[17])) < 1e-12


def place_logical_rows(pool, block_table_row, rows, page_size):
    """Write a sequence's logical rows into a [num_pages, Hkv, P, ...] pool by
    the page mapping itself, token by token: token t goes to page
    block_table_row[t // P], row t % P (the test's own restatement; the oracle's
    layout functions are not used)."""
    for t in range(len(rows)):
        pool[int(block_table_row[t // page_size]), :, t % page_size] = rows[t]


def check_verify(paged_verify, seed=9):
    """Causal verification against pure-Python attention over each query token's
    visible prefix (tiny pools, brute force), and its single-token case against
    decode-style attention over the whole sequence.  The pools are filled with
    random bytes and then each sequence's logical rows are placed page by page;
    the brute force reads the logical rows, so a slip in the oracle's page
    mapping (page and row swapped, a wrong block-table index) fails here."""
    from oracle import brute

    rng = np.random.default_rng(seed)
    P, Hkv, G, D = 4, 2, 3, 8
    for (lens, T) in [([9, 5], 3), ([4], 4), ([2, 7], 3), ([6], 1), ([13], 2)]:
        B = len(lens)
        npages = sum(-(-L // P) for L in lens) + 2  # two pages no sequence uses
        perm = rng.permutation(npages)
        bt = np.full((B, max(-(-L // P) for L in lens)), -1, dtype=np.int32)
        o = 0
        for b, L in enumerate(lens):
            n = -(-L // P)
            bt[b, :n] = perm[o:o + n]
            o += n
        # INT8 codes with per-row scales; the brute force dequantizes by c * s itself
        kc = rng.integers(-127, 128, (npages, Hkv, P, D)).astype(np.int8)
        vc = rng.integers(-127, 128, (npages, Hkv, P, D)).astype(np.int8)
        ks = rng.uniform(0.001, 0.05, (npages, Hkv, P)).astype(np.float32)
        vs = rng.uniform(0.001, 0.05, (npages, Hkv, P)).astype(np.float32)
        logical = []
        for b, L in enumerate(lens):
            lk = rng.integers(-127, 128, (L, Hkv, D)).astype(np.int8)
            lv = rng.integers(-127, 128, (L, Hkv, D)).astype(np.int8)
            lks = rng.uniform(0.001, 0.05, (L, Hkv)).astype(np.float32)
            lvs = rng.uniform(0.001, 0.05, (L, Hkv)).astype(np.float32)
            for pool, rows in ((kc, lk), (vc, lv), (ks, lks), (vs, lvs)):
                place_logical_rows(pool, bt[b], rows, P)
            logical.append((lk.astype(np.float64) * lks.astype(np.float64)[..., None],
                            lv.astype(np.float64) * lvs.astype(np.float64)[..., None]))
        pools = {"k_codes": kc.view(np.uint8), "v_codes": vc.view(np.uint8), "k_scales": ks, "v_scales": vs}
        q = rng.standard_normal((B, T, G * Hkv, D))
        sm = 1.0 / math.sqrt(D)
        out, lse = paged_verify("int8", pools, q, bt, np.array(lens), sm, page_size=P)
        for b, L in enumerate(lens):
            kx, vx = logical[b]
            for i in range(T):
                vis = max(0, L - T + i + 1)
                for h in range(Hkv):
                    kr = [list(kx[t, h]) for t in range(vis)]
                    vr = [list(vx[t, h]) for t in range(vis)]
                    qs = q[b, i, h * G:(h + 1) * G].tolist()
                    if vis == 0:
                        assert np.all(out[b, i, h * G:(h + 1) * G] == 0) and np.all(np.isneginf(lse[b, i, h * G:(h + 1) * G]))
                        continue
                    ob, sb = brute.attend_brute(qs, kr, vr, sm)
                    assert np.max(np.abs(out[b, i, h * G:(h + 1) * G] - np.array(ob))) < 1e-12
                    assert np.max(np.abs(lse[b, i, h * G:(h + 1) * G] - np.array(sb))) < 1e-12


def check_paged_decode(paged_decode, seed=13):
    """Decode over hand-placed pools (INT8 per-row scales, NVFP4 with a global
    scale, BF16) against pure-Python attention over the logical rows, each
    dequantized by its format's definition written out here: c * s; e2m1(c) *
    e4m3(sf) / gs with the E2M1 grid and the E4M3 value read from the golden grid
    and torch's float8_e4m3fn; the bf16 bits widened."""
    from oracle import brute

    rng = np.random.default_rng(seed)
    P, Hkv, G, D = 4, 2, 2, 32
    lens = [11, 3, 0, 8]
    B = len(lens)
    npages = sum(-(-L // P) for L in lens) + 1
    perm = rng.permutation(npages)
    bt = np.zeros((B, max(1, max(-(-L // P) for L in lens))), dtype=np.int32)
    o = 0
    for b, L in enumerate(lens):
        n = -(-L // P)
        bt[b, :n] = perm[o:o + n]
        o += n
    grid = [float(x) for x in read_golden("e2m1_grid.txt")]
    e4 = torch_e4m3_values()
    q = rng.standard_normal((B, G * Hkv, D))
    sm = 1.0 / math.sqrt(D)
    for fmt in ("int8", "nvfp4", "bf16"):
        rb = {"int8": D, "nvfp4": D // 2, "bf16": 2 * D}[fmt]
        pools = {}
        logical = [[None, None] for _ in lens]
        for which, name in enumerate(("k", "v")):
            codes = rng.integers(0, 256, (npages, Hkv, P, rb)).astype(np.uint8)
            if fmt == "int8":
                scales = rng.uniform(0.001, 0.05, (npages, Hkv, P)).astype(np.float32)
            elif fmt == "nvfp4":
                scales = rng.integers(0, 0x7F, (npages, Hkv, P, D // 16)).astype(np.uint8)
            else:
                scales = None
            for b, L in enumerate(lens):
                lc = rng.integers(0, 256, (L, Hkv, rb)).astype(np.uint8)
                if fmt == "bf16":  # finite bf16 values: exponent field kept below all-ones
                    lc[..., 1::2] &= 0xBF
                place_logical_rows(codes, bt[b], lc, P)
                x = np.zeros((L, Hkv, D))
                if fmt == "int8":
                    ls = rng.uniform(0.001, 0.05, (L, Hkv)).astype(np.float32)
                    place_logical_rows(scales, bt[b], ls, P)
                    x = lc.view(np.int8).astype(np.float64) * ls.astype(np.float64)[..., None]
                elif fmt == "nvfp4":
                    ls = rng.integers(0, 0x7F, (L, Hkv, D // 16)).astype(np.uint8)
                    place_logical_rows(scales, bt[b], ls, P)
                    for t in range(L):
                        for h in range(Hkv):
                            for d in range(D):
                                nib = (int(lc[t, h, d // 2]) >> (4 * (d % 2))) & 0xF
                                val = (-1.0 if nib & 8 else 1.0) * grid[nib & 7]
                                x[t, h, d] = val * float(e4[int(ls[t, h, d // 16])]) / 3.5
                else:
                    x = (lc.view(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
                logical[b][which] = x
            pools[name + "_codes"], pools[name + "_scales"] = codes, scales
        if fmt == "nvfp4":
            pools["k_global_scale"] = pools["v_global_scale"] = 3.5
        out, lse = paged_decode(fmt, pools, q, bt, np.array(lens), sm, page_size=P)
        for b, L in enumerate(lens):
            kx, vx = logical[b]
            for h in range(Hkv):
                rows = slice(h * G, (h + 1) * G)
                if L == 0:
                    assert np.all(out[b, rows] == 0) and np.all(np.isneginf(lse[b, rows]))
                    continue
                ob, sb = brute.attend_brute(q[b, rows].tolist(), kx[:, h].tolist(), vx[:, h].tolist(), sm)
                assert np.max(np.abs(out[b, rows] - np.array(ob))) < 1e-9 * max(1.0, np.max(np.abs(ob))), (fmt, b, h)
                assert np.max(np.abs(lse[b, rows] - np.array(sb))) < 1e-9 * max(1.0, np.max(np.abs(sb))), (fmt, b, h)


# ---------------------------------------------------------------------------
# pool layout (the page mapping)
# ---------------------------------------------------------------------------
def _expand_ranges(tokens):
    out = []
    for tok in tokens:
        if ".." in tok:
            a, b = tok.split("..")
            out.extend(range(int(a), int(b) + 1))
        else:
            out.append(int(tok))
    return out


def check_token_slots(token_slots):
    """Slot lists worked by hand (tests/golden/page_mapping.txt)."""
    rows = read_golden("page_mapping.txt")
    assert len(rows) >= 6
    for row in rows:
        lhs, rhs = row.split("->")
        P, bt, L = [s.strip() for s in lhs.split("|")]
        table = np.array([int(x) for x in bt.split()], dtype=np.int32)
        got = [int(s) for s in token_slots(table, int(L), int(P))]
        assert got == _expand_ranges(rhs.split()), (row, got)


def coordinate_pool(num_pages, hkv, P):
    """A pool whose cell (page, head, row) holds the triple (page, head, row)."""
    pool = np.zeros((num_pages, hkv, P, 3), np.int64)
    for p in range(num_pages):
        for h in range(hkv):
            for r in range(P):
                pool[p, h, r] = (p, h, r)
    return pool


def check_gather_scatter(gather_rows, scatter_rows):
    """Row gather / scatter on pools whose cells name their own coordinates; the
    expected cells are worked by hand from slot = page * P + row."""
    pool = coordinate_pool(20, 3, 16)
    # slot 37 = page 2 row 5; 2 = page 0 row 2; 16 = page 1 row 0; 63 = page 3 row 15; 305 = page 19 row 1
    got = gather_rows(pool, np.array([37, 2, 16, 63, 305]), 1)
    assert np.array_equal(got, [[2, 1, 5], [0, 1, 2], [1, 1, 0], [3, 1, 15], [19, 1, 1]]), got
    dst = np.full((20, 3, 16, 2), -1, np.int64)
    scatter_rows(dst, np.array([37, 2]), 2, np.array([[10, 11], [20, 21]]))
    assert dst[2, 2, 5].tolist() == [10, 11] and dst[0, 2, 2].tolist() == [20, 21]
    assert int((dst != -1).sum()) == 4
    # a scale pool [pages, heads, P] with P = 4: slot 5 = page 1 row 1, slot 11 = page 2 row 3
    sp = np.zeros((6, 2, 4))
    scatter_rows(sp, np.array([5, 11]), 0, np.array([1.5, 2.5]))
    assert sp[1, 0, 1] == 1.5 and sp[2, 0, 3] == 2.5 and np.count_nonzero(sp) == 2
    assert gather_rows(sp, np.array([11, 5, 0]), 0).tolist() == [2.5, 1.5, 0.0]


def check_group_major(group_major_scales):
    """The device's group-major per-32 scales [pages, heads, groups, P] read as
    [pages, heads, P, groups]: cells worked by hand on a 2 x 2 x 3 x 16 array
    whose cell (p, h, g, r) holds p*10000 + h*1000 + g*100 + r."""
    a = np.zeros((2, 2, 3, 16))
    for p in range(2):
        for h in range(2):
            for g in range(3):
                for r in range(16):
                    a[p, h, g, r] = p * 10000 + h * 1000 + g * 100 + r
    out = group_major_scales(a)
    assert out.shape == (2, 2, 16, 3)
    assert out[1, 0, 7, 2] == 10207 and out[0, 1, 15, 0] == 1015 and out[1, 1, 0, 1] == 11100
    assert out[0, 0, 3].tolist() == [3, 103, 203]  # one slot row: its three group scales
