"""Reference codecs for the KV-cache formats — TEST INFRASTRUCTURE ONLY (oracle).

Everything here is written from the format definitions on the pages, as plain
numpy on exact values; nothing is shared with the CUDA library.

Formats
-------
INT8   One signed 8-bit code per element plus one fp32 scale per (token, KV head),
       scale = absmax / 127.  Source: "half-the-memory-int8-kv-cache" page,
       section "An 8-bit cache was already available" (vLLM's
       int8_per_token_head format: 8-bit integers with a shared 32-bit scale,
       520 bytes per token per head at D = 256) and section "Is 8 bits enough?"
       (one scale per 256 values).  The symmetric clamp to [-127, 127] and the
       round-to-nearest step follow the gllm page, section "Quantization Design"
       (amax / 127, round-to-nearest, clamped to [-127, 127]).  The tie rule
       (round half to even) and "scale in fp32" are the plainest reading of the
       problem statement and are used on both sides.
NVFP4  E2M1 element codes (sign + magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6), two per
       byte with element 2j in the low nibble and 2j+1 in the high nibble, one
       FP8 E4M3 scale per 16 elements and an fp32 per-tensor global scale;
       decode = fp4 * group_scale / global_scale.  Source: "Building an NVFP4 KV
       cache for a hybrid Qwen model" page, section "How 2,048 bytes became 576";
       the writer steps (group maxima -> FP8 scales -> E2M1 rounding -> pack
       pairs) are from its section "Writing and reading the packed cache".
INT8/32  The same INT8 codec applied to each group of 32 consecutive elements of
       a row instead of the whole row: one fp32 scale per 32 values, scale =
       absmax of the group / 127.  Source: "half-the-memory-int8-kv-cache" page,
       section "Is 8 bits enough?" (llama.cpp's Q8_0 KV format keeps one scale per
       32 values; one per 256 is cheaper but more exposed to outlier channels).
       The page does not give the scale's type or the rounding; the reading is
       the per-token codec's (fp32 scale, fp32 quotient, ties to even).
BF16   Values stored as bfloat16 (the comparison format of the pages' BF16 FA2
       runs); "decoding" is widening.

Readings where the pages leave a step open:
  * INT8 quotient: q = fp32(x / s) with IEEE fp32 division by the stored scale,
    then round half to even, then clamp to [-127, 127]; s == 0 gives all-zero codes.
  * NVFP4 encoder: t = fp32(amax_g / 6), t2 = fp32(t * gs), scale byte =
    E4M3(t2) rounded to nearest-even and saturated to 448; y = fp32(fp32(x * gs)
    / sd) with sd the decoded scale; code = E2M1(y) nearest-even, saturated to 6;
    sign bit = sign bit of x (so -0.1 -> 0x8); sd == 0 gives all codes 0x0.
"""
from __future__ import annotations

import numpy as np

# ---------------------------------------------------------------------------
# INT8, per token and KV head
# ---------------------------------------------------------------------------
INT8_QMAX = 127


def int8_quantize(x):
    """Quantize rows of ``x`` ([..., D], float32 holding bf16 values).

    Returns ``(codes int8 [..., D], scale float32 [...])``.

    scale = fp32(absmax / 127) ("half-the-memory-int8-kv-cache", section "An
    8-bit cache was already available"); codes = clamp(rne(fp32(x / scale)),
    -127, 127) ("gllm", section "Quantization Design").
    """
    x = np.asarray(x, dtype=np.float32)
    amax = np.max(np.abs(x), axis=-1)
    scale = (amax / np.float32(INT8_QMAX)).astype(np.float32)  # IEEE fp32 division
    safe = np.where(scale > 0, scale, np.float32(1.0)).astype(np.float32)
    q = (x / safe[..., None]).astype(np.float32)  # IEEE fp32 division
    codes = np.clip(np.rint(q), -INT8_QMAX, INT8_QMAX)  # np.rint: ties to even
    codes = np.where(scale[..., None] > 0, codes, 0)
    return codes.astype(np.int8), scale


def int8_dequantize(codes, scale):
    """x_hat = code * scale, exact in float64."""
    return np.asarray(codes, dtype=np.float64) * np.asarray(scale, dtype=np.float64)[..., None]


# ---------------------------------------------------------------------------
# INT8 with one scale per 32 values
# ---------------------------------------------------------------------------
INT8_GROUP = 32


def int8_group_quantize(x, group=INT8_GROUP):
    """Quantize rows of ``x`` ([..., D], D a multiple of ``group``) with one INT8
    scale per ``group`` consecutive elements ("half-the-memory-int8-kv-cache",
    section "Is 8 bits enough?").

    Returns ``(codes int8 [..., D], scales float32 [..., D / group])``: each group
    is coded exactly as ``int8_quantize`` codes a row.
    """
    x = np.asarray(x, dtype=np.float32)
    D = x.shape[-1]
    assert D % group == 0
    codes, scales = int8_quantize(x.reshape(x.shape[:-1] + (D // group, group)))
    return codes.reshape(x.shape), scales


def int8_group_dequantize(codes, scales, group=INT8_GROUP):
    """x_hat = code * scale of its group, exact in float64."""
    c = np.asarray(codes, dtype=np.float64)
    D = c.shape[-1]
    g = c.reshape(c.shape[:-1] + (D // group, group)) * np.asarray(scales, dtype=np.float64)[..., None]
    return g.reshape(c.shape)


# ---------------------------------------------------------------------------
# FP8 E4M3 (the NVFP4 group-scale format)
# ---------------------------------------------------------------------------
# Layout of a byte: sign (bit 7) | exponent (bits 6..3, bias 7) | mantissa (bits 2..0).
# exponent 0 -> subnormal  mantissa/8 * 2^-6;  exponent 1..15 -> (1 + mantissa/8) * 2^(e-7);
# exponent 15 with mantissa 7 is NaN; there is no infinity; largest finite = 448.
E4M3_MAX = 448.0


def e4m3_value(byte):
    """Decode E4M3 bytes (array of uint8) to float64 (NaN for 0x7F / 0xFF)."""
    b = np.asarray(byte, dtype=np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = (b & 0x7).astype(np.float64)
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    mag = np.where((e == 15) & ((b & 0x7) == 7), np.nan, mag)
    return sign * mag


# the 127 non-negative finite values, codes 0x00..0x7E, in increasing order
_E4M3_POS = e4m3_value(np.arange(0x7F, dtype=np.uint8))


def _round_to_grid(a, grid):
    """Index of the grid value nearest to each a >= 0; ties go to the even index;
    values beyond the last grid point saturate to it.  ``grid`` is increasing and
    index parity equals the format's mantissa lsb (true for E4M3 and E2M1)."""
    a = np.asarray(a, dtype=np.float64)
    hi = np.searchsorted(grid, a, side="left")  # first grid >= a
    hi = np.clip(hi, 0, len(grid) - 1)
    lo = np.clip(hi - 1, 0, len(grid) - 1)
    d_lo = np.abs(a - grid[lo])
    d_hi = np.abs(grid[hi] - a)
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    idx = np.where(pick_hi, hi, lo)
    idx = np.where(a >= grid[-1], len(grid) - 1, idx)
    return idx.astype(np.int64)


def e4m3_encode_satfinite(t):
    """Round float64 values to E4M3 bytes: nearest, ties to even, |t| > 448 -> 448."""
    t = np.asarray(t, dtype=np.float64)
    idx = _round_to_grid(np.abs(t), _E4M3_POS)
    sign = np.where(np.signbit(t), 0x80, 0)
    return (idx | sign).astype(np.uint8)


# ---------------------------------------------------------------------------
# FP4 E2M1 and the NVFP4 packed record
# ---------------------------------------------------------------------------
# Magnitudes of the eight non-negative codes 0..7, as listed on the NVFP4 page.
E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
NVFP4_GROUP = 16


def e2m1_value(code):
    """Decode 4-bit E2M1 codes (sign = bit 3) to float64."""
    c = np.asarray(code, dtype=np.int64)
    return np.where(c & 0x8, -1.0, 1.0) * E2M1_GRID[c & 0x7]


def e2m1_encode(y):
    """Round float64 values to 4-bit E2M1 codes: nearest, ties to even, saturate
    at 6; the sign bit copies the sign bit of y (so -0.1 becomes 0x8)."""
    y = np.asarray(y, dtype=np.float64)
    idx = _round_to_grid(np.abs(y), E2M1_GRID)
    return (idx | np.where(np.signbit(y), 0x8, 0)).astype(np.uint8)


def pack_nibbles(codes):
    """[..., D] 4-bit codes -> [..., D/2] bytes, element 2j low nibble, 2j+1 high."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def unpack_nibbles(packed):
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def nvfp4_quantize(x, global_scale):
    """Quantize rows of ``x`` ([..., D], float32 holding bf16 values) to NVFP4.

    Returns ``(codes uint8 [..., D/2], scales uint8 [..., D/16])``.  Steps in the
    order of the NVFP4 page's writer ("Writing and reading the packed cache"):
    group maxima, FP8 E4M3 scales, E2M1 rounding, packing of pairs.
    """
    x = np.asarray(x, dtype=np.float32)
    gs = np.float32(global_scale)
    D = x.shape[-1]
    assert D % NVFP4_GROUP == 0
    xg = x.reshape(x.shape[:-1] + (D // NVFP4_GROUP, NVFP4_GROUP))
    amax = np.max(np.abs(xg), axis=-1)
    t = (amax / np.float32(6.0)).astype(np.float32)  # fp32 division
    t2 = (t * gs).astype(np.float32)  # fp32 multiply
    sf = e4m3_encode_satfinite(t2.astype(np.float64))
    sd = e4m3_value(sf).astype(np.float32)  # exact in fp32
    safe = np.where(sd > 0, sd, np.float32(1.0)).astype(np.float32)
    y = ((xg * gs).astype(np.float32) / safe[..., None]).astype(np.float32)
    codes = e2m1_encode(y.astype(np.float64))
    codes = np.where(sd[..., None] > 0, codes, 0).astype(np.uint8)
    return pack_nibbles(codes.reshape(x.shape)), sf


def nvfp4_dequantize(codes, scales, global_scale):
    """x_hat = fp4 * group_scale / global_scale (NVFP4 page, "How 2,048 bytes
    became 576"), in float64."""
    vals = e2m1_value(unpack_nibbles(codes))
    D = vals.shape[-1]
    vg = vals.reshape(vals.shape[:-1] + (D // NVFP4_GROUP, NVFP4_GROUP))
    sd = e4m3_value(scales)
    return (vg * sd[..., None] / np.float64(np.float32(global_scale))).reshape(vals.shape)


def nvfp4_tensor_global_scale(x):
    """The standalone-test choice of global scale on the NVFP4 page ("Some
    standalone numerical tests instead choose a global scale from the tensor's
    absolute maximum"): gs = 448 * 6 / amax(tensor), so that the tensor's largest
    group maps onto the largest E4M3 scale times the largest E2M1 value.  The
    constant 448 * 6 is a reading; the page names only 'absolute maximum'."""
    amax = float(np.max(np.abs(np.asarray(x, dtype=np.float32))))
    return np.float32(1.0) if amax == 0.0 else np.float32(np.float32(E4M3_MAX * 6.0) / np.float32(amax))


# ---------------------------------------------------------------------------
# bf16 helpers (the comparison format and the query dtype)
# ---------------------------------------------------------------------------
def bf16_bits_to_f32(bits):
    """uint16 bfloat16 bit patterns -> float32 (exact widening)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32)
