"""Rotation of K/V rows before 4-bit quantization — TEST INFRASTRUCTURE ONLY (oracle).

Source: "Smaller KV cache, faster first token", section "Lever one: 4-bit KV
with TurboQuant": the K and V vectors are rotated before they are quantized, so
that outliers spread over all dimensions and 4 bits per value lose little.

The page fixes neither the rotation nor its arithmetic.  The reading used on
both sides:
  * R(x) = D^(-1/2) * H_D (s * x): elementwise signs s, then the Sylvester
    Hadamard matrix H_D (H_1 = [1], H_2n = [[H_n, H_n], [H_n, -H_n]]), then the
    normalisation.  R is orthogonal: R(q) . R(k) = q . k, so attention scores
    are unchanged when q and K are both rotated, and the output of attention
    over rotated V is R(o), undone by R^-1(y) = s * (D^(-1/2) H_D y).
  * s_i = -1 if bit 31 of ((i + 1) * 2654435761 mod 2^32) is set, else +1
    (Knuth's multiplicative hash, The Art of Computer Programming vol. 3,
    section 6.4), the same for every head and token.
  * The stored values are the rotation computed in fp32 as a butterfly network,
    stages h = 1, 2, 4, ..., D/2 in that order, each pair (a, b) at positions
    (i, i + h) with bit h of i clear becoming (a + b, a - b); then one multiply
    by fp32(D^(-1/2)) (exact for D = 256); then rounding to the output type
    (bf16: nearest, ties to even).  Forward: signs first; inverse: signs last.

``hadamard`` and ``rotate_exact`` state the definition in float64 (the pins
check the butterfly against them); ``rotate_fp32`` is the arithmetic the CUDA
kernel follows.
"""
from __future__ import annotations

import numpy as np
import torch


def signs(D):
    """The sign vector s (float64, +-1) of length D."""
    i = np.arange(D, dtype=np.uint64)
    h = ((i + np.uint64(1)) * np.uint64(2654435761)) & np.uint64(0xFFFFFFFF)
    return np.where((h >> np.uint64(31)) & np.uint64(1), -1.0, 1.0)


def hadamard(D):
    """Sylvester Hadamard matrix H_D (float64), D a power of two."""
    assert D >= 1 and D & (D - 1) == 0
    H = np.ones((1, 1))
    while H.shape[0] < D:
        H = np.block([[H, H], [H, -H]])
    return H


def rotate_exact(x, inverse=False):
    """R(x) (or R^-1(x)) of the rows of x [..., D] in float64, by the matrix."""
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    H = hadamard(D) / np.sqrt(D)
    s = signs(D)
    if inverse:
        return (x @ H.T) * s
    return (x * s) @ H.T


def _butterfly_fp32(y):
    """The fp32 butterfly network on the last axis, stages h = 1, 2, ..., D/2."""
    y = np.array(y, dtype=np.float32, copy=True)
    D = y.shape[-1]
    h = 1
    while h < D:
        idx = np.arange(D)
        lo = idx[(idx & h) == 0]
        a = y[..., lo].copy()
        b = y[..., lo + h].copy()
        y[..., lo] = (a + b).astype(np.float32)
        y[..., lo + h] = (a - b).astype(np.float32)
        h *= 2
    return y


def rotate_fp32(x, inverse=False, out="bf16"):
    """The stored rotation: fp32 butterfly as described above, rounded to `out`
    ("bf16": float32 array holding bf16 values; "f32": float32)."""
    x = np.asarray(x, dtype=np.float32)
    D = x.shape[-1]
    s = signs(D).astype(np.float32)
    norm = np.float32(1.0 / np.sqrt(D))
    if inverse:
        y = _butterfly_fp32(x)
        y = (y * norm).astype(np.float32) * s
    else:
        y = _butterfly_fp32(x * s)
        y = (y * norm).astype(np.float32)
    y = y.astype(np.float32)
    if out == "bf16":
        return torch.from_numpy(np.ascontiguousarray(y)).to(torch.bfloat16).to(torch.float32).numpy()
    return y
