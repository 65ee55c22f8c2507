"""Seeded synthetic decode workloads — input generation only.

This module draws random inputs with the shapes, value distributions and page
layouts of the decode workloads the pages describe (24 query / 4 KV heads of
dimension 256, i.e. 6:1 GQA; a batch-64 serving mix at 32 / 8 heads of 128; a
long-context NVFP4 batch), and nothing else: it holds none of the method's
arithmetic (no quantization, no attention).  Both the CUDA path (through the
package) and the CPU oracle (in the tests) are fed from it.

All randomness is numpy ``Generator(PCG64)`` seeded from (seed, purpose, index);
values are drawn in float32 and rounded to bfloat16 (round-to-nearest-even, by
torch), so every array below holds bf16-representable float32 values.

Workload recipes (name -> what is drawn):
  tiny_int8     B=1, Hq=24, Hkv=4, D=256, L=512, 32 pages in a random permutation;
                q ~ N(0,1); K, V ~ N(0,1) with 4 outlier channels x8 per (tensor, KV head).
  long_int8     as tiny_int8 with L=32768 (2048 pages, permuted).
  serving_int8  B=64, Hq=32, Hkv=8, D=128, L_b ~ U{512..8192}; pages of all sequences
                shuffled across one shared pool; q ~ N(0,1); K, V ~ N(0, 0.5^2).
  append_int8   B=8, Hq=24, Hkv=4, D=256, L_b ~ U{4096..16384}; K, V ~ N(0,1) with
                1% of the values (i.i.d.) x20; the last 1024 tokens of every sequence
                (8192 in all) are the "new" tokens written by one append call.
  long_nvfp4    B=12, Hq=24, Hkv=4, D=256, L_b = floor(exp(U(ln 4096, ln 131072)));
                q, K, V ~ N(0,1); per-tensor NVFP4 global scale 448*6/amax(tensor).
  (any)         q_tokens(T): T query tokens a sequence for a verify step, N(0,1).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

PAGE = 16


def _rng(seed, *key):
    return np.random.Generator(np.random.PCG64([int(seed)] + [int(k) for k in key]))


def bf16_round(x):
    """float32 array -> float32 array of the nearest bf16 values (ties to even)."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).to(torch.float32).numpy()


@dataclasses.dataclass
class Workload:
    name: str
    seed: int
    B: int
    Hq: int
    Hkv: int
    D: int
    seq_lens: np.ndarray        # int32 [B]
    block_tables: np.ndarray    # int32 [B, max_pages]
    num_pages: int
    out_dtype: str              # "f32" or "bf16"
    value_std: float = 1.0
    outlier_channels: int = 0
    outlier_gain: float = 1.0
    spike_prob: float = 0.0
    spike_gain: float = 1.0
    append_tail: int = 0        # tokens per sequence written by the measured append
    splits: tuple = (0,)

    @property
    def G(self):
        return self.Hq // self.Hkv

    @property
    def sm_scale(self):
        return float(np.float32(1.0 / math.sqrt(self.D)))

    @property
    def total_tokens(self):
        return int(self.seq_lens.sum())

    def q(self):
        g = _rng(self.seed, 1)
        return bf16_round(g.standard_normal((self.B, self.Hq, self.D), dtype=np.float32))

    def q_tokens(self, T):
        """Queries of T tokens a sequence (a verify step): bf16 values [B, T, Hq, D]."""
        g = _rng(self.seed, 6, T)
        return bf16_round(g.standard_normal((self.B, T, self.Hq, self.D), dtype=np.float32))

    def _outlier_channels(self, which):
        g = _rng(self.seed, 2, which)
        return [g.choice(self.D, self.outlier_channels, replace=False) for _ in range(self.Hkv)]

    def kv(self, b):
        """bf16-valued float32 K and V of sequence b, [L_b, Hkv, D] each."""
        L = int(self.seq_lens[b])
        out = []
        for which in (0, 1):
            g = _rng(self.seed, 3, b, which)
            x = g.standard_normal((L, self.Hkv, self.D), dtype=np.float32) * np.float32(self.value_std)
            if self.outlier_channels:
                for h, ch in enumerate(self._outlier_channels(which)):
                    x[:, h, ch] *= np.float32(self.outlier_gain)
            if self.spike_prob > 0:
                mask = g.random((L, self.Hkv, self.D)) < self.spike_prob
                x[mask] *= np.float32(self.spike_gain)
            out.append(bf16_round(x))
        return out[0], out[1]

    def slots(self, b):
        """Physical slot of every token 0..L_b-1 of sequence b."""
        t = np.arange(int(self.seq_lens[b]), dtype=np.int64)
        return self.block_tables[b, t // PAGE].astype(np.int64) * PAGE + t % PAGE

    def tensor_amax(self):
        """max |K| and max |V| over the whole batch (for the NVFP4 global scales)."""
        ka = va = 0.0
        for b in range(self.B):
            k, v = self.kv(b)
            ka = max(ka, float(np.abs(k).max(initial=0.0)))
            va = max(va, float(np.abs(v).max(initial=0.0)))
        return ka, va


def _paged(seed, seq_lens, extra_pages=0):
    """Block tables that scatter every sequence's pages over one shuffled pool."""
    npages = [(int(L) + PAGE - 1) // PAGE for L in seq_lens]
    total = sum(npages) + extra_pages
    perm = _rng(seed, 0).permutation(total).astype(np.int32)
    maxp = max(max(npages), 1)
    bt = np.zeros((len(seq_lens), maxp), dtype=np.int32)
    off = 0
    for b, n in enumerate(npages):
        bt[b, :n] = perm[off:off + n]
        off += n
    return bt, max(total, 1)


def make(name, seed=None, **over):
    """Build one of the named workloads (see the module docstring); keyword
    arguments override fields (e.g. a shorter context for a quick test)."""
    recipes = {
        "tiny_int8": dict(B=1, Hq=24, Hkv=4, D=256, lens=("fixed", 512), out_dtype="f32",
                          outlier_channels=4, outlier_gain=8.0, splits=(1, 4), seed=0),
        "long_int8": dict(B=1, Hq=24, Hkv=4, D=256, lens=("fixed", 32768), out_dtype="f32",
                          outlier_channels=4, outlier_gain=8.0, splits=(1, 2, 4, 8, 16, 32, 64, 0), seed=1),
        "serving_int8": dict(B=64, Hq=32, Hkv=8, D=128, lens=("uniform", 512, 8192), out_dtype="bf16",
                             value_std=0.5, seed=2),
        "append_int8": dict(B=8, Hq=24, Hkv=4, D=256, lens=("uniform", 4096, 16384), out_dtype="bf16",
                            spike_prob=0.01, spike_gain=20.0, append_tail=1024, seed=3),
        "long_nvfp4": dict(B=12, Hq=24, Hkv=4, D=256, lens=("loguniform", 4096, 131072), out_dtype="bf16",
                           seed=4),
    }
    r = dict(recipes[name])
    r.update({k: v for k, v in over.items() if k in ("B", "lens", "out_dtype", "splits")})
    seed = r.pop("seed") if seed is None else seed
    r.pop("seed", None)
    lens = r.pop("lens")
    B = r["B"]
    g = _rng(seed, 9)
    if lens[0] == "fixed":
        seq_lens = np.full(B, lens[1], dtype=np.int32)
    elif lens[0] == "uniform":
        seq_lens = g.integers(lens[1], lens[2] + 1, size=B).astype(np.int32)
    elif lens[0] == "loguniform":
        seq_lens = np.floor(np.exp(g.uniform(math.log(lens[1]), math.log(lens[2]), size=B))).astype(np.int32)
    elif lens[0] == "list":
        seq_lens = np.asarray(lens[1], dtype=np.int32)
    else:
        raise ValueError(lens)
    bt, num_pages = _paged(seed, seq_lens, over.get("extra_pages", 0))
    fields = {k: v for k, v in r.items()}
    fields["B"] = int(len(seq_lens))
    fields.update({k: v for k, v in over.items() if k in ("value_std", "outlier_channels", "outlier_gain",
                                                          "spike_prob", "spike_gain", "append_tail")})
    return Workload(name=name, seed=seed, seq_lens=seq_lens, block_tables=bt, num_pages=num_pages, **fields)


def device_kv(wl, b, layer=0, device="cuda"):
    """K and V of sequence b for one layer, drawn on the device with torch's
    generator (same recipe as ``Workload.kv``, different random stream), as bf16
    tensors [L_b, Hkv, D].  Used where the CPU oracle does not need the values
    (benchmark pools)."""
    L = int(wl.seq_lens[b])
    out = []
    for which in (0, 1):
        g = torch.Generator(device=device)
        g.manual_seed(int(_rng(wl.seed, 5, layer, b, which).integers(1 << 62)))
        x = torch.randn((L, wl.Hkv, wl.D), generator=g, device=device) * wl.value_std
        if wl.outlier_channels:
            for h, ch in enumerate(wl._outlier_channels(which)):
                x[:, h, torch.as_tensor(ch, device=device)] *= wl.outlier_gain
        if wl.spike_prob > 0:
            mask = torch.rand((L, wl.Hkv, wl.D), generator=g, device=device) < wl.spike_prob
            x = torch.where(mask, x * wl.spike_gain, x)
        out.append(x.to(torch.bfloat16))
    return out[0], out[1]
