"""Shared test plumbing: build pools on the GPU through the C ABI, and the same
pools independently with the CPU oracle, from one seeded workload."""
from __future__ import annotations

import os

import numpy as np
import torch

from oracle import attention as oatt
from oracle import layout as olay

SENTINEL = 0xFF  # unwritten slots: NaN scales (fp32 and E4M3), -1 / -6 codes, NaN bf16


def ensure_built():
    import quantized_paged_kv_gb300 as kvq
    from quantized_paged_kv_gb300 import build as kbuild

    lib = kbuild.LIB
    srcs = [os.path.join(kbuild.CSRC, f) for f in os.listdir(kbuild.CSRC)]
    srcs.append(os.path.join(kbuild.INCLUDE, "kvq.h"))
    if not os.path.exists(lib) or os.path.getmtime(lib) < max(os.path.getmtime(s) for s in srcs):
        kbuild.build()
    return kvq.lib()


def global_scales(wl, fmt):
    if fmt != "nvfp4":
        return 1.0, 1.0
    ka, va = wl.tensor_amax()
    return (float(np.float32(2688.0) / np.float32(ka)) if ka else 1.0,
            float(np.float32(2688.0) / np.float32(va)) if va else 1.0)


def gpu_cache(wl, fmt, gs=(1.0, 1.0), seqs=None, device="cuda", fill=SENTINEL, extra_pages=0):
    """Sentinel-filled pool with every token of the chosen sequences appended
    through kvq_quant_append (one call per sequence)."""
    from quantized_paged_kv_gb300 import KVCache

    cache = KVCache(fmt, wl.num_pages + extra_pages, wl.Hkv, wl.D, device=device,
                    k_global_scale=gs[0], v_global_scale=gs[1], fill=fill)
    for b in (range(wl.B) if seqs is None else seqs):
        if wl.seq_lens[b] == 0:
            continue
        k, v = wl.kv(b)
        kt = torch.from_numpy(k).to(torch.bfloat16).to(device)
        vt = torch.from_numpy(v).to(torch.bfloat16).to(device)
        st = torch.from_numpy(wl.slots(b)).to(device)
        cache.append(kt, vt, st)
    return cache


def oracle_pools(wl, fmt, gs=(1.0, 1.0), seqs=None, heads=None):
    """The same pools built by the oracle's codecs and layout (numpy)."""
    P = 16
    row = {"bf16": 2 * wl.D, "int8": wl.D, "int8_g32": wl.D, "nvfp4": wl.D // 2}[fmt]
    shp = (wl.num_pages, wl.Hkv, P)
    pools = {"k_codes": np.full(shp + (row,), SENTINEL, np.uint8), "v_codes": np.full(shp + (row,), SENTINEL, np.uint8),
             "k_global_scale": gs[0], "v_global_scale": gs[1]}
    if fmt == "int8":
        pools["k_scales"] = np.full(shp, np.nan, np.float32)
        pools["v_scales"] = np.full(shp, np.nan, np.float32)
    elif fmt == "int8_g32":  # the oracle's slot-major form [pages, Hkv, P, D/32]
        pools["k_scales"] = np.full(shp + (wl.D // 32,), np.nan, np.float32)
        pools["v_scales"] = np.full(shp + (wl.D // 32,), np.nan, np.float32)
    elif fmt == "nvfp4":
        pools["k_scales"] = np.full(shp + (wl.D // 16,), SENTINEL, np.uint8)
        pools["v_scales"] = np.full(shp + (wl.D // 16,), SENTINEL, np.uint8)
    else:
        pools["k_scales"] = pools["v_scales"] = None
    for b in (range(wl.B) if seqs is None else seqs):
        if wl.seq_lens[b] == 0:
            continue
        k, v = wl.kv(b)
        slots = wl.slots(b)
        for name, x, g in (("k", k, gs[0]), ("v", v, gs[1])):
            for h in (range(wl.Hkv) if heads is None else heads):
                c, s = oatt.quantize_rows(fmt, x[:, h, :], g)
                olay.scatter_rows(pools[name + "_codes"], slots, h, c)
                if s is not None:
                    olay.scatter_rows(pools[name + "_scales"], slots, h, s)
    return pools


def gpu_views_numpy(cache):
    """Codes and scales as numpy, scales in the oracle's slot-major form
    ([pages, Hkv, P, ...]; the per-32 format's device order is group-major)."""
    kc, vc, ks, vs = cache.views()
    f = lambda t: None if t is None else t.cpu().numpy()
    ks, vs = f(ks), f(vs)
    if cache.fmt == "int8_g32":
        ks, vs = olay.group_major_scales(ks), olay.group_major_scales(vs)
    return f(kc), f(vc), ks, vs


def run_decode(cache, wl, split=0, q=None, out_dtype=None, target_ctas=0, checked=True, lse=True, device="cuda"):
    from quantized_paged_kv_gb300 import DecodePlan, decode

    q = wl.q() if q is None else q
    qt = torch.from_numpy(q).to(torch.bfloat16).to(device)
    od = {"f32": torch.float32, "bf16": torch.bfloat16}[out_dtype or wl.out_dtype]
    out = torch.full((wl.B, wl.Hq, wl.D), float("nan"), dtype=od, device=device)
    lse_t = torch.full((wl.B, wl.Hq), float("nan"), dtype=torch.float32, device=device) if lse else None
    plan = DecodePlan(cache, wl.seq_lens, wl.Hq, split_override=split, target_ctas=target_ctas, device=device)
    bt = torch.from_numpy(wl.block_tables).to(device)
    sl = torch.from_numpy(wl.seq_lens).to(device)
    decode(cache, plan, qt, bt, sl, out, wl.sm_scale, lse_out=lse_t, checked=checked)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), (lse_t.cpu().numpy() if lse else None), plan


def oracle_decode(wl, fmt, pools, units=None, q=None):
    q = wl.q() if q is None else q
    return oatt.paged_decode(fmt, pools, q, wl.block_tables, wl.seq_lens, wl.sm_scale, heads=units)


def tol(out_dtype):
    return 2e-3 if out_dtype == "f32" else 1e-2


def bound(out_dtype, ref):
    """Per-element max-abs bound for outputs compared with the reference values
    ``ref``: 2e-3 for fp32 output; for bf16 output max(1e-2, 2^-8 |ref|), because
    rounding the exact result to bf16 alone moves it by up to 2^-8 |ref| (half a
    bf16 ulp), which exceeds 1e-2 once |ref| > 2.56."""
    if out_dtype == "f32":
        return np.full(np.shape(ref), 2e-3)
    return np.maximum(1e-2, 2.0 ** -8 * np.abs(ref))
