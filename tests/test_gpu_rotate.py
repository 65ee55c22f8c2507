"""kvq_rotate_rows on the GPU: bit-exact against the oracle's fp32 butterfly; the
rotation inside the append (KVQ_ROTATE) bit-exact against the oracle and the
two-call path, also on the full 8,192-token append workload; and the rotated
decode pipeline (rotate K/V before the append, rotate q, decode, rotate the
output back) against the oracle."""
import functools

import numpy as np
import pytest
import torch

from oracle import attention as oatt
from oracle import formats as ofmt
from oracle import layout as olay
from oracle import rotation as orot
from quantized_paged_kv_gb300 import workloads as W
from tests import harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    H.ensure_built()


def _rows(n, D, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((n, D)) * np.exp(rng.uniform(-4, 4, (n, 1)))
    x[:, [1, D // 3, D - 2]] *= 8.0
    return x.astype(np.float32)


@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("inverse", [False, True])
@pytest.mark.parametrize("din,dout", [("bf16", "bf16"), ("f32", "f32"), ("bf16", "f32"), ("f32", "bf16")])
def test_rotate_bit_exact(D, inverse, din, dout):
    from quantized_paged_kv_gb300 import kvq_rotate_rows

    x = _rows(1000, D, seed=D + inverse)
    if din == "bf16":
        x = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    tdt = {"bf16": torch.bfloat16, "f32": torch.float32}
    xt = torch.from_numpy(x).to(tdt[din]).cuda()
    out = torch.empty(xt.shape, dtype=tdt[dout], device="cuda")
    kvq_rotate_rows(xt, out, inverse=inverse)
    torch.cuda.synchronize()
    ref = orot.rotate_fp32(x, inverse, out=dout)
    got = out.float().cpu().numpy()
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), np.argwhere(got != ref)[:5]


def test_rotate_round_trip_and_in_place():
    from quantized_paged_kv_gb300 import kvq_rotate_rows

    x = torch.from_numpy(_rows(77, 256, seed=9)).cuda()
    y = kvq_rotate_rows(x)
    kvq_rotate_rows(y, y, inverse=True)  # in place
    torch.cuda.synchronize()
    assert torch.allclose(y, x, rtol=1e-5, atol=1e-6 * float(x.abs().max()))


def _rotated_pipeline(wl, fmt):
    """GPU: rotate K/V rows, append, rotate q, decode (fp32 out), rotate back."""
    from quantized_paged_kv_gb300 import DecodePlan, KVCache, decode, kvq_rotate_rows

    cache = KVCache(fmt, wl.num_pages, wl.Hkv, wl.D, fill=H.SENTINEL)
    for b in range(wl.B):
        k, v = wl.kv(b)
        kt = kvq_rotate_rows(torch.from_numpy(k).to(torch.bfloat16).cuda())
        vt = kvq_rotate_rows(torch.from_numpy(v).to(torch.bfloat16).cuda())
        cache.append(kt, vt, torch.from_numpy(wl.slots(b)).cuda())
    qt = kvq_rotate_rows(torch.from_numpy(wl.q()).to(torch.bfloat16).cuda())
    out = torch.empty((wl.B, wl.Hq, wl.D), dtype=torch.float32, device="cuda")
    plan = DecodePlan(cache, wl.seq_lens, wl.Hq)
    decode(cache, plan, qt, torch.from_numpy(wl.block_tables).cuda(), torch.from_numpy(wl.seq_lens).cuda(), out,
           wl.sm_scale, checked=True)
    kvq_rotate_rows(out, out, inverse=True)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def _oracle_rotated(wl, fmt):
    """Oracle: the same rotated bf16 rows (fp32 butterfly), quantized, attended in
    float64, rotated back exactly."""
    P = 16
    row = {"int8": wl.D, "nvfp4": wl.D // 2}[fmt]
    shp = (wl.num_pages, wl.Hkv, P)
    pools = {"k_codes": np.zeros(shp + (row,), np.uint8), "v_codes": np.zeros(shp + (row,), np.uint8),
             "k_global_scale": 1.0, "v_global_scale": 1.0}
    if fmt == "int8":
        pools["k_scales"], pools["v_scales"] = np.zeros(shp, np.float32), np.zeros(shp, np.float32)
    else:
        pools["k_scales"] = np.zeros(shp + (wl.D // 16,), np.uint8)
        pools["v_scales"] = np.zeros(shp + (wl.D // 16,), np.uint8)
    for b in range(wl.B):
        k, v = wl.kv(b)
        for name, x in (("k", k), ("v", v)):
            xr = orot.rotate_fp32(x, out="bf16")
            for h in range(wl.Hkv):
                c, s = oatt.quantize_rows(fmt, xr[:, h, :], 1.0)
                olay.scatter_rows(pools[name + "_codes"], wl.slots(b), h, c)
                olay.scatter_rows(pools[name + "_scales"], wl.slots(b), h, s)
    qr = orot.rotate_fp32(wl.q(), out="bf16")
    o, _ = oatt.paged_decode(fmt, pools, qr, wl.block_tables, wl.seq_lens, wl.sm_scale)
    return orot.rotate_exact(o, inverse=True)


@pytest.mark.parametrize("fmt", ["int8", "nvfp4"])
def test_rotated_decode_matches_the_oracle(fmt):
    wl = W.make("tiny_int8", lens=("list", [700, 45]), seed=21)
    got = _rotated_pipeline(wl, fmt)
    ref = _oracle_rotated(wl, fmt)
    assert np.abs(got - ref).max() <= H.tol("f32")


def test_rotation_brings_int8_closer_to_exact_attention():
    # outlier channels x8: with one INT8 scale per (token, head) the rotated cache
    # gives the attention of the unquantized bf16 K/V more closely
    from quantized_paged_kv_gb300 import DecodePlan, decode

    wl = W.make("tiny_int8", lens=("list", [700]), seed=22)
    exact, _ = oatt.paged_decode("bf16", H.oracle_pools(wl, "bf16"), wl.q(), wl.block_tables, wl.seq_lens,
                                 wl.sm_scale)
    rotated = _rotated_pipeline(wl, "int8")
    cache = H.gpu_cache(wl, "int8")
    out, _, _ = H.run_decode(cache, wl, out_dtype="f32")
    err_plain = np.abs(out - exact).max()
    err_rot = np.abs(rotated - exact).max()
    assert err_rot < 0.7 * err_plain, (err_rot, err_plain)


def _fused_rows(rng, n, Hkv, D):
    """bf16-valued K/V rows with a spread of magnitudes, outlier channels, an
    all-zero row, a tiny row and a huge row."""
    x = rng.standard_normal((n, Hkv, D)) * np.exp(rng.uniform(-3, 3, (n, Hkv, 1)))
    x[:, :, [2, D // 5, D - 3]] *= 8.0
    x[0] = 0.0
    x[1] *= 1e-30
    x[2] *= 3e4
    return torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).to(torch.float32).numpy()


@pytest.mark.parametrize("fmt,D", [("int8", 128), ("int8", 256), ("int8_g32", 128), ("int8_g32", 256),
                                   ("nvfp4", 128), ("nvfp4", 256), ("bf16", 128), ("bf16", 256)])
@pytest.mark.parametrize("n", [5, 301])
def test_fused_rotated_append_bit_exact(fmt, D, n):
    # KVQ_ROTATE on the append: codes and scales equal the oracle's quantization of
    # its rotated bf16 rows, and the two-call GPU path (rotate, then append)
    from quantized_paged_kv_gb300 import KVCache, kvq_rotate_rows

    Hkv, num_pages = 4, 40
    rng = np.random.default_rng(1000 * D + n)
    k, v = _fused_rows(rng, n, Hkv, D), _fused_rows(rng, n, Hkv, D)
    gs = (0.37, 1234.5) if fmt == "nvfp4" else (1.0, 1.0)
    slots = rng.permutation(num_pages * 16)[:n].astype(np.int64)
    slots[1::7] = -1                                   # padding tokens: not written
    dev = lambda a: torch.from_numpy(a).cuda()
    kb, vb, sl = dev(k).to(torch.bfloat16), dev(v).to(torch.bfloat16), dev(slots)
    fused = KVCache(fmt, num_pages, Hkv, D, k_global_scale=gs[0], v_global_scale=gs[1], fill=H.SENTINEL)
    fused.append(kb, vb, sl, rotate=True)
    two = KVCache(fmt, num_pages, Hkv, D, k_global_scale=gs[0], v_global_scale=gs[1], fill=H.SENTINEL)
    rk = kvq_rotate_rows(kb.reshape(-1, D)).reshape(kb.shape)
    rv = kvq_rotate_rows(vb.reshape(-1, D)).reshape(vb.shape)
    two.append(rk, rv, sl)
    torch.cuda.synchronize()
    got, ref_gpu = H.gpu_views_numpy(fused), H.gpu_views_numpy(two)
    for a, b in zip(got, ref_gpu):
        if a is not None:
            assert np.array_equal(a.view(np.uint8), b.view(np.uint8))
    valid = slots >= 0
    sv = slots[valid]
    for x, codes, scales, g in ((k, got[0], got[2], gs[0]), (v, got[1], got[3], gs[1])):
        xr = orot.rotate_fp32(x, out="bf16")
        for h in range(Hkv):
            c_exp, s_exp = oatt.quantize_rows(fmt, xr[valid, h, :], g)
            got_c = codes[sv // 16, h, sv % 16]
            assert np.array_equal(got_c, c_exp), (fmt, h, np.argwhere(got_c != c_exp)[:5])
            if s_exp is not None:
                got_s = scales[sv // 16, h, sv % 16]
                assert np.array_equal(got_s.view(np.uint8), np.asarray(s_exp).view(np.uint8)), (fmt, h)
    # unwritten slots keep the sentinel
    written = np.zeros(num_pages * 16, bool)
    written[sv] = True
    kc = got[0]
    assert np.all(kc.transpose(0, 2, 1, 3).reshape(num_pages * 16, Hkv, -1)[~written] == H.SENTINEL)


@pytest.mark.parametrize("fmt", ["int8", "nvfp4"])
def test_rotated_decode_with_fused_append_matches_the_oracle(fmt):
    from quantized_paged_kv_gb300 import DecodePlan, KVCache, decode, kvq_rotate_rows

    wl = W.make("tiny_int8", lens=("list", [700, 45]), seed=21)
    cache = KVCache(fmt, wl.num_pages, wl.Hkv, wl.D, fill=H.SENTINEL)
    for b in range(wl.B):
        k, v = wl.kv(b)
        cache.append(torch.from_numpy(k).to(torch.bfloat16).cuda(), torch.from_numpy(v).to(torch.bfloat16).cuda(),
                     torch.from_numpy(wl.slots(b)).cuda(), rotate=True)
    qt = kvq_rotate_rows(torch.from_numpy(wl.q()).to(torch.bfloat16).cuda())
    out = torch.empty((wl.B, wl.Hq, wl.D), dtype=torch.float32, device="cuda")
    plan = DecodePlan(cache, wl.seq_lens, wl.Hq)
    decode(cache, plan, qt, torch.from_numpy(wl.block_tables).cuda(), torch.from_numpy(wl.seq_lens).cuda(), out,
           wl.sm_scale, checked=True)
    kvq_rotate_rows(out, out, inverse=True)
    torch.cuda.synchronize()
    assert np.abs(out.cpu().numpy() - _oracle_rotated(wl, fmt)).max() <= H.tol("f32")


@functools.lru_cache(maxsize=1)
def _append_workload_rows():
    """The append workload's 8,192 new tokens (the last 1,024 of each of its 8
    sequences): K, V [8192, 4, 256] bf16-valued float32 and their slots."""
    wl = W.make("append_int8")
    ks, vs, ss = [], [], []
    for b in range(wl.B):
        k, v = wl.kv(b)
        ks.append(k[-wl.append_tail:])
        vs.append(v[-wl.append_tail:])
        ss.append(wl.slots(b)[-wl.append_tail:])
    return wl, np.concatenate(ks), np.concatenate(vs), np.concatenate(ss)


@pytest.mark.parametrize("fmt", ["int8", "nvfp4"])
@pytest.mark.parametrize("rotate", [False, True])
def test_append_workload_full_size_bit_exact(fmt, rotate):
    # every code and scale of the 8,192-token append (as timed), plain and with the
    # rotation inside the append, against the oracle's quantization
    from quantized_paged_kv_gb300 import KVCache

    wl, k, v, slots = _append_workload_rows()
    kr = orot.rotate_fp32(k, out="bf16") if rotate else k
    vr = orot.rotate_fp32(v, out="bf16") if rotate else v
    gs = (float(ofmt.nvfp4_tensor_global_scale(kr)), float(ofmt.nvfp4_tensor_global_scale(vr))) \
        if fmt == "nvfp4" else (1.0, 1.0)
    cache = KVCache(fmt, wl.num_pages, wl.Hkv, wl.D, k_global_scale=gs[0], v_global_scale=gs[1], fill=H.SENTINEL)
    dev = lambda a: torch.from_numpy(a).cuda()
    cache.append(dev(k).to(torch.bfloat16), dev(v).to(torch.bfloat16), dev(slots), rotate=rotate)
    torch.cuda.synchronize()
    kc, vc, ks, vs = H.gpu_views_numpy(cache)
    for x, codes, scales, g in ((kr, kc, ks, gs[0]), (vr, vc, vs, gs[1])):
        for h in range(wl.Hkv):
            c_exp, s_exp = oatt.quantize_rows(fmt, x[:, h, :], g)
            assert np.array_equal(codes[slots // 16, h, slots % 16], c_exp), (fmt, rotate, h)
            got_s = scales[slots // 16, h, slots % 16]
            assert np.array_equal(got_s.view(np.uint8), np.asarray(s_exp).view(np.uint8)), (fmt, rotate, h)
