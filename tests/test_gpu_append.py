"""kvq_quant_append on the GPU against the oracle: codes and scales bit-exact."""
import numpy as np
import pytest
import torch

from oracle import attention as oatt
from oracle import formats as ofmt
from tests import harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    H.ensure_built()


def _rows(rng, n, Hkv, D, kind):
    x = rng.standard_normal((n, Hkv, D)).astype(np.float32)
    if kind == "outliers":
        x[:, :, [3, 40, 77, 200 % D]] *= 8.0
    elif kind == "spikes":
        x[rng.random(x.shape) < 0.01] *= 20.0
    elif kind == "edge":
        x[0] = 0.0                                    # all-zero rows -> scale 0, codes 0
        x[1] *= 1e-30                                 # tiny (subnormal-scale) rows
        x[2] = np.where(rng.random((Hkv, D)) < 0.5, -0.0, 0.0)
        x[3] *= 3e4                                   # large
        x[4, :, :] = 1.0                              # constant row
        x[5, :, 0] = 127.0 / 8                        # exact INT8 midpoints: scale = 1/8
        x[5, :, 1:11] = (np.array([0.5, 1.5, 2.5, 3.5, -0.5, -1.5, -2.5, 125.5, 126.5, -126.5]) / 8)
        x[5, :, 11:] = 0.0
    return torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()


def _append_and_compare(fmt, Hkv, D, kind, n=300, num_pages=64, gs=(1.0, 1.0), seed=0):
    from quantized_paged_kv_gb300 import KVCache

    rng = np.random.default_rng(seed)
    k, v = _rows(rng, n, Hkv, D, kind), _rows(rng, n, Hkv, D, kind)
    if gs == "tensor":
        gs = (float(ofmt.nvfp4_tensor_global_scale(k)), float(ofmt.nvfp4_tensor_global_scale(v)))
    cap = num_pages * 16
    slots = rng.permutation(cap)[:n].astype(np.int64)
    slots[::17] = -1                                   # padding tokens: not written
    cache = KVCache(fmt, num_pages, Hkv, D, k_global_scale=gs[0], v_global_scale=gs[1], fill=H.SENTINEL)
    dev = lambda a: torch.from_numpy(a).to("cuda")
    cache.append(dev(k).to(torch.bfloat16), dev(v).to(torch.bfloat16), dev(slots))
    torch.cuda.synchronize()
    kc, vc, ks, vs = H.gpu_views_numpy(cache)
    valid = slots >= 0
    for x, codes, scales, g in ((k, kc, ks, gs[0]), (v, vc, vs, gs[1])):
        for h in range(Hkv):
            c_exp, s_exp = oatt.quantize_rows(fmt, x[valid, h, :], g)
            sl = slots[valid]
            got_c = codes[sl // 16, h, sl % 16]
            assert np.array_equal(got_c, c_exp), (fmt, kind, h, np.argwhere(got_c != c_exp)[:5])
            if s_exp is not None:
                got_s = scales[sl // 16, h, sl % 16]
                assert np.array_equal(got_s.view(np.uint8), np.asarray(s_exp).view(np.uint8)), (fmt, kind, h)
    # slots that were not written keep the sentinel
    written = np.zeros(cap, bool)
    written[slots[valid]] = True
    assert np.all(kc.reshape(num_pages, Hkv, 16, -1).transpose(0, 2, 1, 3).reshape(cap, Hkv, -1)[~written] == H.SENTINEL)


@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("kind", ["normal", "outliers", "spikes", "edge"])
def test_int8_append_bit_exact(D, kind):
    _append_and_compare("int8", 4, D, kind)


@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("kind", ["normal", "outliers", "spikes", "edge"])
def test_int8_g32_append_bit_exact(D, kind):
    _append_and_compare("int8_g32", 4, D, kind)


@pytest.mark.parametrize("kind", ["normal", "outliers", "spikes", "edge"])
@pytest.mark.parametrize("gs", [(1.0, 1.0), "tensor", (0.37, 1234.5)])
@pytest.mark.parametrize("D", [128, 256])
def test_nvfp4_append_bit_exact(kind, gs, D):
    _append_and_compare("nvfp4", 2, D, kind, gs=gs)


@pytest.mark.parametrize("fmt,D", [("int8", 128), ("int8", 256), ("int8_g32", 128), ("int8_g32", 256), ("nvfp4", 128),
                                   ("nvfp4", 256), ("bf16", 256)])
@pytest.mark.parametrize("n", [1, 5, 33, 301])
def test_append_ragged_token_counts(fmt, D, n):
    # a block carries several rows a thread group: token counts that leave the
    # last block partly empty, down to a single token
    _append_and_compare(fmt, 3, D, "normal", n=n, seed=n)


@pytest.mark.parametrize("D", [128, 256])
def test_bf16_append_copies(D):
    _append_and_compare("bf16", 3, D, "normal")


def test_nvfp4_scale_rounding_sweep():
    """Group maxima that put fp32(amax/6 * gs) on and between every E4M3 value
    (midpoints included) and across the subnormal range."""
    from quantized_paged_kv_gb300 import KVCache

    vals = ofmt.e4m3_value(np.arange(0x7F, dtype=np.uint8))
    mids = (vals[:-1] + vals[1:]) / 2
    targets = np.concatenate([vals, mids, mids * (1 + 2 ** -20), mids * (1 - 2 ** -20)])
    amax = (targets * 6.0).astype(np.float32)
    amax = torch.from_numpy(amax).to(torch.bfloat16).to(torch.float32).numpy()
    n = (len(amax) + 15) // 16
    x = np.zeros((n, 1, 256), np.float32)
    flat = x.reshape(-1, 16)
    flat[: len(amax), 5] = amax
    flat[: len(amax), 6] = -amax * 0.6
    flat[: len(amax), 7] = amax * 0.25
    x = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    cache = KVCache("nvfp4", (n + 15) // 16, 1, 256, fill=H.SENTINEL)
    slots = np.arange(n, dtype=np.int64)
    xt = torch.from_numpy(x).to(torch.bfloat16).cuda()
    cache.append(xt, xt, torch.from_numpy(slots).cuda())
    torch.cuda.synchronize()
    kc, _, ks, _ = H.gpu_views_numpy(cache)
    c_exp, s_exp = ofmt.nvfp4_quantize(x[:, 0, :], 1.0)
    assert np.array_equal(ks[slots // 16, 0, slots % 16], s_exp)
    assert np.array_equal(kc[slots // 16, 0, slots % 16], c_exp)


def _bf16_upto(a):
    """Every bf16 value v with |v| <= a (both signs, zero once), as float32."""
    bits = np.arange(0x7F80, dtype=np.uint32)          # all finite non-negative bf16 patterns
    v = (bits << 16).view(np.float32)
    v = v[v <= a]
    return np.concatenate([v, -v[1:]])


def _dense_maxima(rng, n):
    """bf16 row / group maxima over many binades, with random mantissas plus the
    all-ones and power-of-two mantissas."""
    e = rng.integers(-40, 40, n)
    m = rng.integers(0, 128, n)
    m[::7] = 127
    m[1::7] = 0
    a = ((1.0 + m / 128.0) * np.exp2(e)).astype(np.float32)
    return torch.from_numpy(a).to(torch.bfloat16).to(torch.float32).numpy()


def _append_rows(fmt, x, gs=1.0):
    from quantized_paged_kv_gb300 import KVCache

    n = x.shape[0]
    cache = KVCache(fmt, (n + 15) // 16, 1, x.shape[-1], k_global_scale=gs, v_global_scale=gs, fill=H.SENTINEL)
    slots = np.arange(n, dtype=np.int64)
    xt = torch.from_numpy(np.ascontiguousarray(x[:, None, :])).to(torch.bfloat16).cuda()
    cache.append(xt, xt, torch.from_numpy(slots).cuda())
    torch.cuda.synchronize()
    kc, _, ks, _ = H.gpu_views_numpy(cache)
    return kc[slots // 16, 0, slots % 16], ks[slots // 16, 0, slots % 16]


def test_int8_append_dense_quotients():
    """Each row holds its maximum and then every bf16 value up to it: every
    quotient x / scale the row can produce, the half-integer ties included,
    over many binades of the scale."""
    rng = np.random.default_rng(11)
    rows = []
    for a in _dense_maxima(rng, 24):
        v = _bf16_upto(a)
        v = np.concatenate([v, np.zeros((-len(v)) % 255, np.float32)])
        r = v.reshape(-1, 255)
        rows.append(np.concatenate([np.full((len(r), 1), a, np.float32), r], axis=1))
    x = np.concatenate(rows)
    got_c, got_s = _append_rows("int8", x)
    c_exp, s_exp = oatt.quantize_rows("int8", x)
    assert np.array_equal(got_s.view(np.uint32), s_exp.view(np.uint32))
    bad = np.argwhere(got_c != c_exp)
    assert len(bad) == 0, (len(bad), bad[:5], x[tuple(bad[0])] if len(bad) else None)


def test_int8_g32_append_dense_quotients():
    """Groups of 32 holding their maximum and 31 bf16 values up to it: every
    quotient each group's scale can produce, ties included."""
    rng = np.random.default_rng(13)
    groups = []
    for a in _dense_maxima(rng, 16):
        v = _bf16_upto(a)
        v = np.concatenate([v, np.zeros((-len(v)) % 31, np.float32)])
        g = v.reshape(-1, 31)
        groups.append(np.concatenate([np.full((len(g), 1), a, np.float32), g], axis=1))
    g = np.concatenate(groups)
    g = g[rng.permutation(len(g))]  # neighbouring groups of a row from different maxima
    g = np.concatenate([g, np.zeros(((-len(g)) % 8, 32), np.float32)])
    x = g.reshape(-1, 256)
    got_c, got_s = _append_rows("int8_g32", x)
    c_exp, s_exp = oatt.quantize_rows("int8_g32", x)
    assert np.array_equal(got_s.view(np.uint32), s_exp.view(np.uint32))
    bad = np.argwhere(got_c != c_exp)
    assert len(bad) == 0, (len(bad), bad[:5])


@pytest.mark.parametrize("gs", [1.0, 0.37, 1234.5])
@pytest.mark.parametrize("D", [128, 256])
def test_nvfp4_append_dense_quotients(gs, D):
    """Groups of 16 holding their maximum and 15 bf16 values up to it, so that
    every value up to each maximum meets the group's E4M3 scale."""
    rng = np.random.default_rng(12)
    groups = []
    for a in _dense_maxima(rng, 16):
        v = _bf16_upto(a)
        v = np.concatenate([v, np.zeros((-len(v)) % 15, np.float32)])
        g = v.reshape(-1, 15)
        groups.append(np.concatenate([np.full((len(g), 1), a, np.float32), g], axis=1))
    g = np.concatenate(groups)
    g = np.concatenate([g, np.zeros(((-len(g)) % 16, 16), np.float32)])
    x = g.reshape(-1, D)
    got_c, got_s = _append_rows("nvfp4", x, gs)
    c_exp, s_exp = oatt.quantize_rows("nvfp4", x, gs)
    assert np.array_equal(got_s, s_exp)
    bad = np.argwhere(got_c != c_exp)
    assert len(bad) == 0, (len(bad), bad[:5])


def test_slot_overwrite():
    from quantized_paged_kv_gb300 import KVCache

    rng = np.random.default_rng(5)
    cache = KVCache("int8", 4, 2, 128, fill=H.SENTINEL)
    slots = torch.tensor([3, 9, 40], dtype=torch.int64, device="cuda")
    for it in range(2):
        k = _rows(rng, 3, 2, 128, "normal")
        kt = torch.from_numpy(k).to(torch.bfloat16).cuda()
        cache.append(kt, kt, slots)
    torch.cuda.synchronize()
    kc, _, ks, _ = H.gpu_views_numpy(cache)
    c_exp, s_exp = oatt.quantize_rows("int8", k[:, 1, :])
    sl = slots.cpu().numpy()
    assert np.array_equal(kc[sl // 16, 1, sl % 16], c_exp)
    assert np.array_equal(ks[sl // 16, 1, sl % 16], s_exp)


def test_checked_append_rejects_bad_metadata():
    from quantized_paged_kv_gb300 import KVCache, KvqError

    cache = KVCache("int8", 2, 1, 128, fill=H.SENTINEL)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    k = torch.randn(3, 1, 128, device="cuda").to(torch.bfloat16)
    with pytest.raises(KvqError) as e:
        cache.append(k, k, torch.tensor([1, 5, 1], device="cuda"), dev_status=status, checked=True)
    assert e.value.code == 1 and "duplicate" in str(e.value)
    with pytest.raises(KvqError) as e:
        cache.append(k, k, torch.tensor([1, 5, 32], device="cuda"), dev_status=status, checked=True)
    assert e.value.code == 1
    bad = k.clone()
    bad[1, 0, 7] = float("inf")
    with pytest.raises(KvqError) as e:
        cache.append(bad, k, torch.tensor([1, 5, 6], device="cuda"), dev_status=status, checked=True)
    assert e.value.code == 5
    # raw mode: an out-of-range slot is skipped and reported in the status word
    cache.append(k, k, torch.tensor([0, 99, 2], device="cuda"), dev_status=status)
    from quantized_paged_kv_gb300 import kvq_read_status
    rc, bits = kvq_read_status(status)
    assert rc == 5 and bits & 16
