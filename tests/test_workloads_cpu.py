"""The seeded input recipes (quantized_paged_kv_gb300.workloads) against their
stated shapes, length distributions, page layouts and value distributions
(CPU only).  Both the GPU path and the oracle are fed from these generators."""
import numpy as np

from quantized_paged_kv_gb300 import workloads as W


def _is_bf16(x):
    return np.array_equal(x, W.bf16_round(x))


def _pages_are_one_shuffled_pool(wl):
    npages = -(-wl.seq_lens.astype(np.int64) // 16)
    used = np.concatenate([wl.block_tables[b, :n] for b, n in enumerate(npages)])
    assert used.size == wl.num_pages  # no page left over, none shared
    assert np.array_equal(np.sort(used), np.arange(wl.num_pages))
    assert not np.array_equal(used, np.arange(wl.num_pages))  # shuffled


def test_shapes_and_lengths():
    t = W.make("tiny_int8")
    assert (t.B, t.Hq, t.Hkv, t.D, t.G, t.out_dtype) == (1, 24, 4, 256, 6, "f32")
    assert list(t.seq_lens) == [512] and t.num_pages == 32
    l32 = W.make("long_int8")
    assert list(l32.seq_lens) == [32768] and l32.num_pages == 2048 and l32.out_dtype == "f32"
    s = W.make("serving_int8")
    assert (s.B, s.Hq, s.Hkv, s.D, s.G, s.out_dtype) == (64, 32, 8, 128, 4, "bf16")
    assert s.seq_lens.min() >= 512 and s.seq_lens.max() <= 8192 and len(set(s.seq_lens)) > 40
    a = W.make("append_int8")
    assert (a.B, a.Hq, a.Hkv, a.D, a.append_tail) == (8, 24, 4, 256, 1024)
    assert a.seq_lens.min() >= 4096 and a.seq_lens.max() <= 16384
    n = W.make("long_nvfp4")
    assert (n.B, n.Hq, n.Hkv, n.D, n.out_dtype) == (12, 24, 4, 256, "bf16")
    assert n.seq_lens.min() >= 4096 and n.seq_lens.max() <= 131072
    # log-uniform: the logs spread over [ln 4096, ln 131072], not bunched at the top
    lg = np.log(n.seq_lens)
    assert lg.min() < np.log(16384) and lg.max() > np.log(32768)
    for wl in (t, l32, s, a, n):
        _pages_are_one_shuffled_pool(wl)
        assert wl.sm_scale == np.float32(1.0 / np.sqrt(wl.D))


def test_draws_are_seeded_and_bf16():
    a, b = W.make("tiny_int8"), W.make("tiny_int8")
    assert np.array_equal(a.q(), b.q())
    ka, va = a.kv(0)
    kb, vb = b.kv(0)
    assert np.array_equal(ka, kb) and np.array_equal(va, vb)
    assert not np.array_equal(ka, va)
    assert _is_bf16(a.q()) and _is_bf16(ka) and _is_bf16(va)
    c = W.make("tiny_int8", seed=7)
    assert not np.array_equal(c.q(), a.q())


def test_value_distributions():
    t = W.make("tiny_int8")
    q = t.q()
    assert abs(q.mean()) < 0.02 and abs(q.std() - 1.0) < 0.02
    k, v = t.kv(0)
    for x, which in ((k, 0), (v, 1)):
        chans = t._outlier_channels(which)
        for h in range(t.Hkv):
            std = x[:, h, :].std(axis=0)
            assert len(set(chans[h])) == 4
            out = np.zeros(t.D, bool)
            out[chans[h]] = True
            assert np.all(std[out] > 6.0) and np.all(std[~out] < 1.3)  # 4 channels x8, the rest N(0,1)
    s = W.make("serving_int8", lens=("list", [3000]))
    k, _ = s.kv(0)
    assert abs(k.std() - 0.5) < 0.01
    a = W.make("append_int8", lens=("list", [4096]))
    k, _ = a.kv(0)
    big = np.abs(k) > 6.0  # N(0,1) alone almost never exceeds 6; the x20 spikes often do
    frac = big.mean()
    assert 0.005 < frac < 0.012


def test_slots_follow_the_block_table():
    wl = W.make("serving_int8")
    for b in (0, 17, 63):
        sl = wl.slots(b)
        assert sl.size == wl.seq_lens[b]
        t = np.arange(sl.size)
        assert np.array_equal(sl // 16, wl.block_tables[b, t // 16])
        assert np.array_equal(sl % 16, t % 16)
