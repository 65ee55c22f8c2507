"""The oracle's attention against brute force and invariants (CPU only)."""
import numpy as np

from oracle import attention, brute, layout
from tests import oracle_pins as pins


def test_attend_matches_pure_python_brute_force():
    pins.check_attend_brute(attention.attend, brute.attend_brute)


def test_split_then_merge_equals_unsplit():
    pins.check_split_merge(attention.attend, attention.attend_split)


def test_merge_is_not_an_average():
    pins.check_merge_not_average(attention.attend, attention.merge)


def test_attention_invariants():
    pins.check_attention_invariants(attention.attend, attention.probabilities)


def test_merge_skips_empty_segments():
    o = np.ones((3, 2, 4))
    s = np.array([[0.0, -np.inf], [-np.inf, -np.inf], [0.0, -np.inf]])
    om, sm = attention.merge(o, s)
    assert np.allclose(om[0], 1.0) and not om[1].any()
    assert np.isclose(sm[0], np.log(2.0)) and np.isneginf(sm[1])


def _paged_pool(rng, fmt, L, D, Hkv, perm):
    """Quantized pools with the sequence's rows placed page by page (the test's
    own placement, not the oracle's layout functions); also returns the logical
    (codes, scales) of K and V."""
    P = 16
    npages = -(-L // P)
    k = pins.bf16_values(rng, (L, Hkv, D))
    v = pins.bf16_values(rng, (L, Hkv, D))
    pools, logical = {}, {}
    for name, x in (("k", k), ("v", v)):
        c, s = attention.quantize_rows(fmt, x.reshape(-1, D))
        c = c.reshape(L, Hkv, -1)
        cp = np.zeros((npages, Hkv, P, c.shape[-1]), np.uint8)
        pins.place_logical_rows(cp, perm, c, P)
        sp = None
        if s is not None:
            s = s.reshape(L, Hkv, *s.shape[1:])
            sp = np.zeros((npages, Hkv, P) + s.shape[2:], s.dtype)
            pins.place_logical_rows(sp, perm, s, P)
        pools[name + "_codes"], pools[name + "_scales"] = cp, sp
        logical[name] = (c, s)
    return pools, logical


def test_block_table_permutation_does_not_change_the_result():
    rng = np.random.default_rng(11)
    L, D, Hkv, G = 70, 16, 2, 3
    npages = -(-L // 16)
    q = pins.bf16_values(rng, (1, Hkv * G, D))
    for fmt in ("int8", "nvfp4", "bf16"):
        state = rng.bit_generator.state
        outs = []
        for perm in (np.arange(npages), rng.permutation(npages)):
            rng.bit_generator.state = state
            pools, _ = _paged_pool(np.random.default_rng(5), fmt, L, D, Hkv, perm)
            o, s = attention.paged_decode(fmt, pools, q, perm[None, :], [L], 0.25)
            outs.append((o, s))
        assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])


def test_paged_decode_equals_dense_attend_over_dequantized_rows():
    rng = np.random.default_rng(12)
    L, D, Hkv, G = 45, 16, 2, 2
    perm = rng.permutation(3)
    pools, logical = _paged_pool(rng, "int8", L, D, Hkv, perm)
    q = pins.bf16_values(rng, (1, Hkv * G, D))
    o, s = attention.paged_decode("int8", pools, q, perm[None, :], [L], 0.25)
    (kc, ks), (vc, vs) = logical["k"], logical["v"]
    for h in range(Hkv):
        # logical rows dequantized by their definition c * s
        k = kc[:, h].view(np.int8).astype(np.float64) * ks[:, h].astype(np.float64)[:, None]
        v = vc[:, h].view(np.int8).astype(np.float64) * vs[:, h].astype(np.float64)[:, None]
        ob, sb = brute.attend_brute(q[0, h * G:(h + 1) * G].tolist(), k.tolist(), v.tolist(), 0.25)
        assert np.max(np.abs(o[0, h * G:(h + 1) * G] - np.array(ob))) < 1e-12


def test_verify_matches_brute_force_over_each_visible_prefix():
    pins.check_verify(attention.paged_verify)


def test_paged_decode_over_hand_placed_pools_of_each_format():
    pins.check_paged_decode(attention.paged_decode)


def test_token_slots_hand_worked():
    pins.check_token_slots(layout.token_slots)


def test_gather_and_scatter_rows_on_coordinate_pools():
    pins.check_gather_scatter(layout.gather_rows, layout.scatter_rows)


def test_group_major_scales_hand_worked():
    pins.check_group_major(layout.group_major_scales)
    # the inverse restores the device order
    a = np.arange(2 * 2 * 3 * 16, dtype=np.float64).reshape(2, 2, 3, 16)
    assert np.array_equal(layout.to_group_major_scales(layout.group_major_scales(a)), a)


def test_hand_worked_two_key_softmax():
    # logits 0 and ln 2 (q . k scaled): p = (1/3, 2/3); V rows e0, e1 -> out = (1/3, 2/3);
    # lse = log(1 + 2) = ln 3
    q = np.array([[1.0, 0.0]])
    k = np.array([[0.0, 0.0], [np.log(2.0), 0.0]])
    v = np.array([[1.0, 0.0], [0.0, 1.0]])
    o, lse = attention.attend(q, k, v, 1.0)
    assert np.allclose(o[0], [1.0 / 3.0, 2.0 / 3.0], rtol=0, atol=1e-15)
    assert abs(float(np.ravel(lse)[0]) - np.log(3.0)) < 1e-15


def test_hand_worked_merge():
    # two splits with lse 0 and ln 3 (weights 1 : 3), outputs e0 and e1:
    # out = (1/4, 3/4), lse = ln 4
    o = np.array([[[1.0, 0.0]], [[0.0, 1.0]]])  # [split][row][D]
    s = np.array([[0.0], [np.log(3.0)]])        # [split][row]
    om, sm = attention.merge(o, s)
    assert np.allclose(om[0], [0.25, 0.75], rtol=0, atol=1e-15)
    assert abs(float(sm[0]) - np.log(4.0)) < 1e-15
