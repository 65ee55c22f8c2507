"""Pins of the rotation oracle (CPU): the Hadamard matrix against its closed
form, the sign generator against hand-computed hash values, the fp32 butterfly
against the matrix product, orthogonality, and invariance of attention."""
import numpy as np
import pytest

from oracle import attention as oatt
from oracle import formats as ofmt
from oracle import rotation as orot


def test_hadamard_closed_form():
    H4 = np.array([[1, 1, 1, 1], [1, -1, 1, -1], [1, 1, -1, -1], [1, -1, -1, 1]], dtype=np.float64)
    assert np.array_equal(orot.hadamard(4), H4)
    for D in (8, 128, 256):
        H = orot.hadamard(D)
        assert np.array_equal(H @ H.T, D * np.eye(D))
        assert np.array_equal(H, H.T)
        # entry (i, j) = (-1)^popcount(i & j)
        i, j = np.meshgrid(np.arange(D), np.arange(D), indexing="ij")
        pc = np.vectorize(lambda v: bin(v).count("1"))(i & j)
        assert np.array_equal(H, np.where(pc % 2, -1.0, 1.0))


def test_signs_from_hand_computed_hash_values():
    # (i + 1) * 2654435761 mod 2^32 for i = 0, 1, 2 is 0x9E3779B1, 0x3C6EF362,
    # 0xDAA66D13: bit 31 set, clear, set
    assert list(orot.signs(3)) == [-1.0, 1.0, -1.0]
    s = orot.signs(256)
    assert set(np.unique(s)) == {-1.0, 1.0}
    assert abs(s.sum()) < 64  # a spread of signs, not a constant


@pytest.mark.parametrize("D", [128, 256])
def test_rotation_is_orthogonal(D):
    rng = np.random.default_rng(0)
    x = rng.standard_normal((50, D))
    y = orot.rotate_exact(x)
    assert np.allclose(orot.rotate_exact(y, inverse=True), x, atol=1e-12)
    assert np.allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-12)
    k = rng.standard_normal((7, D))
    assert np.allclose(y @ orot.rotate_exact(k).T, x @ k.T, atol=1e-10)


@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("inverse", [False, True])
def test_fp32_butterfly_matches_the_matrix(D, inverse):
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((40, D)) * np.exp(rng.uniform(-3, 3, (40, 1)))).astype(np.float32)
    ref = orot.rotate_exact(x.astype(np.float64), inverse)
    got = orot.rotate_fp32(x, inverse, out="f32").astype(np.float64)
    # fp32 butterfly: log2(D) roundings of partial sums bounded by the row's 1-norm
    bound = 2.0 ** -23 * (np.log2(D) + 2) * np.abs(x).sum(axis=1, keepdims=True) / np.sqrt(D)
    assert np.all(np.abs(got - ref) <= bound)
    # bf16 output: the fp32 result rounded to nearest bf16
    b = orot.rotate_fp32(x, inverse, out="bf16").astype(np.float64)
    assert np.all(np.abs(b - got) <= 2.0 ** -8 * np.abs(got))


def test_attention_is_invariant_under_the_rotation():
    rng = np.random.default_rng(2)
    D, L = 256, 90
    q = rng.standard_normal((3, D))
    k = rng.standard_normal((L, D))
    v = rng.standard_normal((L, D))
    sm = 1.0 / 16
    o, lse = oatt.attend(q, k, v, sm)
    o_r, lse_r = oatt.attend(orot.rotate_exact(q), orot.rotate_exact(k), orot.rotate_exact(v), sm)
    assert np.allclose(orot.rotate_exact(o_r, inverse=True), o, atol=1e-12)
    assert np.allclose(lse_r, lse, atol=1e-12)


def test_rotation_lowers_per_token_int8_error_on_outlier_channels():
    # the page's motivation: outlier channels force a large per-row scale; spread
    # over all dimensions they cost less.  One scale per 256 values (the INT8
    # format) gains; NVFP4's 16-element groups already isolate such channels.
    rng = np.random.default_rng(3)
    D = 256
    x = rng.standard_normal((256, D))
    x[:, [3, 70, 131, 200]] *= 8.0
    x = x.astype(np.float32)

    def rel_err(rows):
        back = ofmt.int8_dequantize(*ofmt.int8_quantize(rows))
        return np.sqrt(((back - rows) ** 2).sum() / (rows.astype(np.float64) ** 2).sum())

    xr = orot.rotate_fp32(x, out="bf16")
    assert rel_err(xr) < 0.5 * rel_err(x)
