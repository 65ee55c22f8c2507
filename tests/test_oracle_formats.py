"""The oracle's codecs against independent pins (CPU only)."""
import numpy as np

from oracle import formats
from tests import oracle_pins as pins


def test_int8_matches_exact_rational_arithmetic():
    pins.check_int8_exact(formats.int8_quantize)


def test_int8_every_bf16_value_at_fixed_scales():
    pins.check_int8_exhaustive_bf16(formats.int8_quantize)


def test_nvfp4_every_bf16_value_at_fixed_group_scales():
    pins.check_nvfp4_exhaustive_bf16(formats.nvfp4_quantize, formats.unpack_nibbles)


def test_int8_ties_round_half_to_even():
    pins.check_int8_ties(formats.int8_quantize)


def test_int8_invariants():
    pins.check_int8_invariants(formats.int8_quantize, formats.int8_dequantize)


def test_int8_group_matches_exact_rational_arithmetic():
    pins.check_int8_group_exact(formats.int8_group_quantize)


def test_int8_group_hand_example():
    pins.check_int8_group_hand_example(formats.int8_group_quantize, formats.int8_group_dequantize)


def test_int8_group_invariants():
    pins.check_int8_group_invariants(formats.int8_group_quantize, formats.int8_group_dequantize,
                                     formats.int8_quantize)


def test_e4m3_decode_matches_torch_float8():
    pins.check_e4m3_decode(formats.e4m3_value)


def test_e4m3_encode_matches_torch_float8():
    pins.check_e4m3_encode(formats.e4m3_encode_satfinite)


def test_e2m1_grid_is_the_pages_grid():
    pins.check_e2m1_grid(formats.e2m1_value)


def test_e2m1_ties_and_signed_zero():
    pins.check_e2m1_ties(formats.e2m1_encode)


def test_nibble_order_is_the_pages_order():
    pins.check_nibble_order(formats.pack_nibbles)
    rng = np.random.default_rng(0)
    c = rng.integers(0, 16, (5, 32)).astype(np.uint8)
    assert np.array_equal(formats.unpack_nibbles(formats.pack_nibbles(c)), c)


def test_nvfp4_matches_exact_rational_arithmetic():
    pins.check_nvfp4_exact(formats.nvfp4_quantize, formats.unpack_nibbles)


def test_nvfp4_invariants():
    pins.check_nvfp4_invariants(formats.nvfp4_quantize, formats.nvfp4_dequantize, formats.e4m3_value)


def test_nvfp4_group_max_maps_to_six_when_scale_is_exact():
    # amax = 6 * 2^k with gs = 1 -> t2 = 2^k is an exact E4M3 value -> code 7 (= 6)
    x = np.zeros((1, 32), np.float32)
    x[0, 3] = 6.0 * 0.25
    x[0, 20] = -6.0 * 4.0
    x[0, 21] = 4.0
    codes, scales = formats.nvfp4_quantize(x, 1.0)
    c = formats.unpack_nibbles(codes)[0]
    assert c[3] == 7 and c[20] == 15 and c[21] == 2  # 4 / 4 = 1.0 -> code 2
    assert list(formats.e4m3_value(scales[0])) == [0.25, 4.0]


def test_nvfp4_tensor_global_scale():
    x = np.array([[0.5, -3.0, 2.0]], np.float32)
    assert formats.nvfp4_tensor_global_scale(x) == np.float32(2688.0) / np.float32(3.0)
    assert formats.nvfp4_tensor_global_scale(np.zeros(4, np.float32)) == 1.0
