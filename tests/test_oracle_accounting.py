"""Byte accounting of the oracle against the closed forms the pages print."""
from oracle import accounting as acc
from tests import oracle_pins as pins

GiB = 1 << 30
MiB = 1 << 20


def test_closed_forms():
    cf = pins.closed_forms()
    assert acc.bytes_per_token("bf16", 16, 4, 256) == cf["bf16_bytes_per_token_16L_4H_D256"]
    assert acc.token_slots(GiB, acc.bytes_per_token("bf16", 16, 4, 256)) == cf["slots_per_gib_bf16_16L_4H_D256"]
    assert acc.bytes_per_token_head("int8", 256) == cf["int8_bytes_per_token_head_D256"]
    assert acc.bytes_per_token_head("bf16", 256) == cf["bf16_bytes_per_token_head_D256"]
    assert round(1000 * acc.bytes_per_token_head("int8", 256) / acc.bytes_per_token_head("bf16", 256)) == cf["int8_over_bf16_ratio_x1000"]
    assert acc.record_bytes("int8", 256) == cf["int8_record_stride_D256"]
    assert acc.bytes_per_token_layer("nvfp4", 2, 256) == cf["nvfp4_bytes_per_token_layer_2H_D256"]
    assert acc.bytes_per_token_layer("bf16", 2, 256) == cf["bf16_bytes_per_token_layer_2H_D256"]
    assert acc.bytes_per_token_layer("fp8", 2, 256) == cf["fp8_bytes_per_token_layer_2H_D256"]
    n, b, f = (acc.bytes_per_token_layer(x, 2, 256) for x in ("nvfp4", "bf16", "fp8"))
    assert round(100 * b / n) == cf["nvfp4_vs_bf16_x100"]
    assert round(100 * f / n) == cf["nvfp4_vs_fp8_x100"]
    assert round(10000 * (1 - n / f)) == cf["nvfp4_smaller_than_fp8_pct_x100"]
    assert acc.bytes_per_token_head("nvfp4", 256) == cf["nvfp4_bytes_per_kv_head_D256"]
    assert acc.record_bytes("nvfp4", 256) == cf["nvfp4_record_bytes_D256"]
    assert 3136 * n == cf["nvfp4_page_bytes_3136_tokens"]
    assert acc.token_slots(3207168, n) == cf["nvfp4_tokens_in_3207168_byte_page"]
    kv32k = acc.decode_kv_bytes("bf16", [32768], 16 * 4, 256)  # 16 layers x 4 KV heads
    assert round(kv32k / 1e8) == cf["bf16_kv_bytes_32k_context_x100M"]
    assert round(kv32k / 3.5e-3 / 1e9, -1) == cf["bf16_32k_read_rate_gbs_3p5ms"]
    assert acc.conversion_scratch_bytes(131072, 4, 256) // MiB == cf["fp16_scratch_128k_mib"]
    assert acc.conversion_scratch_bytes(32768, 4, 256) // MiB == cf["fp16_scratch_32k_mib"]
    assert round(acc.attention_flops(64, 131072, 256, 4) / 1e9) == cf["verify_gflop_128k_64rows"]


def test_per_32_scale_record():
    # one fp32 scale per 32 values: 256 codes + 8 scales, 128 codes + 4 scales
    assert acc.record_bytes("int8_g32", 256) == 256 + 8 * 4
    assert acc.record_bytes("int8_g32", 128) == 128 + 4 * 4
    # 28 bytes more than one scale per 256 values at D = 256
    assert acc.record_bytes("int8_g32", 256) - acc.record_bytes("int8", 256) == 28
