"""Byte and flop accounting against the pages' formulas (no GPU)."""
from decode_attention_kv_split_gb300 import accounting as acc


def test_moa_traffic_formula_single_head_fp32():
    # "MoA-Structured Decode Attention", introduction item 1:
    # M = (d_k + n d_k + n d_v + d_v) x 4 bytes for one head.
    for n, d_k, d_v in [(256, 64, 64), (257, 64, 64), (4096, 128, 128), (3, 2, 2), (10, 64, 32)]:
        assert acc.decode_bytes([n], 1, 1, d_k, d_v, 4) == (d_k + n * d_k + n * d_v + d_v) * 4


def test_gqa_reads_cache_once_per_kv_head():
    # Introduction item 4: traffic for the cache falls by h_q / h_kv.
    mha = acc.decode_bytes([1000], 32, 32, 128, 128, 2) - 32 * 128 * (2 + 4)
    gqa = acc.decode_bytes([1000], 32, 8, 128, 128, 2) - 32 * 128 * (2 + 4)
    assert mha == 4 * gqa


def test_arithmetic_intensity_is_group_ratio_for_bf16():
    # "Attention over the KV cache in the decode step": AI = n_q / n_kv for
    # bf16 KV, independent of batch and context (cache bytes only).
    for h_q, h_kv in [(32, 32), (32, 8), (64, 8), (32, 1)]:
        for lens in ([4096], [1024, 8192, 77]):
            flops = acc.decode_flops(lens, h_q, 128, 128)
            cache = sum(lens) * h_kv * 256 * 2
            assert flops / cache == h_q / h_kv


def test_kv_bytes_per_token_examples():
    # Same page: 2 * layers * n_kv * d_h * 2 bytes per token.
    per_token = lambda layers, n_kv: layers * (acc.decode_bytes([1], n_kv, n_kv, 128, 128, 2)
                                              - n_kv * 128 * (2 + 4))
    assert per_token(32, 32) == 512 * 1024      # Llama-2-7B
    assert per_token(80, 8) == 320 * 1024       # Llama-2-70B
    assert per_token(32, 8) == 128 * 1024       # Llama-3-8B


def test_q8_bytes_per_row():
    """An 8-bit row: d codes of one byte plus a float32 scale, for K and for V."""
    from decode_attention_kv_split_gb300 import accounting
    one = accounting.decode_bytes_q8([1], 1, 1, 128, 128) - accounting.decode_bytes_q8([0], 1, 1, 128, 128)
    assert one == 2 * (128 + 4)
    # bf16 q and fp32 out around them
    assert accounting.decode_bytes_q8([0], 4, 1, 128, 128) == 4 * 128 * 2 + 4 * 128 * 4
    assert accounting.append_bytes_q8(2, 3, 64, 64) == 2 * 2 * 3 * (64 + 4 + 64 + 4)
