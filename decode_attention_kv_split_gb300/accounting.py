"""Algorithmic bytes and flops of one decode-attention call.

Traffic follows the minimal-traffic count of "MoA-Structured Decode
Attention" (introduction item 1): per head, the query (d_k elements), every
cached key and value row (n * d_k + n * d_v elements) and the output (d_v
elements), each moved once, i.e. (d_k + n d_k + n d_v + d_v) x 4 bytes for
fp32.  Lifted to a batch with GQA/MQA (introduction item 4), the cache is
read once per KV head, not once per query head, and q/out are per query head.
The output is float32 whatever the input dtype.  Split-KV partials are not
algorithmic: they are overhead and are measured, not counted here.

Flops follow "Attention over the KV cache in the decode step":
4 * L * d_h * n_q per token (2 for q.K, 2 for p.V).
"""
from __future__ import annotations

from collections.abc import Sequence

ELEM_BYTES = {"fp32": 4, "bf16": 2}


def decode_bytes(seq_lens: Sequence[int], h_q: int, h_kv: int, d_k: int, d_v: int,
                 elem_bytes: int, out_bytes: int = 4) -> int:
    """Bytes one decode_attn call must move: K/V rows read, q read, out written."""
    rows = sum(int(n) for n in seq_lens)
    B = len(seq_lens)
    kv = rows * h_kv * (d_k + d_v) * elem_bytes
    q = B * h_q * d_k * elem_bytes
    out = B * h_q * d_v * out_bytes
    return kv + q + out


def append_bytes(B: int, h_kv: int, d_k: int, d_v: int, elem_bytes: int) -> int:
    """Bytes one kv_append call moves: the new rows read once and written once."""
    return 2 * B * h_kv * (d_k + d_v) * elem_bytes


def decode_bytes_q8(seq_lens: Sequence[int], h_q: int, h_kv: int, d_k: int, d_v: int,
                    out_bytes: int = 4) -> int:
    """decode_bytes for an 8-bit cache: every cached K and V row is one byte per
    element plus one float32 scale; q is bf16."""
    rows = sum(n for n in seq_lens)
    B = len(seq_lens)
    kv = rows * h_kv * (d_k + 4 + d_v + 4)
    return int(kv + B * h_q * d_k * 2 + B * h_q * d_v * out_bytes)


def append_bytes_q8(B: int, h_kv: int, d_k: int, d_v: int) -> int:
    """append_bytes for an 8-bit cache: code rows and their scales, read once and written once."""
    return 2 * B * h_kv * (d_k + 4 + d_v + 4)


def decode_flops(seq_lens: Sequence[int], h_q: int, d_k: int, d_v: int) -> int:
    """Multiply-adds x 2 for q.K over every row and p.V over every row."""
    rows = sum(int(n) for n in seq_lens)
    return 2 * rows * h_q * (d_k + d_v)
