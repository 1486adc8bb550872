"""The C-ABI library builds, loads and exports every declared symbol (no GPU).

Only argument checks that return before any CUDA call are exercised here;
nothing is launched.
"""
import ctypes
import os
import re

import pytest

from decode_attention_kv_split_gb300 import api
from decode_attention_kv_split_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")


def declared_symbols():
    names = set()
    for fn in os.listdir(HEADER_DIR):
        if fn.endswith(".h"):
            text = open(os.path.join(HEADER_DIR, fn)).read()
            names |= set(re.findall(r"DA_API\s+[\w\s\*]+?\b(\w+)\s*\(", text))
    return names


@pytest.fixture(scope="module")
def lib():
    build()
    return api.load()


def test_header_declares_expected_entry_points():
    names = declared_symbols()
    assert {"decode_attn", "decode_attn_ex", "kv_append", "decode_attn_workspace_bytes"} <= names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
    # and the binding declares a signature for each of them
    assert declared_symbols() == set(api.SIGNATURES)


def test_status_strings(lib):
    for st in range(0, -9, -1):
        s = lib.decode_attn_status_string(st).decode()
        assert s and s != "unknown status"
    assert lib.decode_attn_status_string(5).decode() == "unknown status"


def _decode_ex(lib, q=16, K=16, V=16, lens=16, out=16, B=1, h_q=1, h_kv=1, d_k=64, d_v=64,
               n_max=8, scale=0.125, dtype=0, splits=0):
    P = ctypes.c_void_p
    return lib.decode_attn_ex(P(q) if q else None, P(K) if K else None, P(V) if V else None,
                              P(lens) if lens else None, P(out) if out else None, B, h_q, h_kv,
                              d_k, d_v, n_max, scale, dtype, splits, None, 0, None, None)


def test_argument_errors_return_before_touching_cuda(lib):
    assert _decode_ex(lib, q=0) == -1                      # DA_ERR_NULL
    assert _decode_ex(lib, out=0) == -1
    assert _decode_ex(lib, h_q=3, h_kv=2) == -2            # DA_ERR_SHAPE: h_q % h_kv
    assert _decode_ex(lib, B=0) == -2
    assert _decode_ex(lib, n_max=0) == -2
    assert _decode_ex(lib, n_max=(1 << 30) + 1) == -2
    assert _decode_ex(lib, dtype=7) == -3                  # DA_ERR_DTYPE
    assert _decode_ex(lib, dtype=0x200) == -3              # unknown flag bit
    assert _decode_ex(lib, dtype=api.DA_OUT_BF16 | 7) == -3
    assert _decode_ex(lib, d_k=96, d_v=96) == -8           # DA_ERR_UNSUPPORTED
    assert _decode_ex(lib, d_k=64, d_v=128) == -8
    assert _decode_ex(lib, d_k=256, d_v=256) == -8         # d = 256 only for bf16 caches
    assert _decode_ex(lib, d_k=192, d_v=128) == -8         # d_k 192 / d_v 128 likewise
    assert _decode_ex(lib, d_k=192, d_v=64, dtype=api.DA_BF16) == -8
    assert _decode_ex(lib, d_k=128, d_v=256, dtype=api.DA_BF16) == -8
    assert _decode_ex(lib, scale=float("nan")) == -2
    assert _decode_ex(lib, q=24) == -4                     # DA_ERR_ALIGN
    assert _decode_ex(lib, K=8) == -4


def test_kv_append_argument_errors(lib):
    P = ctypes.c_void_p
    ok = P(16)
    assert lib.kv_append(None, ok, ok, ok, ok, 1, 1, 64, 64, 8, 0, None, None) == -1
    assert lib.kv_append(ok, ok, ok, ok, ok, 1, 1, 64, 64, 8, 5, None, None) == -3
    # no output, so no output-type flag
    assert lib.kv_append(ok, ok, ok, ok, ok, 1, 1, 64, 64, 8, api.DA_OUT_BF16, None, None) == -3
    assert lib.kv_append(ok, ok, ok, ok, ok, 0, 1, 64, 64, 8, 0, None, None) == -2
    assert lib.kv_append(ok, ok, ok, ok, ok, 1, 1, 6, 64, 8, 1, None, None) == -2   # 12-byte rows
    assert lib.kv_append(ok, P(20), ok, ok, ok, 1, 1, 64, 64, 8, 0, None, None) == -4


def test_q8_argument_errors(lib):
    """8-bit caches: wrong entry point, missing scales, bad sizes; all before any CUDA call."""
    P = ctypes.c_void_p
    ok = P(16)

    def q8(dtype=api.DA_FP8_E4M3, ks=16, vs=16, n_max=8, d=64):
        return lib.decode_attn_q8_ex(ok, ok, ok, P(ks) if ks else None, P(vs) if vs else None, ok,
                                     ok, 1, 1, 1, d, d, n_max, 0.125, dtype, 0, None, 0, None, None)
    assert q8(dtype=api.DA_BF16) == -3                 # not an 8-bit type
    assert q8(ks=0) == -1                              # scales required
    assert q8(n_max=6) == -2                           # n_max % 4
    assert q8(d=96) == -8
    assert q8(ks=8) == -4                              # scales 16-byte aligned
    assert _decode_ex(lib, dtype=api.DA_INT8) == -3    # 8-bit cache through the 16/32-bit entry
    assert _decode_ex(lib, dtype=api.DA_FP8_E4M3 | api.DA_OUT_BF16) == -3
    assert lib.kv_append(ok, ok, ok, ok, ok, 1, 1, 64, 64, 8, api.DA_INT8, None, None) == -3
    assert lib.kv_append_q8(ok, ok, None, ok, ok, ok, ok, ok, ok, 1, 1, 64, 64, 8, api.DA_INT8,
                            None, None) == -1
    assert lib.kv_append_q8(ok, ok, ok, ok, ok, ok, ok, ok, ok, 1, 1, 64, 64, 8, api.DA_BF16,
                            None, None) == -3
    assert lib.kv_quantize(ok, api.DA_FP32, ok, ok, 4, 48, api.DA_INT8, None) == -2   # d % 32
    assert lib.kv_quantize(ok, api.DA_FP32, ok, ok, 4, 512, api.DA_INT8, None) == -2  # d > 256
    assert lib.kv_quantize(ok, api.DA_INT8, ok, ok, 4, 64, api.DA_INT8, None) == -3   # x type
    assert lib.kv_quantize(ok, api.DA_FP32, ok, ok, 4, 64, api.DA_BF16, None) == -3   # code type
    assert lib.kv_quantize(None, api.DA_FP32, ok, ok, 4, 64, api.DA_INT8, None) == -1
    assert lib.kv_quantize(ok, api.DA_FP32, ok, ok, 0, 64, api.DA_INT8, None) == 0    # nothing to do


def test_header_constants_match_binding():
    text = open(os.path.join(HEADER_DIR, "decode_attn.h")).read()
    defs = dict(re.findall(r"#define\s+(DA_\w+)\s+(0x[0-9a-fA-F]+|\d+)", text))
    assert int(defs["DA_OUT_BF16"], 0) == api.DA_OUT_BF16
    enum = dict(re.findall(r"(DA_(?:FP32|BF16|INT8|FP8_E4M3))\s*=\s*(\d+)", text))
    assert {k: int(v) for k, v in enum.items()} == {
        "DA_FP32": api.DA_FP32, "DA_BF16": api.DA_BF16, "DA_INT8": api.DA_INT8,
        "DA_FP8_E4M3": api.DA_FP8_E4M3}
    assert int(defs["DA_DEVERR_SEQ_LEN"], 0) == api.DEVERR_SEQ_LEN
    assert int(defs["DA_DEVERR_POS"], 0) == api.DEVERR_POS
    assert int(defs["DA_DEVERR_TIMEOUT"], 0) == api.DEVERR_TIMEOUT
    assert int(defs["DA_DEVERR_BOUNDS"], 0) == api.DEVERR_BOUNDS


def test_no_fallback_when_library_missing(tmp_path, monkeypatch):
    monkeypatch.setattr(api, "_lib", None)
    with pytest.raises(RuntimeError, match="no fallback"):
        api.load(str(tmp_path / "missing.so"))
