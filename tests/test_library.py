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


def test_header_constants_match_binding():
    text = open(os.path.join(HEADER_DIR, "decode_attn.h")).read()
    defs = dict(re.findall(r"#define\s+(DA_\w+)\s+(0x[0-9a-fA-F]+|\d+)", text))
    assert int(defs["DA_OUT_BF16"], 0) == api.DA_OUT_BF16
    assert int(defs["DA_DEVERR_SEQ_LEN"], 0) == api.DEVERR_SEQ_LEN
    assert int(defs["DA_DEVERR_POS"], 0) == api.DEVERR_POS
    assert int(defs["DA_DEVERR_TIMEOUT"], 0) == api.DEVERR_TIMEOUT


def test_no_fallback_when_library_missing(tmp_path, monkeypatch):
    monkeypatch.setattr(api, "_lib", None)
    with pytest.raises(RuntimeError, match="no fallback"):
        api.load(str(tmp_path / "missing.so"))
