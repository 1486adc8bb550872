"""Plain CPU oracle for decode-step attention (fp64).

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product
library never imports, links or calls it, and the two share no code.

The arithmetic lives in ``decode_oracle.c`` (plain C, IEEE double, three
literal passes per head as in "MoA-Structured Decode Attention", section 2,
Steps I-III).  This module only compiles it with gcc and marshals numpy
arrays through ctypes.  Inputs are float32 arrays: a bf16 cache is widened
to float32 by the caller first, which is exact, so the oracle computes on
the same rounded values the GPU reads.
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "decode_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, f"liboracle_{platform.machine()}.so")

_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH,
          extra_flags: tuple[str, ...] = ()) -> str:
    """Compile the C oracle into a shared library with gcc (OpenMP on)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-fno-fast-math", "-ffp-contract=off", *extra_flags, src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def load_library(path: str) -> ctypes.CDLL:
    """Load a compiled oracle library and declare its C signatures."""
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    I = ctypes.c_int
    I64 = ctypes.c_int64
    D = ctypes.c_double
    lib.oracle_decode_head.argtypes = [P, P, P, I64, I, I, D, P, P, P]
    lib.oracle_decode_head.restype = I
    lib.oracle_decode.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I64, D, I]
    lib.oracle_decode.restype = I
    lib.oracle_lse_combine.argtypes = [P, P, I, I, P, P]
    lib.oracle_lse_combine.restype = I
    lib.oracle_kv_append.argtypes = [P, P, P, P, P, I, I, I, I, I64, I]
    lib.oracle_kv_append.restype = I
    lib.oracle_causal_attention.argtypes = [P, P, P, I, I, I, I, D, P]
    lib.oracle_causal_attention.restype = I
    lib.oracle_code_value.argtypes = [I, I]
    lib.oracle_code_value.restype = D
    lib.oracle_quantize_rows.argtypes = [P, I64, I, I, P, P]
    lib.oracle_quantize_rows.restype = I
    lib.oracle_dequant_rows.argtypes = [P, P, I64, I, I, P]
    lib.oracle_dequant_rows.restype = I
    lib.oracle_max_threads.argtypes = []
    lib.oracle_max_threads.restype = I
    return lib


def _get() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(build())
        return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


class Oracle:
    """Bound view of one compiled oracle library (the default, or a variant)."""

    def __init__(self, lib: ctypes.CDLL):
        self.lib = lib

    def decode_head(self, q, K, V, scale: float, want_weights: bool = False):
        """Decode one head over all rows of K/V ([n, d_k], [n, d_v]).

        Returns ``(out[d_v], lse)`` or ``(out, lse, a[n])`` with the softmax
        weights when ``want_weights`` is set.  lse = m + log(Z) in natural log.
        """
        q, K, V = _f32(q), _f32(K), _f32(V)
        if K.ndim != 2 or V.ndim != 2 or K.shape[0] != V.shape[0]:
            raise ValueError("K and V must be [n, d] arrays with the same n")
        n = K.shape[0]
        d_k, d_v = q.shape[0], V.shape[1]
        out = np.zeros(d_v, dtype=np.float64)
        a = np.zeros(max(n, 1), dtype=np.float64) if want_weights else None
        lse = np.zeros(1, dtype=np.float64)
        _check(self.lib.oracle_decode_head(_ptr(q), _ptr(K), _ptr(V), n, d_k, d_v,
                                           float(scale), _ptr(out), _ptr(a), _ptr(lse)),
               "decode_head")
        if want_weights:
            return out, float(lse[0]), a[:n]
        return out, float(lse[0])

    def decode(self, q, K, V, seq_lens, scale: float, threads: int = 1):
        """Batched GQA decode over a padded cache.

        q [B, h_q, d_k], K [B, h_kv, n_max, d_k], V [B, h_kv, n_max, d_v],
        seq_lens [B] -> (out [B, h_q, d_v] float64, lse [B, h_q] float64).
        """
        q, K, V = _f32(q), _f32(K), _f32(V)
        seq = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32))
        B, h_q, d_k = q.shape
        _, h_kv, n_max, _ = K.shape
        d_v = V.shape[3]
        out = np.zeros((B, h_q, d_v), dtype=np.float64)
        lse = np.zeros((B, h_q), dtype=np.float64)
        _check(self.lib.oracle_decode(_ptr(q), _ptr(K), _ptr(V), _ptr(seq), _ptr(out),
                                      _ptr(lse), B, h_q, h_kv, d_k, d_v, n_max,
                                      float(scale), int(threads)), "decode")
        return out, lse

    def lse_combine(self, o_parts, lse_parts):
        """Merge partial (o_s, lse_s) over disjoint row ranges -> (out, lse)."""
        o = np.ascontiguousarray(np.asarray(o_parts, dtype=np.float64))
        lp = np.ascontiguousarray(np.asarray(lse_parts, dtype=np.float64))
        S, d_v = o.shape
        out = np.zeros(d_v, dtype=np.float64)
        lse = np.zeros(1, dtype=np.float64)
        _check(self.lib.oracle_lse_combine(_ptr(o), _ptr(lp), S, d_v, _ptr(out), _ptr(lse)),
               "lse_combine")
        return out, float(lse[0])

    def kv_append(self, k_new: np.ndarray, v_new: np.ndarray, K: np.ndarray,
                  V: np.ndarray, pos) -> int:
        """Write row pos[b] of every (b, h) in place; returns #skipped sequences.

        Arrays may be any fixed-size dtype (bf16 caches are passed as uint16
        views); all four must share it.
        """
        for a in (k_new, v_new, K, V):
            if not a.flags.c_contiguous:
                raise ValueError("kv_append oracle needs C-contiguous arrays")
        es = K.dtype.itemsize
        if not (k_new.dtype.itemsize == v_new.dtype.itemsize == V.dtype.itemsize == es):
            raise ValueError("element sizes differ")
        p = np.ascontiguousarray(np.asarray(pos, dtype=np.int32))
        B, h_kv, n_max, d_k = K.shape
        d_v = V.shape[3]
        rc = self.lib.oracle_kv_append(_ptr(k_new), _ptr(v_new), _ptr(K), _ptr(V), _ptr(p),
                                       B, h_kv, d_k, d_v, n_max, es)
        if rc < 0:
            raise RuntimeError(f"oracle kv_append failed with code {rc}")
        return rc

    def causal_attention(self, Q, K, V, scale: float):
        """Full causal attention per head: Q,K [H,T,d_k], V [H,T,d_v] -> [H,T,d_v]."""
        Q, K, V = _f32(Q), _f32(K), _f32(V)
        H, T, d_k = Q.shape
        d_v = V.shape[2]
        out = np.zeros((H, T, d_v), dtype=np.float64)
        _check(self.lib.oracle_causal_attention(_ptr(Q), _ptr(K), _ptr(V), H, T, d_k, d_v,
                                                float(scale), _ptr(out)), "causal_attention")
        return out

    # ---- 8-bit caches (kind 1: int8, kind 2: fp8 e4m3; see decode_oracle.c)
    def code_value(self, code: int, kind: int) -> float:
        """The value one 8-bit code stands for."""
        return float(self.lib.oracle_code_value(int(code), int(kind)))

    def quantize(self, x, kind: int):
        """Rows x [..., d] (float32) -> (codes uint8 [..., d], scales float32 [...])."""
        x = _f32(x)
        d = x.shape[-1]
        rows = x.size // d
        codes = np.zeros(x.shape, dtype=np.uint8)
        scales = np.zeros(x.shape[:-1], dtype=np.float32)
        _check(self.lib.oracle_quantize_rows(_ptr(x), rows, d, int(kind), _ptr(codes),
                                             _ptr(scales)), "quantize_rows")
        return codes, scales

    def dequant(self, codes, scales, kind: int) -> np.ndarray:
        """codes uint8 [..., d], scales float32 [...] -> values float64 [..., d]."""
        codes = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8))
        scales = _f32(scales)
        d = codes.shape[-1]
        rows = codes.size // d
        if scales.size != rows:
            raise ValueError("one scale per row")
        out = np.zeros(codes.shape, dtype=np.float64)
        _check(self.lib.oracle_dequant_rows(_ptr(codes), _ptr(scales), rows, d, int(kind),
                                            _ptr(out)), "dequant_rows")
        return out

    def max_threads(self) -> int:
        return int(self.lib.oracle_max_threads())


def get() -> Oracle:
    """The oracle compiled from ``decode_oracle.c`` as committed."""
    return Oracle(_get())


# Module-level conveniences bound to the default build.
def decode_head(*a, **k):
    return get().decode_head(*a, **k)


def decode(*a, **k):
    return get().decode(*a, **k)


def lse_combine(*a, **k):
    return get().lse_combine(*a, **k)


def kv_append(*a, **k):
    return get().kv_append(*a, **k)


def causal_attention(*a, **k):
    return get().causal_attention(*a, **k)


def max_threads() -> int:
    return get().max_threads()
