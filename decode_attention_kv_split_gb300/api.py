"""Python binding over libdecode_attn.so (ctypes; argument marshalling only).

Every step of the computation runs in the library's CUDA kernels.  This
module checks tensor shapes/dtypes/devices, takes raw device pointers and the
current CUDA stream from PyTorch, allocates the split workspace with PyTorch,
and calls the C entry points of the same names.  There is no CPU fallback:
if the shared library is missing the first call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdecode_attn.so")

DA_FP32 = 0
DA_BF16 = 1
DA_INT8 = 2          # 8-bit caches: one-byte codes + a float32 scale per cached row
DA_FP8_E4M3 = 3
DA_OUT_BF16 = 0x100  # dtype flag: out is bfloat16
DEVERR_SEQ_LEN = 1
DEVERR_POS = 2
DEVERR_TIMEOUT = 4
DEVERR_BOUNDS = 8    # set only by the bounds-checked test build

_DTYPES = {torch.float32: DA_FP32, torch.bfloat16: DA_BF16}
# 8-bit caches are passed as torch.int8 / torch.float8_e4m3fn tensors of codes
_Q8_DTYPES = {torch.int8: DA_INT8, torch.float8_e4m3fn: DA_FP8_E4M3}
_ALL_DTYPES = {**_DTYPES, **_Q8_DTYPES}

_lock = threading.Lock()
_lib = None

# Every entry point of include/decode_attn.h with its ctypes signature.
_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_SZ = ctypes.c_size_t
SIGNATURES = {
    "decode_attn_resolve_splits": (_I, [_I, _I, _I, _I, _I, _I, _I, _I]),
    "decode_attn_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I, _I, _I, _I, ctypes.POINTER(_I)]),
    "decode_attn_ex": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _I, _P, _SZ, _P, _P]),
    "decode_attn": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _P]),
    "decode_attn_append": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _I,
                                _P, _SZ, _P, _P]),
    "decode_attn_noalloc": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _I, _P, _P]),
    "kv_append": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P]),
    "decode_attn_status_string": (ctypes.c_char_p, [_I]),
    "decode_attn_last_cuda_error": (ctypes.c_char_p, []),
    "decode_attn_launch_count": (ctypes.c_uint64, []),
    "decode_attn_q8_ex": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _I, _P,
                               _SZ, _P, _P]),
    "decode_attn_q8_append": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I,
                                   _I, _I, _F, _I, _I, _P, _SZ, _P, _P]),
    "kv_append_q8": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P]),
    "kv_quantize": (_I, [_P, _I, _P, _P, ctypes.c_longlong, _I, _I, _P]),
    "decode_attn_partial": (_I, [_P, _P, _P, _P, _I, _I, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I,
                                 _I, _P, _SZ, _P, _P]),
    "decode_attn_combine": (_I, [_P, _P, _I, _P, _P, _I, _I, _I, _I, _P]),
}


class DecodeAttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        lib = load()
        msg = lib.decode_attn_status_string(status).decode()
        if status == -6:
            msg += ": " + lib.decode_attn_last_cuda_error().decode()
        super().__init__(f"{where}: {msg} (status {status})")
        self.status = status


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the shared library once; raise if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{path} is missing: build it with __graft_entry__.build() "
                    "(there is no fallback implementation)")
            lib = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
        return _lib


def _check(status: int, where: str) -> None:
    if status != 0:
        raise DecodeAttnError(status, where)


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(t: torch.Tensor, stream) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream(t.device)
    return ctypes.c_void_p(s.cuda_stream)


class _on_device:
    """Make t's device current for the call (a no-op when it already is)."""

    def __init__(self, t: torch.Tensor):
        self.idx = t.device.index
        self.prev = None

    def __enter__(self):
        cur = torch.cuda.current_device()
        if self.idx is not None and cur != self.idx:
            self.prev = cur
            torch.cuda.set_device(self.idx)

    def __exit__(self, *exc):
        if self.prev is not None:
            torch.cuda.set_device(self.prev)


def _cache_dims(q, K, V, seq_lens):
    if q.dim() != 3 or K.dim() != 4 or V.dim() != 4:
        raise ValueError("expected q [B, h_q, d_k], K [B, h_kv, n_max, d_k], V [B, h_kv, n_max, d_v]")
    B, h_q, d_k = q.shape
    Bk, h_kv, n_max, d_k2 = K.shape
    Bv, h_kv2, n_max2, d_v = V.shape
    if (Bk, Bv) != (B, B) or h_kv2 != h_kv or n_max2 != n_max or d_k2 != d_k:
        raise ValueError("q, K and V shapes disagree")
    if seq_lens.shape != (B,) or seq_lens.dtype != torch.int32:
        raise ValueError("seq_lens must be an int32 tensor of shape [B]")
    for name, t in (("q", q), ("K", K), ("V", V), ("seq_lens", seq_lens)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if not (q.dtype == K.dtype == V.dtype) or q.dtype not in _DTYPES:
        raise ValueError("q, K, V must share dtype float32 or bfloat16")
    return B, h_q, h_kv, d_k, d_v, n_max


def resolve_splits(B, h_q, h_kv, d_k, d_v, n_max, dtype: torch.dtype, num_splits: int = 0) -> int:
    """Splits per (b, kv head) the library uses for this request (on the current device).
    ``dtype`` is the cache's element type (torch.int8 / torch.float8_e4m3fn: 8-bit caches)."""
    r = load().decode_attn_resolve_splits(B, h_q, h_kv, d_k, d_v, n_max, _ALL_DTYPES[dtype],
                                          num_splits)
    if r < 0:
        raise DecodeAttnError(r, "decode_attn_resolve_splits")
    return r


_ws_bytes_cache: dict = {}


def workspace_bytes(B, h_q, h_kv, d_k, d_v, n_max, dtype: torch.dtype, num_splits: int = 0) -> int:
    key = (torch.cuda.current_device(), B, h_q, h_kv, d_k, d_v, n_max, dtype, num_splits)
    hit = _ws_bytes_cache.get(key)
    if hit is not None:
        return hit
    st = ctypes.c_int(0)
    n = load().decode_attn_workspace_bytes(B, h_q, h_kv, d_k, d_v, n_max, _ALL_DTYPES[dtype],
                                           num_splits, ctypes.byref(st))
    _check(st.value, "decode_attn_workspace_bytes")
    _ws_bytes_cache[key] = int(n)
    return int(n)


_ws_cache: dict = {}


def _out(out: torch.Tensor | None, out_dtype: torch.dtype | None, B: int, h_q: int, d_v: int,
         device: torch.device) -> tuple[torch.Tensor, int]:
    """The output tensor (allocated when None) and its dtype flag."""
    if out is None:
        out = torch.empty((B, h_q, d_v), dtype=out_dtype or torch.float32, device=device)
    if (out.shape != (B, h_q, d_v) or out.dtype not in (torch.float32, torch.bfloat16)
            or not out.is_contiguous() or out.device != device
            or (out_dtype is not None and out.dtype != out_dtype)):
        raise ValueError("out must be a contiguous float32 or bfloat16 tensor [B, h_q, d_v] "
                         "on the query's device")
    return out, (DA_OUT_BF16 if out.dtype == torch.bfloat16 else 0)


def _workspace(device: torch.device, nbytes: int) -> torch.Tensor | None:
    if nbytes == 0:
        return None
    key = (device.index, torch.cuda.current_stream(device).cuda_stream)
    ws = _ws_cache.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
        _ws_cache[key] = ws
    return ws


def decode_attn(q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, seq_lens: torch.Tensor,
                out: torch.Tensor | None = None, scale: float | None = None, num_splits: int = 0,
                workspace: torch.Tensor | None = None, dev_error: torch.Tensor | None = None,
                stream: torch.cuda.Stream | None = None,
                out_dtype: torch.dtype | None = None) -> torch.Tensor:
    """Decode attention (calls ``decode_attn_ex``); returns ``out`` [B, h_q, d_v], float32
    or bfloat16 (``out_dtype``, or the dtype of a given ``out``).

    ``scale`` defaults to 1/sqrt(d_k).  ``workspace`` (uint8 CUDA tensor) is
    allocated and cached per stream when not given.  ``dev_error`` is an
    optional int32 CUDA scalar the kernels OR error bits into.
    """
    B, h_q, h_kv, d_k, d_v, n_max = _cache_dims(q, K, V, seq_lens)
    if scale is None:
        scale = 1.0 / math.sqrt(d_k)
    out, oflag = _out(out, out_dtype, B, h_q, d_v, q.device)
    dt = _DTYPES[q.dtype] | oflag
    lib = load()
    with _on_device(q):
        need = workspace_bytes(B, h_q, h_kv, d_k, d_v, n_max, q.dtype, num_splits)
        if workspace is None:
            workspace = _workspace(q.device, need)
        nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        st = lib.decode_attn_ex(_ptr(q), _ptr(K), _ptr(V), _ptr(seq_lens), _ptr(out), B, h_q, h_kv,
                                d_k, d_v, n_max, float(scale), dt, int(num_splits), _ptr(workspace),
                                nbytes, _ptr(dev_error), _stream(q, stream))
    _check(st, "decode_attn_ex")
    return out


def decode_attn_append(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor, K: torch.Tensor,
                       V: torch.Tensor, seq_lens: torch.Tensor, out: torch.Tensor | None = None,
                       seq_lens_out: torch.Tensor | None = None, scale: float | None = None,
                       num_splits: int = 0, workspace: torch.Tensor | None = None,
                       dev_error: torch.Tensor | None = None,
                       stream: torch.cuda.Stream | None = None,
                       out_dtype: torch.dtype | None = None) -> torch.Tensor:
    """Append row seq_lens[b] of every kv head and decode over seq_lens[b] + 1 rows,
    in one launch (calls ``decode_attn_append``); returns ``out``."""
    B, h_q, h_kv, d_k, d_v, n_max = _cache_dims(q, K, V, seq_lens)
    if k_new.shape != (B, h_kv, d_k) or v_new.shape != (B, h_kv, d_v):
        raise ValueError("k_new/v_new must be [B, h_kv, d]")
    for name, t in (("k_new", k_new), ("v_new", v_new)):
        if not t.is_cuda or not t.is_contiguous() or t.dtype != K.dtype:
            raise ValueError(f"{name} must be a contiguous CUDA tensor of the cache dtype")
    if seq_lens_out is not None and (seq_lens_out.shape != (B,) or seq_lens_out.dtype != torch.int32):
        raise ValueError("seq_lens_out must be an int32 tensor of shape [B]")
    if scale is None:
        scale = 1.0 / math.sqrt(d_k)
    out, oflag = _out(out, out_dtype, B, h_q, d_v, q.device)
    lib = load()
    with _on_device(q):
        need = workspace_bytes(B, h_q, h_kv, d_k, d_v, n_max, q.dtype, num_splits)
        if workspace is None:
            workspace = _workspace(q.device, need)
        nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        st = lib.decode_attn_append(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(K), _ptr(V),
                                    _ptr(seq_lens), _ptr(seq_lens_out), _ptr(out), B, h_q, h_kv,
                                    d_k, d_v, n_max, float(scale), _DTYPES[q.dtype] | oflag,
                                    int(num_splits), _ptr(workspace), nbytes, _ptr(dev_error),
                                    _stream(q, stream))
    _check(st, "decode_attn_append")
    return out


def decode_attn_owned(q, K, V, seq_lens, out=None, scale=None, stream=None,
                      out_dtype=None) -> torch.Tensor:
    """Decode attention through ``decode_attn`` (library-owned workspace)."""
    B, h_q, h_kv, d_k, d_v, n_max = _cache_dims(q, K, V, seq_lens)
    if scale is None:
        scale = 1.0 / math.sqrt(d_k)
    out, oflag = _out(out, out_dtype, B, h_q, d_v, q.device)
    with _on_device(q):
        st = load().decode_attn(_ptr(q), _ptr(K), _ptr(V), _ptr(seq_lens), _ptr(out), B, h_q, h_kv,
                                d_k, d_v, n_max, float(scale), _DTYPES[q.dtype] | oflag,
                                _stream(q, stream))
    _check(st, "decode_attn")
    return out


def decode_attn_noalloc(q, K, V, seq_lens, out=None, scale=None, num_splits: int = 0,
                        dev_error=None, stream=None, out_dtype=None) -> torch.Tensor:
    """Decode attention through ``decode_attn_noalloc``: the split scratch is the
    library's own fixed device buffer, so nothing is allocated for it.  Calls
    whose kernels may overlap on the GPU share that buffer and must be
    serialised by the caller."""
    B, h_q, h_kv, d_k, d_v, n_max = _cache_dims(q, K, V, seq_lens)
    if scale is None:
        scale = 1.0 / math.sqrt(d_k)
    out, oflag = _out(out, out_dtype, B, h_q, d_v, q.device)
    with _on_device(q):
        st = load().decode_attn_noalloc(_ptr(q), _ptr(K), _ptr(V), _ptr(seq_lens), _ptr(out), B, h_q,
                                        h_kv, d_k, d_v, n_max, float(scale),
                                        _DTYPES[q.dtype] | oflag,
                                        int(num_splits), _ptr(dev_error), _stream(q, stream))
    _check(st, "decode_attn_noalloc")
    return out


def decode_attn_partial(q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, seq_lens: torch.Tensor,
                        row_begin: int = 0, row_end: int | None = None,
                        o: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                        scale: float | None = None, num_splits: int = 0,
                        workspace: torch.Tensor | None = None,
                        dev_error: torch.Tensor | None = None,
                        stream: torch.cuda.Stream | None = None):
    """One shard of a sequence-sharded decode (calls ``decode_attn_partial``): the
    decode of rows [row_begin, row_end) of every sequence (clipped to its length).
    Returns ``(o, lse)``: the normalised output [B, h_q, d_v] float32 and the
    natural-log log-sum-exp of those rows' scores [B, h_q] float32 (-inf when a
    sequence has no rows in the range)."""
    B, h_q, h_kv, d_k, d_v, n_max = _cache_dims(q, K, V, seq_lens)
    if row_end is None:
        row_end = n_max
    if scale is None:
        scale = 1.0 / math.sqrt(d_k)
    o, _ = _out(o, torch.float32, B, h_q, d_v, q.device)
    if lse is None:
        lse = torch.empty((B, h_q), dtype=torch.float32, device=q.device)
    if lse.shape != (B, h_q) or lse.dtype != torch.float32 or not lse.is_contiguous() \
            or lse.device != q.device:
        raise ValueError("lse must be a contiguous float32 tensor [B, h_q] on the query's device")
    lib = load()
    with _on_device(q):
        need = workspace_bytes(B, h_q, h_kv, d_k, d_v, n_max, q.dtype, num_splits)
        if workspace is None:
            workspace = _workspace(q.device, need)
        nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        st = lib.decode_attn_partial(_ptr(q), _ptr(K), _ptr(V), _ptr(seq_lens), int(row_begin),
                                     int(row_end), _ptr(o), _ptr(lse), B, h_q, h_kv, d_k, d_v,
                                     n_max, float(scale), _DTYPES[q.dtype], int(num_splits),
                                     _ptr(workspace), nbytes, _ptr(dev_error), _stream(q, stream))
    _check(st, "decode_attn_partial")
    return o, lse


def decode_attn_combine(o_parts: torch.Tensor, lse_parts: torch.Tensor,
                        out: torch.Tensor | None = None, lse_out: torch.Tensor | None = None,
                        out_dtype: torch.dtype | None = None,
                        stream: torch.cuda.Stream | None = None):
    """Merge S partial results over disjoint row sets (calls ``decode_attn_combine``):
    ``o_parts`` [S, B, h_q, d_v] and ``lse_parts`` [S, B, h_q] (float32, natural log,
    on this GPU).  Returns ``(out, lse_out)``."""
    if o_parts.dim() != 4 or lse_parts.dim() != 3 or o_parts.shape[:3] != lse_parts.shape:
        raise ValueError("expected o_parts [S, B, h_q, d_v] and lse_parts [S, B, h_q]")
    for name, t in (("o_parts", o_parts), ("lse_parts", lse_parts)):
        if not t.is_cuda or not t.is_contiguous() or t.dtype != torch.float32:
            raise ValueError(f"{name} must be a contiguous float32 CUDA tensor")
    S, B, h_q, d_v = o_parts.shape
    out, oflag = _out(out, out_dtype, B, h_q, d_v, o_parts.device)
    if lse_out is None:
        lse_out = torch.empty((B, h_q), dtype=torch.float32, device=o_parts.device)
    if lse_out.shape != (B, h_q) or lse_out.dtype != torch.float32 or not lse_out.is_contiguous():
        raise ValueError("lse_out must be a contiguous float32 tensor [B, h_q]")
    with _on_device(o_parts):
        st = load().decode_attn_combine(_ptr(o_parts), _ptr(lse_parts), S, _ptr(out), _ptr(lse_out),
                                        B, h_q, d_v, DA_FP32 | oflag, _stream(o_parts, stream))
    _check(st, "decode_attn_combine")
    return out, lse_out


def kv_append(k_new: torch.Tensor, v_new: torch.Tensor, K: torch.Tensor, V: torch.Tensor,
              pos: torch.Tensor, dev_error: torch.Tensor | None = None,
              stream: torch.cuda.Stream | None = None) -> None:
    """Write row pos[b] of every (b, kv head) of K and V in place (exact copy)."""
    if K.dim() != 4 or V.dim() != 4:
        raise ValueError("K, V must be [B, h_kv, n_max, d]")
    B, h_kv, n_max, d_k = K.shape
    d_v = V.shape[3]
    if k_new.shape != (B, h_kv, d_k) or v_new.shape != (B, h_kv, d_v) or V.shape[:3] != K.shape[:3]:
        raise ValueError("k_new/v_new/K/V shapes disagree")
    if pos.shape != (B,) or pos.dtype != torch.int32:
        raise ValueError("pos must be an int32 tensor of shape [B]")
    for name, t in (("k_new", k_new), ("v_new", v_new), ("K", K), ("V", V), ("pos", pos)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if not (k_new.dtype == v_new.dtype == K.dtype == V.dtype) or K.dtype not in _DTYPES:
        raise ValueError("k_new, v_new, K, V must share dtype float32 or bfloat16")
    with _on_device(K):
        st = load().kv_append(_ptr(k_new), _ptr(v_new), _ptr(K), _ptr(V), _ptr(pos), B, h_kv, d_k,
                              d_v, n_max, _DTYPES[K.dtype], _ptr(dev_error), _stream(K, stream))
    _check(st, "kv_append")


# ----------------------------------------------------------------- 8-bit caches
def _q8_dims(q, K, V, k_scale, v_scale, seq_lens):
    if q.dim() != 3 or K.dim() != 4 or V.dim() != 4:
        raise ValueError("expected q [B, h_q, d], K/V codes [B, h_kv, n_max, d]")
    B, h_q, d_k = q.shape
    Bk, h_kv, n_max, d_k2 = K.shape
    if V.shape != K.shape or Bk != B or d_k2 != d_k:
        raise ValueError("q, K and V shapes disagree")
    if K.dtype not in _Q8_DTYPES or V.dtype != K.dtype:
        raise ValueError("K and V must be torch.int8 or torch.float8_e4m3fn code tensors")
    if q.dtype != torch.bfloat16:
        raise ValueError("q must be bfloat16 with an 8-bit cache")
    for name, t in (("k_scale", k_scale), ("v_scale", v_scale)):
        if t.shape != (B, h_kv, n_max) or t.dtype != torch.float32:
            raise ValueError(f"{name} must be a float32 tensor [B, h_kv, n_max]")
    if seq_lens.shape != (B,) or seq_lens.dtype != torch.int32:
        raise ValueError("seq_lens must be an int32 tensor of shape [B]")
    for name, t in (("q", q), ("K", K), ("V", V), ("k_scale", k_scale), ("v_scale", v_scale),
                    ("seq_lens", seq_lens)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    return B, h_q, h_kv, d_k, d_k, n_max


def kv_quantize(x: torch.Tensor, code_dtype: torch.dtype, stream=None):
    """Rows x [..., d] (float32 or bfloat16, CUDA) -> (codes [..., d] of ``code_dtype``
    (torch.int8 or torch.float8_e4m3fn), scales float32 [...]) by absmax scaling
    (calls ``kv_quantize``)."""
    if x.dtype not in _DTYPES or not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous float32 or bfloat16 CUDA tensor")
    d = x.shape[-1]
    codes = torch.empty(x.shape, dtype=code_dtype, device=x.device)
    scales = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device)
    with _on_device(x):
        st = load().kv_quantize(_ptr(x), _DTYPES[x.dtype], _ptr(codes), _ptr(scales),
                                x.numel() // d if d else 0, d, _Q8_DTYPES[code_dtype],
                                _stream(x, stream))
    _check(st, "kv_quantize")
    return codes, scales


def decode_attn_q8(q, K, V, k_scale, v_scale, seq_lens, out=None, scale=None, num_splits: int = 0,
                   workspace=None, dev_error=None, stream=None, out_dtype=None) -> torch.Tensor:
    """Decode over an 8-bit cache (calls ``decode_attn_q8_ex``): K, V codes
    [B, h_kv, n_max, d] (torch.int8 or torch.float8_e4m3fn) with row scales
    [B, h_kv, n_max]; q bf16 [B, h_q, d].  Returns ``out``."""
    B, h_q, h_kv, d_k, d_v, n_max = _q8_dims(q, K, V, k_scale, v_scale, seq_lens)
    if scale is None:
        scale = 1.0 / math.sqrt(d_k)
    out, oflag = _out(out, out_dtype, B, h_q, d_v, q.device)
    lib = load()
    with _on_device(q):
        need = workspace_bytes(B, h_q, h_kv, d_k, d_v, n_max, K.dtype, num_splits)
        if workspace is None:
            workspace = _workspace(q.device, need)
        nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        st = lib.decode_attn_q8_ex(_ptr(q), _ptr(K), _ptr(V), _ptr(k_scale), _ptr(v_scale),
                                   _ptr(seq_lens), _ptr(out), B, h_q, h_kv, d_k, d_v, n_max,
                                   float(scale), _Q8_DTYPES[K.dtype] | oflag, int(num_splits),
                                   _ptr(workspace), nbytes, _ptr(dev_error), _stream(q, stream))
    _check(st, "decode_attn_q8_ex")
    return out


def decode_attn_q8_append(q, k_new, v_new, k_new_scale, v_new_scale, K, V, k_scale, v_scale,
                          seq_lens, out=None, seq_lens_out=None, scale=None, num_splits: int = 0,
                          workspace=None, dev_error=None, stream=None, out_dtype=None):
    """Append the code rows k_new/v_new [B, h_kv, d] (scales [B, h_kv]) at row
    seq_lens[b] of an 8-bit cache and decode over seq_lens[b] + 1 rows in one
    launch (calls ``decode_attn_q8_append``).  Returns ``out``."""
    B, h_q, h_kv, d_k, d_v, n_max = _q8_dims(q, K, V, k_scale, v_scale, seq_lens)
    for name, t, shape, dt in (("k_new", k_new, (B, h_kv, d_k), K.dtype),
                               ("v_new", v_new, (B, h_kv, d_v), K.dtype),
                               ("k_new_scale", k_new_scale, (B, h_kv), torch.float32),
                               ("v_new_scale", v_new_scale, (B, h_kv), torch.float32)):
        if t.shape != shape or t.dtype != dt or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor {list(shape)} of {dt}")
    if seq_lens_out is not None and (seq_lens_out.shape != (B,) or seq_lens_out.dtype != torch.int32):
        raise ValueError("seq_lens_out must be an int32 tensor of shape [B]")
    if scale is None:
        scale = 1.0 / math.sqrt(d_k)
    out, oflag = _out(out, out_dtype, B, h_q, d_v, q.device)
    lib = load()
    with _on_device(q):
        need = workspace_bytes(B, h_q, h_kv, d_k, d_v, n_max, K.dtype, num_splits)
        if workspace is None:
            workspace = _workspace(q.device, need)
        nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        st = lib.decode_attn_q8_append(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_new_scale),
                                       _ptr(v_new_scale), _ptr(K), _ptr(V), _ptr(k_scale),
                                       _ptr(v_scale), _ptr(seq_lens), _ptr(seq_lens_out), _ptr(out),
                                       B, h_q, h_kv, d_k, d_v, n_max, float(scale),
                                       _Q8_DTYPES[K.dtype] | oflag, int(num_splits),
                                       _ptr(workspace), nbytes, _ptr(dev_error), _stream(q, stream))
    _check(st, "decode_attn_q8_append")
    return out


def kv_append_q8(k_new, v_new, k_new_scale, v_new_scale, K, V, k_scale, v_scale, pos,
                 dev_error=None, stream=None) -> None:
    """Write code row pos[b] and its scale into every (b, kv head) of an 8-bit cache."""
    if K.dim() != 4 or V.shape != K.shape or K.dtype not in _Q8_DTYPES or V.dtype != K.dtype:
        raise ValueError("K, V must be 8-bit code tensors [B, h_kv, n_max, d] of one dtype")
    B, h_kv, n_max, d = K.shape
    for name, t, shape, dt in (("k_new", k_new, (B, h_kv, d), K.dtype),
                               ("v_new", v_new, (B, h_kv, d), K.dtype),
                               ("k_new_scale", k_new_scale, (B, h_kv), torch.float32),
                               ("v_new_scale", v_new_scale, (B, h_kv), torch.float32),
                               ("k_scale", k_scale, (B, h_kv, n_max), torch.float32),
                               ("v_scale", v_scale, (B, h_kv, n_max), torch.float32),
                               ("pos", pos, (B,), torch.int32)):
        if t.shape != shape or t.dtype != dt or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor {list(shape)} of {dt}")
    with _on_device(K):
        st = load().kv_append_q8(_ptr(k_new), _ptr(v_new), _ptr(k_new_scale), _ptr(v_new_scale),
                                 _ptr(K), _ptr(V), _ptr(k_scale), _ptr(v_scale), _ptr(pos), B, h_kv,
                                 d, d, n_max, _Q8_DTYPES[K.dtype], _ptr(dev_error),
                                 _stream(K, stream))
    _check(st, "kv_append_q8")


def launch_count() -> int:
    """Kernels launched by the library in this process so far."""
    return int(load().decode_attn_launch_count())
