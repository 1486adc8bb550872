"""Seeded synthetic inputs for decode attention: shapes, seeds, distributions.

This module only draws random numbers and fixes shapes.  It holds none of the
attention arithmetic, so both the CUDA path's tests/bench and the CPU oracle
can take their inputs from it without sharing any of the method.

Every tensor is drawn on the CPU with ``torch.Generator`` in float32 and then
cast to the workload's dtype; the oracle is handed ``.float()`` of the cast
tensor, which is exact for bf16, so both sides see identical values.

Seeds: K uses ``seed + 0``, V ``seed + 1``, q ``seed + 2``, the per-sequence
lengths ``seed + 3``; the key row appended at step t uses ``seed + 100 + 2t``
and the value row ``seed + 101 + 2t``.

Workloads follow the model shapes the pages discuss (page "Attention over the
KV cache in the decode step": Llama-3-8B with 32 query / 8 KV heads,
Llama-2-70B with 64 / 8, MQA with 32 query heads; all head_dim 128; page
"MoA-Structured Decode Attention": fp32 multi-head decode).
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    h_q: int
    h_kv: int
    d_k: int
    d_v: int
    n: int                      # cached rows before the first append (all sequences)
    n_max: int                  # cache capacity per sequence
    dtype: torch.dtype          # q, K, V element type; torch.int8 / torch.float8_e4m3fn:
                                # an 8-bit cache of codes with float32 row scales (q bf16)
    kv_std: float = 1.0         # standard deviation of the K/V entries
    q_std: float = 1.0
    ragged: tuple[int, int] | None = None   # lengths ~ U[lo, hi] (inclusive) when set
    steps: int = 0              # append + decode steps the workload describes
    num_splits: int = 0         # 0 = let the library choose; -1 = balanced pieces
    description: str = ""

    @property
    def group(self) -> int:
        return self.h_q // self.h_kv

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d_k)


WORKLOADS: dict[str, Workload] = {
    "single_head": Workload(
        "single_head", B=1, h_q=1, h_kv=1, d_k=64, d_v=64, n=256, n_max=512,
        dtype=torch.float32, steps=1,
        description="single-head decode, fp32, d=64, n=256 then one append and a re-decode at n=257"),
    "mha_fp32": Workload(
        "mha_fp32", B=4, h_q=32, h_kv=32, d_k=128, d_v=128, n=4096, n_max=4096 + 16,
        dtype=torch.float32, steps=16,
        description="MHA fp32, B=4, h_q=h_kv=32, d=128, n=4096, 16 append+decode steps"),
    "gqa_llama3_8b": Workload(
        "gqa_llama3_8b", B=16, h_q=32, h_kv=8, d_k=128, d_v=128, n=8192, n_max=8192,
        dtype=torch.bfloat16, ragged=(1024, 8192),
        description="GQA g=4 (Llama-3-8B shape), bf16, B=16, lengths ~ U[1024, 8192], n_max=8192"),
    "mqa_g32": Workload(
        "mqa_g32", B=8, h_q=32, h_kv=1, d_k=128, d_v=128, n=32768, n_max=32768,
        dtype=torch.bfloat16,
        description="MQA g=32, bf16, B=8, n=32768"),
    "long_llama2_70b": Workload(
        "long_llama2_70b", B=2, h_q=64, h_kv=8, d_k=128, d_v=128, n=131072, n_max=131072,
        dtype=torch.bfloat16, kv_std=0.5, num_splits=256,
        description="long context g=8 (Llama-2-70B shape), bf16, B=2, n=131072, 256 splits, K/V ~ N(0, 0.5^2)"),
    "gqa_llama3_8b_fp8": Workload(
        "gqa_llama3_8b_fp8", B=16, h_q=32, h_kv=8, d_k=128, d_v=128, n=8192, n_max=8192,
        dtype=torch.float8_e4m3fn, ragged=(1024, 8192), num_splits=-1,
        description="GQA g=4 (Llama-3-8B shape), fp8 e4m3 KV cache with float32 row scales, "
                    "bf16 q, B=16, lengths ~ U[1024, 8192], n_max=8192, balanced pieces"),
    "gqa_llama3_8b_int8": Workload(
        "gqa_llama3_8b_int8", B=16, h_q=32, h_kv=8, d_k=128, d_v=128, n=8192, n_max=8192,
        dtype=torch.int8, ragged=(1024, 8192), num_splits=-1,
        description="GQA g=4 (Llama-3-8B shape), int8 KV cache with float32 row scales, "
                    "bf16 q, B=16, lengths ~ U[1024, 8192], n_max=8192, balanced pieces"),
    "long_llama2_70b_fp8": Workload(
        "long_llama2_70b_fp8", B=2, h_q=64, h_kv=8, d_k=128, d_v=128, n=131072, n_max=131072,
        dtype=torch.float8_e4m3fn, kv_std=0.5,
        description="long context g=8 (Llama-2-70B shape), fp8 e4m3 KV cache with float32 row "
                    "scales, bf16 q, B=2, n=131072, library's splits"),
}

Q8_DTYPES = (torch.int8, torch.float8_e4m3fn)


def is_q8(w: "Workload") -> bool:
    """An 8-bit cache: codes plus float32 row scales, q in bf16."""
    return w.dtype in Q8_DTYPES


def _values(w: Workload) -> torch.dtype:
    """Element type of the generated K/V values: float32 before 8-bit quantization."""
    return torch.float32 if is_q8(w) else w.dtype


def _randn(shape, seed: int, std: float, device="cpu") -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    t = torch.randn(*shape, generator=g, dtype=torch.float32, device=device)
    if std != 1.0:
        t.mul_(std)
    return t


def seq_lens(w: Workload, seed: int = 0) -> torch.Tensor:
    """Per-sequence cached lengths (int32, CPU)."""
    if w.ragged is None:
        return torch.full((w.B,), w.n, dtype=torch.int32)
    g = torch.Generator(device="cpu")
    g.manual_seed(seed + 3)
    lo, hi = w.ragged
    return torch.randint(lo, hi + 1, (w.B,), generator=g, dtype=torch.int32)


def cache(w: Workload, seed: int = 0, poison: bool = False, device="cpu"):
    """K [B, h_kv, n_max, d_k] and V [B, h_kv, n_max, d_v] in ``w.dtype`` (float32
    values, to be quantized, for an 8-bit cache).

    Rows at or beyond each sequence's length are filled with NaN when
    ``poison`` is set (a cache's unused rows may hold anything), otherwise
    they hold random values like the rest.  ``device`` picks where the
    generator runs: a CUDA generator draws other numbers than the CPU one
    from the same seed, so parity inputs are always made on the CPU.
    """
    K = _randn((w.B, w.h_kv, w.n_max, w.d_k), seed + 0, w.kv_std, device).to(_values(w))
    V = _randn((w.B, w.h_kv, w.n_max, w.d_v), seed + 1, w.kv_std, device).to(_values(w))
    if poison:
        lens = seq_lens(w, seed)
        for b in range(w.B):
            K[b, :, int(lens[b]):, :] = float("nan")
            V[b, :, int(lens[b]):, :] = float("nan")
    return K, V


def query(w: Workload, seed: int = 0) -> torch.Tensor:
    """q [B, h_q, d_k] in ``w.dtype`` (bf16 for an 8-bit cache) (CPU)."""
    return _randn((w.B, w.h_q, w.d_k), seed + 2, w.q_std).to(
        torch.bfloat16 if is_q8(w) else w.dtype)


def new_rows(w: Workload, step: int, seed: int = 0):
    """The key and value rows appended at decode step ``step``: [B, h_kv, d]."""
    k = _randn((w.B, w.h_kv, w.d_k), seed + 100 + 2 * step, w.kv_std).to(_values(w))
    v = _randn((w.B, w.h_kv, w.d_v), seed + 101 + 2 * step, w.kv_std).to(_values(w))
    return k, v


def custom(name: str = "custom", **kw) -> Workload:
    """A workload with explicit fields, for parity sweeps."""
    kw.setdefault("n_max", kw.get("n", 1))
    kw.setdefault("d_v", kw.get("d_k"))
    return Workload(name=name, **kw)
