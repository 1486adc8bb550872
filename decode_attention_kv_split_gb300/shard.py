"""Sequence-sharded decode across ranks (host plumbing over the C ABI).

When the cached rows of every sequence are spread over several GPUs, each
rank decodes the rows it holds (``decode_attn_partial``: a normalised output
and the natural-log log-sum-exp of its scores per query head), the ranks
all-gather those partials into each GPU's own memory, and
``decode_attn_combine`` merges them by the log-sum-exp identity into the
decode over all rows.  Page "Phase 3, Section 6: StoryLM-0 head-parallel
attention" shards attention across devices and gathers the per-device
results (sections 3-4); cut along the cached rows instead of the heads, the
gather carries (o, lse) and the merge is exact.

The only exchange is the all-gather of B * h_q * (d_v + 1) floats per rank.
No kernel is ever handed a peer's memory: the collective copies the
partials into local tensors first.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from . import api


def gather_partials(o: torch.Tensor, lse: torch.Tensor, group=None):
    """All-gather every rank's partial ``(o [B, h_q, d_v], lse [B, h_q])`` into
    local tensors ``(o_parts [S, B, h_q, d_v], lse_parts [S, B, h_q])``, part s
    from rank s of ``group``."""
    world = dist.get_world_size(group)
    o, lse = o.contiguous(), lse.contiguous()
    o_parts = torch.empty((world, *o.shape), dtype=o.dtype, device=o.device)
    lse_parts = torch.empty((world, *lse.shape), dtype=lse.dtype, device=lse.device)
    if dist.get_backend(group) == "nccl":
        dist.all_gather_into_tensor(o_parts, o, group=group)
        dist.all_gather_into_tensor(lse_parts, lse, group=group)
    else:
        dist.all_gather(list(o_parts.unbind(0)), o, group=group)
        dist.all_gather(list(lse_parts.unbind(0)), lse, group=group)
    return o_parts, lse_parts


def sharded_decode(q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, seq_lens: torch.Tensor,
                   group=None, scale: float | None = None, out: torch.Tensor | None = None,
                   out_dtype: torch.dtype | None = None, num_splits: int = 0):
    """Decode attention over a cache whose rows are spread across the ranks of
    ``group``: this rank holds ``K``/``V`` [B, h_kv, n_local_max, d] with
    ``seq_lens`` [B] rows of each sequence (any disjoint assignment of rows to
    ranks).  Every rank receives the full result.  Returns ``(out, lse)``."""
    o, lse = api.decode_attn_partial(q, K, V, seq_lens, 0, None, scale=scale,
                                     num_splits=num_splits)
    o_parts, lse_parts = gather_partials(o, lse, group)
    return api.decode_attn_combine(o_parts, lse_parts, out=out, out_dtype=out_dtype)
