"""GB300-native split-KV decode attention.

The compute lives in a C-ABI shared library of hand-written sm_103a CUDA
kernels (``libdecode_attn.so``, built in-tree by ``__graft_entry__.build()``);
this package is the thin Python binding over it.  Importing the package does
not load the library; the first call does, and raises if it is missing.
"""
from . import workloads  # noqa: F401  (seeded inputs; no attention arithmetic)
from .api import (  # noqa: F401
    DecodeAttnError,
    decode_attn,
    decode_attn_append,
    decode_attn_noalloc,
    decode_attn_owned,
    kv_append,
    launch_count,
    resolve_splits,
    workspace_bytes,
)
