"""decode_attn_noalloc against decode_attn_ex (needs a GB300).

The no-allocation entry point serves callers that cannot call cudaMalloc
(for instance a serving loop where an allocation would synchronise the
device, or code whose device memory is owned by another allocator).  Its
split scratch is the library's own fixed device buffer.  This file is named
to be collected last, so that a run stopping at the first failure has run
every other test before it.  It calls the entry point through the C ABI
twice in a row, since the buffer keeps the previous call's contents, and
compares each result with decode_attn_ex on a caller-provided workspace.
"""
import ctypes

import pytest
import torch

from decode_attention_kv_split_gb300 import api, workloads as W

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-5, torch.bfloat16: 2e-3}
SCRATCH_LIMIT = 32 * 1024 * 1024


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return api.load()


def _inputs(B, h_q, h_kv, d, n_max, lens, dtype, seed):
    w = W.custom(B=B, h_q=h_q, h_kv=h_kv, d_k=d, n=max(lens), n_max=n_max, dtype=dtype)
    K, V = W.cache(w, seed)
    for b, n in enumerate(lens):
        K[b, :, n:] = float("nan")
        V[b, :, n:] = float("nan")
    dev = torch.device("cuda")
    return (W.query(w, seed).to(dev), K.to(dev), V.to(dev),
            torch.tensor(lens, dtype=torch.int32, device=dev), w.scale)


def _call_noalloc(lib, q, K, V, lens, out, scale, splits):
    B, h_q, d = q.shape
    _, h_kv, n_max, _ = K.shape
    dt = 1 if q.dtype == torch.bfloat16 else 0
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    return lib.decode_attn_noalloc(P(q), P(K), P(V), P(lens), P(out), B, h_q, h_kv, d, d, n_max,
                                   float(scale), dt, int(splits), None, stream)


CASES = [
    # B, h_q, h_kv, d, n_max, lens, dtype, splits
    (2, 16, 4, 128, 3000, [3000, 1234], torch.bfloat16, 0),
    (2, 16, 4, 128, 3000, [2999, 17], torch.bfloat16, 7),
    (1, 32, 1, 128, 8192, [8192], torch.bfloat16, 32),
    (3, 8, 8, 64, 777, [777, 1, 400], torch.float32, 5),
    (2, 4, 4, 128, 300, [300, 0], torch.float32, 1),
    (2, 8, 2, 128, 2000, [2000, 333], torch.bfloat16, -1),   # balanced: per-unit table too
]


@pytest.mark.parametrize("case", CASES, ids=[f"case{i}" for i in range(len(CASES))])
def test_noalloc_matches_ex_on_two_calls_in_a_row(lib, case):
    B, h_q, h_kv, d, n_max, lens, dtype, splits = case
    q, K, V, lens_t, scale = _inputs(B, h_q, h_kv, d, n_max, lens, dtype, seed=B + d)
    ref = api.decode_attn(q, K, V, lens_t, scale=scale, num_splits=splits)
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        st = _call_noalloc(lib, q, K, V, lens_t, out, scale, splits)
        assert st == 0, lib.decode_attn_status_string(st).decode()
        torch.cuda.synchronize()
        assert torch.isfinite(out).all()
        assert torch.max(torch.abs(out - ref)).item() <= TOL[dtype]
    # a different request in between must not disturb the next result
    q2, K2, V2, l2, s2 = _inputs(1, 8, 2, 128, 500, [500], torch.bfloat16, seed=99)
    out2 = torch.empty((1, 8, 128), dtype=torch.float32, device="cuda")
    assert _call_noalloc(lib, q2, K2, V2, l2, out2, s2, 3) == 0
    out = torch.full_like(ref, float("nan"))
    assert _call_noalloc(lib, q, K, V, lens_t, out, scale, splits) == 0
    torch.cuda.synchronize()
    assert torch.max(torch.abs(out - ref)).item() <= TOL[dtype]


def test_noalloc_rejects_requests_beyond_its_scratch(lib):
    # 64 x 64 query heads x 1024 splits of 129 floats needs ~2 GB of scratch.
    B, h_q, h_kv, d, n_max = 64, 64, 8, 128, 131072
    need = api.workspace_bytes(B, h_q, h_kv, d, d, n_max, torch.bfloat16, 1024)
    assert need > SCRATCH_LIMIT
    # Real (small) device buffers: the call must refuse on the sizes alone, but
    # nothing it is handed is a bogus address should that order ever change.
    dev = torch.device("cuda")
    bufs = [torch.zeros(64, dtype=torch.int32, device=dev) for _ in range(5)]
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = lib.decode_attn_noalloc(*[P(t) for t in bufs], B, h_q, h_kv, d, d, n_max, 0.1, 1, 1024,
                                 None, stream)
    assert st == -5   # DA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert all(bool((t == 0).all()) for t in bufs)


def test_noalloc_takes_one_split_when_balanced_pieces_do_not_fit(lib):
    """The library's choice here is balanced pieces (128 units on a 152-SM grid),
    whose partials (~40 MB) exceed the buffer: the call takes one split per
    sequence instead, exactly as num_splits = 1 computes it."""
    B, h_q, h_kv, d, n_max = 16, 32, 8, 128, 8192
    lens = [8192, 1024, 5000, 7777, 3000, 8191, 1500, 6000, 2048, 4096, 100, 8000, 512, 7000, 2500, 6500]
    if api.resolve_splits(B, h_q, h_kv, d, d, n_max, torch.bfloat16, 0) <= 1:
        pytest.skip("the library takes one split on this device's grid")
    assert api.workspace_bytes(B, h_q, h_kv, d, d, n_max, torch.bfloat16, 0) > SCRATCH_LIMIT
    q, K, V, lens_t, scale = _inputs(B, h_q, h_kv, d, n_max, lens, torch.bfloat16, seed=7)
    ref = api.decode_attn(q, K, V, lens_t, scale=scale, num_splits=1)
    out = torch.full_like(ref, float("nan"))
    st = _call_noalloc(lib, q, K, V, lens_t, out, scale, 0)
    assert st == 0, lib.decode_attn_status_string(st).decode()
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
