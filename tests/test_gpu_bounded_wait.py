"""A pipeline wait that runs out: the kernels' timeout path (needs a GB300).

Every wait inside the split kernels is bounded; when one runs out the kernel
sets DA_DEVERR_TIMEOUT in the caller's error word, stops waiting, lets its
own copies in flight land, frees what it holds and returns, so the context
stays usable.  To take that path on purpose, the tests load a test build of
the library (the same sources compiled with DA_TEST_HOOKS: waits give up
after 2 ms, and ``decode_attn_test_withhold(cta)`` makes the producer of one
CTA never fill the last stage of its first work item, a flag that nothing
sets).  No fault, trap or endless loop is involved.  Each case checks that
the call returns, that the error word carries DA_DEVERR_TIMEOUT, that the
test build decodes correctly once the hook is off, and that the product
library's next call on the same stream matches the oracle.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from decode_attention_kv_split_gb300 import api, workloads as W
from decode_attention_kv_split_gb300.build import build

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-5, torch.bfloat16: 2e-3}


@pytest.fixture(scope="module")
def test_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    api.load()
    lib = ctypes.CDLL(build(test_hooks=True))
    P, I, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.decode_attn_ex.argtypes = [P, P, P, P, P, I, I, I, I, I, I, F, I, I, P, SZ, P, P]
    lib.decode_attn_ex.restype = I
    lib.decode_attn_q8_ex.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, F, I, I, P, SZ, P, P]
    lib.decode_attn_q8_ex.restype = I
    lib.decode_attn_test_withhold.argtypes = [I]
    lib.decode_attn_test_withhold.restype = None
    yield lib
    lib.decode_attn_test_withhold(-1)


@pytest.fixture(scope="module")
def o():
    return oracle.get()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _run_test_lib(lib, q, K, V, lens, out, err, splits, q8=None):
    B, h_q, d = q.shape
    _, h_kv, n_max, _ = K.shape
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if q8 is None:
        dt = api.DA_BF16 if q.dtype == torch.bfloat16 else api.DA_FP32
        need = api.workspace_bytes(B, h_q, h_kv, d, d, n_max, q.dtype, splits)
        ws = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")
        return lib.decode_attn_ex(_ptr(q), _ptr(K), _ptr(V), _ptr(lens), _ptr(out), B, h_q, h_kv,
                                  d, d, n_max, 1.0 / d ** 0.5, dt, splits, _ptr(ws), need,
                                  _ptr(err), stream)
    ks, vs = q8
    need = api.workspace_bytes(B, h_q, h_kv, d, d, n_max, K.dtype, splits)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")
    dt = api.DA_INT8 if K.dtype == torch.int8 else api.DA_FP8_E4M3
    return lib.decode_attn_q8_ex(_ptr(q), _ptr(K), _ptr(V), _ptr(ks), _ptr(vs), _ptr(lens),
                                 _ptr(out), B, h_q, h_kv, d, d, n_max, 1.0 / d ** 0.5, dt, splits,
                                 _ptr(ws), need, _ptr(err), stream)


CASES = [
    # name, B, h_q, h_kv, d, n_max, lens, dtype, splits
    ("fp32", 2, 4, 4, 128, 1000, [1000, 700], torch.float32, 3),
    ("bf16_mma", 2, 16, 4, 128, 2000, [2000, 1500], torch.bfloat16, 3),
    ("bf16_tc5", 2, 32, 1, 128, 3000, [3000, 2100], torch.bfloat16, 4),
    ("bf16_single_split", 2, 8, 2, 64, 600, [600, 599], torch.bfloat16, 1),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_withheld_stage_times_out_and_context_survives(test_lib, o, case):
    name, B, h_q, h_kv, d, n_max, lens, dtype, splits = case
    w = W.custom(B=B, h_q=h_q, h_kv=h_kv, d_k=d, n=n_max, n_max=n_max, dtype=dtype)
    K, V = W.cache(w, 2)
    q = W.query(w, 2)
    lens_t = torch.tensor(lens, dtype=torch.int32)
    dev = torch.device("cuda")
    qd, Kd, Vd, ld = q.to(dev), K.to(dev), V.to(dev), lens_t.to(dev)
    want, _ = o.decode(q.float().numpy(), K.float().numpy(), V.float().numpy(), lens_t.numpy(),
                       w.scale, threads=8)
    err = torch.zeros((), dtype=torch.int32, device=dev)
    out = torch.zeros((B, h_q, d), device=dev)
    # 1. CTA 0 never receives the last stage of its first item: a wait runs out
    test_lib.decode_attn_test_withhold(0)
    try:
        assert _run_test_lib(test_lib, qd, Kd, Vd, ld, out, err, splits) == 0
        torch.cuda.synchronize()  # the kernel returned (a hang would never get here)
    finally:
        test_lib.decode_attn_test_withhold(-1)
    assert int(err.item()) & api.DEVERR_TIMEOUT, f"{name}: no timeout reported"
    # 2. the same build without the hook: correct, no error bits
    err.zero_()
    out2 = torch.full((B, h_q, d), float("nan"), device=dev)
    assert _run_test_lib(test_lib, qd, Kd, Vd, ld, out2, err, splits) == 0
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.max(np.abs(out2.double().cpu().numpy() - want)) <= TOL[dtype]
    # 3. the product library on the same stream
    out3 = api.decode_attn(qd, Kd, Vd, ld, num_splits=splits)
    torch.cuda.synchronize()
    assert np.max(np.abs(out3.double().cpu().numpy() - want)) <= TOL[dtype]


@pytest.mark.parametrize("kind", ["int8", "e4m3"])
def test_q8_withheld_stage_times_out(test_lib, o, kind):
    from test_gpu_q8 import KINDS, _codes_tensor, make_q8_case, oracle_decode_q8

    k, tdt = KINDS[kind]
    w, q, kc, ks, vc, vs, lens_t = make_q8_case(o, k, 2, 16, 2, 128, 1000, [1000, 640], seed=4)
    dev = torch.device("cuda")
    args = (q.to(dev), _codes_tensor(kc, tdt).to(dev), _codes_tensor(vc, tdt).to(dev))
    scales = (torch.from_numpy(ks).to(dev), torch.from_numpy(vs).to(dev))
    ld = lens_t.to(dev)
    err = torch.zeros((), dtype=torch.int32, device=dev)
    out = torch.zeros((2, 16, 128), device=dev)
    test_lib.decode_attn_test_withhold(0)
    try:
        assert _run_test_lib(test_lib, *args, ld, out, err, 3, q8=scales) == 0
        torch.cuda.synchronize()
    finally:
        test_lib.decode_attn_test_withhold(-1)
    assert int(err.item()) & api.DEVERR_TIMEOUT
    want = oracle_decode_q8(o, k, q, kc, ks, vc, vs, lens_t, w.scale)
    got = api.decode_attn_q8(*args, *scales, ld, num_splits=3)
    torch.cuda.synchronize()
    assert np.max(np.abs(got.double().cpu().numpy() - want)) <= 2e-4
