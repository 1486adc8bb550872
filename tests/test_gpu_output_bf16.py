"""bf16 output (the DA_OUT_BF16 dtype flag) on the GPU (needs a GB300).

The kernels compute the float32 result and round it once to bf16 (round to
nearest even), so with the same inputs and launch configuration the bf16
output equals the float32 output converted by PyTorch, bit for bit; against
the fp64 oracle it is within the cache's tolerance plus half a bf16 unit.
"""
import numpy as np
import pytest
import torch

import oracle
from decode_attention_kv_split_gb300 import api, workloads as W

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-5, torch.bfloat16: 2e-3}
CASES = [
    # B, h_q, h_kv, d, n_max, lens
    (2, 4, 4, 128, 300, [300, 1]),          # fp32 / bf16 group 1
    (3, 8, 2, 128, 200, [200, 0, 77]),      # group 4, an empty sequence
    (2, 16, 2, 64, 129, [129, 64]),         # group 8, d = 64
    (2, 32, 1, 128, 700, [700, 321]),       # group 32 (tcgen05 kernel for bf16)
]


@pytest.fixture(scope="module")
def o():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    api.load()
    return oracle.get()


def _case(B, h_q, h_kv, d, n_max, lens, dtype, seed):
    w = W.custom(B=B, h_q=h_q, h_kv=h_kv, d_k=d, n=max(lens), n_max=n_max, dtype=dtype)
    K, V = W.cache(w, seed, poison=True)
    return w, W.query(w, seed), K, V, torch.tensor(lens, dtype=torch.int32)


def _check_bf16(o, q, K, V, lens, scale, out16, out32, tol):
    assert out16.dtype == torch.bfloat16
    assert torch.equal(out16.cpu(), out32.cpu().to(torch.bfloat16)), "bf16 output is not RNE(fp32 output)"
    want, _ = o.decode(q.float().numpy(), K.float().numpy(), V.float().numpy(), lens.numpy(), scale,
                       threads=8)
    got = out16.cpu().double().numpy()
    assert np.all(np.isfinite(got))
    bound = tol + 2.0 ** -8 * np.abs(want)
    assert np.all(np.abs(got - want) <= bound), float(np.max(np.abs(got - want) - bound))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["fp32", "bf16"])
@pytest.mark.parametrize("case", CASES, ids=[f"hq{c[1]}_hkv{c[2]}_d{c[3]}" for c in CASES])
@pytest.mark.parametrize("splits", [0, 1, 3])
def test_decode_bf16_output(o, dtype, case, splits):
    B, h_q, h_kv, d, n_max, lens = case
    w, q, K, V, lens_t = _case(B, h_q, h_kv, d, n_max, lens, dtype, seed=d + h_q)
    dev = torch.device("cuda")
    args = (q.to(dev), K.to(dev), V.to(dev), lens_t.to(dev))
    out32 = api.decode_attn(*args, num_splits=splits)
    out16 = torch.full((B, h_q, d), float("nan"), dtype=torch.bfloat16, device=dev)
    api.decode_attn(*args, out=out16, num_splits=splits)
    torch.cuda.synchronize()
    _check_bf16(o, q, K, V, lens_t, w.scale, out16, out32, TOL[dtype])


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["fp32", "bf16"])
def test_fused_append_bf16_output(o, dtype):
    B, h_q, h_kv, d, n_max, lens = 3, 32, 2, 128, 300, [0, 127, 200]
    w, q, K, V, lens_t = _case(B, h_q, h_kv, d, n_max, lens, dtype, seed=5)
    kn, vn = W.new_rows(w, 0, seed=9)
    dev = torch.device("cuda")
    outs = {}
    for odt in (torch.float32, torch.bfloat16):
        Kd, Vd = K.to(dev), V.to(dev)
        outs[odt] = api.decode_attn_append(q.to(dev), kn.to(dev), vn.to(dev), Kd, Vd, lens_t.to(dev),
                                           num_splits=3, out_dtype=odt)
    torch.cuda.synchronize()
    # the oracle sees the cache with the new rows written
    K2, V2 = K.clone(), V.clone()
    for b in range(B):
        K2[b, :, lens[b]] = kn[b]
        V2[b, :, lens[b]] = vn[b]
    _check_bf16(o, q, K2, V2, lens_t + 1, w.scale, outs[torch.bfloat16], outs[torch.float32],
                TOL[dtype])


def test_other_entry_points_bf16_output(o):
    B, h_q, h_kv, d, n_max, lens = 2, 8, 2, 128, 400, [400, 55]
    w, q, K, V, lens_t = _case(B, h_q, h_kv, d, n_max, lens, torch.bfloat16, seed=11)
    dev = torch.device("cuda")
    args = (q.to(dev), K.to(dev), V.to(dev), lens_t.to(dev))
    ref32 = api.decode_attn_owned(*args)
    for fn in (api.decode_attn_owned, api.decode_attn_noalloc):
        out16 = fn(*args, out_dtype=torch.bfloat16)
        torch.cuda.synchronize()
        _check_bf16(o, q, K, V, lens_t, w.scale, out16, ref32, TOL[torch.bfloat16])
