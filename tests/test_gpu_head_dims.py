"""Head dims beyond 64/128 on the bf16 path: d = 256, and d_k = 192 with d_v = 128
(needs a GB300).  Same checks as the main parity sweep: against the fp64
oracle, NaN in every unused cache row and in the pre-filled output, the fused
append bit-exact, bf16 output equal to the rounded float32 output.
"""
import numpy as np
import pytest
import torch

import oracle
from decode_attention_kv_split_gb300 import api, workloads as W

pytestmark = pytest.mark.gpu
TOL = 2e-3  # bf16 cache

CASES = [
    # B, h_q, h_kv, d_k, d_v, n_max, lens
    (2, 8, 2, 256, 256, 300, [300, 77]),
    (3, 16, 2, 256, 256, 200, [200, 0, 129]),      # group 8
    (2, 32, 2, 256, 256, 130, [130, 65]),          # group 16: two head chunks
    (1, 1, 1, 256, 256, 1000, [999]),
    (2, 8, 8, 192, 128, 300, [300, 1]),
    (2, 32, 4, 192, 128, 260, [257, 128]),         # group 8
    (1, 4, 1, 192, 128, 1000, [999]),
    (4, 12, 4, 192, 128, 130, [63, 64, 65, 130]),  # group 3
]


@pytest.fixture(scope="module")
def o():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    api.load()
    return oracle.get()


def _case(B, h_q, h_kv, dk, dv, n_max, lens, seed):
    w = W.custom(B=B, h_q=h_q, h_kv=h_kv, d_k=dk, d_v=dv, n=max(lens), n_max=n_max,
                 dtype=torch.bfloat16)
    K, V = W.cache(w, seed, poison=True)
    return w, W.query(w, seed), K, V, torch.tensor(lens, dtype=torch.int32)


def _want(o, q, K, V, lens, scale):
    want, _ = o.decode(q.float().numpy(), K.float().numpy(), V.float().numpy(), lens.numpy(),
                       scale, threads=8)
    return want


def _check(got, want):
    got = got.double().cpu().numpy()
    assert np.all(np.isfinite(got)), "non-finite output (unwritten element or padding read)"
    err = float(np.max(np.abs(got - want)))
    assert err <= TOL, f"max abs error {err:.3e}"


@pytest.mark.parametrize("case", CASES, ids=[f"hq{c[1]}_hkv{c[2]}_dk{c[3]}_dv{c[4]}_n{c[5]}" for c in CASES])
@pytest.mark.parametrize("splits", [0, 1, 3, -1])
def test_decode_wide_heads(o, case, splits):
    B, h_q, h_kv, dk, dv, n_max, lens = case
    w, q, K, V, lens_t = _case(B, h_q, h_kv, dk, dv, n_max, lens, seed=dk + h_q)
    dev = torch.device("cuda")
    out = torch.full((B, h_q, dv), float("nan"), device=dev)
    api.decode_attn(q.to(dev), K.to(dev), V.to(dev), lens_t.to(dev), out=out, num_splits=splits)
    out16 = api.decode_attn(q.to(dev), K.to(dev), V.to(dev), lens_t.to(dev), num_splits=splits,
                            out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    _check(out, _want(o, q, K, V, lens_t, w.scale))
    assert torch.equal(out16.cpu(), out.cpu().to(torch.bfloat16))


@pytest.mark.parametrize("dims", [(256, 256), (192, 128)], ids=["d256", "dk192_dv128"])
@pytest.mark.parametrize("splits", [0, 3])
def test_fused_append_wide_heads(o, dims, splits):
    dk, dv = dims
    B, h_q, h_kv, n_max, lens = 3, 16, 2, 200, [0, 127, 200]  # the last one has no room
    w, q, K, V, lens_t = _case(B, h_q, h_kv, dk, dv, n_max, lens, seed=dk)
    kn, vn = W.new_rows(w, 1, seed=4)
    dev = torch.device("cuda")
    Kd, Vd = K.to(dev), V.to(dev)
    err = torch.zeros((), dtype=torch.int32, device=dev)
    out = api.decode_attn_append(q.to(dev), kn.to(dev), vn.to(dev), Kd, Vd, lens_t.to(dev),
                                 num_splits=splits, dev_error=err)
    torch.cuda.synchronize()
    K2, V2 = K.clone(), V.clone()
    kb, vb = K2.view(torch.int16).numpy(), V2.view(torch.int16).numpy()
    skipped = o.kv_append(kn.view(torch.int16).numpy(), vn.view(torch.int16).numpy(), kb, vb,
                          lens_t.numpy())
    assert skipped == 1 and int(err.item()) == api.DEVERR_POS
    assert torch.equal(Kd.cpu().view(torch.int16), K2.view(torch.int16))
    assert torch.equal(Vd.cpu().view(torch.int16), V2.view(torch.int16))
    new_lens = torch.tensor([min(n + 1, n_max) if n < n_max else n for n in lens], dtype=torch.int32)
    _check(out, _want(o, q, K2, V2, new_lens, w.scale))
