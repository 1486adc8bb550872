"""Launches where a CTA holds more than 64 work items (needs a GB300).

A CTA decodes its first 64 work items into shared memory once and decodes any
later ones on the fly from the work list.  These cases give every kernel
family (fp32, bf16 mma.sync, bf16 tcgen05, 8-bit) well over 64 x 152 items in
one launch, in both list modes: fixed splits (many splits of many units) and
balanced pieces (many short units per piece).  Every head is compared with
the oracle; rows past each length hold NaN.
"""
import numpy as np
import pytest
import torch

import oracle
from decode_attention_kv_split_gb300 import api, workloads as W

from test_gpu_q8 import KINDS, _codes_tensor, oracle_decode_q8

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-5, torch.bfloat16: 2e-3}
SMS = 152
ITEM_CACHE = 64


@pytest.fixture(scope="module")
def o():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    api.load()
    return oracle.get()


def _lens(B, lo, hi, seed):
    rng = np.random.default_rng(seed)
    return [int(x) for x in rng.integers(lo, hi + 1, B)]


def _units(B, h_q, h_kv, heads_per_item):
    return B * h_kv * -(-(h_q // h_kv) // heads_per_item)


# name, B, h_q, h_kv, d, n_max, lens (lo, hi), splits, heads per work item, rows per split
CASES = [
    ("fp32_fixed", 512, 8, 8, 64, 256, (129, 256), 4, 1, 64),
    ("fp32_balanced", 512, 32, 32, 64, 32, (0, 32), -1, 1, None),
    ("bf16_mma_fixed", 512, 32, 8, 128, 384, (257, 384), 3, 8, 128),
    ("bf16_mma_balanced", 512, 128, 32, 64, 64, (0, 64), -1, 8, None),
    ("bf16_tc5_fixed", 512, 128, 8, 128, 384, (257, 384), 3, 16, 128),
    ("bf16_tc5_balanced", 512, 384, 24, 128, 128, (0, 128), -1, 16, None),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_more_than_64_items_per_cta(o, case):
    name, B, h_q, h_kv, d, n_max, (lo, hi), splits, hpi, chunk = case
    dtype = torch.float32 if name.startswith("fp32") else torch.bfloat16
    lens = _lens(B, lo, hi, seed=B + h_q)
    units = _units(B, h_q, h_kv, hpi)
    items = units * (sum(-(-n // chunk) for n in lens) / B if chunk else 1)
    assert items > ITEM_CACHE * SMS, (name, items)
    w = W.custom(B=B, h_q=h_q, h_kv=h_kv, d_k=d, n=n_max, n_max=n_max, dtype=dtype)
    K, V = W.cache(w, 3)
    for b, n in enumerate(lens):
        K[b, :, n:] = float("nan")
        V[b, :, n:] = float("nan")
    q = W.query(w, 3)
    lens_t = torch.tensor(lens, dtype=torch.int32)
    dev = torch.device("cuda")
    out = torch.full((B, h_q, d), float("nan"), device=dev)
    api.decode_attn(q.to(dev), K.to(dev), V.to(dev), lens_t.to(dev), out=out, num_splits=splits)
    torch.cuda.synchronize()
    want, _ = o.decode(q.float().numpy(), K.float().numpy(), V.float().numpy(), lens_t.numpy(),
                       w.scale, threads=max(1, o.max_threads()))
    got = out.double().cpu().numpy()
    assert np.all(np.isfinite(got))
    err = float(np.max(np.abs(got - want)))
    assert err <= TOL[dtype], f"{name}: max abs error {err:.3e}"


Q8_CASES = [
    # name, B, h_q, h_kv, d, n_max, lens (lo, hi), splits, rows per split
    ("q8_fixed", 512, 32, 8, 128, 384, (257, 384), 3, 128),
    ("q8_balanced", 512, 96, 24, 64, 64, (0, 64), -1, None),
]


@pytest.mark.parametrize("kind", list(KINDS))
@pytest.mark.parametrize("case", Q8_CASES, ids=[c[0] for c in Q8_CASES])
def test_q8_more_than_64_items_per_cta(o, kind, case):
    name, B, h_q, h_kv, d, n_max, (lo, hi), splits, chunk = case
    k, tdt = KINDS[kind]
    lens = _lens(B, lo, hi, seed=B + h_q + k)
    units = _units(B, h_q, h_kv, 8)
    items = units * (sum(-(-n // chunk) for n in lens) / B if chunk else 1)
    assert items > ITEM_CACHE * SMS, (name, items)
    w = W.custom(B=B, h_q=h_q, h_kv=h_kv, d_k=d, n=n_max, n_max=n_max, dtype=torch.float32)
    K, V = W.cache(w, 4)
    kc, ks = o.quantize(K.numpy(), k)
    vc, vs = o.quantize(V.numpy(), k)
    del K, V
    for b, n in enumerate(lens):
        kc[b, :, n:] = 0x7F
        vc[b, :, n:] = 0x7F
        ks[b, :, n:] = np.nan
        vs[b, :, n:] = np.nan
    q = W.query(w, 4).to(torch.bfloat16)
    lens_t = torch.tensor(lens, dtype=torch.int32)
    dev = torch.device("cuda")
    out = api.decode_attn_q8(q.to(dev), _codes_tensor(kc, tdt).to(dev),
                             _codes_tensor(vc, tdt).to(dev), torch.from_numpy(ks).to(dev),
                             torch.from_numpy(vs).to(dev), lens_t.to(dev), num_splits=splits)
    torch.cuda.synchronize()
    want = oracle_decode_q8(o, k, q, kc, ks, vc, vs, lens_t, w.scale)
    got = out.double().cpu().numpy()
    assert np.all(np.isfinite(got))
    err = float(np.max(np.abs(got - want)))
    assert err <= 2e-4, f"{name}/{kind}: max abs error {err:.3e}"
