"""Sequence-sharded decode on one GPU against the fp64 oracle (needs a GB300).

Each sequence's cached rows are cut into 2-4 ranges (some empty, some past
the sequence's end); ``decode_attn_partial`` decodes each range and
``decode_attn_combine`` merges the parts.  Every part is compared with the
oracle run on that range alone (normalised output and natural-log
log-sum-exp), and the merge with the oracle's decode over all rows.

Tolerances: outputs as the other parity tests (1e-5 fp32, 2e-3 bf16 cache).
The log-sum-exp is log2(sum of up to a few thousand float32 exponentials)
plus the running max, converted by ln 2: its float32 sum carries a relative
error of at most a few 1e-5 at these lengths, so 1e-4 absolute bounds it.
"""
import numpy as np
import pytest
import torch

import oracle
from decode_attention_kv_split_gb300 import api, workloads as W

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-5, torch.bfloat16: 2e-3}
LSE_TOL = 1e-4


@pytest.fixture(scope="module")
def o():
    return oracle.get()


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    api.load()


def _case(B, h_q, h_kv, d, n_max, lens, dtype, seed):
    w = W.custom(B=B, h_q=h_q, h_kv=h_kv, d_k=d, n=max(lens), n_max=n_max, dtype=dtype)
    K, V = W.cache(w, seed)
    for b, n in enumerate(lens):
        K[b, :, n:] = float("nan")
        V[b, :, n:] = float("nan")
    return W.query(w, seed), K, V, torch.tensor(lens, dtype=torch.int32), w.scale


def _oracle_range(o, q, K, V, lens, r0, r1, scale):
    """The oracle's decode of rows [r0, r1) of every sequence (clipped to its length)."""
    lo = [min(r0, int(n)) for n in lens]
    hi = [min(r1, int(n)) for n in lens]
    width = max(1, max(h - l for l, h in zip(lo, hi)))
    Ks = np.zeros((K.shape[0], K.shape[1], width, K.shape[3]), dtype=np.float32)
    Vs = np.zeros((V.shape[0], V.shape[1], width, V.shape[3]), dtype=np.float32)
    Kf, Vf = K.float().numpy(), V.float().numpy()
    for b, (l, h) in enumerate(zip(lo, hi)):
        Ks[b, :, :h - l] = Kf[b, :, l:h]
        Vs[b, :, :h - l] = Vf[b, :, l:h]
    return o.decode(q.float().numpy(), Ks, Vs, np.array([h - l for l, h in zip(lo, hi)],
                                                         dtype=np.int32), scale, threads=8)


def _close_lse(got, want, tol):
    got = np.asarray(got, dtype=np.float64)
    both_empty = np.isneginf(got) & np.isneginf(want)
    assert np.array_equal(np.isneginf(got), np.isneginf(want)), "empty ranges differ"
    err = np.max(np.abs(np.where(both_empty, 0.0, got - np.where(both_empty, 0.0, want))))
    assert err <= tol, f"lse max abs error {err:.3e} > {tol:.1e}"


CASES = [
    # B, h_q, h_kv, d, n_max, lens, cuts (range boundaries; the last one past every length)
    (3, 8, 2, 128, 700, [700, 0, 333], [0, 200, 450, 10**6]),      # g=4 mma.sync, an empty sequence
    (2, 4, 4, 64, 300, [300, 17], [0, 128, 129, 300]),             # g=1, a one-row range
    (2, 32, 1, 128, 1000, [1000, 640], [0, 640, 640, 999, 5000]),  # MQA tcgen05, an empty range
    (2, 16, 2, 128, 777, [777, 500], [0, 390, 10**6]),             # g=8 (two parts)
    (1, 64, 1, 64, 520, [520], [0, 100, 300, 400, 520]),           # two head chunks, four parts
]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["fp32", "bf16"])
@pytest.mark.parametrize("case", CASES, ids=[f"case{i}" for i in range(len(CASES))])
@pytest.mark.parametrize("splits", [0, 1, 3])
def test_partials_and_merge_match_oracle(o, dtype, case, splits):
    B, h_q, h_kv, d, n_max, lens, cuts = case
    q, K, V, lens_t, scale = _case(B, h_q, h_kv, d, n_max, lens, dtype, seed=B + d)
    dev = torch.device("cuda")
    qd, Kd, Vd, ld = q.to(dev), K.to(dev), V.to(dev), lens_t.to(dev)
    parts_o, parts_l = [], []
    for r0, r1 in zip(cuts[:-1], cuts[1:]):
        po = torch.full((B, h_q, d), float("nan"), device=dev)
        pl = torch.full((B, h_q), float("nan"), device=dev)
        api.decode_attn_partial(qd, Kd, Vd, ld, r0, r1, o=po, lse=pl, num_splits=splits)
        torch.cuda.synchronize()
        want_o, want_l = _oracle_range(o, q, K, V, lens, r0, r1, scale)
        got = po.double().cpu().numpy()
        assert np.all(np.isfinite(got))
        assert np.max(np.abs(got - want_o)) <= TOL[dtype]
        _close_lse(pl.cpu().numpy(), want_l, LSE_TOL)
        parts_o.append(po)
        parts_l.append(pl)
    out, lse = api.decode_attn_combine(torch.stack(parts_o), torch.stack(parts_l))
    torch.cuda.synchronize()
    want, want_l = o.decode(q.float().numpy(), K.float().numpy(), V.float().numpy(),
                            lens_t.numpy(), scale, threads=8)
    assert np.max(np.abs(out.double().cpu().numpy() - want)) <= TOL[dtype]
    _close_lse(lse.cpu().numpy(), want_l, LSE_TOL)


def test_merge_with_bf16_out_and_no_parts(o):
    q, K, V, lens_t, scale = _case(2, 8, 2, 128, 400, [400, 250], torch.bfloat16, seed=3)
    dev = torch.device("cuda")
    qd, Kd, Vd, ld = q.to(dev), K.to(dev), V.to(dev), lens_t.to(dev)
    parts = [api.decode_attn_partial(qd, Kd, Vd, ld, r0, r1) for r0, r1 in ((0, 256), (256, 400))]
    o_parts = torch.stack([p[0] for p in parts])
    l_parts = torch.stack([p[1] for p in parts])
    out32, _ = api.decode_attn_combine(o_parts, l_parts)
    out16, _ = api.decode_attn_combine(o_parts, l_parts, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert torch.equal(out16.cpu(), out32.cpu().to(torch.bfloat16))
    # no parts at all: the softmax over an empty set, out = 0 and lse = -inf
    out0, lse0 = api.decode_attn_combine(o_parts[:0], l_parts[:0])
    torch.cuda.synchronize()
    assert torch.all(out0 == 0) and torch.all(torch.isneginf(lse0))


def test_full_cache_partial_equals_decode(o):
    """The whole row range is the ordinary decode, and its lse is the oracle's."""
    q, K, V, lens_t, scale = _case(4, 32, 8, 128, 3000, [3000, 1, 0, 2047], torch.bfloat16, seed=9)
    dev = torch.device("cuda")
    qd, Kd, Vd, ld = q.to(dev), K.to(dev), V.to(dev), lens_t.to(dev)
    po, pl = api.decode_attn_partial(qd, Kd, Vd, ld)
    ref = api.decode_attn(qd, Kd, Vd, ld)
    torch.cuda.synchronize()
    assert torch.max(torch.abs(po - ref)).item() <= TOL[torch.bfloat16]
    _, want_l = o.decode(q.float().numpy(), K.float().numpy(), V.float().numpy(), lens_t.numpy(),
                         scale, threads=8)
    _close_lse(pl.cpu().numpy(), want_l, LSE_TOL)


def test_long_context_in_four_shards(o):
    """The long-context g=8 shape (n = 131072, Llama-2-70B heads) cut into four row
    ranges of one cache, as four GPUs would hold it; every head against the oracle."""
    w = W.WORKLOADS["long_llama2_70b"]
    K, V = W.cache(w)
    lens = W.seq_lens(w)
    q = W.query(w)
    dev = torch.device("cuda")
    qd, Kd, Vd, ld = q.to(dev), K.to(dev), V.to(dev), lens.to(dev)
    cuts = [0, 40000, 65536, 100001, w.n_max]
    parts = [api.decode_attn_partial(qd, Kd, Vd, ld, r0, r1) for r0, r1 in zip(cuts[:-1], cuts[1:])]
    out, lse = api.decode_attn_combine(torch.stack([p[0] for p in parts]),
                                       torch.stack([p[1] for p in parts]))
    torch.cuda.synchronize()
    want, want_l = o.decode(q.float().numpy(), K.float().numpy(), V.float().numpy(),
                            lens.numpy(), w.scale, threads=max(1, o.max_threads()))
    assert np.max(np.abs(out.double().cpu().numpy() - want)) <= TOL[w.dtype]
    _close_lse(lse.cpu().numpy(), want_l, LSE_TOL)


def test_partial_rejects_bad_ranges():
    q, K, V, lens_t, _ = _case(1, 4, 4, 64, 64, [64], torch.float32, seed=1)
    dev = torch.device("cuda")
    with pytest.raises(api.DecodeAttnError):
        api.decode_attn_partial(q.to(dev), K.to(dev), V.to(dev), lens_t.to(dev), 10, 5)
    with pytest.raises(api.DecodeAttnError):
        api.decode_attn_partial(q.to(dev), K.to(dev), V.to(dev), lens_t.to(dev), -1, 5)
