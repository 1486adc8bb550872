"""8-bit KV caches (int8, fp8 e4m3 codes with float32 row scales) on the GPU.

The oracle quantizes on the CPU and dequantizes in float64; the decode oracle
then runs on the dequantized values rounded to float32 (within 2^-24 of the
exact products, far below the tolerance).  Quantization, append and the
cache rows an append writes are compared bit for bit.  Rows past each
sequence's length hold NaN-coded values and NaN scales, so any read of them
into a result shows up as a NaN.

Decode tolerance: the GPU multiplies the codes' exact fp16 values on tensor
cores with fp32 accumulation, applies the scales in fp32 and carries the
softmax weights as an fp16 head plus an fp16 remainder (~22 bits), so its
error is a few float32 roundings per row: 2e-4 absolute on outputs of
magnitude up to ~4.
"""
import numpy as np
import pytest
import torch

import oracle
from decode_attention_kv_split_gb300 import api, workloads as W

pytestmark = pytest.mark.gpu

KINDS = {"int8": (1, torch.int8), "e4m3": (2, torch.float8_e4m3fn)}
TOL = 2e-4


@pytest.fixture(scope="module")
def o():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    api.load()
    return oracle.get()


def _codes_tensor(codes_u8: np.ndarray, dtype) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(codes_u8)).view(dtype)


def make_q8_case(o, kind, B, h_q, h_kv, d, n_max, lens, seed=0):
    w = W.custom(B=B, h_q=h_q, h_kv=h_kv, d_k=d, n=max(lens), n_max=n_max, dtype=torch.float32)
    K, V = W.cache(w, seed)
    kc, ks = o.quantize(K.numpy(), kind)
    vc, vs = o.quantize(V.numpy(), kind)
    for b in range(B):  # unused rows: NaN codes (0x7F for e4m3; 127 for int8) and NaN scales
        kc[b, :, lens[b]:] = 0x7F
        vc[b, :, lens[b]:] = 0x7F
        ks[b, :, lens[b]:] = np.nan
        vs[b, :, lens[b]:] = np.nan
    q = W.query(w, seed).to(torch.bfloat16)
    return w, q, kc, ks, vc, vs, torch.tensor(lens, dtype=torch.int32)


def oracle_decode_q8(o, kind, q, kc, ks, vc, vs, lens, scale):
    Kd = o.dequant(kc, ks, kind)
    Vd = o.dequant(vc, vs, kind)
    for b in range(len(lens)):  # the oracle only reads rows below lens[b]
        Kd[b, :, int(lens[b]):] = 0.0
        Vd[b, :, int(lens[b]):] = 0.0
    want, _ = o.decode(q.float().numpy(), Kd.astype(np.float32), Vd.astype(np.float32),
                       lens.numpy(), scale, threads=8)
    return want


def gpu_decode_q8(kind, q, kc, ks, vc, vs, lens, num_splits=0, out_dtype=None):
    dev = torch.device("cuda")
    tdt = KINDS[kind][1]
    args = (q.to(dev), _codes_tensor(kc, tdt).to(dev), _codes_tensor(vc, tdt).to(dev),
            torch.from_numpy(ks).to(dev), torch.from_numpy(vs).to(dev), lens.to(dev))
    out = api.decode_attn_q8(*args, num_splits=num_splits, out_dtype=out_dtype)
    torch.cuda.synchronize()
    return out.cpu()


def _check(got, want, tol):
    got = got.double().numpy()
    assert np.all(np.isfinite(got)), "non-finite output (unwritten element or padding read)"
    err = float(np.max(np.abs(got - want))) if got.size else 0.0
    assert err <= tol, f"max abs error {err:.3e} > {tol:.1e}"
    return err


# ----------------------------------------------------------------- quantization
@pytest.mark.parametrize("kind", list(KINDS))
@pytest.mark.parametrize("x_dtype", [torch.float32, torch.bfloat16], ids=["fp32", "bf16"])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_kv_quantize_bit_exact(o, kind, x_dtype, d):
    rng = np.random.default_rng(d)
    x = (rng.standard_normal((300, d)) * rng.uniform(0.01, 30, (300, 1))).astype(np.float32)
    x[5] = 0.0                       # zero row
    x[6, 3] = 1e4                    # one huge element
    x[7] = -x[7]
    xt = torch.from_numpy(x).to(x_dtype)
    codes, scales = api.kv_quantize(xt.cuda(), KINDS[kind][1])
    torch.cuda.synchronize()
    want_c, want_s = o.quantize(xt.float().numpy(), KINDS[kind][0])
    got_c = codes.cpu().view(torch.uint8).numpy()
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), want_s.view(np.uint32))
    assert np.array_equal(got_c, want_c), int((got_c != want_c).sum())


# ----------------------------------------------------------------- decode
CASES = [
    # B, h_q, h_kv, d, n_max, lens
    (1, 1, 1, 64, 512, [256]),
    (2, 4, 4, 128, 300, [300, 1]),
    (3, 8, 2, 128, 200, [200, 0, 77]),
    (2, 16, 2, 64, 132, [129, 64]),
    (2, 32, 2, 128, 260, [257, 130]),       # group 16: two head chunks
    (4, 8, 1, 128, 520, [520, 128, 127, 1]),
    (2, 12, 4, 128, 388, [385, 129]),       # group 3 (padded heads)
]


@pytest.mark.parametrize("kind", list(KINDS))
@pytest.mark.parametrize("case", CASES, ids=[f"B{c[0]}_hq{c[1]}_hkv{c[2]}_d{c[3]}_n{c[4]}" for c in CASES])
@pytest.mark.parametrize("splits", [0, 1, 3, -1])
def test_q8_decode_matches_oracle(o, kind, case, splits):
    B, h_q, h_kv, d, n_max, lens = case
    k = KINDS[kind][0]
    w, q, kc, ks, vc, vs, lens_t = make_q8_case(o, k, B, h_q, h_kv, d, n_max, lens, seed=d + h_q)
    out = gpu_decode_q8(kind, q, kc, ks, vc, vs, lens_t, num_splits=splits)
    want = oracle_decode_q8(o, k, q, kc, ks, vc, vs, lens_t, w.scale)
    _check(out, want, TOL)


def _gpu_q8_checked(kind, q, kc, ks, vc, vs, lens, num_splits=0, scale=None):
    """decode_attn_q8 with an explicit scale and the device error word: (out, error bits)."""
    dev = torch.device("cuda")
    tdt = KINDS[kind][1]
    err = torch.zeros((), dtype=torch.int32, device=dev)
    out = api.decode_attn_q8(q.to(dev), _codes_tensor(kc, tdt).to(dev), _codes_tensor(vc, tdt).to(dev),
                             torch.from_numpy(ks).to(dev), torch.from_numpy(vs).to(dev), lens.to(dev),
                             scale=scale, num_splits=num_splits, dev_error=err)
    torch.cuda.synchronize()
    return out.cpu(), int(err.item())


@pytest.mark.parametrize("kind", list(KINDS))
def test_q8_all_sequences_empty(o, kind):
    """No rows anywhere (every cached row NaN-coded), chunked and balanced
    lists: every output is exactly zero and no error bit is set."""
    k = KINDS[kind][0]
    for d in (64, 128):
        _, q, kc, ks, vc, vs, lens_t = make_q8_case(o, k, 3, 8, 2, d, 64, [0, 0, 0], seed=d)
        for splits in (0, 1, 4, -1):
            out, err = _gpu_q8_checked(kind, q, kc, ks, vc, vs, lens_t, splits)
            assert torch.all(out == 0)
            assert err == 0


@pytest.mark.parametrize("kind", list(KINDS))
def test_q8_zero_rows(o, kind):
    """Cached rows that are entirely zero quantize to zero codes with scale 0
    (the format's degenerate row): a zero K row scores 0, a zero V row adds
    weight and no value."""
    k = KINDS[kind][0]
    B, h_q, h_kv, d, n_max, lens = 2, 8, 2, 128, 300, [300, 130]
    w = W.custom(B=B, h_q=h_q, h_kv=h_kv, d_k=d, n=max(lens), n_max=n_max, dtype=torch.float32)
    K, V = W.cache(w, 7)
    K[:, :, ::3] = 0.0
    V[:, :, 1::4] = 0.0
    kc, ks = o.quantize(K.numpy(), k)
    vc, vs = o.quantize(V.numpy(), k)
    assert np.all(ks[:, :, ::3] == 0) and np.all(vs[:, :, 1::4] == 0)
    for b in range(B):  # unused rows: NaN codes and scales, as in make_q8_case
        kc[b, :, lens[b]:] = 0x7F
        vc[b, :, lens[b]:] = 0x7F
        ks[b, :, lens[b]:] = np.nan
        vs[b, :, lens[b]:] = np.nan
    q = W.query(w, 7).to(torch.bfloat16)
    lens_t = torch.tensor(lens, dtype=torch.int32)
    want = oracle_decode_q8(o, k, q, kc, ks, vc, vs, lens_t, w.scale)
    for splits in (0, 3, -1):
        out, err = _gpu_q8_checked(kind, q, kc, ks, vc, vs, lens_t, splits)
        assert err == 0
        _check(out, want, TOL)


@pytest.mark.parametrize("kind", list(KINDS))
def test_q8_peaked_softmax(o, kind):
    """Large scores concentrate the weight on few rows (stresses the score
    arithmetic and the fp16 head + remainder of P): scale 0.5 and 1.0 instead
    of 1/sqrt(128)."""
    k = KINDS[kind][0]
    _, q, kc, ks, vc, vs, lens_t = make_q8_case(o, k, 2, 8, 2, 128, 400, [400, 37], seed=3)
    for scale in (0.5, 1.0):
        want = oracle_decode_q8(o, k, q, kc, ks, vc, vs, lens_t, scale)
        out, err = _gpu_q8_checked(kind, q, kc, ks, vc, vs, lens_t, 4, scale=scale)
        assert err == 0
        _check(out, want, TOL)


@pytest.mark.parametrize("kind", list(KINDS))
def test_q8_tile_boundaries(o, kind):
    lens = [1, 2, 15, 16, 17, 31, 32, 33, 63, 64, 65, 127, 128, 129, 255, 256, 257]
    k = KINDS[kind][0]
    for d in (64, 128):
        w, q, kc, ks, vc, vs, lens_t = make_q8_case(o, k, len(lens), 8, 1, d, 260, lens, seed=d)
        want = oracle_decode_q8(o, k, q, kc, ks, vc, vs, lens_t, w.scale)
        for splits in (0, 1, 2):
            _check(gpu_decode_q8(kind, q, kc, ks, vc, vs, lens_t, num_splits=splits), want, TOL)


@pytest.mark.parametrize("kind", list(KINDS))
def test_q8_bf16_output(o, kind):
    k = KINDS[kind][0]
    w, q, kc, ks, vc, vs, lens_t = make_q8_case(o, k, 3, 8, 2, 128, 300, [300, 5, 160], seed=3)
    out32 = gpu_decode_q8(kind, q, kc, ks, vc, vs, lens_t, num_splits=3)
    out16 = gpu_decode_q8(kind, q, kc, ks, vc, vs, lens_t, num_splits=3, out_dtype=torch.bfloat16)
    assert torch.equal(out16, out32.to(torch.bfloat16))
    want = oracle_decode_q8(o, k, q, kc, ks, vc, vs, lens_t, w.scale)
    got = out16.double().numpy()
    assert np.all(np.abs(got - want) <= TOL + 2.0 ** -8 * np.abs(want))


# ----------------------------------------------------------------- append
@pytest.mark.parametrize("kind", list(KINDS))
def test_kv_append_q8_bit_exact(o, kind):
    k, tdt = KINDS[kind]
    B, h_kv, d, n_max = 3, 2, 128, 40
    rng = np.random.default_rng(1)
    kc = rng.integers(0, 255, (B, h_kv, n_max, d), dtype=np.uint8)
    vc = rng.integers(0, 255, (B, h_kv, n_max, d), dtype=np.uint8)
    ks = rng.standard_normal((B, h_kv, n_max)).astype(np.float32)
    vs = rng.standard_normal((B, h_kv, n_max)).astype(np.float32)
    kn = rng.integers(0, 255, (B, h_kv, d), dtype=np.uint8)
    vn = rng.integers(0, 255, (B, h_kv, d), dtype=np.uint8)
    kns = rng.standard_normal((B, h_kv)).astype(np.float32)
    vns = rng.standard_normal((B, h_kv)).astype(np.float32)
    pos = np.array([0, 39, 40], dtype=np.int32)  # the last one is out of range: not written
    dev = torch.device("cuda")
    Kd, Vd = _codes_tensor(kc, tdt).to(dev), _codes_tensor(vc, tdt).to(dev)
    ksd, vsd = torch.from_numpy(ks).to(dev), torch.from_numpy(vs).to(dev)
    err = torch.zeros((), dtype=torch.int32, device=dev)
    api.kv_append_q8(_codes_tensor(kn, tdt).to(dev), _codes_tensor(vn, tdt).to(dev),
                     torch.from_numpy(kns).to(dev), torch.from_numpy(vns).to(dev), Kd, Vd, ksd, vsd,
                     torch.from_numpy(pos).to(dev), dev_error=err)
    torch.cuda.synchronize()
    skipped = o.kv_append(kn, vn, kc, vc, pos)
    for b in range(B):  # the scales of the written rows
        if 0 <= pos[b] < n_max:
            ks[b, :, pos[b]] = kns[b]
            vs[b, :, pos[b]] = vns[b]
    assert skipped == 1 and int(err.item()) == api.DEVERR_POS
    assert np.array_equal(Kd.cpu().view(torch.uint8).numpy(), kc)
    assert np.array_equal(Vd.cpu().view(torch.uint8).numpy(), vc)
    assert np.array_equal(ksd.cpu().numpy().view(np.uint32), ks.view(np.uint32))
    assert np.array_equal(vsd.cpu().numpy().view(np.uint32), vs.view(np.uint32))


APPEND_CASES = [
    (3, 8, 2, 128, 300, [0, 127, 299]),
    (2, 8, 1, 64, 260, [128, 255]),
    (4, 4, 4, 64, 200, [63, 64, 65, 200]),  # last one has no room: no append, flagged
]


@pytest.mark.parametrize("kind", list(KINDS))
@pytest.mark.parametrize("case", APPEND_CASES, ids=[f"case{i}" for i in range(len(APPEND_CASES))])
@pytest.mark.parametrize("splits", [0, 1, 3, -1])
def test_q8_fused_append_decode(o, kind, case, splits):
    k, tdt = KINDS[kind]
    B, h_q, h_kv, d, n_max, lens = case
    w, q, kc, ks, vc, vs, lens_t = make_q8_case(o, k, B, h_q, h_kv, d, n_max, lens, seed=B + h_q)
    kn_f, vn_f = W.new_rows(W.custom(B=B, h_q=h_q, h_kv=h_kv, d_k=d, n=1, dtype=torch.float32), 3, 7)
    knc, kns = o.quantize(kn_f.numpy(), k)
    vnc, vns = o.quantize(vn_f.numpy(), k)
    dev = torch.device("cuda")
    Kd, Vd = _codes_tensor(kc, tdt).to(dev), _codes_tensor(vc, tdt).to(dev)
    ksd, vsd = torch.from_numpy(ks.copy()).to(dev), torch.from_numpy(vs.copy()).to(dev)
    err = torch.zeros((), dtype=torch.int32, device=dev)
    lens_out = torch.full((B,), -7, dtype=torch.int32, device=dev)
    out = api.decode_attn_q8_append(q.to(dev), _codes_tensor(knc, tdt).to(dev),
                                    _codes_tensor(vnc, tdt).to(dev), torch.from_numpy(kns).to(dev),
                                    torch.from_numpy(vns).to(dev), Kd, Vd, ksd, vsd, lens_t.to(dev),
                                    seq_lens_out=lens_out, num_splits=splits, dev_error=err)
    torch.cuda.synchronize()
    # cache after the append (oracle: byte copies of the code rows and scales)
    pos = lens_t.numpy().copy()
    skipped = o.kv_append(knc, vnc, kc, vc, pos)
    new_lens = lens_t.clone()
    for b in range(B):
        if pos[b] < n_max:
            ks[b, :, pos[b]] = kns[b]
            vs[b, :, pos[b]] = vns[b]
            new_lens[b] += 1
    assert np.array_equal(Kd.cpu().view(torch.uint8).numpy(), kc)
    assert np.array_equal(Vd.cpu().view(torch.uint8).numpy(), vc)
    assert np.array_equal(ksd.cpu().numpy().view(np.uint32), ks.view(np.uint32))
    assert np.array_equal(vsd.cpu().numpy().view(np.uint32), vs.view(np.uint32))
    assert torch.equal(lens_out.cpu(), new_lens)
    assert (int(err.item()) == api.DEVERR_POS) == (skipped > 0)
    want = oracle_decode_q8(o, k, q, kc, ks, vc, vs, new_lens, w.scale)
    _check(out.cpu(), want, TOL)


# ----------------------------------------------------------------- full-size workloads
@pytest.mark.parametrize("name", ["gqa_llama3_8b_fp8", "gqa_llama3_8b_int8", "long_llama2_70b_fp8"])
def test_q8_full_size_workload_every_head(o, name):
    """The bench's 8-bit workloads at full size (ragged GQA in balanced pieces; the
    131072-row long context with the library's splits): the oracle quantizes the
    seeded values, the GPU decodes the codes, every head is compared."""
    w = W.WORKLOADS[name]
    k = 1 if w.dtype == torch.int8 else 2
    K, V = W.cache(w)
    kc, ks = o.quantize(K.numpy(), k)
    vc, vs = o.quantize(V.numpy(), k)
    del K, V
    lens = W.seq_lens(w)
    for b, n in enumerate(lens.tolist()):
        kc[b, :, n:] = 0x7F
        vc[b, :, n:] = 0x7F
        ks[b, :, n:] = np.nan
        vs[b, :, n:] = np.nan
    q = W.query(w)
    dev = torch.device("cuda")
    out = api.decode_attn_q8(q.to(dev), _codes_tensor(kc, w.dtype).to(dev),
                             _codes_tensor(vc, w.dtype).to(dev), torch.from_numpy(ks).to(dev),
                             torch.from_numpy(vs).to(dev), lens.to(dev), num_splits=w.num_splits)
    torch.cuda.synchronize()
    Kd = o.dequant(kc, ks, k)
    Vd = o.dequant(vc, vs, k)
    del kc, vc
    for b, n in enumerate(lens.tolist()):
        Kd[b, :, n:] = 0.0
        Vd[b, :, n:] = 0.0
    want, _ = o.decode(q.float().numpy(), Kd.astype(np.float32), Vd.astype(np.float32),
                       lens.numpy(), w.scale, threads=max(1, o.max_threads()))
    _check(out.cpu(), want, TOL)
