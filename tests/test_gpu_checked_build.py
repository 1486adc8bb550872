"""The bounds-checked test build against the product library (needs a GB300).

The test library is the same sources compiled with DA_BOUNDS_CHECK (and
DA_TEST_HOOKS): every global index the kernels compute for a store, a
per-row load or a bulk copy is checked against the size of its buffer, and
an index outside it skips the access and sets DA_DEVERR_BOUNDS in the
caller's error word.  It stands in for a memory checker: each case runs one
entry point of the C ABI through both libraries on the same inputs (every
kernel family, both work-list modes, appends, 8-bit caches, row ranges and
the merge) and checks that the checked build found no index out of range,
reports the same error word as the product build, and writes bit for bit the
same outputs and caches.
"""
import ctypes

import pytest
import torch

from decode_attention_kv_split_gb300 import api
from decode_attention_kv_split_gb300.build import build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def libs():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    prod = api.load()
    chk = ctypes.CDLL(build(test_hooks=True))
    for name, (res, args) in api.SIGNATURES.items():
        fn = getattr(chk, name)
        fn.restype = res
        fn.argtypes = args
    chk.decode_attn_test_withhold.argtypes = [ctypes.c_int]
    chk.decode_attn_test_withhold.restype = None
    chk.decode_attn_test_withhold(-1)
    return prod, chk


def _both(libs, monkeypatch, run):
    """run(err) -> tensors, once through each library; compare them."""
    got = []
    for lib in libs:
        monkeypatch.setattr(api, "_lib", lib)
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        outs = run(err)
        torch.cuda.synchronize()
        got.append(([t.clone() for t in outs], int(err.item())))
    monkeypatch.setattr(api, "_lib", libs[0])
    (want, err_p), (have, err_c) = got
    assert err_c & api.DEVERR_BOUNDS == 0, f"checked build found an index out of range ({err_c:#x})"
    assert err_c == err_p, f"error words differ: product {err_p:#x}, checked {err_c:#x}"
    for a, b in zip(want, have):
        torch.testing.assert_close(b, a, rtol=0, atol=0, equal_nan=True)
    return err_p


def _gen(seed):
    g = torch.Generator().manual_seed(seed)
    return lambda *shape: torch.randn(*shape, generator=g)


def _inputs(B, h_q, h_kv, dk, dv, n_max, lens, dtype, seed=0):
    r = _gen(seed)
    q = r(B, h_q, dk).to(dtype)
    K = r(B, h_kv, n_max, dk).to(dtype)
    V = r(B, h_kv, n_max, dv).to(dtype)
    for b, n in enumerate(lens):  # rows past the length are never read
        n = min(max(n, 0), n_max)
        K[b, :, n:] = float("nan")
        V[b, :, n:] = float("nan")
    lens = torch.tensor(lens, dtype=torch.int32)
    return [t.cuda() for t in (q, K, V, lens)]


# name, B, h_q, h_kv, d_k, d_v, n_max, lens, dtype
SHAPES = [
    ("fp32_mha_d64", 3, 8, 8, 64, 64, 700, [700, 0, 333], torch.float32),
    ("bf16_gqa_g8", 4, 32, 4, 128, 128, 2000, [2000, 1, 999, 1500], torch.bfloat16),
    ("bf16_mqa_g32", 2, 32, 1, 128, 128, 3000, [3000, 1234], torch.bfloat16),
    ("bf16_d256", 2, 32, 2, 256, 256, 260, [260, 65], torch.bfloat16),
    ("bf16_dk192_dv128", 2, 32, 4, 192, 128, 260, [257, 128], torch.bfloat16),
    ("bf16_clamped_lens", 3, 16, 2, 128, 128, 500, [-5, 5000, 100], torch.bfloat16),
]


@pytest.mark.parametrize("splits", [0, 1, 3, -1])
@pytest.mark.parametrize("shape", SHAPES, ids=[s[0] for s in SHAPES])
def test_decode(libs, monkeypatch, shape, splits):
    _, B, h_q, h_kv, dk, dv, n_max, lens, dtype = shape
    q, K, V, sl = _inputs(B, h_q, h_kv, dk, dv, n_max, lens, dtype)
    out_dtype = torch.bfloat16 if splits == 3 and dtype == torch.bfloat16 else None
    err = _both(libs, monkeypatch, lambda e: [
        api.decode_attn(q, K, V, sl, num_splits=splits, dev_error=e, out_dtype=out_dtype)])
    clamped = any(n < 0 or n > n_max for n in lens)
    assert bool(err & api.DEVERR_SEQ_LEN) == clamped


def test_many_items_per_cta(libs, monkeypatch):
    g = torch.Generator().manual_seed(7)
    lens = torch.randint(0, 65, (512,), generator=g).tolist()
    q, K, V, sl = _inputs(512, 128, 32, 64, 64, 64, lens, torch.bfloat16, seed=7)
    for splits in (-1, 0):
        _both(libs, monkeypatch, lambda e: [api.decode_attn(q, K, V, sl, num_splits=splits,
                                                            dev_error=e)])


APPEND = [
    ("fp32", 2, 4, 4, 64, 300, [299, 300], torch.float32),
    ("bf16_gqa_g8", 3, 32, 4, 128, 1000, [0, 999, 1000], torch.bfloat16),
    ("bf16_mqa_g32", 2, 32, 1, 128, 2000, [1999, 700], torch.bfloat16),
]


@pytest.mark.parametrize("splits", [0, -1])
@pytest.mark.parametrize("case", APPEND, ids=[c[0] for c in APPEND])
def test_decode_append(libs, monkeypatch, case, splits):
    _, B, h_q, h_kv, d, n_max, lens, dtype = case
    q, K, V, sl = _inputs(B, h_q, h_kv, d, d, n_max, lens, dtype, seed=3)
    r = _gen(4)
    k_new = r(B, h_kv, d).to(dtype).cuda()
    v_new = r(B, h_kv, d).to(dtype).cuda()

    def run(e):
        Kc, Vc = K.clone(), V.clone()
        lens_out = torch.full_like(sl, -7)
        out = api.decode_attn_append(q, k_new, v_new, Kc, Vc, sl, seq_lens_out=lens_out,
                                     num_splits=splits, dev_error=e)
        return [out, Kc, Vc, lens_out]

    err = _both(libs, monkeypatch, run)
    assert bool(err & api.DEVERR_POS) == any(n >= n_max for n in lens)


def test_kv_append(libs, monkeypatch):
    B, h_kv, n_max, d = 4, 8, 100, 128
    _, K, V, _ = _inputs(B, 8, h_kv, d, d, n_max, [n_max] * B, torch.bfloat16, seed=5)
    r = _gen(6)
    k_new = r(B, h_kv, d).to(torch.bfloat16).cuda()
    v_new = r(B, h_kv, d).to(torch.bfloat16).cuda()
    pos = torch.tensor([0, 99, -1, 100], dtype=torch.int32, device="cuda")

    def run(e):
        Kc, Vc = K.clone(), V.clone()
        api.kv_append(k_new, v_new, Kc, Vc, pos, dev_error=e)
        return [Kc, Vc]

    assert _both(libs, monkeypatch, run) & api.DEVERR_POS


def _codes(shape, dtype, g):
    if dtype == torch.int8:
        return torch.randint(-127, 128, shape, generator=g, dtype=torch.int8)
    c = torch.randint(0, 0x7F, shape, generator=g, dtype=torch.uint8)  # finite e4m3 codes
    sign = torch.randint(0, 2, shape, generator=g, dtype=torch.uint8) << 7
    return (c | sign).view(torch.float8_e4m3fn)


def _q8_inputs(B, h_q, h_kv, d, n_max, lens, cdt, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, h_q, d, generator=g).to(torch.bfloat16)
    K, V = _codes((B, h_kv, n_max, d), cdt, g), _codes((B, h_kv, n_max, d), cdt, g)
    ks = torch.rand(B, h_kv, n_max, generator=g) * 0.05 + 0.01
    vs = torch.rand(B, h_kv, n_max, generator=g) * 0.05 + 0.01
    for b, n in enumerate(lens):
        ks[b, :, n:] = float("nan")
        vs[b, :, n:] = float("nan")
    lens = torch.tensor(lens, dtype=torch.int32)
    return [t.cuda() for t in (q, K, V, ks, vs, lens)]


Q8 = [
    ("int8_d128_g8", 3, 32, 4, 128, 1500, [1500, 3, 777], torch.int8),
    ("e4m3_d128_g8", 2, 32, 4, 128, 1500, [1499, 1024], torch.float8_e4m3fn),
    ("int8_d64_g4", 2, 16, 4, 64, 600, [600, 129], torch.int8),
    ("e4m3_d128_mha", 2, 4, 4, 128, 900, [900, 65], torch.float8_e4m3fn),
]


@pytest.mark.parametrize("splits", [0, 1, -1])
@pytest.mark.parametrize("case", Q8, ids=[c[0] for c in Q8])
def test_q8(libs, monkeypatch, case, splits):
    _, B, h_q, h_kv, d, n_max, lens, cdt = case
    q, K, V, ks, vs, sl = _q8_inputs(B, h_q, h_kv, d, n_max, lens, cdt, seed=11)
    _both(libs, monkeypatch, lambda e: [api.decode_attn_q8(q, K, V, ks, vs, sl, num_splits=splits,
                                                           dev_error=e)])


@pytest.mark.parametrize("case", Q8[:3], ids=[c[0] for c in Q8[:3]])
def test_q8_append(libs, monkeypatch, case):
    _, B, h_q, h_kv, d, n_max, lens, cdt = case
    lens = [min(n, n_max - 1) for n in lens[:-1]] + [n_max]  # the last one cannot append
    q, K, V, ks, vs, sl = _q8_inputs(B, h_q, h_kv, d, n_max, lens, cdt, seed=12)
    g = torch.Generator().manual_seed(13)
    k_new, v_new = _codes((B, h_kv, d), cdt, g).cuda(), _codes((B, h_kv, d), cdt, g).cuda()
    kns = (torch.rand(B, h_kv, generator=g) * 0.05 + 0.01).cuda()
    vns = (torch.rand(B, h_kv, generator=g) * 0.05 + 0.01).cuda()

    def run(e):
        Kc, Vc, ksc, vsc = K.clone(), V.clone(), ks.clone(), vs.clone()
        out = api.decode_attn_q8_append(q, k_new, v_new, kns, vns, Kc, Vc, ksc, vsc, sl,
                                        dev_error=e)
        return [out, Kc.view(torch.uint8), Vc.view(torch.uint8), ksc, vsc]

    assert _both(libs, monkeypatch, run) & api.DEVERR_POS


@pytest.mark.parametrize("splits", [0, -1])
def test_partial_and_combine(libs, monkeypatch, splits):
    B, h_q, h_kv, d, n_max, lens = 3, 32, 4, 128, 2000, [2000, 600, 1001]
    q, K, V, sl = _inputs(B, h_q, h_kv, d, d, n_max, lens, torch.bfloat16, seed=9)
    ranges = [(0, 700), (700, 1400), (1400, 2000)]

    def run(e):
        parts = [api.decode_attn_partial(q, K, V, sl, r0, r1, num_splits=splits, dev_error=e)
                 for r0, r1 in ranges]
        o = torch.stack([p[0] for p in parts]).contiguous()
        lse = torch.stack([p[1] for p in parts]).contiguous()
        out, lse_out = api.decode_attn_combine(o, lse, out_dtype=torch.bfloat16)
        return [o, lse, out, lse_out]

    _both(libs, monkeypatch, run)


def test_kv_quantize(libs, monkeypatch):
    x = torch.randn(3, 5, 77, 128, generator=torch.Generator().manual_seed(2)).cuda()
    for cdt in (torch.int8, torch.float8_e4m3fn):
        _both(libs, monkeypatch,
              lambda e: [t.view(torch.uint8) if t.dtype == cdt else t
                         for t in api.kv_quantize(x, cdt)])
