"""CUDA path against the fp64 CPU oracle, element by element (needs a GB300).

Tolerances (max abs error against the oracle run on the same rounded inputs):
1e-5 for an fp32 cache, 2e-3 for a bf16 cache; kv_append is bit-exact.
Cache rows past each sequence's length are filled with NaN, so any read of
them into a result shows up as a NaN.  Outputs are pre-filled with NaN, so
any element a kernel fails to write shows up too.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from decode_attention_kv_split_gb300 import api, workloads as W

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-5, torch.bfloat16: 2e-3}


@pytest.fixture(scope="module")
def o():
    return oracle.get()


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    api.load()


def _f32(t):
    return t.float().contiguous().numpy()


def gpu_decode(q, K, V, lens, num_splits=0, scale=None, dev_error=None):
    dev = torch.device("cuda")
    qd, Kd, Vd = q.to(dev), K.to(dev), V.to(dev)
    ld = lens.to(dev)
    out = torch.full((q.shape[0], q.shape[1], V.shape[3]), float("nan"), device=dev)
    api.decode_attn(qd, Kd, Vd, ld, out=out, scale=scale, num_splits=num_splits, dev_error=dev_error)
    torch.cuda.synchronize()
    return out.cpu()


def check_against_oracle(o, q, K, V, lens, scale, out, tol):
    want, _ = o.decode(_f32(q), _f32(K), _f32(V), lens.numpy(), scale, threads=8)
    got = out.double().numpy()
    assert np.all(np.isfinite(got)), "non-finite output (unwritten element or padding read)"
    err = np.max(np.abs(got - want)) if got.size else 0.0
    assert err <= tol, f"max abs error {err:.3e} > {tol:.1e}"
    return err


def make_case(B, h_q, h_kv, d, n_max, lens, dtype, seed=0, kv_std=1.0):
    w = W.custom(B=B, h_q=h_q, h_kv=h_kv, d_k=d, n=max(lens) if lens else 0, n_max=n_max,
                 dtype=dtype, kv_std=kv_std)
    K, V = W.cache(w, seed)
    lens_t = torch.tensor(lens, dtype=torch.int32)
    for b in range(B):
        K[b, :, lens[b]:] = float("nan")
        V[b, :, lens[b]:] = float("nan")
    q = W.query(w, seed)
    return q, K, V, lens_t, w.scale


# ----------------------------------------------------------------- decode sweeps
SWEEP = [
    # B, h_q, h_kv, d, n_max, lens
    (1, 1, 1, 64, 512, [256]),
    (2, 4, 4, 128, 300, [300, 1]),
    (3, 8, 2, 128, 200, [200, 0, 77]),
    (2, 16, 2, 64, 129, [129, 64]),
    (2, 32, 2, 128, 257, [257, 130]),       # group 16
    (1, 8, 8, 128, 1000, [999]),
    (2, 32, 1, 128, 700, [700, 321]),       # MQA group 32
    (1, 64, 1, 64, 300, [300]),             # group 64 (two head chunks)
    (2, 12, 4, 128, 385, [385, 129]),       # group 3 (padded heads)
    (4, 8, 1, 128, 520, [520, 128, 127, 1]),
]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["fp32", "bf16"])
@pytest.mark.parametrize("case", SWEEP, ids=[f"B{c[0]}_hq{c[1]}_hkv{c[2]}_d{c[3]}_n{c[4]}" for c in SWEEP])
@pytest.mark.parametrize("splits", [0, 1, 3, 1000, -1])
def test_decode_matches_oracle(o, dtype, case, splits):
    B, h_q, h_kv, d, n_max, lens = case
    q, K, V, lens_t, scale = make_case(B, h_q, h_kv, d, n_max, lens, dtype, seed=len(lens) + d)
    out = gpu_decode(q, K, V, lens_t, num_splits=splits)
    check_against_oracle(o, q, K, V, lens_t, scale, out, TOL[dtype])


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["fp32", "bf16"])
def test_tile_boundaries(o, dtype):
    """Lengths one short of, equal to and one past multiples of every stage height."""
    lens = [1, 2, 15, 16, 17, 31, 32, 33, 63, 64, 65, 127, 128, 129, 255, 256, 257]
    for d in (64, 128):
        for g in (1, 4, 32):
            q, K, V, lens_t, scale = make_case(len(lens), g, 1, d, 260, lens, dtype, seed=g + d)
            for splits in (0, 1, 2):
                out = gpu_decode(q, K, V, lens_t, num_splits=splits)
                check_against_oracle(o, q, K, V, lens_t, scale, out, TOL[dtype])


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["fp32", "bf16"])
def test_peaked_softmax(o, dtype):
    """Large scores concentrate the weight on few rows (stresses the P precision)."""
    q, K, V, lens_t, _ = make_case(2, 8, 2, 128, 400, [400, 37], dtype, seed=3)
    for scale in (1.0, 0.5):
        out = gpu_decode(q, K, V, lens_t, scale=scale, num_splits=4)
        check_against_oracle(o, q, K, V, lens_t, scale, out, TOL[dtype])


def test_all_sequences_empty(o):
    q, K, V, lens_t, scale = make_case(3, 8, 2, 128, 64, [0, 0, 0], torch.bfloat16)
    for splits in (0, 1, 4):
        out = gpu_decode(q, K, V, lens_t, num_splits=splits)
        assert torch.all(out == 0)


@pytest.mark.parametrize("dtype,h_q", [(torch.float32, 8), (torch.bfloat16, 8), (torch.bfloat16, 64)],
                         ids=["fp32_g4", "bf16_g4", "bf16_g32"])
def test_all_sequences_empty_every_family(o, dtype, h_q):
    """No rows anywhere, in every list mode (balanced pieces count an empty
    sequence as one row so that its zero output is still written): every
    output is exactly zero and no error bit is set."""
    q, K, V, lens_t, _ = make_case(3, h_q, 2, 128, 64, [0, 0, 0], dtype)
    for splits in (0, 1, 4, -1):
        err = torch.zeros((), dtype=torch.int32, device="cuda")
        out = gpu_decode(q, K, V, lens_t, num_splits=splits, dev_error=err)
        assert torch.all(out == 0)
        assert int(err.item()) == 0


@pytest.mark.parametrize("dtype,h_q,h_kv", [(torch.float32, 8, 2), (torch.bfloat16, 8, 2),
                                            (torch.bfloat16, 32, 1)],
                         ids=["fp32_g4", "bf16_g4", "bf16_g32"])
def test_zero_scale_is_the_mean_of_v(o, dtype, h_q, h_kv):
    """scale = 0 makes every score 0, so every weight is 1/n and each query
    head's output is the plain mean of its KV head's first n rows of V:
    checked against the oracle and against that mean taken directly."""
    lens = [300, 129, 1]
    q, K, V, lens_t, _ = make_case(3, h_q, h_kv, 128, 300, lens, dtype, seed=11)
    g = h_q // h_kv
    for splits in (0, 3, -1):
        out = gpu_decode(q, K, V, lens_t, num_splits=splits, scale=0.0)
        check_against_oracle(o, q, K, V, lens_t, 0.0, out, TOL[dtype])
        for b, n in enumerate(lens):
            mean = V[b, :, :n].double().mean(dim=1)        # [h_kv, d_v]
            want = mean.repeat_interleave(g, dim=0)         # query head h reads kv head h // g
            assert torch.max(torch.abs(out[b].double() - want)).item() <= TOL[dtype]


def test_large_n_max_few_rows(o):
    """A cache sized for 262144 rows that holds a few hundred: the host plans
    for n_max, the device splits the actual lengths.  Only the rows below the
    lengths reach the oracle (the rest are NaN and must never be read)."""
    B, h_q, h_kv, d, n_max = 2, 16, 2, 64, 1 << 18
    q, K, V, lens_t, scale = make_case(B, h_q, h_kv, d, n_max, [5, 200], torch.bfloat16, seed=5)
    for splits in (0, 2, 300, -1):
        out = gpu_decode(q, K, V, lens_t, num_splits=splits)
        check_against_oracle(o, q, K[:, :, :256], V[:, :, :256], lens_t, scale, out,
                             TOL[torch.bfloat16])


def test_out_of_range_lengths_are_clamped_and_flagged(o):
    q, K, V, _, scale = make_case(2, 4, 2, 64, 100, [100, 50], torch.float32)
    err = torch.zeros((), dtype=torch.int32, device="cuda")
    bad = torch.tensor([150, -3], dtype=torch.int32)
    out = gpu_decode(q, K, V, bad, dev_error=err)
    assert int(err.item()) & api.DEVERR_SEQ_LEN
    clamped = torch.tensor([100, 0], dtype=torch.int32)
    check_against_oracle(o, q, K, V, clamped, scale, out, TOL[torch.float32])


def test_repeatable_bit_for_bit(o):
    q, K, V, lens_t, _ = make_case(2, 32, 8, 128, 3000, [3000, 1777], torch.bfloat16)
    a = gpu_decode(q, K, V, lens_t, num_splits=5)
    b = gpu_decode(q, K, V, lens_t, num_splits=5)
    assert torch.equal(a, b)


def test_gqa_equals_replicated_mha_on_gpu(o):
    """Introduction item 4 on the device: reading KV head h // g equals running
    MHA on a cache with every KV head repeated g times."""
    for dtype in (torch.float32, torch.bfloat16):
        q, K, V, lens_t, _ = make_case(2, 16, 4, 128, 300, [300, 200], dtype)
        a = gpu_decode(q, K, V, lens_t, num_splits=2)
        Kr = K.repeat_interleave(4, dim=1).contiguous()
        Vr = V.repeat_interleave(4, dim=1).contiguous()
        b = gpu_decode(q, Kr, Vr, lens_t, num_splits=2)
        assert torch.max(torch.abs(a - b)).item() <= TOL[dtype]


def test_owned_workspace_entry_point(o):
    q, K, V, lens_t, scale = make_case(2, 32, 8, 128, 5000, [5000, 4000], torch.bfloat16)
    dev = torch.device("cuda")
    out = api.decode_attn_owned(q.to(dev), K.to(dev), V.to(dev), lens_t.to(dev))
    torch.cuda.synchronize()
    check_against_oracle(o, q, K, V, lens_t, scale, out.cpu(), TOL[torch.bfloat16])


# ----------------------------------------------------------------- kv_append
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["fp32", "bf16"])
def test_kv_append_bit_exact(o, dtype):
    B, h_kv, n_max, d = 5, 3, 40, 128
    w = W.custom(B=B, h_q=h_kv, h_kv=h_kv, d_k=d, n=n_max, n_max=n_max, dtype=dtype)
    K, V = W.cache(w, 1)
    kn, vn = W.new_rows(w, 0, 1)
    pos = torch.tensor([0, 39, 17, -1, 40], dtype=torch.int32)   # last two out of range
    dev = torch.device("cuda")
    Kd, Vd = K.to(dev), V.to(dev)
    err = torch.zeros((), dtype=torch.int32, device=dev)
    api.kv_append(kn.to(dev), vn.to(dev), Kd, Vd, pos.to(dev), dev_error=err)
    torch.cuda.synchronize()
    view = np.uint16 if dtype == torch.bfloat16 else np.uint32
    Kw = K.view(torch.int16 if dtype == torch.bfloat16 else torch.int32).numpy().view(view).copy()
    Vw = V.view(torch.int16 if dtype == torch.bfloat16 else torch.int32).numpy().view(view).copy()
    kw = kn.view(torch.int16 if dtype == torch.bfloat16 else torch.int32).numpy().view(view).copy()
    vw = vn.view(torch.int16 if dtype == torch.bfloat16 else torch.int32).numpy().view(view).copy()
    skipped = o.kv_append(kw, vw, Kw, Vw, pos.numpy())
    assert skipped == 2
    got_K = Kd.cpu().view(torch.int16 if dtype == torch.bfloat16 else torch.int32).numpy().view(view)
    got_V = Vd.cpu().view(torch.int16 if dtype == torch.bfloat16 else torch.int32).numpy().view(view)
    assert np.array_equal(got_K, Kw)
    assert np.array_equal(got_V, Vw)
    assert int(err.item()) & api.DEVERR_POS


def test_append_then_decode_is_causal_last_row(o):
    """After appending row t, a decode over rows 0..t equals row t of full causal
    attention computed by the oracle from the same q, k, v rows."""
    T, d, h = 9, 64, 2
    rng = np.random.default_rng(7)
    Q = rng.standard_normal((h, T, d)).astype(np.float32)
    Kf = rng.standard_normal((h, T, d)).astype(np.float32)
    Vf = rng.standard_normal((h, T, d)).astype(np.float32)
    scale = 1 / math.sqrt(d)
    full = o.causal_attention(Q, Kf, Vf, scale)
    dev = torch.device("cuda")
    K = torch.full((1, h, 16, d), float("nan"), device=dev)
    V = torch.full((1, h, 16, d), float("nan"), device=dev)
    for t in range(T):
        pos = torch.tensor([t], dtype=torch.int32, device=dev)
        api.kv_append(torch.from_numpy(Kf[:, t][None].copy()).to(dev),
                      torch.from_numpy(Vf[:, t][None].copy()).to(dev), K, V, pos)
        out = api.decode_attn(torch.from_numpy(Q[:, t][None].copy()).to(dev), K, V, pos + 1)
        torch.cuda.synchronize()
        err = np.max(np.abs(out.cpu().double().numpy()[0] - full[:, t]))
        assert err <= 1e-5, (t, err)


# ----------------------------------------------------------------- full-size workloads
def _sampled_parity(o, w, q, Kd, Vd, lens, out, units):
    tol = TOL[w.dtype]
    worst = 0.0
    for b, h in units:
        kvh = h // w.group
        n = int(lens[b])
        qv = q[b, h].float().numpy()
        Kb = Kd[b, kvh, :n].float().cpu().numpy()
        Vb = Vd[b, kvh, :n].float().cpu().numpy()
        want, _ = o.decode_head(qv, Kb, Vb, w.scale)
        got = out[b, h].double().cpu().numpy()
        assert np.all(np.isfinite(got))
        worst = max(worst, float(np.max(np.abs(got - want))))
    assert worst <= tol, f"{w.name}: max abs error {worst:.3e} > {tol:.1e}"


def _units(w, k, seed):
    rng = np.random.default_rng(seed)
    picks = {(0, 0), (w.B - 1, w.h_q - 1)}
    while len(picks) < min(k, w.B * w.h_q):
        picks.add((int(rng.integers(w.B)), int(rng.integers(w.h_q))))
    return sorted(picks)


@pytest.mark.parametrize("name", ["gqa_llama3_8b", "mqa_g32", "long_llama2_70b"])
def test_full_size_workload_every_head(o, name):
    """The full-size bf16 workloads in the bench's split configuration, every
    head of every sequence against the oracle (on all host cores)."""
    w = W.WORKLOADS[name]
    dev = torch.device("cuda")
    K, V = W.cache(w)
    lens = W.seq_lens(w)
    q = W.query(w)
    out = torch.full((w.B, w.h_q, w.d_v), float("nan"), device=dev)
    api.decode_attn(q.to(dev), K.to(dev), V.to(dev), lens.to(dev), out=out,
                    num_splits=w.num_splits)
    torch.cuda.synchronize()
    want, _ = o.decode(q.float().numpy(), K.float().numpy(), V.float().numpy(), lens.numpy(),
                       w.scale, threads=max(1, o.max_threads()))
    got = out.double().cpu().numpy()
    assert np.all(np.isfinite(got))
    err = float(np.max(np.abs(got - want)))
    assert err <= TOL[w.dtype], f"{name}: max abs error {err:.3e}"


def test_single_head_workload_append_and_redecode(o):
    w = W.WORKLOADS["single_head"]
    dev = torch.device("cuda")
    K, V = W.cache(w, poison=True)
    lens = W.seq_lens(w)
    q = W.query(w)
    Kd, Vd = K.to(dev), V.to(dev)
    out = gpu_decode(q, K, V, lens)
    check_against_oracle(o, q, K, V, lens, w.scale, out, TOL[w.dtype])
    kn, vn = W.new_rows(w, 0)
    api.kv_append(kn.to(dev), vn.to(dev), Kd, Vd, lens.to(dev))
    lens2 = lens + 1
    out2 = torch.full((1, 1, w.d_v), float("nan"), device=dev)
    api.decode_attn(q.to(dev), Kd, Vd, lens2.to(dev), out=out2)
    torch.cuda.synchronize()
    K[0, 0, 256], V[0, 0, 256] = kn[0, 0], vn[0, 0]
    check_against_oracle(o, q, K, V, lens2, w.scale, out2.cpu(), TOL[w.dtype])


def test_mha_fp32_workload_sixteen_steps(o):
    """All heads, at the first and the last of 16 append+decode steps."""
    w = W.WORKLOADS["mha_fp32"]
    dev = torch.device("cuda")
    K, V = W.cache(w, poison=True)
    lens = W.seq_lens(w)
    q = W.query(w)
    Kd, Vd, ld, qd = K.to(dev), V.to(dev), lens.to(dev), q.to(dev)
    for t in range(w.steps):
        kn, vn = W.new_rows(w, t)
        api.kv_append(kn.to(dev), vn.to(dev), Kd, Vd, ld)
        ld += 1
        out = torch.full((w.B, w.h_q, w.d_v), float("nan"), device=dev)
        api.decode_attn(qd, Kd, Vd, ld, out=out)
        K[:, :, w.n + t] = kn
        V[:, :, w.n + t] = vn
        if t in (0, w.steps - 1):
            torch.cuda.synchronize()
            check_against_oracle(o, q, K, V, lens + t + 1, w.scale, out.cpu(), TOL[w.dtype])
    assert torch.equal(Kd.cpu()[:, :, w.n:w.n + w.steps], K[:, :, w.n:w.n + w.steps])


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["fp32", "bf16"])
def test_batch_larger_than_one_launch_slice(o, dtype):
    """More than 1024 sequences run as several launches sharing one workspace."""
    B = 1100
    rng = np.random.default_rng(4)
    lens = [int(x) for x in rng.integers(0, 70, B)]
    q, K, V, lens_t, scale = make_case(B, 4, 2, 64, 70, lens, dtype, seed=5)
    for splits in (0, 1, 3, -1):
        out = gpu_decode(q, K, V, lens_t, num_splits=splits)
        check_against_oracle(o, q, K, V, lens_t, scale, out, TOL[dtype])


# ----------------------------------------------------------------- balanced pieces (num_splits = -1)
BALANCED = [
    # B, h_q, h_kv, d, n_max, dtype; lengths drawn in [0, n_max] with zeros and full rows forced
    (16, 32, 8, 128, 3000, torch.bfloat16),   # GQA group 4 (mma.sync kernel)
    (6, 32, 1, 128, 5000, torch.bfloat16),    # MQA (tcgen05 kernel)
    (12, 8, 8, 64, 2000, torch.float32),      # MHA (fp32 kernel)
    (40, 16, 2, 64, 700, torch.bfloat16),     # many short units, group 8, d = 64
    (3, 64, 1, 64, 900, torch.bfloat16),      # group 64: two head chunks
]


@pytest.mark.parametrize("case", BALANCED, ids=[f"B{c[0]}_hq{c[1]}_hkv{c[2]}_d{c[3]}_{str(c[5])[6:]}" for c in BALANCED])
def test_balanced_pieces_ragged(o, case):
    """One equal piece of the concatenated rows per CTA: units cut at arbitrary
    tile boundaries, several units per CTA, empty and full sequences."""
    B, h_q, h_kv, d, n_max, dtype = case
    rng = np.random.default_rng(B + d)
    lens = [int(x) for x in rng.integers(0, n_max + 1, B)]
    lens[0], lens[-1] = 0, n_max
    q, K, V, lens_t, scale = make_case(B, h_q, h_kv, d, n_max, lens, dtype, seed=B)
    out = gpu_decode(q, K, V, lens_t, num_splits=-1)
    check_against_oracle(o, q, K, V, lens_t, scale, out, TOL[dtype])


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["fp32", "bf16"])
def test_library_choice_balances_an_uneven_grid(o, dtype):
    """With the library's choice, where one split per unit would be taken but
    the units leave much of the grid idle (16 sequences x 8 kv heads = 128
    units on 152 CTAs), the units get balanced pieces instead; units that fill
    whole rounds keep one split each."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    B, h_q, h_kv, d, n_max = 16, 32, 8, 128, 4096
    if 128 >= 0.9 * sms:
        pytest.skip("128 units fill this device's grid")
    assert api.resolve_splits(B, h_q, h_kv, d, d, n_max, dtype, 0) == sms
    if sms % 8 == 0:  # sms / 8 sequences x 8 kv heads: exactly one round of units
        assert api.resolve_splits(sms // 8, h_q, h_kv, d, d, n_max, dtype, 0) == 1
    rng = np.random.default_rng(12)
    lens = [int(x) for x in rng.integers(1, n_max + 1, B)]
    lens[0] = n_max
    q, K, V, lens_t, scale = make_case(B, h_q, h_kv, d, n_max, lens, dtype, seed=12)
    out = gpu_decode(q, K, V, lens_t, num_splits=0)
    check_against_oracle(o, q, K, V, lens_t, scale, out, TOL[dtype])


@pytest.mark.parametrize("d", [64, 128, 256])
def test_balanced_long_unit_among_short_ones(o, d):
    """Balanced pieces over many short units and one long one: the combine is
    the one-warp-per-head kind (few pieces per unit on average), and the long
    unit's heads have many more pieces than one pass of it holds."""
    B, h_q, h_kv, n_max = 64, 8, 2, 16384
    lens = [64 + (7 * b) % 61 for b in range(B)]
    lens[5] = n_max
    dtype = torch.bfloat16
    q, K, V, lens_t, scale = make_case(B, h_q, h_kv, d, n_max, lens, dtype, seed=d)
    out = gpu_decode(q, K, V, lens_t, num_splits=-1)
    check_against_oracle(o, q, K, V, lens_t, scale, out, TOL[dtype])


# ----------------------------------------------------------------- fused append + decode
def _bits(t):
    return t.view(torch.int16 if t.dtype == torch.bfloat16 else torch.int32).numpy()


APPEND_CASES = [
    # B, h_q, h_kv, d, n_max, lens before the append
    (3, 8, 2, 128, 300, [0, 127, 299]),       # empty, a stage boundary, the last free row
    (2, 32, 1, 128, 700, [699, 320]),         # MQA
    (2, 64, 1, 64, 260, [128, 255]),          # two head chunks
    (4, 4, 4, 64, 200, [63, 64, 65, 200]),    # last one has no room: no append, flagged
]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["fp32", "bf16"])
@pytest.mark.parametrize("case", APPEND_CASES, ids=[f"case{i}" for i in range(len(APPEND_CASES))])
@pytest.mark.parametrize("splits", [0, 1, 3, -1])
def test_fused_append_decode(o, dtype, case, splits):
    B, h_q, h_kv, d, n_max, lens = case
    q, K, V, lens_t, scale = make_case(B, h_q, h_kv, d, n_max, lens, dtype, seed=B + h_q)
    w = W.custom(B=B, h_q=h_q, h_kv=h_kv, d_k=d, n=max(lens), n_max=n_max, dtype=dtype)
    kn, vn = W.new_rows(w, 3, seed=7)
    dev = torch.device("cuda")
    Kd, Vd = K.to(dev), V.to(dev)
    err = torch.zeros((), dtype=torch.int32, device=dev)
    lens_out = torch.full((B,), -7, dtype=torch.int32, device=dev)
    out = torch.full((B, h_q, d), float("nan"), device=dev)
    api.decode_attn_append(q.to(dev), kn.to(dev), vn.to(dev), Kd, Vd, lens_t.to(dev), out=out,
                           seq_lens_out=lens_out, num_splits=splits, dev_error=err)
    torch.cuda.synchronize()
    # oracle: append, then decode over the grown lengths
    Kw, Vw = _bits(K).copy(), _bits(V).copy()
    skipped = o.kv_append(_bits(kn).copy(), _bits(vn).copy(), Kw, Vw, lens_t.numpy())
    grown = torch.tensor([n + 1 if n < n_max else n for n in lens], dtype=torch.int32)
    assert np.array_equal(_bits(Kd.cpu()), Kw) and np.array_equal(_bits(Vd.cpu()), Vw)
    assert torch.equal(lens_out.cpu(), grown)
    assert bool(int(err.item()) & api.DEVERR_POS) == (skipped > 0)
    K2 = torch.from_numpy(Kw).view(dtype)
    V2 = torch.from_numpy(Vw).view(dtype)
    check_against_oracle(o, q, K2, V2, grown, scale, out.cpu(), TOL[dtype])


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["fp32", "bf16"])
def test_fused_append_sixteen_steps(o, dtype):
    """Sixteen fused steps, lengths ping-ponged through seq_lens_out, equal the
    oracle's sixteen appends and decodes."""
    B, h_q, h_kv, d, n0, steps = 2, 8, 4, 128, 250, 16
    n_max = n0 + steps
    q, K, V, lens_t, scale = make_case(B, h_q, h_kv, d, n_max, [n0, n0 - 100], dtype, seed=11)
    w = W.custom(B=B, h_q=h_q, h_kv=h_kv, d_k=d, n=n0, n_max=n_max, dtype=dtype)
    dev = torch.device("cuda")
    Kd, Vd, qd = K.to(dev), V.to(dev), q.to(dev)
    la, lb = lens_t.to(dev), torch.empty(B, dtype=torch.int32, device=dev)
    Kw, Vw = _bits(K).copy(), _bits(V).copy()
    lens_np = lens_t.numpy().copy()
    for t in range(steps):
        kn, vn = W.new_rows(w, t, seed=13)
        out = api.decode_attn_append(qd, kn.to(dev), vn.to(dev), Kd, Vd, la, seq_lens_out=lb,
                                     num_splits=2)
        o.kv_append(_bits(kn).copy(), _bits(vn).copy(), Kw, Vw, lens_np)
        lens_np += 1
        la, lb = lb, la
        if t in (0, steps - 1):
            torch.cuda.synchronize()
            check_against_oracle(o, q, torch.from_numpy(Kw).view(dtype),
                                 torch.from_numpy(Vw).view(dtype), torch.from_numpy(lens_np),
                                 scale, out.cpu(), TOL[dtype])
    torch.cuda.synchronize()
    assert np.array_equal(_bits(Kd.cpu()), Kw) and np.array_equal(_bits(Vd.cpu()), Vw)


# ----------------------------------------------------------------- combine variants
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["fp32", "bf16"])
@pytest.mark.parametrize("splits", [40, 100, 200, 300])
def test_combine_variants(o, dtype, splits):
    """Split counts that select each merge layout: 8-warp CTAs (up to 136 splits,
    one pass) and 16-warp CTAs (hundreds of splits, more than one pass at 300)."""
    n_max = 300 * 128
    lens = [n_max, n_max - 5000, 129]
    q, K, V, lens_t, scale = make_case(3, 8, 2, 128, n_max, lens, dtype, seed=splits)
    # the split length is a whole number of pipeline stages near n_max / splits;
    # the counts still land in the layout each case is meant for
    got = api.resolve_splits(3, 8, 2, 128, 128, n_max, dtype, splits)
    lo, hi = {40: (2, 68), 100: (69, 136), 200: (137, 10**6), 300: (137, 10**6)}[splits]
    assert lo <= got <= hi, got
    out = gpu_decode(q, K, V, lens_t, num_splits=splits)
    check_against_oracle(o, q, K, V, lens_t, scale, out, TOL[dtype])
