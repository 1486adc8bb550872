"""Pins for the CPU oracle: facts the pages and plain mathematics fix.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises ``AssertionError`` when
the oracle disagrees with something that does not come from the oracle
itself: values printed in "MoA-Structured Decode Attention" (section 2,
concrete example), closed forms, invariants of softmax attention, brute
force in pure Python, and PyTorch's float64 scaled_dot_product_attention.
They are plain functions so that ``test_oracle.py`` can run them against the
committed oracle and ``test_oracle_mutants.py`` against copies with a
planted mistake (each mistake must trip at least one pin).
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
EPS = np.finfo(np.float64).eps


def _rng(seed):
    return np.random.default_rng(seed)


def _normal(rng, *shape):
    return rng.standard_normal(shape).astype(np.float32)


def _worked():
    with open(os.path.join(GOLDEN, "moa_worked_example.json")) as f:
        return json.load(f)


def pin_worked_example_closed_form(o):
    """Section 2 example: out = ((2+6e)/(1+e), (4+8e)/(1+e)), e = exp(-1/sqrt 2)."""
    g = _worked()["inputs"]
    out, lse, a = o.decode_head(g["q"], g["K"], g["V"], g["scale"], want_weights=True)
    e = math.exp(-1.0 / math.sqrt(2.0))
    want = np.array([(2 + 6 * e) / (1 + e), (4 + 8 * e) / (1 + e)])
    assert np.max(np.abs(out - want)) <= 1e-12, (out, want)
    assert np.max(np.abs(a - np.array([1 / (1 + e), e / (1 + e)]))) <= 1e-12, a
    m = 1.0 / math.sqrt(2.0)          # the largest score, s[0]
    assert abs(math.exp(lse - m) - (1 + e)) <= 1e-12, lse   # Z = 1 + e


def pin_worked_example_printed(o):
    """Section 2 example against the rounded values the page prints."""
    g = _worked()
    inp, pr = g["inputs"], g["printed"]
    tol = pr["printed_digits_tolerance"]
    out, lse, a = o.decode_head(inp["q"], inp["K"], inp["V"], inp["scale"], want_weights=True)
    assert np.max(np.abs(out - np.array(pr["out"]))) <= tol, out
    assert np.max(np.abs(a - np.array(pr["a"]))) <= tol, a
    assert abs(math.exp(lse - pr["m"]) - pr["Z"]) <= tol, lse
    assert abs(a[1] / a[0] - pr["e"][1]) <= tol, a    # e[1]/e[0] = a[1]/a[0]


def pin_weights_sum_to_one(o):
    """Step II: the weights a[l] = e[l]/Z sum to 1 (to n rounding steps)."""
    rng = _rng(11)
    n, d = 1000, 64
    q, K, V = _normal(rng, d), _normal(rng, n, d), _normal(rng, n, d)
    _, _, a = o.decode_head(q, K, V, 1 / math.sqrt(d), want_weights=True)
    assert np.all(a > 0)
    assert abs(a.sum() - 1.0) <= n * EPS, a.sum()


def pin_gqa_equals_replicated_mha(o):
    """Introduction item 4: query head h reads KV head h // g; replicating each
    KV head g times and running plain MHA must give the same numbers."""
    rng = _rng(12)
    B, h_kv, g, n_max, d = 2, 3, 4, 37, 16
    h_q = h_kv * g
    q = _normal(rng, B, h_q, d)
    K = _normal(rng, B, h_kv, n_max, d)
    V = _normal(rng, B, h_kv, n_max, d)
    lens = np.array([37, 21], dtype=np.int32)
    out, lse = o.decode(q, K, V, lens, 0.25)
    Kr = np.ascontiguousarray(np.repeat(K, g, axis=1))
    Vr = np.ascontiguousarray(np.repeat(V, g, axis=1))
    out_r, lse_r = o.decode(q, Kr, Vr, lens, 0.25)
    assert np.array_equal(out, out_r)
    assert np.array_equal(lse, lse_r)


def pin_causal_last_row(o):
    """A decode over rows 0..t after appending row t equals row t of full causal
    attention (page "StoryLM-0 head-parallel attention", section 3)."""
    rng = _rng(13)
    T, d_k, d_v, n_max = 9, 8, 6, 12
    Q, Kf, Vf = _normal(rng, T, d_k), _normal(rng, T, d_k), _normal(rng, T, d_v)
    scale = 1 / math.sqrt(d_k)
    full = o.causal_attention(Q[None], Kf[None], Vf[None], scale)[0]
    K = np.full((1, 1, n_max, d_k), np.nan, dtype=np.float32)
    V = np.full((1, 1, n_max, d_v), np.nan, dtype=np.float32)
    for t in range(T):
        skipped = o.kv_append(np.ascontiguousarray(Kf[t][None, None]),
                              np.ascontiguousarray(Vf[t][None, None]), K, V, [t])
        assert skipped == 0
        out, _ = o.decode(Q[t][None, None], K, V, [t + 1], scale)
        assert np.max(np.abs(out[0, 0] - full[t])) <= 1e-12, (t, out[0, 0], full[t])


def pin_head_parallel_instance(o):
    """Page "StoryLM-0 head-parallel attention", sections 3-4 and 7: B=1, T=4,
    H=2, Dh=2.  Per-head shards concatenated on the head axis equal the
    unsharded two-head result, and changing the last token leaves earlier rows
    unchanged.  (The page's trained weights are not given; Q, K, V are seeded.)"""
    rng = _rng(14)
    H, T, Dh = 2, 4, 2
    Q, K, V = _normal(rng, H, T, Dh), _normal(rng, H, T, Dh), _normal(rng, H, T, Dh)
    scale = 1 / math.sqrt(Dh)
    whole = o.causal_attention(Q, K, V, scale)
    shards = [o.causal_attention(Q[h:h + 1], K[h:h + 1], V[h:h + 1], scale) for h in range(H)]
    assert np.array_equal(np.concatenate(shards, axis=0), whole)
    Q2, K2, V2 = Q.copy(), K.copy(), V.copy()
    Q2[:, T - 1] += 1.5
    K2[:, T - 1] -= 2.0
    V2[:, T - 1] *= -3.0
    changed = o.causal_attention(Q2, K2, V2, scale)
    assert np.array_equal(changed[:, :T - 1], whole[:, :T - 1])
    assert not np.allclose(changed[:, T - 1], whole[:, T - 1])
    # and a decode of the last row reproduces the last causal row per head
    for h in range(H):
        out, _ = o.decode_head(Q[h, T - 1], K[h], V[h], scale)
        assert np.max(np.abs(out - whole[h, T - 1])) <= 1e-12


def pin_single_row_returns_it(o):
    """n = 1: the only weight is exp(0)/exp(0) = 1, so out is V[0] exactly."""
    rng = _rng(15)
    q, K, V = _normal(rng, 32), _normal(rng, 1, 32), _normal(rng, 1, 24)
    out, lse, a = o.decode_head(q, K, V, 0.3, want_weights=True)
    assert np.array_equal(a, [1.0])
    assert np.array_equal(out, V[0].astype(np.float64))
    assert abs(lse - 0.3 * float(np.dot(q.astype(np.float64), K[0].astype(np.float64)))) <= 1e-12


def pin_equal_scores_average(o):
    """Equal scores (identical keys, or scale 0) weight every row 1/n: out = mean(V)."""
    rng = _rng(16)
    n, d = 50, 16
    q, V = _normal(rng, d), _normal(rng, n, d)
    K = np.repeat(_normal(rng, 1, d), n, axis=0)
    out, lse = o.decode_head(q, K, V, 0.7)
    mean = V.astype(np.float64).mean(axis=0)
    assert np.max(np.abs(out - mean)) <= 1e-12
    s0 = 0.7 * float(np.dot(q.astype(np.float64), K[0].astype(np.float64)))
    assert abs(lse - (s0 + math.log(n))) <= 1e-12
    out0, lse0 = o.decode_head(q, _normal(rng, n, d), V, 0.0)
    assert np.max(np.abs(out0 - mean)) <= 1e-12
    assert abs(lse0 - math.log(n)) <= 1e-12


def pin_dominant_row_selected(o):
    """One score far above the rest puts all the weight on that row."""
    rng = _rng(17)
    n, d = 40, 16
    q = _normal(rng, d)
    K = _normal(rng, n, d) * 0.01
    j = 23
    K[j] = q * (60.0 / float(np.dot(q, q)))      # s[j] = 60 * scale, others ~ 0
    V = _normal(rng, n, d)
    out, _ = o.decode_head(q, K, V, 1.0)
    assert np.max(np.abs(out - V[j])) <= 1e-12


def pin_row_permutation_invariant(o):
    """Softmax attention is a sum over rows: permuting (K, V) rows together
    leaves out unchanged (up to rounding), permuting only V does not."""
    rng = _rng(18)
    n, d = 64, 16
    q, K, V = _normal(rng, d), _normal(rng, n, d), _normal(rng, n, d)
    out, lse = o.decode_head(q, K, V, 0.25)
    p = rng.permutation(n)
    out_p, lse_p = o.decode_head(q, K[p], V[p], 0.25)
    assert np.max(np.abs(out - out_p)) <= 1e-12
    assert abs(lse - lse_p) <= 1e-12
    out_v, _ = o.decode_head(q, K, V[p], 0.25)
    assert np.max(np.abs(out - out_v)) > 1e-6


def pin_split_merge_equals_whole(o):
    """Splitting the rows into disjoint ranges, decoding each, and merging by
    log-sum-exp gives the whole decode (an empty range contributes nothing)."""
    rng = _rng(19)
    n, d_k, d_v = 300, 32, 24
    q, K, V = _normal(rng, d_k), _normal(rng, n, d_k), _normal(rng, n, d_v)
    out, lse = o.decode_head(q, K, V, 0.2)
    cuts = [0, 1, 77, 77, 200, 300]          # includes an empty range [77, 77)
    parts = [o.decode_head(q, K[a:b], V[a:b], 0.2) for a, b in zip(cuts[:-1], cuts[1:])]
    o_parts = np.stack([p[0] for p in parts])
    lse_parts = np.array([p[1] for p in parts])
    assert lse_parts[2] == -np.inf and np.all(o_parts[2] == 0)
    merged, lse_m = o.lse_combine(o_parts, lse_parts)
    assert np.max(np.abs(merged - out)) <= 1e-12
    assert abs(lse_m - lse) <= 1e-12
    empty, lse_e = o.lse_combine(np.zeros((3, d_v)), np.full(3, -np.inf))
    assert np.all(empty == 0) and lse_e == -np.inf


def pin_brute_force_tiny(o):
    """n <= 4 against sums written out in pure Python with math.exp."""
    rng = _rng(20)
    for n in range(1, 5):
        for trial in range(3):
            d_k, d_v = 3, 2
            q, K, V = _normal(rng, d_k), _normal(rng, n, d_k), _normal(rng, n, d_v)
            scale = 0.5 + trial
            s = [scale * sum(float(q[j]) * float(K[l][j]) for j in range(d_k)) for l in range(n)]
            e = [math.exp(x) for x in s]               # no max shift: tiny scores
            Z = math.fsum(e)
            want = [math.fsum(e[l] / Z * float(V[l][c]) for l in range(n)) for c in range(d_v)]
            out, lse = o.decode_head(q, K, V, scale)
            assert np.max(np.abs(out - np.array(want))) <= 1e-12, (n, out, want)
            assert abs(lse - math.log(Z)) <= 1e-12


def pin_matches_torch_sdpa_float64(o):
    """PyTorch's float64 scaled_dot_product_attention on CPU, one call per
    sequence with (B, H, S, D) = (1, h_q, n_b, d) and GQA heads repeated, as the
    page's verification against SDPA does with dummy dimensions."""
    import torch
    rng = _rng(21)
    B, h_kv, g, n_max, d_k, d_v = 3, 2, 3, 45, 16, 8
    h_q = h_kv * g
    q = _normal(rng, B, h_q, d_k)
    K = _normal(rng, B, h_kv, n_max, d_k)
    V = _normal(rng, B, h_kv, n_max, d_v)
    lens = np.array([45, 1, 30], dtype=np.int32)
    scale = 0.3
    out, _ = o.decode(q, K, V, lens, scale)
    for b in range(B):
        n = int(lens[b])
        qt = torch.from_numpy(q[b]).double()[None, :, None, :]               # [1,h_q,1,d_k]
        kt = torch.from_numpy(K[b, :, :n]).double().repeat_interleave(g, 0)[None]
        vt = torch.from_numpy(V[b, :, :n]).double().repeat_interleave(g, 0)[None]
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)
        ref = ref[0, :, 0, :].numpy()
        assert np.max(np.abs(out[b] - ref)) <= 1e-12, b


def pin_empty_sequence(o):
    """n_b = 0 (a reading the pages leave open): out = 0 and lse = -inf."""
    rng = _rng(22)
    q = _normal(rng, 2, 4, 8)
    K = np.full((2, 2, 5, 8), np.nan, dtype=np.float32)
    V = np.full((2, 2, 5, 8), np.nan, dtype=np.float32)
    K[1, :, :3] = _normal(rng, 2, 3, 8)
    V[1, :, :3] = _normal(rng, 2, 3, 8)
    out, lse = o.decode(q, K, V, [0, 3], 0.35)
    assert np.all(out[0] == 0) and np.all(lse[0] == -np.inf)
    assert np.all(np.isfinite(out[1]))


def pin_kv_append_rows(o):
    """KV accumulation writes row pos[b] of every (b, h) at its gamma offset and
    nothing else, byte for byte; numpy fancy indexing is the independent check.
    Out-of-range positions are skipped and counted."""
    rng = _rng(23)
    B, h_kv, n_max, d_k, d_v = 3, 2, 6, 8, 4
    for dtype in (np.float32, np.uint16):
        if dtype == np.float32:
            K = _normal(rng, B, h_kv, n_max, d_k)
            V = _normal(rng, B, h_kv, n_max, d_v)
            kn, vn = _normal(rng, B, h_kv, d_k), _normal(rng, B, h_kv, d_v)
        else:   # bf16 bit patterns
            K = rng.integers(0, 65535, (B, h_kv, n_max, d_k), dtype=np.uint16)
            V = rng.integers(0, 65535, (B, h_kv, n_max, d_v), dtype=np.uint16)
            kn = rng.integers(0, 65535, (B, h_kv, d_k), dtype=np.uint16)
            vn = rng.integers(0, 65535, (B, h_kv, d_v), dtype=np.uint16)
        pos = np.array([0, n_max - 1, 3], dtype=np.int32)
        K0, V0 = K.copy(), V.copy()
        assert o.kv_append(kn, vn, K, V, pos) == 0
        Kw, Vw = K0.copy(), V0.copy()
        for b in range(B):
            Kw[b, :, pos[b]] = kn[b]
            Vw[b, :, pos[b]] = vn[b]
        assert np.array_equal(K.view(np.uint8), Kw.view(np.uint8))
        assert np.array_equal(V.view(np.uint8), Vw.view(np.uint8))
        K1, V1 = K.copy(), V.copy()
        assert o.kv_append(kn, vn, K, V, [-1, n_max, 2]) == 2
        K1[2, :, 2] = kn[2]
        V1[2, :, 2] = vn[2]
        assert np.array_equal(K.view(np.uint8), K1.view(np.uint8))
        assert np.array_equal(V.view(np.uint8), V1.view(np.uint8))


# ----------------------------------------------------------------- 8-bit caches
# The fp8 e4m3 format is fixed by its definition (1 sign, 4 exponent bits with
# bias 7, 3 mantissa bits, subnormals below 2^-6, S.1111.111 the only NaN, no
# infinities); int8 by two's complement.  These pins use values that follow
# from those definitions and PyTorch's own float8_e4m3fn implementation.

def pin_e4m3_code_values(o):
    """Values the e4m3 definition fixes, and all 256 codes against PyTorch's float8_e4m3fn."""
    fixed = {0x00: 0.0, 0x38: 1.0, 0x3C: 1.5, 0x40: 2.0, 0x7E: 448.0, 0x08: 2.0 ** -6,
             0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0xB8: -1.0, 0xFE: -448.0, 0x30: 0.5}
    for c, v in fixed.items():
        assert o.code_value(c, 2) == v, (hex(c), o.code_value(c, 2), v)
    assert math.isnan(o.code_value(0x7F, 2)) and math.isnan(o.code_value(0xFF, 2))
    assert math.copysign(1.0, o.code_value(0x80, 2)) == -1.0
    try:
        import torch
    except ImportError:  # pragma: no cover - torch is part of the test image
        return
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    got = np.array([o.code_value(c, 2) for c in range(256)])
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all(), [hex(c) for c in np.nonzero(~same)[0]]


def pin_int8_code_values(o):
    """Two's complement: 0x7F = 127, 0x80 = -128, 0xFF = -1."""
    for c in range(256):
        want = c - 256 if c >= 128 else c
        assert o.code_value(c, 1) == want, (c, o.code_value(c, 1))


def pin_quantize_absmax_maps_to_limit(o):
    """The largest |x| of a row becomes the code for +-Q, and its scale is absmax / Q."""
    rng = _rng(40)
    x = _normal(rng, 16, 64)
    for kind, Q, top in ((1, 127, 0x7F), (2, 448, 0x7E)):
        codes, scales = o.quantize(x, kind)
        for r in range(x.shape[0]):
            j = int(np.argmax(np.abs(x[r])))
            assert scales[r] == np.float32(np.abs(x[r]).max()) / np.float32(Q)
            want = top if x[r, j] > 0 else (0x81 if kind == 1 else 0xFE)
            assert codes[r, j] == want, (kind, r, hex(codes[r, j]))


def pin_quantize_round_trip_error(o):
    """|s * value(c) - x| is at most half a code step times s (plus the division's rounding)."""
    rng = _rng(41)
    x = _normal(rng, 32, 128) * np.float32(3.0)
    for kind in (1, 2):
        codes, scales = o.quantize(x, kind)
        back = o.dequant(codes, scales, kind)
        for r in range(x.shape[0]):
            s = float(scales[r])
            v = np.abs(x[r].astype(np.float64)) / s
            if kind == 1:
                step = np.ones_like(v)
            else:  # e4m3 spacing: 2^-9 below 2^-6, else 2^(floor(log2 v) - 3)
                e = np.floor(np.log2(np.maximum(v, 2.0 ** -6)))
                step = 2.0 ** (e - 3)
            bound = s * (0.5 * step + 1e-6 * v + 1e-12)
            err = np.abs(back[r] - x[r].astype(np.float64))
            assert np.all(err <= bound), (kind, r, float(np.max(err - bound)))


def pin_quantize_ties_to_even(o):
    """x / s exactly halfway between two codes goes to the even one."""
    # int8: absmax 127 makes s = 1 exactly, so x / s = x
    x = np.array([[127.0, 2.5, 3.5, -2.5, -3.5, 0.5, -0.5, 1.5] + [0.0] * 8], dtype=np.float32)
    codes, scales = o.quantize(x, 1)
    assert scales[0] == 1.0
    assert list(codes[0, :8].view(np.int8)) == [127, 2, 4, -2, -4, 0, 0, 2]
    # e4m3: absmax 448 makes s = 1.  In [8, 16) the step is 1: 8.5 lies halfway between
    # 8 (M=0) and 9 (M=1) -> 8, 9.5 between 9 (M=1) and 10 (M=2) -> 10; in [16, 32) the
    # step is 2: 17 -> 16; 2^-10 is half the first subnormal -> 0; 3 * 2^-10 lies between
    # 2^-9 (M=1) and 2^-8 (M=2) -> 2^-8; 440 lies between 416 and 448, nearer 448.
    x = np.array([[448.0, 8.5, 9.5, -8.5, 2.0 ** -10, 3 * 2.0 ** -10, 17.0, 440.0] + [0.0] * 8],
                 dtype=np.float32)
    codes, scales = o.quantize(x, 2)
    assert scales[0] == 1.0
    vals = [o.code_value(c, 2) for c in codes[0, :8]]
    assert vals == [448.0, 8.0, 10.0, -8.0, 0.0, 2.0 ** -8, 16.0, 448.0], vals


def pin_quantize_zero_row(o):
    """An all-zero row has scale 0 and all-zero codes."""
    x = np.zeros((2, 32), dtype=np.float32)
    for kind in (1, 2):
        codes, scales = o.quantize(x, kind)
        assert np.all(codes == 0) and np.all(scales == 0)


def pin_quantize_matches_torch_e4m3_cast(o):
    """The e4m3 codes equal PyTorch's round-to-nearest-even cast of x / s (|x / s| <= 448)."""
    try:
        import torch
    except ImportError:  # pragma: no cover
        return
    rng = _rng(42)
    x = _normal(rng, 64, 128)
    codes, scales = o.quantize(x, 2)
    v = np.clip(x / scales[:, None], -448.0, 448.0).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ref, codes), int((ref != codes).sum())


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
