"""Pins for the fp64 oracle, against things other than the oracle itself.

Each test ties the oracle to something the pages or the mathematics fix:
hand-derived closed forms (tests/golden/), high-precision brute force on tiny
inputs, invariants of softmax attention, and the hand-written All-to-All table.
The last test plants plausible mistakes in a private copy of the oracle source
and checks that at least one pin catches each of them.
"""
import ctypes
import json
import math
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
import xsgen

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16(a):
    a = np.asarray(a, dtype=np.float32)
    bits = xsgen.f32_to_bf16_bits(a)
    assert np.array_equal(xsgen.bf16_bits_to_f32(bits), a), "fixture value not exact in bf16"
    return bits


def _scale(s):
    return {"ln3": math.log(3.0), "ln2": math.log(2.0)}[s] if isinstance(s, str) else float(s)


def _brute(q, k, v, B, S, H, D, P, scale, dps=40, causal=False):
    """exp(s_j) / sum_k exp(s_k) without max subtraction, in 40-digit arithmetic;
    with causal, query i sums over keys j <= i only."""
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = dps
    qf, kf, vf = (xsgen.bf16_bits_to_f32(x).astype(np.float64) for x in (q, k, v))
    Hl = H // P
    out = np.zeros((P, B, S, Hl, D))
    sc = mp.mpf(scale)
    for r in range(P):
        for b in range(B):
            for hl in range(Hl):
                for i in range(S):
                    keys = range(i + 1) if causal else range(S)
                    w = [mp.exp(sc * mp.fsum(mp.mpf(qf[r, b, i, hl, d]) * mp.mpf(kf[r, b, j, hl, d])
                                            for d in range(D))) for j in keys]
                    tot = mp.fsum(w)
                    for d in range(D):
                        out[r, b, i, hl, d] = float(mp.fsum(w[n] * mp.mpf(vf[r, b, j, hl, d])
                                                            for n, j in enumerate(keys)) / tot)
    return out


# ------------------------------------------------------------------ golden pins

def test_golden_closed_form_cases():
    g = json.load(open(os.path.join(GOLDEN, "attn_closed_form.json")))
    for c in g["cases"]:
        q, k, v = _bf16(c["q"]), _bf16(c["k"]), _bf16(c["v"])
        o = oracle.attention(q, k, v, c["B"], c["S"], c["H"], c["D"], c["P"], _scale(c["scale"]))
        np.testing.assert_allclose(o, np.array(c["o"]), rtol=0, atol=1e-12, err_msg=c["name"])


def test_golden_fused_case():
    c = json.load(open(os.path.join(GOLDEN, "attn_closed_form.json")))["fused"]
    q, k, v = _bf16(c["q"]), _bf16(c["k"]), _bf16(c["v"])
    out = oracle.attention_a2a(q, k, v, c["B"], c["S"], c["H"], c["D"], c["P"], _scale(c["scale"]))
    np.testing.assert_allclose(out, np.array(c["out"]), rtol=0, atol=1e-12)


def test_golden_a2a_table():
    g = json.load(open(os.path.join(GOLDEN, "a2a_map_tiny.json")))
    B, S, H, D, P = g["B"], g["S"], g["H"], g["D"], g["P"]
    Hl = H // P
    x = np.zeros((P, B, S, Hl, D), dtype=np.int32)
    for r in range(P):
        for b in range(B):
            for s in range(S):
                for hl in range(Hl):
                    x[r, b, s, hl, 0] = 1000 * r + 100 * b + 10 * s + hl
    y = oracle.a2a(x, B, S, H, D, P)
    assert np.array_equal(y, np.array(g["out"], dtype=np.int32))
    assert np.array_equal(oracle.a2a_inverse(y, B, S, H, D, P), x)


# ------------------------------------------------------------ brute force pins

TINY = [  # (B, S, H, D, P, scale, sigma)
    (1, 1, 1, 1, 1, 0.5, 1.0),
    (1, 4, 2, 3, 1, 0.7, 1.0),
    (2, 4, 2, 2, 2, 1.0, 1.0),
    (1, 8, 4, 4, 4, 0.5, 1.0),
    (2, 6, 4, 4, 2, 0.35, 1.5),
    (1, 8, 4, 4, 2, 0.125, 2.0),
]


@pytest.mark.parametrize("case", TINY)
def test_brute_force_tiny(case):
    B, S, H, D, P, scale, sigma = case
    q, k, v = xsgen.random_inputs(77 + S * 10 + D, P, B, S, H, D, sigma, 1.0)
    o = oracle.attention(q, k, v, B, S, H, D, P, scale)
    ref = _brute(q, k, v, B, S, H, D, P, scale)
    np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)


def test_brute_force_large_logits():
    """Logits of several hundred: the max subtraction keeps exp finite."""
    B, S, H, D, P = 1, 6, 2, 4, 2
    q, k, v = xsgen.random_inputs(5, P, B, S, H, D, 3.0, 1.0)
    scale = 40.0
    o = oracle.attention(q, k, v, B, S, H, D, P, scale)
    assert np.isfinite(o).all()
    np.testing.assert_allclose(o, _brute(q, k, v, B, S, H, D, P, scale, dps=60), rtol=0, atol=1e-12)


# ------------------------------------------------------------------ causal pins
# The causal reading: query token i sees keys 0..i of its own sequence.

@pytest.mark.parametrize("case", TINY)
def test_causal_brute_force_tiny(case):
    B, S, H, D, P, scale, sigma = case
    q, k, v = xsgen.random_inputs(91 + S * 10 + D, P, B, S, H, D, sigma, 1.0)
    o = oracle.attention(q, k, v, B, S, H, D, P, scale, causal=True)
    np.testing.assert_allclose(o, _brute(q, k, v, B, S, H, D, P, scale, causal=True), rtol=0, atol=1e-12)


def test_causal_first_row_is_its_own_value():
    """Token 0 sees only key 0: its output is v_0 exactly, for every head."""
    B, S, H, D, P = 2, 10, 4, 8, 2
    q, k, v = xsgen.random_inputs(12, P, B, S, H, D, 2.0, 1.0)
    o = oracle.attention(q, k, v, B, S, H, D, P, 0.3, causal=True)
    assert np.array_equal(o[:, :, 0], xsgen.bf16_bits_to_f32(v[:, :, 0]).astype(np.float64))


def test_causal_last_row_sees_everything():
    B, S, H, D, P = 1, 12, 4, 8, 2
    q, k, v = xsgen.random_inputs(13, P, B, S, H, D)
    c = oracle.attention(q, k, v, B, S, H, D, P, 0.3, causal=True)
    f = oracle.attention(q, k, v, B, S, H, D, P, 0.3)
    assert np.array_equal(c[:, :, S - 1], f[:, :, S - 1])
    assert not np.allclose(c[:, :, : S - 1], f[:, :, : S - 1])


def test_causal_row_is_full_attention_over_its_prefix():
    """Row i of causal attention equals row i of full attention over tokens 0..i."""
    B, S, H, D, P = 1, 10, 2, 4, 1
    q, k, v = xsgen.random_inputs(14, P, B, S, H, D)
    c = oracle.attention(q, k, v, B, S, H, D, P, 0.5, causal=True)
    for i in (0, 3, 9):
        pre = [np.ascontiguousarray(x[:, :, : i + 1]) for x in (q, k, v)]
        f = oracle.attention(*pre, B, i + 1, H, D, P, 0.5)
        np.testing.assert_allclose(c[:, :, i], f[:, :, i], rtol=0, atol=1e-15)


def test_causal_rows_and_a2a_apis_agree():
    B, S, H, D, P = 2, 8, 4, 4, 2
    q, k, v = xsgen.random_inputs(15, P, B, S, H, D)
    full = oracle.attention(q, k, v, B, S, H, D, P, 0.4, causal=True)
    rows = np.array([0, 5, 17, P * B * S * (H // P) - 1])
    np.testing.assert_array_equal(oracle.attention_rows(q, k, v, B, S, H, D, P, 0.4, rows, causal=True),
                                  full.reshape(-1, D)[rows])
    np.testing.assert_array_equal(oracle.attention_a2a(q, k, v, B, S, H, D, P, 0.4, causal=True),
                                  oracle.a2a(full, B, S, H, D, P))


# ------------------------------------------------------------------ FP8 inputs

def test_e4m3_decode_standard_values():
    g = json.load(open(os.path.join(GOLDEN, "e4m3_values.json")))["values"]
    codes = np.array([int(c, 16) for c in g], dtype=np.uint8)
    got = oracle.e4m3_decode(codes)
    for c, want, v in zip(g, g.values(), got):
        if want == "nan":
            assert math.isnan(v), c
        else:
            assert v == want and math.copysign(1.0, v) == math.copysign(1.0, want), c


def test_e4m3_codes_are_ordered_and_symmetric():
    pos = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    assert (np.diff(pos) > 0).all()
    neg = oracle.e4m3_decode(np.arange(0x80, 0xFF, dtype=np.uint8))
    np.testing.assert_array_equal(neg, -pos)


def test_attention_q8_equals_bf16_on_widened_inputs():
    """Every E4M3 value is exact in bf16, so attention on E4M3 q and k must equal
    the (separately pinned) bf16 attention on their widened values, bit for bit."""
    B, S, H, D, P = 2, 12, 4, 8, 2
    q8 = xsgen.normal_e4m3(21, 1, (P, B, S, H // P, D), 2.0)
    k8 = xsgen.normal_e4m3(21, 2, (P, B, S, H // P, D), 2.0)
    _, _, v = xsgen.random_inputs(21, P, B, S, H, D)
    widen = lambda c: xsgen.f32_to_bf16_bits(oracle.e4m3_decode(c).astype(np.float32))
    for causal in (False, True):
        a = oracle.attention_q8(q8, k8, v, B, S, H, D, P, 0.3, causal=causal)
        b = oracle.attention(widen(q8), widen(k8), v, B, S, H, D, P, 0.3, causal=causal)
        np.testing.assert_array_equal(a, b)
    rows = np.array([0, 7, 30, P * B * S * (H // P) - 1])
    np.testing.assert_array_equal(oracle.attention_rows_q8(q8, k8, v, B, S, H, D, P, 0.3, rows),
                                  oracle.attention(widen(q8), widen(k8), v, B, S, H, D, P, 0.3).reshape(-1, D)[rows])


def test_attention_e4m3_values_equal_bf16_on_widened_inputs():
    """E4M3 v as well: still exactly the bf16 attention on the widened q, k, v."""
    B, S, H, D, P = 2, 12, 4, 8, 2
    shape = (P, B, S, H // P, D)
    q8, k8, v8 = (xsgen.normal_e4m3(31, i, shape, s) for i, s in ((1, 2.0), (2, 2.0), (3, 24.0)))
    widen = lambda c: xsgen.f32_to_bf16_bits(oracle.e4m3_decode(c).astype(np.float32))
    assert (oracle.e4m3_decode(v8) < 0).any() and (np.abs(oracle.e4m3_decode(v8)) >= 64).any()
    for causal in (False, True):
        a = oracle.attention_q8(q8, k8, v8, B, S, H, D, P, 0.3, causal=causal)
        b = oracle.attention(widen(q8), widen(k8), widen(v8), B, S, H, D, P, 0.3, causal=causal)
        np.testing.assert_array_equal(a, b)
    rows = np.array([0, 5, 41, P * B * S * (H // P) - 1])
    np.testing.assert_array_equal(oracle.attention_rows_q8(q8, k8, v8, B, S, H, D, P, 0.3, rows, causal=True),
                                  oracle.attention(widen(q8), widen(k8), widen(v8), B, S, H, D, P, 0.3,
                                                   causal=True).reshape(-1, D)[rows])


def test_attention_e4m3_values_special_cases():
    """Hand-checkable E4M3 cases: equal keys give the plain mean of the decoded
    values; one dominant key returns its value row (the largest code, 448, and
    the smallest subnormal, 2^-9, among them)."""
    B, S, H, D, P = 1, 4, 1, 2, 1
    q8 = np.zeros((P, B, S, H, D), dtype=np.uint8)           # q = 0: uniform weights
    k8 = np.full_like(q8, 0x38)                              # 1.0
    v8 = np.array([0x7E, 0x01, 0xC0, 0x30], dtype=np.uint8)  # 448, 2^-9, -2.0, 0.5
    v8 = np.stack([v8, v8[::-1]], axis=-1).reshape(P, B, S, H, D)
    o = oracle.attention_q8(q8, k8, v8, B, S, H, D, P, 1.0)
    want = (448.0 + 2.0 ** -9 - 2.0 + 0.5) / 4.0
    np.testing.assert_allclose(o.reshape(S, D), np.full((S, D), want), rtol=0, atol=1e-13)
    q8 = np.full_like(q8, 0x38)                              # q = 1
    k8 = np.array([0x00, 0x00, 0x78, 0x00], dtype=np.uint8)  # key 2 = 256, the others 0
    k8 = np.repeat(k8, D).reshape(P, B, S, H, D)
    o = oracle.attention_q8(q8, k8, v8, B, S, H, D, P, 1.0)  # logits 512 vs 0: weight 1 - O(e^-512)
    np.testing.assert_array_equal(o.reshape(S, D), np.tile([-2.0, 2.0 ** -9], (S, 1)))


# ------------------------------------------------------------------ invariants

def test_rows_are_probabilities():
    """With V = identity (D = S) the output rows are the softmax rows: >= 0, sum 1."""
    B, S, H, P = 2, 8, 2, 2
    D = S
    q, k, _ = xsgen.random_inputs(11, P, B, S, H, D)
    v = np.zeros((P, B, S, H // P, D), dtype=np.float32)
    for j in range(S):
        v[:, :, j, :, j] = 1.0
    o = oracle.attention(q, k, _bf16(v), B, S, H, D, P, 0.4)
    assert (o >= 0).all()
    np.testing.assert_allclose(o.sum(-1), 1.0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(o, _brute(q, k, _bf16(v), B, S, H, D, P, 0.4), rtol=0, atol=1e-12)


def test_zero_q_gives_mean_v():
    B, S, H, D, P = 2, 64, 4, 16, 2
    _, k, v = xsgen.random_inputs(12, P, B, S, H, D)
    q = np.zeros_like(k)
    o = oracle.attention(q, k, v, B, S, H, D, P, 0.25)
    mean_v = xsgen.bf16_bits_to_f32(v).astype(np.float64).mean(axis=2, keepdims=True)
    np.testing.assert_allclose(o, np.broadcast_to(mean_v, o.shape), rtol=0, atol=1e-12)


def test_constant_v():
    B, S, H, D, P = 1, 32, 4, 8, 4
    q, k, _ = xsgen.random_inputs(13, P, B, S, H, D)
    c = np.linspace(-3, 3, D, dtype=np.float32)
    c = xsgen.bf16_bits_to_f32(xsgen.f32_to_bf16_bits(c))
    v = _bf16(np.broadcast_to(c, (P, B, S, H // P, D)).copy())
    o = oracle.attention(q, k, v, B, S, H, D, P, 0.3)
    np.testing.assert_allclose(o, np.broadcast_to(c.astype(np.float64), o.shape), rtol=0, atol=1e-12)


def test_single_token_returns_v():
    B, S, H, D, P = 2, 1, 3, 8, 1
    q, k, v = xsgen.random_inputs(14, P, B, S, H, D)
    o = oracle.attention(q, k, v, B, S, H, D, P, 0.3)
    np.testing.assert_array_equal(o, xsgen.bf16_bits_to_f32(v).astype(np.float64))


def test_scale_moves_between_q_and_scale():
    """q -> 2q with scale -> scale/2 leaves every logit, hence the output, unchanged."""
    B, S, H, D, P = 1, 48, 2, 8, 2
    q, k, v = xsgen.random_inputs(15, P, B, S, H, D)
    q2 = _bf16(2.0 * xsgen.bf16_bits_to_f32(q))
    o1 = oracle.attention(q, k, v, B, S, H, D, P, 0.5)
    o2 = oracle.attention(q2, k, v, B, S, H, D, P, 0.25)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)


def test_logit_shift_invariance():
    """A key component shared by all keys adds the same constant to every logit of a row."""
    B, S, H, D, P = 1, 32, 2, 4, 1
    q, k, v = xsgen.random_inputs(16, P, B, S, H, D)
    qf, kf = xsgen.bf16_bits_to_f32(q).copy(), xsgen.bf16_bits_to_f32(k).copy()
    qf[..., -1] = 1.0
    kf[..., -1] = 0.0
    o1 = oracle.attention(_bf16(qf), _bf16(kf), v, B, S, H, D, P, 0.5)
    kf[..., -1] = 5.0
    o2 = oracle.attention(_bf16(qf), _bf16(kf), v, B, S, H, D, P, 0.5)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)


def test_heads_stay_in_their_slots():
    """Head h has V == h+1 everywhere, so after the All-to-All slot h holds h+1."""
    B, S, H, D, P = 2, 16, 8, 4, 4
    q, k, _ = xsgen.random_inputs(17, P, B, S, H, D)
    Hl = H // P
    v = np.zeros((P, B, S, Hl, D), dtype=np.float32)
    for r in range(P):
        for hl in range(Hl):
            v[r, :, :, hl, :] = r * Hl + hl + 1
    out = oracle.attention_a2a(q, k, _bf16(v), B, S, H, D, P, 0.5)
    want = np.arange(1, H + 1, dtype=np.float64)[None, None, None, :, None]
    np.testing.assert_allclose(out, np.broadcast_to(want, out.shape), rtol=0, atol=1e-12)


def test_rows_api_matches_full():
    B, S, H, D, P = 2, 40, 4, 8, 2
    q, k, v = xsgen.random_inputs(18, P, B, S, H, D)
    full = oracle.attention(q, k, v, B, S, H, D, P, 0.3).reshape(-1, D)
    rows = np.random.default_rng(0).choice(full.shape[0], 37, replace=False)
    np.testing.assert_array_equal(oracle.attention_rows(q, k, v, B, S, H, D, P, 0.3, rows), full[rows])


def test_thread_count_does_not_change_result():
    B, S, H, D, P = 1, 64, 4, 16, 2
    q, k, v = xsgen.random_inputs(19, P, B, S, H, D)
    a = oracle.attention(q, k, v, B, S, H, D, P, 0.3, nthreads=1)
    b = oracle.attention(q, k, v, B, S, H, D, P, 0.3, nthreads=7)
    np.testing.assert_array_equal(a, b)


# --------------------------------------------------------------- All-to-All map

@pytest.mark.parametrize("shape", [(1, 8, 2, 3, 1), (2, 8, 4, 2, 2), (1, 12, 6, 1, 3), (3, 16, 8, 2, 4),
                                   (1, 32, 8, 4, 8)])
def test_a2a_is_bijection_with_inverse(shape):
    B, S, H, D, P = shape
    n = B * S * H * D
    x = np.arange(n, dtype=np.int64).reshape(P, B, S, H // P, D)
    y = oracle.a2a(x, B, S, H, D, P)
    assert np.array_equal(np.sort(y.ravel()), np.arange(n))           # every slot hit once
    assert np.array_equal(oracle.a2a_inverse(y, B, S, H, D, P), x)      # inverse restores


def test_a2a_single_rank_is_identity():
    B, S, H, D = 2, 8, 3, 4
    x = np.arange(B * S * H * D, dtype=np.int32).reshape(1, B, S, H, D)
    assert np.array_equal(oracle.a2a(x, B, S, H, D, 1), x)


def test_a2a_rows_move_whole():
    """A row of D elements stays contiguous and in order (only rows move)."""
    B, S, H, D, P = 2, 8, 4, 5, 2
    x = np.arange(B * S * H * D, dtype=np.int64).reshape(P, B, S, H // P, D)
    y = oracle.a2a(x, B, S, H, D, P).reshape(-1, D)
    assert np.array_equal(y - y[:, :1], np.broadcast_to(np.arange(D), y.shape))
    assert (y[:, 0] % D == 0).all()


def test_oracle_rejects_bad_shapes():
    q = np.zeros(8, dtype=np.uint16)
    with pytest.raises(ValueError):
        oracle.attention(q, q, q, 1, 3, 2, 1, 2, 1.0)    # S % P != 0
    with pytest.raises(ValueError):
        oracle.a2a(q, 1, 4, 3, 1, 2)                     # H % P != 0


# ---------------------------------------------------------------- mutation check

_MUTANTS = {
    "no max subtraction": ("p[t] = exp(p[t] - m);", "p[t] = exp(p[t]);"),
    "no normalisation": ("o[d] /= l;", "o[d] /= 1.0;"),
    "wrong exp sign": ("p[t] = exp(p[t] - m);", "p[t] = exp(m - p[t]);"),
    "scale dropped": ("p[t] = j->scale * acc;", "p[t] = acc;"),
    "query row used as key": ("j->k + head_base + t * row_stride", "j->k + head_base + s_i * row_stride"),
    "value row index": ("j->v + head_base + t * row_stride", "j->v + head_base + (S - 1 - t) * row_stride"),
    "q/k transposed head": ("(rb * S * Hl + hl) * D", "(rb * S * Hl + (Hl - 1 - hl)) * D"),
    "token slot": ("int64_t sl = s - rd * Sl;", "int64_t sl = s % P;"),
    "head order": ("int64_t h = r * Hl + hl;", "int64_t h = hl * P + r;"),
    "rank of token": ("int64_t rd = s / Sl;", "int64_t rd = s % P;"),
    "causal drops the diagonal": ("j->causal ? s_i + 1 : S", "j->causal ? s_i : S"),
    "causal looks ahead": ("const int64_t t0 = 0, t1 = j->causal ? s_i + 1 : S;",
                           "const int64_t t0 = j->causal ? s_i : 0, t1 = S;"),
    "causal mask ignored": ("j->causal ? s_i + 1 : S", "S"),
    "e4m3 exponent bias": ("v = ldexp(1.0 + (double)m / 8.0, e - 7);", "v = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    "e4m3 subnormal scale": ("v = ldexp((double)m / 8.0, -6);", "v = ldexp((double)m / 8.0, -7);"),
    "e4m3 mantissa width": ("v = ldexp(1.0 + (double)m / 8.0, e - 7);", "v = ldexp(1.0 + (double)m / 16.0, e - 7);"),
    "e4m3 value row index": ("const uint8_t *vt = j->v8 + head_base + t * row_stride;",
                             "const uint8_t *vt = j->v8 + head_base + (S - 1 - t) * row_stride;"),
    "e4m3 value weight": ("o[d] += p[t] * e4m3_to_double(vt[d]);", "o[d] += e4m3_to_double(vt[d]);"),
    "e4m3 value read as key": ("o[d] += p[t] * e4m3_to_double(vt[d]);",
                               "o[d] += p[t] * e4m3_to_double(j->k8[head_base + t * row_stride + d]);"),
}


def _pins_pass(lib):
    """The pins above, re-run against an arbitrary compiled copy of the oracle."""
    vp, i64, dbl = ctypes.c_void_p, ctypes.c_int64, ctypes.c_double
    lib.xs_oracle_attention.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, dbl, ctypes.c_int]
    lib.xs_oracle_a2a.argtypes = [vp, vp, i64, i64, i64, i64, i64, i64]
    lib.xs_oracle_attention_ex.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, dbl, ctypes.c_int,
                                           ctypes.c_int]

    def attn(q, k, v, B, S, H, D, P, sc):
        o = np.empty((P, B, S, H // P, D))
        lib.xs_oracle_attention(q.ctypes.data, k.ctypes.data, v.ctypes.data, o.ctypes.data,
                                B, S, H, D, P, sc, 2)
        return o

    def attn_causal(q, k, v, B, S, H, D, P, sc):
        o = np.empty((P, B, S, H // P, D))
        lib.xs_oracle_attention_ex(q.ctypes.data, k.ctypes.data, v.ctypes.data, o.ctypes.data,
                                   B, S, H, D, P, sc, 1, 2)
        return o

    lib.xs_oracle_e4m3_decode.argtypes = [vp, vp, i64]
    g8 = json.load(open(os.path.join(GOLDEN, "e4m3_values.json")))["values"]
    codes = np.array([int(c, 16) for c in g8], dtype=np.uint8)
    dec = np.empty(codes.size)
    lib.xs_oracle_e4m3_decode(codes.ctypes.data, dec.ctypes.data, codes.size)
    want = np.array([np.nan if x == "nan" else x for x in g8.values()])
    ok = bool(np.array_equal(np.isnan(dec), np.isnan(want)) and np.array_equal(dec[~np.isnan(want)], want[~np.isnan(want)]))
    # E4M3 q, k, v against the bf16 path on the widened values (exact)
    lib.xs_oracle_attention_q8.argtypes = [vp, vp, vp, ctypes.c_int, vp, i64, i64, i64, i64, i64, dbl,
                                           ctypes.c_int, ctypes.c_int]
    B, S, H, D, P = 2, 12, 4, 8, 2
    sh = (P, B, S, H // P, D)
    q8, k8, v8 = (xsgen.normal_e4m3(31, i, sh, s) for i, s in ((1, 2.0), (2, 2.0), (3, 24.0)))
    wid = lambda c: xsgen.f32_to_bf16_bits(_decode_ref(c).astype(np.float32))
    o8 = np.empty(sh)
    lib.xs_oracle_attention_q8(q8.ctypes.data, k8.ctypes.data, v8.ctypes.data, 1, o8.ctypes.data,
                               B, S, H, D, P, 0.3, 0, 2)
    ok &= bool(np.array_equal(o8, attn(wid(q8), wid(k8), wid(v8), B, S, H, D, P, 0.3)))
    B, S, H, D, P, scale, sigma = TINY[3]
    q, k, v = xsgen.random_inputs(91 + S * 10 + D, P, B, S, H, D, sigma, 1.0)
    ok &= bool(np.allclose(attn_causal(q, k, v, B, S, H, D, P, scale),
                           _brute(q, k, v, B, S, H, D, P, scale, causal=True), rtol=0, atol=1e-12))
    g = json.load(open(os.path.join(GOLDEN, "attn_closed_form.json")))
    for c in g["cases"]:
        o = attn(_bf16(c["q"]), _bf16(c["k"]), _bf16(c["v"]), c["B"], c["S"], c["H"], c["D"], c["P"],
                 _scale(c["scale"]))
        ok &= bool(np.allclose(o, np.array(c["o"]), rtol=0, atol=1e-12))
    for case in TINY[2:5]:
        B, S, H, D, P, scale, sigma = case
        q, k, v = xsgen.random_inputs(77 + S * 10 + D, P, B, S, H, D, sigma, 1.0)
        ok &= bool(np.allclose(attn(q, k, v, B, S, H, D, P, scale), _brute(q, k, v, B, S, H, D, P, scale),
                               rtol=0, atol=1e-12))
    B, S, H, D, P = 1, 6, 2, 4, 2
    q, k, v = xsgen.random_inputs(5, P, B, S, H, D, 3.0, 1.0)
    o = attn(q, k, v, B, S, H, D, P, 40.0)
    ok &= bool(np.isfinite(o).all())
    a2a = json.load(open(os.path.join(GOLDEN, "a2a_map_tiny.json")))
    B, S, H, D, P = a2a["B"], a2a["S"], a2a["H"], a2a["D"], a2a["P"]
    x = np.zeros((P, B, S, H // P, D), dtype=np.int32)
    for r in range(P):
        for b in range(B):
            for s in range(S):
                for hl in range(H // P):
                    x[r, b, s, hl, 0] = 1000 * r + 100 * b + 10 * s + hl
    y = np.zeros((P, B, S // P, H, D), dtype=np.int32)
    lib.xs_oracle_a2a(x.ctypes.data, y.ctypes.data, B, S, H, D, P, 4)
    ok &= bool(np.array_equal(y, np.array(a2a["out"], dtype=np.int32)))
    return ok


def _decode_ref(codes):
    """E4M3 decode by the generator's independent value table (not the oracle's)."""
    vals = xsgen._e4m3_positive_values()
    c = np.asarray(codes)
    mag = vals[np.minimum(c & 0x7F, 0x7E)]
    return np.where(c & 0x80, -mag, mag)


def test_pins_catch_planted_mistakes(tmp_path):
    pytest.importorskip("mpmath")
    src = open(os.path.join(os.path.dirname(oracle.__file__), "xs_oracle.c")).read()
    # the unmodified source passes
    assert _pins_pass(ctypes.CDLL(oracle.build()))
    for name, (old, new) in _MUTANTS.items():
        assert src.count(old) >= 1, f"mutation anchor missing: {name}"
        path = tmp_path / f"m_{abs(hash(name))}.c"
        path.write_text(src.replace(old, new))
        so = str(path)[:-2] + ".so"
        subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread", str(path),
                               "-o", so, "-lm"])
        assert not _pins_pass(ctypes.CDLL(so)), f"no pin caught the planted mistake: {name}"
