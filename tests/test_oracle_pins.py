"""Pins of the float64 oracle against what the pages and mathematics fix.

None of these re-type the oracle's formulas: each checks it against exact
rational arithmetic, a closed form, a printed number, an invariant, or a
textbook library routine, chosen so that a dropped term, a wrong sign or index,
a transposed operand or the wrong rounding rule fails at least one test.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import kvq_oracle as O
from synth import f32_to_bf16_bits

RNG = np.random.default_rng(1234)


# ---------------------------------------------------------------- exact helpers (test-side)
def rne_int(r: Fraction) -> int:
    """Round a rational to the nearest integer, ties to even (exact)."""
    fl = math.floor(r)
    rem = r - fl
    if rem > Fraction(1, 2):
        return fl + 1
    if rem < Fraction(1, 2):
        return fl
    return fl if fl % 2 == 0 else fl + 1


def rn_float32(r: Fraction) -> Fraction:
    """Round a positive rational to the nearest binary32 value (ties to even),
    including the subnormal range, exactly."""
    assert r > 0
    e = math.floor(math.log2(r.numerator) - math.log2(r.denominator))
    while Fraction(2) ** e > r:
        e -= 1
    while Fraction(2) ** (e + 1) <= r:
        e += 1
    e = max(e, -126)                     # subnormals share the minimum exponent
    ulp = Fraction(2) ** (e - 23)
    return rne_int(r / ulp) * ulp


def exact_quantize(xs, bits):
    """Exact rational restatement of the page definition (float32 stored scale)."""
    qmax = {8: 127, 4: 7, 2: 1}[bits]
    lo, hi = {8: (-127, 127), 4: (-8, 7), 2: (-2, 1)}[bits]
    fr = [Fraction(float(x)) for x in xs]
    amax = max(abs(f) for f in fr)
    if amax == 0:
        return [0] * len(fr), Fraction(1)
    s = rn_float32(amax / qmax)
    return [min(hi, max(lo, rne_int(f / s))) for f in fr], s


def bf16_vec(n, scale=1.0, dist="normal"):
    x = RNG.standard_normal(n).astype(np.float32) * np.float32(scale)
    if dist == "t3":
        x = RNG.standard_t(3, n).astype(np.float32)
    return O.bf16_to_f64(f32_to_bf16_bits(x))


# ---------------------------------------------------------------- quantizer pins
@pytest.mark.parametrize("bits", [8, 4])
def test_quantizer_matches_exact_rational_brute_force(bits):
    for trial in range(300):
        n = int(RNG.integers(1, 40))
        dist = "t3" if trial % 3 == 0 else "normal"
        x = bf16_vec(n, scale=float(2.0 ** RNG.integers(-20, 20)), dist=dist)
        codes, s = O.quantize(x, bits)
        ref_codes, ref_s = exact_quantize(x, bits)
        assert Fraction(float(s)) == ref_s
        assert list(map(int, codes)) == ref_codes


@pytest.mark.parametrize("bits", [8, 4])
def test_quantizer_exact_ties_round_to_even(bits):
    qmax = O.QMAX[bits]
    for k in range(-10, 10):
        s = 2.0 ** k
        # amax = qmax * s makes the stored scale exactly s; the rest sit on ties
        halves = [n + 0.5 for n in range(-qmax, qmax)]
        x = np.array([qmax * s] + [h * s for h in halves])
        codes, sc = O.quantize(x, bits)
        assert float(sc) == s
        expect = [qmax] + [rne_int(Fraction(h)) for h in halves]
        assert list(map(int, codes)) == expect
        # ties to even: never an odd code on a tie
        assert all(int(c) % 2 == 0 for c in codes[1:])


@pytest.mark.parametrize("bits", [8, 4])
def test_quantizer_near_ties(bits):
    qmax = O.QMAX[bits]
    s = 2.0 ** -3
    for n in range(0, qmax):
        tie = (n + 0.5) * s
        up = np.nextafter(np.float32(tie), np.float32(np.inf)).astype(np.float64)
        dn = np.nextafter(np.float32(tie), np.float32(-np.inf)).astype(np.float64)
        codes, sc = O.quantize(np.array([qmax * s, up, dn, -up, -dn]), bits)
        assert list(map(int, codes)) == [qmax, n + 1, n, -(n + 1), -n]


@pytest.mark.parametrize("bits", [8, 4])
def test_quantizer_invariants(bits):
    qmax = O.QMAX[bits]
    x = O.bf16_to_f64(f32_to_bf16_bits(RNG.standard_normal((500, 128)).astype(np.float32)))
    codes, s = O.quantize(x, bits)
    err = np.abs(x - codes * s.astype(np.float64)[:, None])     # code*s exact in float64
    assert np.all(err <= s.astype(np.float64)[:, None] / 2)
    assert np.all(np.abs(codes).max(axis=1) == qmax)           # amax element hits qmax
    assert codes.min() >= -qmax and codes.max() <= qmax


def test_quantizer_zero_vector():
    for bits in (8, 4):
        codes, s = O.quantize(np.zeros((3, 128)), bits)
        assert np.all(codes == 0) and np.all(s == np.float32(1.0))


def test_quantizer_golden_worked_examples(golden_dir):
    with open(os.path.join(golden_dir, "quantize_worked.txt")) as f:
        rows = [l for l in f if l.strip() and not l.startswith("#")]
    assert len(rows) >= 4
    for row in rows:
        bits, scale, vals, codes = [p.strip() for p in row.split("|")]
        x = np.array([float(v) for v in vals.split(",")])
        c, s = O.quantize(x, int(bits))
        assert float(s) == float(scale)
        assert list(map(int, c)) == [int(v) for v in codes.split(",")]


def _float64_scale_quantizer(vec, qmax):
    """The rule of [P3] "The axis choice is a kernel decision" with the scale
    kept in float64 (the page keeps it as a Python float) instead of the stored
    float32: vectorised, half-to-even rounding of x / scale, clamp to +-qmax."""
    x = np.asarray(vec, dtype=np.float64)
    scale = float(np.abs(x).max()) / qmax
    if scale == 0.0:
        return np.zeros(x.shape, dtype=np.int64), 1.0
    return np.clip(np.rint(x / scale), -qmax, qmax).astype(np.int64), scale


def test_quantizer_agrees_with_page_listing_except_near_ties():
    """Codes from the float32 stored scale agree with the page's float64-scale
    listing except where x/s is within a few float32 ulps of a half-integer."""
    n_checked = 0
    for _ in range(200):
        x = bf16_vec(128)
        codes, s = O.quantize(x, 8)
        ref, scale64 = _float64_scale_quantizer(x, 127)
        assert abs(float(s) - scale64) <= scale64 * 2.0 ** -24
        for xi, c, r in zip(x, codes, ref):
            frac = abs(xi / scale64) % 1.0
            if abs(frac - 0.5) < 1e-5:
                continue
            assert int(c) == r
            n_checked += 1
    assert n_checked > 20000


def test_quantizer_subnormal_inputs():
    # bf16 subnormals (below 2^-126) and the smallest bf16 subnormal 2^-133
    for bits in (8, 4):
        tiny = np.array([2.0 ** -133, -3 * 2.0 ** -133, 5 * 2.0 ** -130, 2.0 ** -127, 0.0])
        codes, s = O.quantize(tiny, bits)
        ref_codes, ref_s = exact_quantize(tiny, bits)
        assert Fraction(float(s)) == ref_s and float(s) > 0
        assert list(map(int, codes)) == ref_codes
        err = np.abs(tiny - codes * float(s))
        assert np.all(err <= float(s) / 2)


def test_channel_factor_division_is_float32_rounded():
    k = bf16_vec(64)
    c = np.abs(bf16_vec(64)) + 0.5
    kp = O.divide_by_channel_factor(k, c.astype(np.float32))
    for a, b, r in zip(k, c.astype(np.float32), kp):
        assert Fraction(float(r)) == (rn_float32(abs(Fraction(float(a)) / Fraction(float(b)))) * (1 if a >= 0 else -1) if a != 0 else 0)


# ---------------------------------------------------------------- fold identities
def test_scale_fold_after_integer_dot_is_exact_in_rationals():
    """(q . k_int) * s == q . (k_int * s) exactly; the float64 oracle's
    dequantize-then-dot agrees with the folded order to a few ulps."""
    for _ in range(50):
        q = bf16_vec(128)
        k = bf16_vec(128)
        codes, s = O.quantize(k, 8)
        qf = [Fraction(float(v)) for v in q]
        sf = Fraction(float(s))
        folded = sum(a * int(c) for a, c in zip(qf, codes)) * sf
        unfolded = sum(a * (int(c) * sf) for a, c in zip(qf, codes))
        assert folded == unfolded
        oracle_dot = float(q @ O.dequantize(codes, s))
        assert abs(oracle_dot - float(folded)) <= 1e-13 * max(1.0, abs(float(folded)))


def test_channel_factor_moved_onto_query_is_exact_in_rationals():
    """(q (.) c) . k' == q . (c (.) k') exactly, and the oracle reconstruction
    c * code * s is what a folded-query dot would see."""
    q = bf16_vec(128)
    k = bf16_vec(128)
    c = (np.abs(bf16_vec(128)) + 0.25).astype(np.float32).astype(np.float64)
    codes, s = O.quantize_keys(k, 4, c)
    kp = O.dequantize(codes, s)
    lhs = sum(Fraction(float(a)) * Fraction(float(cc)) * Fraction(float(b)) for a, cc, b in zip(q, c, kp))
    rhs = sum(Fraction(float(a)) * (Fraction(float(cc)) * Fraction(float(b))) for a, cc, b in zip(q, c, kp))
    assert lhs == rhs
    kh = O.reconstruct_keys(codes, s, c)
    assert abs(float(q @ kh) - float(rhs)) <= 1e-12 * max(1.0, abs(float(rhs)))


# ---------------------------------------------------------------- attention pins
def test_attention_matches_torch_sdpa_float64():
    for T in (1, 2, 7, 64, 300):
        for G in (1, 4, 8):
            q = bf16_vec(G * 128).reshape(G, 128)
            k = bf16_vec(T * 128).reshape(T, 128)
            v = bf16_vec(T * 128).reshape(T, 128)
            o, lse = O.attention(q, k, v)
            tq = torch.from_numpy(q)[None, :, None, :]          # [G, 1 query, D] as batch of heads
            tk = torch.from_numpy(k)[None, None].expand(1, G, T, 128)
            tv = torch.from_numpy(v)[None, None].expand(1, G, T, 128)
            ref = torch.nn.functional.scaled_dot_product_attention(tq.transpose(0, 1).reshape(1, G, 1, 128), tk, tv)
            np.testing.assert_allclose(o, ref[0, :, 0].numpy(), rtol=0, atol=1e-13)
            ref_lse = torch.logsumexp(torch.from_numpy(q @ k.T / math.sqrt(128)), dim=1).numpy()
            np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)


def test_attention_weights_sum_to_one():
    q = bf16_vec(4 * 128).reshape(4, 128)
    k = bf16_vec(1000 * 128).reshape(1000, 128) * 3
    a = O.attention_weights(q, k)
    assert np.all(np.abs(a.sum(axis=1) - 1.0) <= 1e-15 * 1000)
    assert np.all(a >= 0)


def test_attention_single_token_returns_that_value():
    q = bf16_vec(3 * 128).reshape(3, 128)
    k = bf16_vec(128).reshape(1, 128)
    v = bf16_vec(128).reshape(1, 128)
    o, lse = O.attention(q, k, v)
    assert np.array_equal(o, np.repeat(v, 3, axis=0))
    np.testing.assert_allclose(lse, (q @ k[0]) / math.sqrt(128), rtol=0, atol=1e-14)


def test_attention_identical_keys_or_zero_query_gives_mean():
    T = 37
    v = bf16_vec(T * 128).reshape(T, 128)
    k_same = np.repeat(bf16_vec(128).reshape(1, 128), T, axis=0)
    q = bf16_vec(2 * 128).reshape(2, 128)
    o, lse = O.attention(q, k_same, v)
    np.testing.assert_allclose(o, np.repeat(v.mean(axis=0, keepdims=True), 2, axis=0), rtol=0, atol=1e-14)
    o0, lse0 = O.attention(np.zeros((1, 128)), bf16_vec(T * 128).reshape(T, 128), v)
    np.testing.assert_allclose(o0[0], v.mean(axis=0), rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse0, [math.log(T)], rtol=0, atol=1e-14)


def test_attention_empty_sequence_convention():
    o, lse = O.attention(np.ones((2, 128)), np.zeros((0, 128)), np.zeros((0, 128)))
    assert np.all(o == 0) and np.all(np.isneginf(lse))


def test_attention_two_token_closed_form():
    """T = 2: a_0 = 1 / (1 + exp(s_1 - s_0)) (logistic form of softmax)."""
    q = bf16_vec(128).reshape(1, 128)
    k = bf16_vec(256).reshape(2, 128)
    v = bf16_vec(256).reshape(2, 128)
    s0, s1 = (k @ q[0]) / math.sqrt(128)
    a0 = 1.0 / (1.0 + math.exp(s1 - s0))
    o, _ = O.attention(q, k, v)
    np.testing.assert_allclose(o[0], a0 * v[0] + (1 - a0) * v[1], rtol=0, atol=1e-14)


def test_attention_high_precision_brute_force():
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 50
    q = bf16_vec(2 * 8).reshape(2, 8)
    k = bf16_vec(5 * 8).reshape(5, 8)
    v = bf16_vec(5 * 8).reshape(5, 8)
    o, lse = O.attention(q, k, v)
    for g in range(2):
        sc = [mp.fsum(mp.mpf(q[g, j]) * mp.mpf(k[i, j]) for j in range(8)) / mp.sqrt(8) for i in range(5)]
        den = mp.fsum(mp.exp(s) for s in sc)
        for d in range(8):
            num = mp.fsum(mp.exp(sc[i]) * mp.mpf(v[i, d]) for i in range(5))
            assert abs(float(num / den) - o[g, d]) <= 1e-14
        assert abs(float(mp.log(den)) - lse[g]) <= 1e-14


def test_split_merge_equals_single_pass():
    q = bf16_vec(4 * 128).reshape(4, 128)
    T = 517
    k = bf16_vec(T * 128).reshape(T, 128) * 2
    v = bf16_vec(T * 128).reshape(T, 128)
    o, lse = O.attention(q, k, v)
    for cuts in ([100, 300], [1, 2, 3, 516], [256]):
        edges = [0] + cuts + [T]
        parts = [O.attention(q, k[a:b], v[a:b]) for a, b in zip(edges[:-1], edges[1:])]
        om, lm = O.lse_merge(parts)
        np.testing.assert_allclose(om, o, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lm, lse, rtol=0, atol=1e-12)


def test_perturbation_identities():
    """s' - s = q E_K^T / sqrt(d) and, for fixed a, o' - o = a E_V."""
    d = 128
    q = bf16_vec(d).reshape(1, d)
    k = bf16_vec(50 * d).reshape(50, d)
    v = bf16_vec(50 * d).reshape(50, d)
    codes, s = O.quantize(k, 4)
    e_k = O.dequantize(codes, s) - k
    s_exact = (q @ k.T) / math.sqrt(d)
    s_pert = (q @ (k + e_k).T) / math.sqrt(d)
    np.testing.assert_allclose(s_pert - s_exact, (q @ e_k.T) / math.sqrt(d), rtol=0, atol=1e-13)
    a = O.attention_weights(q, k)
    vc, vs = O.quantize(v, 4)
    e_v = O.dequantize(vc, vs) - v
    np.testing.assert_allclose(a @ (v + e_v) - a @ v, a @ e_v, rtol=0, atol=1e-14)
    # with exact keys the oracle output moves by exactly a E_V
    o_exact, _ = O.attention(q, k, v)
    o_q, _ = O.attention(q, k, v + e_v)
    np.testing.assert_allclose(o_q - o_exact, a @ e_v, rtol=0, atol=1e-14)


# ---------------------------------------------------------------- window and sequence assembly
def test_window_covering_whole_sequence_reduces_to_plain_attention():
    L, H, G = 90, 2, 4
    k = bf16_vec(L * H * 128).reshape(L, H, 128)
    v = bf16_vec(L * H * 128).reshape(L, H, 128)
    qb = f32_to_bf16_bits(RNG.standard_normal((H * G, 128)).astype(np.float32))
    st = O.quantize_sequence(k, v, 8, 8, window=128)
    assert st["Lq"] == 0
    o, lse = O.decode_sequence(qb, st, H)
    q = O.bf16_to_f64(qb)
    for h in range(H):
        tk = torch.from_numpy(k[:, h])[None, None]
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q[h * G:(h + 1) * G])[None, :, None], tk.expand(1, G, L, 128),
            torch.from_numpy(v[:, h])[None, None].expand(1, G, L, 128))
        np.testing.assert_allclose(o[h * G:(h + 1) * G], ref[0, :, 0].numpy(), rtol=0, atol=1e-13)


def test_window_split_positions():
    assert O.window_split(4096, 128) == 3968
    assert O.window_split(100, 128) == 0
    assert O.window_split(128, 128) == 0
    assert O.window_split(129, 128) == 1
    assert O.window_split(77, 0) == 77


def test_sequence_reconstruction_orders_quantized_then_window():
    L, H = 40, 1
    k = bf16_vec(L * H * 128).reshape(L, H, 128)
    v = bf16_vec(L * H * 128).reshape(L, H, 128)
    st = O.quantize_sequence(k, v, 8, 4, window=16)
    kh, vh = O.reconstruct_sequence(st, 0)
    assert kh.shape == (L, 128)
    assert np.array_equal(kh[24:], k[24:, 0]) and np.array_equal(vh[24:], v[24:, 0])
    assert np.all(np.abs(kh[:24] - k[:24, 0]) <= np.abs(k[:24, 0]).max(axis=1, keepdims=True) / 127 / 2 * 1.0000001)


def test_grouped_query_heads_read_their_kv_head():
    L, H, G = 20, 3, 2
    k = bf16_vec(L * H * 128).reshape(L, H, 128)
    v = bf16_vec(L * H * 128).reshape(L, H, 128)
    qb = f32_to_bf16_bits(RNG.standard_normal((H * G, 128)).astype(np.float32))
    st = O.quantize_sequence(k, v, 16, 16)
    o, _ = O.decode_sequence(qb, st, H)
    q = O.bf16_to_f64(qb)
    for hq in range(H * G):
        ref, _ = O.attention(q[hq:hq + 1], k[:, hq // G], v[:, hq // G])
        np.testing.assert_allclose(o[hq], ref[0], rtol=0, atol=1e-15)


# ---------------------------------------------------------------- byte accounting
def test_metadata_fractions_match_printed_values(golden_dir):
    with open(os.path.join(golden_dir, "metadata_fractions.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    assert len(rows) == 4
    for d, bits, meta, pct in rows:
        frac = O.metadata_fraction(int(d), int(bits), int(meta))
        assert round(100 * frac) == int(pct) or math.floor(100 * frac) == int(pct)
    assert O.metadata_fraction(128, 8, 4) == 0.03125
    assert O.metadata_fraction(128, 4, 4) == 0.0625
    assert O.metadata_fraction(128, 2, 4) == 0.125


def test_kv_payload_formula(golden_dir):
    with open(os.path.join(golden_dir, "kv_payload.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    for L, H, D, T, b, expect in rows:
        assert O.kv_payload_bytes(int(L), int(H), int(D), int(T), float(b)) == float(expect)
    assert O.kv_payload_bytes(1, 8, 128, 4096, 1) * 2 == O.kv_payload_bytes(1, 8, 128, 4096, 2)


def test_cache_bytes_per_token_include_scales():
    assert O.cache_bytes_per_token_head(128, 8, 8) == 264
    assert O.cache_bytes_per_token_head(128, 4, 4) == 136
    assert O.cache_bytes_per_token_head(128, 4, 8) == 200
    assert O.cache_bytes_per_token_head(128, 16, 16) == 512
    # payload part equals the page formula per token per head (b = bits / 8)
    for kb, vb in ((8, 8), (4, 4), (16, 16)):
        pay = O.kv_payload_bytes(1, 1, 128, 1, kb / 8) if kb == vb else None
        extra = 0 if kb == 16 else 8
        assert O.cache_bytes_per_token_head(128, kb, vb) == pay + extra


# ---------------------------------------------------------------- planted mistakes are caught
def test_pins_catch_a_planted_rounding_mistake(monkeypatch):
    """Half-away-from-zero instead of half-to-even must fail the tie pin."""
    real = np.rint
    monkeypatch.setattr(O.np, "rint", lambda a: np.trunc(a + np.copysign(0.5, a)))
    x = np.array([127 * 0.25, 0.625])          # 0.625 / 0.25 = 2.5 -> 2 (even), not 3
    codes, _ = O.quantize(x, 8)
    assert int(codes[1]) == 3                  # the planted mistake shows ...
    monkeypatch.setattr(O.np, "rint", real)
    codes, _ = O.quantize(x, 8)
    assert int(codes[1]) == 2 == rne_int(Fraction(5, 2))   # ... and the pin distinguishes it


def test_pins_catch_a_planted_missing_sqrt_d(monkeypatch):
    q = bf16_vec(2 * 128).reshape(2, 128)
    k = bf16_vec(9 * 128).reshape(9, 128)
    v = bf16_vec(9 * 128).reshape(9, 128)
    monkeypatch.setattr(O.np, "sqrt", lambda x: 1.0)
    o_bad, _ = O.attention(q, k, v)
    monkeypatch.undo()
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None, :, None], torch.from_numpy(k)[None, None].expand(1, 2, 9, 128),
        torch.from_numpy(v)[None, None].expand(1, 2, 9, 128))[0, :, 0].numpy()
    assert np.max(np.abs(o_bad - ref)) > 1e-3
    o_good, _ = O.attention(q, k, v)
    assert np.max(np.abs(o_good - ref)) < 1e-13


# ---------------------------------------------------------------- asymmetric format (scale + zero point)
def exact_quantize_asym(xs, bits):
    """Exact rational restatement: offset = min, s = RN32((max - min)/qmaxu),
    u = clamp(RNE((x - min)/s), 0, qmaxu)."""
    qmaxu = {8: 255, 4: 15, 2: 3}[bits]
    fr = [Fraction(float(x)) for x in xs]
    lo, hi = min(fr), max(fr)
    if hi == lo:
        return [0] * len(fr), Fraction(1), lo
    s = rn_float32((hi - lo) / qmaxu)
    return [min(qmaxu, max(0, rne_int((f - lo) / s))) for f in fr], s, lo


@pytest.mark.parametrize("bits", [8, 4])
def test_asym_quantizer_matches_exact_rational_brute_force(bits):
    for trial in range(300):
        n = int(RNG.integers(2, 40))
        dist = "t3" if trial % 3 == 0 else "normal"
        x = bf16_vec(n, scale=float(2.0 ** RNG.integers(-10, 10)), dist=dist)
        if trial % 5 == 0:
            x = np.abs(x)                                   # one-signed vectors: min far from 0
        codes, s, m = O.quantize_asym(x, bits)
        ref_codes, ref_s, ref_m = exact_quantize_asym(x, bits)
        assert Fraction(float(s)) == ref_s and Fraction(float(m)) == ref_m
        assert list(map(int, codes)) == ref_codes


@pytest.mark.parametrize("bits", [8, 4])
def test_asym_quantizer_invariants(bits):
    qmaxu = O.QMAXU[bits]
    x = O.bf16_to_f64(f32_to_bf16_bits(RNG.standard_normal((400, 128)).astype(np.float32) + 1.5))
    codes, s, m = O.quantize_asym(x, bits)
    xh = O.dequantize_asym(codes, s, m)
    assert np.all(np.abs(x - xh) <= s.astype(np.float64)[:, None] / 2 * (1 + 1e-12))
    assert np.all(codes.min(axis=1) == 0) and np.all(codes.max(axis=1) == qmaxu)   # min -> 0, max -> top
    assert np.array_equal(m, x.min(axis=1).astype(np.float32))


def test_asym_quantizer_constant_and_tie_cases():
    c = np.full(16, 0.75)
    codes, s, m = O.quantize_asym(c, 8)
    assert np.all(codes == 0) and float(s) == 1.0 and float(m) == 0.75
    assert np.array_equal(O.dequantize_asym(codes, s, m), c)
    # (x - min) / s on exact half-integers rounds to even: s = 2^-4, min = -1
    x = np.array([-1.0, -1.0 + 15 * 2.0 ** -4, -1.0 + 2.5 * 2.0 ** -4, -1.0 + 3.5 * 2.0 ** -4])
    codes, s, m = O.quantize_asym(x, 4)
    assert float(s) == 2.0 ** -4 and float(m) == -1.0
    assert list(map(int, codes)) == [0, 15, 2, 4]


def test_asym_score_fold_is_exact_in_rationals():
    """q . (u*s + m) == s*(q . u) + m*(sum q): the offset moves out of the dot."""
    q = bf16_vec(128)
    k = bf16_vec(128) + 0.5
    u, s, m = O.quantize_asym(k, 8)
    qf = [Fraction(float(a)) for a in q]
    lhs = sum(a * (int(c) * Fraction(float(s)) + Fraction(float(m))) for a, c in zip(qf, u))
    rhs = Fraction(float(s)) * sum(a * int(c) for a, c in zip(qf, u)) + Fraction(float(m)) * sum(qf)
    assert lhs == rhs
    assert abs(float(q @ O.dequantize_asym(u, s, m)) - float(lhs)) <= 1e-12 * max(1.0, abs(float(lhs)))


def rn32_signed(r: Fraction) -> Fraction:
    """Round a rational to binary32 (ties to even), either sign."""
    if r == 0:
        return Fraction(0)
    return rn_float32(r) if r > 0 else -rn_float32(-r)


def _check_asym_keys_under_channel_factor(bits):
    """Asymmetric keys with a per-channel factor c ([P3] "The axis choice is a
    kernel decision": the factor comes out of the keys and onto the query;
    [P1] "Quantization granularity defines which values share a scale": scale
    and zero point per token).  Exact reference: k'_j = RN32(k_j / c_j), the
    asymmetric quantizer on k' in rationals, and k_hat_j = c_j * (u_j * s + m):
    the factor multiplies the zero point as well as the scaled code.  The
    oracle's float64 reconstruction must lie within a few roundings of it, and
    the plausible slip of scaling only the code term (c_j * u_j * s + m) must
    fall far outside that bound."""
    rng = np.random.default_rng(21 + bits)
    L, H, D = 7, 2, 128
    k = O.bf16_to_f64(f32_to_bf16_bits((rng.standard_t(3, (L, H, D)) + 0.7).astype(np.float32)))
    v = O.bf16_to_f64(f32_to_bf16_bits(rng.standard_normal((L, H, D)).astype(np.float32)))
    c = (np.abs(k).max(axis=0) * rng.uniform(0.5, 2.0, (H, D))).astype(np.float32).astype(np.float64)
    st = O.quantize_sequence(k, v, bits, 8, c=c, asym=True)
    slip_caught = 0
    for h in range(H):
        k_hat, _ = O.reconstruct_sequence(st, h)
        for t in range(L):
            kp = [rn32_signed(Fraction(float(k[t, h, j])) / Fraction(float(c[h, j]))) for j in range(D)]
            u, s, m = exact_quantize_asym([float(x) for x in kp], bits)
            assert list(map(int, st["k_codes"][t, h])) == u
            assert Fraction(float(st["k_scale"][t, h])) == s and Fraction(float(st["k_offset"][t, h])) == m
            for j in range(D):
                cj = Fraction(float(c[h, j]))
                ref = cj * (u[j] * s + m)
                bound = 2.0 ** -50 * float(cj * (abs(u[j] * s) + abs(m)))
                assert abs(k_hat[t, j] - float(ref)) <= bound
                slip = float(cj * u[j] * s + m)
                slip_caught += abs(slip - float(ref)) > 1e6 * bound
    assert slip_caught > 0.9 * H * L * D


@pytest.mark.parametrize("bits", [8, 4])
def test_asym_keys_under_channel_factor_match_exact_rationals(bits):
    _check_asym_keys_under_channel_factor(bits)


def test_asym_factor_pin_catches_a_zero_point_left_unscaled(monkeypatch):
    """Plant the slip in the oracle (the factor multiplies u * s but not m):
    the exact-rational pin above must fail."""
    real = O.reconstruct_sequence

    def planted(st, head):
        k_hat, v_hat = real(st, head)
        if st.get("asym") and st["c"] is not None:
            Lq = st["Lq"]
            c = np.asarray(st["c"][head], np.float64)
            m = np.asarray(st["k_offset"][:, head], np.float64)[:, None]
            k_hat = k_hat.copy()
            k_hat[:Lq] = k_hat[:Lq] - c * m + m
        return k_hat, v_hat

    monkeypatch.setattr(O, "reconstruct_sequence", planted)
    with pytest.raises(AssertionError):
        _check_asym_keys_under_channel_factor(8)


def test_asym_metadata_fraction_is_the_printed_six_percent(golden_dir):
    # scale + zero point over 128 int8 codes: the page's "add 6 percent" row
    assert O.metadata_fraction(128, 8, 8) == 0.0625
    assert O.cache_bytes_per_token_head(128, 8, 8, asym=True) == 2 * (128 + 8)


# ---------------------------------------------------------------- quantized query (integer dot)
def test_query_quantizer_is_the_cache_rule_on_the_folded_query():
    """q_int / s_q are the exact symmetric int8 rule applied to q, or to the
    float32 product q * c when a per-channel key factor is folded onto q."""
    for trial in range(100):
        q = bf16_vec(128, scale=float(2.0 ** RNG.integers(-6, 6)))
        codes, s = O.quantize_query(q)
        ref_codes, ref_s = exact_quantize(q, 8)
        assert Fraction(float(s)) == ref_s and list(map(int, codes)) == ref_codes
        c = (np.abs(bf16_vec(128)) + 0.1).astype(np.float32).astype(np.float64)
        codes, s = O.quantize_query(q, c)
        folded = (q * c).astype(np.float32)                         # one float32 rounding per element
        ref_codes, ref_s = exact_quantize(folded, 8)
        assert Fraction(float(s)) == ref_s and list(map(int, codes)) == ref_codes


@pytest.mark.parametrize("k_bits", [8, 4])
@pytest.mark.parametrize("factor", [False, True])
def test_quantized_query_score_is_the_scaled_integer_dot(k_bits, factor):
    """The oracle's score with the effective query equals s_q * s_k *
    (q_int . k_int) / sqrt(D) computed with exact integers, with or without a
    per-channel key factor (which cancels between query and keys)."""
    D = 128
    c = (np.abs(bf16_vec(D)) + 0.25).astype(np.float32).astype(np.float64) if factor else None
    for _ in range(20):
        q = bf16_vec(D)
        k = bf16_vec(D, dist="t3")
        q_int, s_q = O.quantize_query(q, c)
        k_int, s_k = O.quantize_keys(k, k_bits, c)
        acc = sum(int(a) * int(b) for a, b in zip(q_int, k_int))            # integer accumulator
        exact = Fraction(float(s_q)) * Fraction(float(s_k)) * acc
        k_hat = O.reconstruct_keys(k_int, s_k, c)
        oracle_dot = float(O.effective_query(q, c) @ k_hat)
        assert abs(oracle_dot - float(exact)) <= 1e-12 * max(1.0, abs(float(exact)))


def test_integer_accumulator_width_matches_the_page():
    """[P3] "Precision floors and mixed cache formats": a 4-bit key times an
    8-bit query fits easily in 16 bits, the sum over 128 dims needs a few more
    bits.  The extreme codes the two quantizers can produce bear this out."""
    q_int, _ = O.quantize_query(np.ones(128))
    k_int, _ = O.quantize_keys(-np.ones(128), 4)
    assert int(q_int.max()) == 127 and int(k_int.min()) == -7          # -8 is unreachable
    prods = q_int.astype(np.int64) * k_int.astype(np.int64)
    assert np.abs(prods).max() < 2 ** 15                                 # a signed 16-bit product
    acc = int(prods.sum())
    assert 2 ** 15 <= abs(acc) < 2 ** 17                                 # the sum needs 17-18 bits


def test_quantized_query_error_is_bounded_by_half_its_scale():
    """|score(q_int s_q) - score(q)| <= (s_q / 2) * sum|k_hat| / sqrt(D): the
    query quantizer's round-trip bound carried through the dot product (a
    wrong query scale breaks it)."""
    D = 128
    for _ in range(50):
        q = bf16_vec(D)
        k_hat = bf16_vec(D)
        _, s_q = O.quantize_query(q)
        s_exact = float(q @ k_hat) / math.sqrt(D)
        s_quant = float(O.effective_query(q) @ k_hat) / math.sqrt(D)
        bound = float(s_q) / 2 * float(np.abs(k_hat).sum()) / math.sqrt(D)
        assert abs(s_quant - s_exact) <= bound * (1 + 1e-12)
        assert abs(s_quant - s_exact) > 0 or bound == 0


def test_decode_sequence_quantized_query_mode_uses_each_heads_factor():
    """GQA: the quantized-query decode of a sequence equals attention of each
    query group's effective query over its own KV head (factor row h)."""
    H, G, D, L = 2, 3, 128, 40
    rng = np.random.default_rng(5)
    k = O.bf16_to_f64(f32_to_bf16_bits(rng.standard_normal((L, H, D)).astype(np.float32)))
    v = O.bf16_to_f64(f32_to_bf16_bits(rng.standard_normal((L, H, D)).astype(np.float32)))
    qb = f32_to_bf16_bits(rng.standard_normal((H * G, D)).astype(np.float32))
    c = (np.abs(rng.standard_normal((H, D))) + 0.5).astype(np.float32).astype(np.float64)
    st = O.quantize_sequence(k, v, 8, 8, c=c)
    o, lse = O.decode_sequence(qb, st, H, query_bits=8)
    q = O.bf16_to_f64(qb)
    for h in range(H):
        k_hat, v_hat = O.reconstruct_sequence(st, h)
        ref_o, ref_l = O.attention(O.effective_query(q[h * G:(h + 1) * G], c[h]), k_hat, v_hat)
        np.testing.assert_allclose(o[h * G:(h + 1) * G], ref_o, rtol=0, atol=1e-15)
        np.testing.assert_allclose(lse[h * G:(h + 1) * G], ref_l, rtol=0, atol=1e-15)
    o16, _ = O.decode_sequence(qb, st, H)
    assert not np.array_equal(o, o16)                                    # the mode changes the numerics


# ---------------------------------------------------------------- per-channel key scales only
def exact_quantize_per_channel(ks, cs, bits):
    lo, hi = {8: (-127, 127), 4: (-8, 7)}[bits]
    return [min(hi, max(lo, rne_int(Fraction(float(k)) / Fraction(float(c))))) for k, c in zip(ks, cs)]


@pytest.mark.parametrize("bits", [8, 4])
def test_per_channel_key_codes_match_exact_rationals(bits):
    for trial in range(60):
        k = bf16_vec(128, dist="t3" if trial % 2 else "normal")
        c = (np.abs(bf16_vec(128)) * (0.02 if bits == 8 else 0.3) + 1e-3).astype(np.float32).astype(np.float64)
        codes = O.quantize_keys_per_channel(k, bits, c)
        assert list(map(int, codes)) == exact_quantize_per_channel(k, c, bits)


def test_per_channel_key_ties_and_clamp():
    c = np.array([0.25, 0.25, 0.5, 0.5, 0.125, 1.0, 1.0, 1.0])
    k = np.array([0.125, 0.375, 0.25, 0.75, -0.0625, 200.0, -200.0, -7.75])   # quotients .5 1.5 .5 1.5 -.5 200 -200 -7.75
    assert list(map(int, O.quantize_keys_per_channel(k, 8, c))) == [0, 2, 0, 2, 0, 127, -127, -8]
    assert list(map(int, O.quantize_keys_per_channel(k, 4, c))) == [0, 2, 0, 2, 0, 7, -8, -8]   # -8 reachable here


def test_per_channel_keys_round_trip_and_query_fold():
    """|k - code * c| <= c / 2 inside the calibrated range, and the fold onto the
    query is exact: (q * c) . code == q . (c * code) in rationals."""
    k = bf16_vec(128)
    c = (np.abs(k) / 127 * 1.5 + 1e-4).astype(np.float32).astype(np.float64)   # |k / c| < 127
    codes = O.quantize_keys_per_channel(k, 8, c)
    assert np.all(np.abs(k - codes * c) <= c / 2 * (1 + 1e-12))
    q = bf16_vec(128)
    lhs = sum((Fraction(float(a)) * Fraction(float(cc))) * int(b) for a, cc, b in zip(q, c, codes))
    rhs = sum(Fraction(float(a)) * (Fraction(float(cc)) * int(b)) for a, cc, b in zip(q, c, codes))
    assert lhs == rhs


def test_per_channel_sequence_reconstruction_and_bytes():
    rng = np.random.default_rng(9)
    L, H, D = 20, 2, 128
    k = O.bf16_to_f64(f32_to_bf16_bits(rng.standard_normal((L, H, D)).astype(np.float32)))
    v = O.bf16_to_f64(f32_to_bf16_bits(rng.standard_normal((L, H, D)).astype(np.float32)))
    c = (np.abs(k).max(axis=0) / 7).astype(np.float32).astype(np.float64)     # per-channel absmax / qmax
    st = O.quantize_sequence(k, v, 4, 8, window=4, c=c, k_per_channel=True)
    assert "k_scale" not in st
    k_hat, _ = O.reconstruct_sequence(st, 1)
    assert np.array_equal(k_hat[:16], st["k_codes"][:, 1].astype(np.float64) * c[1])
    assert np.array_equal(k_hat[16:], k[16:, 1])
    assert O.cache_bytes_per_token_head(128, 8, 8, k_per_channel=True) == 128 + 128 + 4
    with pytest.raises(ValueError):
        O.quantize_sequence(k, v, 8, 8, c=None, k_per_channel=True)


def test_unit_channel_factor_reduces_to_the_plain_path():
    """c == 1 divides and multiplies by one: codes, scales, reconstruction and the
    decode output equal the path without a factor exactly."""
    rng = np.random.default_rng(13)
    L, H, D = 33, 2, 128
    k = O.bf16_to_f64(f32_to_bf16_bits(rng.standard_normal((L, H, D)).astype(np.float32)))
    v = O.bf16_to_f64(f32_to_bf16_bits(rng.standard_normal((L, H, D)).astype(np.float32)))
    qb = f32_to_bf16_bits(rng.standard_normal((2 * H, D)).astype(np.float32))
    ones = np.ones((H, D))
    for bits in (8, 4):
        a = O.quantize_sequence(k, v, bits, 8, c=ones)
        b = O.quantize_sequence(k, v, bits, 8)
        assert np.array_equal(a["k_codes"], b["k_codes"]) and np.array_equal(a["k_scale"], b["k_scale"])
        oa, la = O.decode_sequence(qb, a, H)
        ob, lb = O.decode_sequence(qb, b, H)
        assert np.array_equal(oa, ob) and np.array_equal(la, lb)


# ---------------------------------------------------------------- 2-bit codes with token-group scales
def test_token_group_quantizer_matches_exact_rationals_per_group():
    """Each 16-position group of each head is one vector for the rule: codes
    and the one scale equal the exact rational quantizer applied to the
    group's values (the last, partial group over the positions it holds)."""
    rng = np.random.default_rng(31)
    for trial in range(12):
        L, H, D = int(rng.integers(1, 40)), 2, 24
        x = O.bf16_to_f64(f32_to_bf16_bits((rng.standard_t(3, (L, H, D)) * 2.0 ** rng.integers(-6, 6))
                                           .astype(np.float32)))
        asym = trial % 2 == 1
        res = O.quantize_token_groups(x, 2, asym=asym)
        for g0 in range(0, L, 16):
            g1 = min(L, g0 + 16)
            for h in range(H):
                flat = x[g0:g1, h].reshape(-1)
                if asym:
                    ref_c, ref_s, ref_m = exact_quantize_asym(flat, 2)
                    assert np.all(res[2][g0:g1, h] == np.float32(float(ref_m)))
                else:
                    ref_c, ref_s = exact_quantize(flat, 2)
                assert list(map(int, res[0][g0:g1, h].reshape(-1))) == ref_c
                assert np.all(res[1][g0:g1, h] == np.float32(float(ref_s)))


def test_token_group_quantizer_invariants_and_ternary_codes():
    """Symmetric 2-bit: qmax = 1, so s = max|x| over the group, codes are in
    {-1, 0, 1} (the clamp's -2 is unreachable), every non-zero group has a code
    of magnitude 1, and |x - code * s| <= s / 2."""
    rng = np.random.default_rng(32)
    x = O.bf16_to_f64(f32_to_bf16_bits(rng.standard_normal((100, 3, 128)).astype(np.float32)))
    codes, s = O.quantize_token_groups(x, 2)
    assert set(np.unique(codes)) <= {-1, 0, 1}
    xh = codes * s.astype(np.float64)[..., None]
    assert np.all(np.abs(x - xh) <= s.astype(np.float64)[..., None] / 2)
    for g0 in range(0, 100, 16):
        for h in range(3):
            grp = x[g0:g0 + 16, h]
            assert float(s[g0, h]) == np.float32(np.abs(grp).max())
            assert np.abs(codes[g0:g0 + 16, h]).max() == 1


def test_token_groups_are_cache_blocks_and_a_single_token_group_is_the_per_token_rule():
    """Groups are positions [16j, 16j + 16): a change inside group 1 leaves
    group 0 untouched; a group of one position is the per-token quantizer."""
    rng = np.random.default_rng(33)
    x = O.bf16_to_f64(f32_to_bf16_bits(rng.standard_normal((40, 2, 128)).astype(np.float32)))
    c0, s0 = O.quantize_token_groups(x, 2)
    y = x.copy()
    y[20, 1, 5] = 1000.0
    c1, s1 = O.quantize_token_groups(y, 2)
    assert np.array_equal(c0[:16], c1[:16]) and np.array_equal(s0[:16], s1[:16])
    assert np.array_equal(c0[32:], c1[32:]) and float(s1[16, 1]) == 1000.0
    one_c, one_s = O.quantize_token_groups(x[:1], 2)
    ref_c, ref_s = O.quantize(x[0], 2)
    assert np.array_equal(one_c[0], ref_c) and np.array_equal(one_s[0], ref_s)


def test_two_bit_sequence_reconstruction_and_bytes():
    """A 2-bit sequence: keys (after the per-channel factor) and values in
    token groups, window positions kept in bf16; one 16-byte metadata record
    per group makes the read 64 + 1 bytes per token per head, against the
    4-byte per-token scale that would add the printed 12 percent."""
    rng = np.random.default_rng(34)
    L, H, D = 45, 2, 128
    k = O.bf16_to_f64(f32_to_bf16_bits(rng.standard_normal((L, H, D)).astype(np.float32)))
    v = O.bf16_to_f64(f32_to_bf16_bits(rng.standard_normal((L, H, D)).astype(np.float32)))
    c = (np.abs(k).max(axis=0)).astype(np.float32).astype(np.float64)
    st = O.quantize_sequence(k, v, 2, 2, window=16, c=c)
    assert st["Lq"] == 29
    kc, ks = O.quantize_token_groups(O.divide_by_channel_factor(k[:29], c), 2)
    assert np.array_equal(st["k_codes"], kc) and np.array_equal(st["k_scale"], ks)
    k_hat, v_hat = O.reconstruct_sequence(st, 1)
    assert np.array_equal(k_hat[:29], kc[:, 1] * ks[:, 1, None].astype(np.float64) * c[1])
    assert np.array_equal(k_hat[29:], k[29:, 1]) and np.array_equal(v_hat[29:], v[29:, 1])
    assert O.cache_bytes_per_token_head(128, 2, 2) == 65
    assert O.metadata_fraction(128, 2, 4) == 0.125               # the per-token cost it avoids
    with pytest.raises(ValueError):
        O.quantize_sequence(k, v, 2, 8)


# ---------------------------------------------------------------- chunked prefill (causal rows)
def test_prefill_rows_match_torch_sdpa_with_a_causal_offset_mask():
    """Rows of a chunk at positions p0..p0+C-1 attend to keys 0..p (plain bf16
    values, no quantization): equal to the library routine with a boolean mask
    key <= position, in float64."""
    rng = np.random.default_rng(41)
    L, H, D, G, C = 37, 2, 128, 4, 9
    k = O.bf16_to_f64(f32_to_bf16_bits(rng.standard_normal((L, H, D)).astype(np.float32)))
    v = O.bf16_to_f64(f32_to_bf16_bits(rng.standard_normal((L, H, D)).astype(np.float32)))
    st = O.quantize_sequence(k, v, 16, 16)
    pos = np.arange(L - C, L)
    q = O.bf16_to_f64(f32_to_bf16_bits(rng.standard_normal((C, G, D)).astype(np.float32)))
    for h in range(H):
        o, lse = O.prefill_attention(q, st, h, pos)
        mask = torch.from_numpy(np.arange(L)[None, :] <= pos[:, None])            # [C, L]
        qt = torch.from_numpy(q.transpose(1, 0, 2))                                 # [G, C, D]
        kt = torch.from_numpy(k[:, h])[None].expand(G, L, D)
        vt = torch.from_numpy(v[:, h])[None].expand(G, L, D)
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask[None])
        np.testing.assert_allclose(o.transpose(1, 0, 2), ref.numpy(), rtol=0, atol=1e-12)
        assert lse.shape == (C, G) and np.all(np.isfinite(lse))


def test_prefill_last_row_is_the_decode_of_the_whole_sequence():
    """The chunk's last row sees every stored position: it is the decode step
    over the whole (quantized) sequence; a row at position 0 sees one key."""
    rng = np.random.default_rng(42)
    L, H, D = 50, 2, 128
    k = O.bf16_to_f64(f32_to_bf16_bits(rng.standard_normal((L, H, D)).astype(np.float32)))
    v = O.bf16_to_f64(f32_to_bf16_bits(rng.standard_normal((L, H, D)).astype(np.float32)))
    st = O.quantize_sequence(k, v, 4, 8)
    qb = f32_to_bf16_bits(rng.standard_normal((2 * H, D)).astype(np.float32))
    o_dec, l_dec = O.decode_sequence(qb, st, H)
    q = O.bf16_to_f64(qb)
    for h in range(H):
        o, lse = O.prefill_attention(q[None, 2 * h:2 * h + 2], st, h, np.array([L - 1]))
        assert np.array_equal(o[0], o_dec[2 * h:2 * h + 2]) and np.array_equal(lse[0], l_dec[2 * h:2 * h + 2])
        o0, _ = O.prefill_attention(q[None, 2 * h:2 * h + 2], st, h, np.array([0]))
        _, v_hat = O.reconstruct_sequence(st, h)
        assert np.array_equal(o0[0], np.broadcast_to(v_hat[0], (2, D)))
