"""Pins of the oracle's primitives against exact arithmetic, closed forms and the
pages' printed values (CPU only)."""
import math
import os
from fractions import Fraction

import mpmath
import numpy as np
import pytest
import torch

from tests import _ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(1234)


def rand_bf16(shape, std=1.0, seed=0):
    r = np.random.default_rng(seed)
    return _ref.f32_to_bf16_bits(r.normal(0, std, size=shape).astype(np.float32))


# ---- bf16 rounding ------------------------------------------------------------

def test_bf16_rounding_matches_bit_twiddle_on_fp32_boundaries(orc):
    # every exponent/mantissa of the upper half, with low halves at and around the tie
    hi = np.arange(0, 1 << 16, dtype=np.uint32)
    lows = np.array([0, 1, 0x7FFF, 0x8000, 0x8001, 0xFFFF, 0x1234, 0xC000], dtype=np.uint32)
    u = (hi[:, None] << 16 | lows[None, :]).ravel()
    f = u.view(np.float32)
    finite = np.isfinite(f)
    f = f[finite]
    got = orc.bf16_round(f.astype(np.float64))
    want = _ref.f32_to_bf16_bits(f)
    assert np.array_equal(got, want)


def test_bf16_rounding_random_fp32_and_torch(orc):
    u = rng.integers(0, 1 << 32, size=1 << 20, dtype=np.uint64).astype(np.uint32)
    f = u.view(np.float32)
    f = f[np.isfinite(f)]
    got = orc.bf16_round(f.astype(np.float64))
    assert np.array_equal(got, _ref.f32_to_bf16_bits(f))
    t = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, t)


def test_bf16_rounding_of_doubles_is_nearest_even(orc):
    # doubles that fp32 cannot hold: a double-rounding mistake (via float) fails here
    base = _ref.bf16_to_float(rand_bf16(4000, std=10.0, seed=3))
    base = base[base != 0]
    sp = 2.0 ** (np.frexp(np.abs(base))[1] - 8)
    for off in (0.5 + 2.0 ** -30, 0.5 - 2.0 ** -30, 0.5, 0.25, 0.75):
        x = base + off * sp * np.sign(base)
        got = _ref.bf16_to_float(orc.bf16_round(x))
        want = np.array([_ref.rnd_bf16(v) for v in x])
        assert np.array_equal(got, want), off


def test_bf16_special_values(orc):
    b = orc.bf16_round(np.array([np.nan, np.inf, -np.inf, 3.5e38, -3.5e38, 0.0, -0.0,
                                 2.0 ** -133, 2.0 ** -134, 1.5 * 2.0 ** -134, 2.0 ** -140]))
    assert b[0] & 0x7FC0 == 0x7FC0
    assert list(b[1:7]) == [0x7F80, 0xFF80, 0x7F80, 0xFF80, 0x0000, 0x8000]
    # smallest subnormal 2^-133; 2^-134 is a tie with 0 -> even (0); 1.5*2^-134 -> 2^-133
    assert list(b[7:]) == [0x0001, 0x0000, 0x0001, 0x0000]


def _golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


def test_bf16_golden_values_from_the_pages(orc):
    for row in _golden("bf16_rounding.txt"):
        kind = row[0]
        x = float(row[1])
        if kind == "round":
            assert orc.bf16_value(orc.bf16_round([x]))[0] == float(row[2]), row
        elif kind == "step":
            b = int(orc.bf16_round([x])[0])
            assert orc.bf16_value(np.array([b + 1], np.uint16))[0] - x == float(row[2]), row
        elif kind == "exact":
            assert orc.bf16_value(orc.bf16_round([x]))[0] == x, row


# ---- residual add -------------------------------------------------------------

def test_residual_add_exact_rounding(orc):
    h = rand_bf16(5000, 3.0, 1)
    y = rand_bf16(5000, 0.05, 2)
    got = orc.residual_add(h, y)
    hv, yv = _ref.bf16_to_float(h), _ref.bf16_to_float(y)
    want = [_ref.bf16_bits(_ref.rnd_bf16(Fraction(a) + Fraction(b))) for a, b in zip(hv, yv)]
    assert np.array_equal(got, np.array(want, np.uint16))


# ---- RMSNorm ------------------------------------------------------------------

def _rmsnorm_exact(x, w, eps):
    xv = [Fraction(v) for v in _ref.bf16_to_float(x)]
    wv = _ref.bf16_to_float(w)
    ms = sum(v * v for v in xv) / len(xv) + Fraction(eps)
    r = 1 / mpmath.sqrt(mpmath.mpf(ms.numerator) / ms.denominator)
    out, ties = [], 0
    for xi, wi in zip(xv, wv):
        prod = mpmath.mpf(xi.numerator) / xi.denominator * r
        ties += _ref.near_tie_bf16(_ref.frac(prod), 1e-13)
        y = _ref.rnd_bf16(_ref.frac(prod))
        out.append(_ref.bf16_bits(_ref.rnd_bf16(Fraction(wi) * Fraction(y))))
    return np.array(out, np.uint16), ties


@pytest.mark.parametrize("H,std", [(64, 1.0), (7168, 0.02)])
def test_rmsnorm_brute_force(orc, H, std):
    x = rand_bf16((1, H), std, 5)
    w = _ref.f32_to_bf16_bits((1 + 0.1 * np.random.default_rng(6).normal(size=H)).astype(np.float32))
    got = orc.rmsnorm(x, w, 1e-5)[0]
    want, ties = _rmsnorm_exact(x[0], w, 1e-5)
    assert ties == 0
    assert np.array_equal(got, want)


def test_rmsnorm_constant_vector_closed_form(orc):
    # x = c everywhere: out = bf16(w * bf16(c / sqrt(c^2 + eps)))
    for c in (0.5, 3.0, 0.0078125):
        x = _ref.f32_to_bf16_bits(np.full((1, 256), c, np.float32))
        w = rand_bf16(256, 1.0, 7)
        got = orc.rmsnorm(x, w, 1e-5)[0]
        y = _ref.rnd_bf16(mpmath.mpf(c) / mpmath.sqrt(mpmath.mpf(c) ** 2 + mpmath.mpf(1e-5)))
        want = [_ref.bf16_bits(_ref.rnd_bf16(Fraction(wi) * Fraction(y))) for wi in _ref.bf16_to_float(w)]
        assert np.array_equal(got, np.array(want, np.uint16))


def test_rmsnorm_scale_invariance(orc):
    x = rand_bf16((3, 512), 1.0, 8)
    w = rand_bf16(512, 1.0, 9)
    x4 = orc.bf16_round(_ref.bf16_to_float(x) * 16.0)   # exact power-of-two scaling
    assert np.array_equal(orc.rmsnorm(x, w, 0.0), orc.rmsnorm(x4, w, 0.0))


def test_rmsnorm_uses_its_own_row(orc):
    x = rand_bf16((2, 128), 1.0, 10)
    w = rand_bf16(128, 1.0, 11)
    both = orc.rmsnorm(x, w, 1e-5)
    assert np.array_equal(both[1], orc.rmsnorm(x[1:2], w, 1e-5)[0])


# ---- projections --------------------------------------------------------------

def test_linear_one_hot_returns_a_column(orc):
    W = rand_bf16((48, 80), 1.0, 12)
    x = np.zeros((80, 80), np.uint16)
    x[np.arange(80), np.arange(80)] = 0x3F80  # 1.0
    out = orc.linear(W, x)            # out[r, n] = W[n, r]
    assert np.array_equal(out, W.T)


def test_linear_brute_force_exact(orc):
    W = rand_bf16((24, 40), 1.0, 13)
    x = rand_bf16((3, 40), 1.0, 14)
    got = orc.linear(W, x)
    Wv, xv = _ref.bf16_to_float(W), _ref.bf16_to_float(x)
    for r in range(3):
        for n in range(24):
            s = sum(Fraction(Wv[n, k]) * Fraction(xv[r, k]) for k in range(40))
            assert not _ref.near_tie_bf16(s, 1e-13)
            assert got[r, n] == _ref.bf16_bits(_ref.rnd_bf16(s)), (r, n)


def test_linear_small_integers_exact(orc):
    r = np.random.default_rng(15)
    Wi = r.integers(-8, 9, size=(16, 1000))
    xi = r.integers(-8, 9, size=(2, 1000))
    W = _ref.f32_to_bf16_bits(Wi.astype(np.float32))
    x = _ref.f32_to_bf16_bits(xi.astype(np.float32))
    got = _ref.bf16_to_float(orc.linear(W, x))
    exact = xi @ Wi.T
    want = np.array([[_ref.rnd_bf16(Fraction(int(v))) for v in row] for row in exact])
    assert np.array_equal(got, want)


def test_linear_fp32_sums_equal_sequential_fp32_cumsum(orc):
    """fp32-sum mode: each output is numpy's sequential float32 cumulative sum of
    the (exact) products in increasing k order, rounded to bf16 by torch."""
    import torch
    W = rand_bf16((12, 700), 1.0, 16)
    x = rand_bf16((3, 700), 1.0, 17)
    with orc.fp32_sums():
        got = orc.linear(W, x)
    assert not orc.get_fp32_sums()
    Wv = _ref.bf16_to_float(W).astype(np.float32)
    xv = _ref.bf16_to_float(x).astype(np.float32)
    for r in range(3):
        for n in range(12):
            acc = np.cumsum(Wv[n] * xv[r], dtype=np.float32)[-1]
            want = torch.tensor(acc, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).item() & 0xFFFF
            assert got[r, n] == want, (r, n)


def test_linear_fp32_sums_truncate_where_double_does_not(orc):
    """1 + 2^20 x 2^-25: fp32 sums in increasing k order lose every small term
    (1 + 2^-25 rounds back to 1), the double sum keeps them all (1 + 2^-5)."""
    K = 1 + (1 << 20)
    W = np.full((1, K), 0x3F80, np.uint16)                      # 1.0
    x = np.full((1, K), _ref.f32_to_bf16_bits(np.float32(2.0 ** -25)), np.uint16)
    x[0, 0] = 0x3F80
    assert _ref.bf16_to_float(orc.linear(W, x))[0, 0] == 1.0 + 2.0 ** -5
    with orc.fp32_sums():
        assert _ref.bf16_to_float(orc.linear(W, x))[0, 0] == 1.0


# ---- RoPE ---------------------------------------------------------------------

THETA = 1.2e8


def test_rope_inv_freq(orc):
    inv = orc.rope_inv_freq(THETA, 128)
    assert inv[0] == 1.0
    assert np.all(np.diff(inv) < 0)
    for i in range(64):
        p = _ref.rnd_f32(mpmath.power(mpmath.mpf(THETA), mpmath.mpf(2 * i) / 128))
        want = _ref.rnd_f32(1 / Fraction(p))
        assert inv[i] == np.float32(want), i


@pytest.mark.parametrize("pos", [0, 1, 2, 4095, 8191, 131071, 262143])
def test_rope_table_against_mpmath(orc, pos):
    c, s = orc.rope_table(THETA, 128, pos + 1)
    inv = orc.rope_inv_freq(THETA, 128)
    for i in range(64):
        a = _ref.rnd_f32(Fraction(pos) * Fraction(float(inv[i])))
        ca = mpmath.cos(mpmath.mpf(a))
        sa = mpmath.sin(mpmath.mpf(a))
        if _ref.near_tie_bf16(_ref.frac(ca), 1e-14) or _ref.near_tie_bf16(_ref.frac(sa), 1e-14):
            continue
        assert c[pos, i] == _ref.bf16_bits(_ref.rnd_bf16(_ref.frac(ca))), (pos, i)
        assert s[pos, i] == _ref.bf16_bits(_ref.rnd_bf16(_ref.frac(sa))), (pos, i)


def test_rope_position_zero_is_identity(orc):
    c, s = orc.rope_table(THETA, 128, 1)
    assert np.all(c == 0x3F80) and np.all(s == 0)
    x = rand_bf16((2, 3, 128), 1.0, 16)
    assert np.array_equal(orc.rope_apply(x, [0, 0], c, s), x)


def test_rope_unit_vectors_give_cos_sin_with_neox_signs(orc):
    # x = e_j (j < 64) rotates to (c_j at j, s_j at j+64); x = e_{j+64} to (-s_j at j, c_j at j+64)
    pos = 5
    c, s = orc.rope_table(THETA, 128, pos + 1)
    for j in (0, 1, 17, 63):
        x = np.zeros((1, 1, 128), np.uint16)
        x[0, 0, j] = 0x3F80
        out = orc.rope_apply(x, [pos], c, s)[0, 0]
        assert out[j] == c[pos, j] and out[j + 64] == s[pos, j]
        assert np.count_nonzero(out & 0x7FFF) <= 2   # signed zeros elsewhere are fine
        x = np.zeros((1, 1, 128), np.uint16)
        x[0, 0, j + 64] = 0x3F80
        out = orc.rope_apply(x, [pos], c, s)[0, 0]
        assert out[j] == (s[pos, j] ^ 0x8000 if s[pos, j] else 0) and out[j + 64] == c[pos, j]
    # textbook values at position 1, pair 0: angle 1 rad
    assert _ref.bf16_to_float(c[1, 0]) == _ref.rnd_bf16(_ref.frac(mpmath.cos(1)))
    assert _ref.bf16_to_float(s[1, 0]) == _ref.rnd_bf16(_ref.frac(mpmath.sin(1)))


def test_rope_brute_force_against_exact_arithmetic(orc):
    c, s = orc.rope_table(THETA, 128, 300)
    x = rand_bf16((3, 2, 128), 2.0, 17)
    pos = [7, 123, 299]
    got = orc.rope_apply(x, pos, c, s)
    xv = _ref.bf16_to_float(x)
    cv, sv = _ref.bf16_to_float(c), _ref.bf16_to_float(s)
    for r, p in enumerate(pos):
        for h in range(2):
            for j in range(128):
                i = j % 64
                rot = -xv[r, h, j + 64] if j < 64 else xv[r, h, j - 64]
                a = _ref.rnd_bf16(Fraction(xv[r, h, j]) * Fraction(cv[p, i]))
                b = _ref.rnd_bf16(Fraction(rot) * Fraction(sv[p, i]))
                assert got[r, h, j] == _ref.bf16_bits(_ref.rnd_bf16(Fraction(a) + Fraction(b)))


def test_rope_relative_position_and_norm(orc):
    n = 40000
    c, s = orc.rope_table(THETA, 128, n)
    q = rand_bf16((1, 1, 128), 1.0, 18)
    k = rand_bf16((1, 1, 128), 1.0, 19)
    dots = []
    for base in (0, 1000, 31000):
        qr = _ref.bf16_to_float(orc.rope_apply(q, [base + 37], c, s))
        kr = _ref.bf16_to_float(orc.rope_apply(k, [base + 5], c, s))
        dots.append(float(np.dot(qr.ravel(), kr.ravel())))
        # pair norms are kept up to bf16 rounding of the products and the sum
        qv = _ref.bf16_to_float(q).ravel()
        nr = qr.ravel() ** 2
        pn = nr[:64] + nr[64:]
        p0 = qv[:64] ** 2 + qv[64:] ** 2
        assert np.allclose(pn, p0, rtol=0.03, atol=1e-3)
    # q.k depends on the offset only (up to rounding of the rotated bf16 vectors)
    assert max(dots) - min(dots) < 0.05 * (abs(dots[0]) + 1)
    # the rotation is really applied: a zero inv_freq would leave these equal
    assert not np.array_equal(orc.rope_apply(q, [1], c, s), q)


# ---- attention ----------------------------------------------------------------

def _attn_exact(q, pos, K, V, NKV):
    rows, NQ, D = q.shape
    G = NQ // NKV
    qv, Kv, Vv = _ref.bf16_to_float(q), _ref.bf16_to_float(K), _ref.bf16_to_float(V)
    out = np.zeros((rows, NQ * D), np.uint16)
    for r in range(rows):
        for h in range(NQ):
            g = h // G
            n = pos[r] + 1
            sc = [mpmath.mpf(float(np.dot(qv[r, h], Kv[t, g]))) / mpmath.sqrt(D) for t in range(n)]
            # np.dot of bf16 values in float64 is exact for D = 8..16 small ints; keep inputs small
            m = max(sc)
            e = [mpmath.exp(v - m) for v in sc]
            l = sum(e)
            for d in range(D):
                o = sum(e[t] * mpmath.mpf(Vv[t, g, d]) for t in range(n)) / l
                assert not _ref.near_tie_bf16(_ref.frac(o), 1e-13)
                out[r, h * D + d] = _ref.bf16_bits(_ref.rnd_bf16(_ref.frac(o)))
    return out


def test_attention_brute_force_gqa(orc):
    D, NQ, NKV, n = 8, 6, 2, 11
    q = _ref.f32_to_bf16_bits(np.random.default_rng(20).integers(-4, 5, (3, NQ, D)).astype(np.float32) / 4)
    K = _ref.f32_to_bf16_bits(np.random.default_rng(21).integers(-4, 5, (n, NKV, D)).astype(np.float32) / 4)
    V = rand_bf16((n, NKV, D), 1.0, 22)
    pos = np.array([0, 5, 10], np.int32)
    got = orc.attention(q, pos, K, V)
    assert np.array_equal(got, _attn_exact(q, pos, K, V, NKV))


def test_attention_single_key_returns_v(orc):
    q = rand_bf16((1, 4, 128), 1.0, 23)
    K = rand_bf16((1, 2, 128), 1.0, 24)
    V = rand_bf16((1, 2, 128), 1.0, 25)
    out = orc.attention(q, [0], K, V).reshape(4, 128)
    assert np.array_equal(out[0], V[0, 0]) and np.array_equal(out[1], V[0, 0])
    assert np.array_equal(out[2], V[0, 1]) and np.array_equal(out[3], V[0, 1])


def test_attention_equal_keys_give_mean_and_ones_give_one(orc):
    n, D = 37, 128
    q = rand_bf16((1, 1, D), 1.0, 26)
    K = np.repeat(rand_bf16((1, 1, D), 1.0, 27), n, axis=0)
    V = rand_bf16((n, 1, D), 1.0, 28)
    out = orc.attention(q, [n - 1], K, V)[0]
    Vv = _ref.bf16_to_float(V)
    want = [_ref.bf16_bits(_ref.rnd_bf16(sum(Fraction(Vv[t, 0, d]) for t in range(n)) / n)) for d in range(D)]
    assert np.array_equal(out, np.array(want, np.uint16))
    ones = np.full((n, 1, D), 0x3F80, np.uint16)
    Kr = rand_bf16((n, 1, D), 1.0, 29)
    assert np.all(orc.attention(q, [n - 1], Kr, ones) == 0x3F80)


def test_attention_two_keys_closed_form_scale(orc):
    # q.k0 = 0, q.k1 = s*sqrt(128) -> weights 1/(1+e^s), e^s/(1+e^s)
    D = 128
    q = np.zeros((1, 1, D), np.uint16); q[0, 0, 0] = _ref.bf16_bits(2.0)
    K = np.zeros((2, 1, D), np.uint16); K[1, 0, 0] = _ref.bf16_bits(4.0)   # q.k1 = 8
    V = np.zeros((2, 1, D), np.uint16); V[1, 0, 1] = 0x3F80               # v1 = e_1
    out = _ref.bf16_to_float(orc.attention(q, [1], K, V)[0])
    s = mpmath.mpf(8) / mpmath.sqrt(128)
    assert out[1] == _ref.rnd_bf16(_ref.frac(mpmath.exp(s) / (1 + mpmath.exp(s))))
    assert out[0] == 0.0


def test_attention_is_causal(orc):
    n = 20
    q = rand_bf16((2, 2, 128), 1.0, 30)
    K = rand_bf16((n, 1, 128), 1.0, 31)
    V = rand_bf16((n, 1, 128), 1.0, 32)
    a = orc.attention(q, [9, 12], K, V)
    K2, V2 = K.copy(), V.copy()
    K2[13:] = rand_bf16((n - 13, 1, 128), 5.0, 33)
    V2[13:] = rand_bf16((n - 13, 1, 128), 5.0, 34)
    b = orc.attention(q, [9, 12], K2, V2)
    assert np.array_equal(a, b)
    K2[12] = K2[13]
    assert not np.array_equal(orc.attention(q, [9, 12], K2, V2)[1], a[1])


def test_attention_head_to_kv_head_mapping(orc):
    # NQ = 4, NKV = 2: heads 0,1 read KV head 0; heads 2,3 read KV head 1 (h // 2, not h % 2)
    q = rand_bf16((1, 4, 128), 1.0, 35)
    K = rand_bf16((3, 2, 128), 1.0, 36)
    V = np.zeros((3, 2, 128), np.uint16)
    V[:, 0, :] = _ref.bf16_bits(1.0)
    V[:, 1, :] = _ref.bf16_bits(-2.0)
    out = _ref.bf16_to_float(orc.attention(q, [2], K, V)).reshape(4, 128)
    assert np.all(out[0] == 1.0) and np.all(out[1] == 1.0)
    assert np.all(out[2] == -2.0) and np.all(out[3] == -2.0)
    # MHA (NKV == NQ): each head its own
    V4 = np.zeros((3, 4, 128), np.uint16)
    for h in range(4):
        V4[:, h, :] = _ref.bf16_bits(float(h + 1))
    out = _ref.bf16_to_float(orc.attention(q, [2], rand_bf16((3, 4, 128), 1.0, 37), V4)).reshape(4, 128)
    assert [out[h, 0] for h in range(4)] == [1.0, 2.0, 3.0, 4.0]


# ---- SwiGLU -------------------------------------------------------------------

def test_swiglu_brute_force_and_limits(orc):
    g = rand_bf16(3000, 3.0, 40)
    u = rand_bf16(3000, 1.0, 41)
    got = orc.swiglu(g, u)
    gv, uv = _ref.bf16_to_float(g), _ref.bf16_to_float(u)
    for i in range(len(g)):
        sg = mpmath.mpf(gv[i]) / (1 + mpmath.exp(-mpmath.mpf(gv[i])))
        if _ref.near_tie_bf16(_ref.frac(sg), 1e-13):
            continue
        a = _ref.rnd_bf16(_ref.frac(sg))
        assert got[i] == _ref.bf16_bits(_ref.rnd_bf16(Fraction(a) * Fraction(uv[i]))), i
    z = orc.swiglu(np.zeros(4, np.uint16), rand_bf16(4, 1.0, 42))
    assert np.all((z & 0x7FFF) == 0)
    big = np.full(4, _ref.bf16_bits(64.0), np.uint16)
    uu = rand_bf16(4, 1.0, 43)
    assert np.array_equal(orc.swiglu(big, uu), orc.bf16_round(64.0 * _ref.bf16_to_float(uu)))


# ---- argmax -------------------------------------------------------------------

def test_argmax_brute_force_ties_and_nonfinite(orc):
    L = rand_bf16((5, 3000), 2.0, 50)
    ids, st = orc.argmax(L)
    assert st == 0
    Lv = _ref.bf16_to_float(L)
    for r in range(5):
        best = 0
        for i in range(3000):
            if Lv[r, i] > Lv[r, best]:
                best = i
        assert ids[r] == best
    # planted exact ties: the lower id wins
    L2 = L.copy()
    L2[0, 100] = L2[0, 2000] = _ref.bf16_bits(64.0)
    L2[1, 7] = L2[1, 6] = _ref.bf16_bits(64.0)
    ids, st = orc.argmax(L2)
    assert st == 0 and ids[0] == 100 and ids[1] == 6
    # planted non-finite values off the winner, and on it
    for bad in (0x7FC0, 0x7F80, 0xFF80):
        L3 = L2.copy()
        L3[2, 2999] = bad
        ids, st = orc.argmax(L3)
        assert st == -1 and ids[2] == -1 and ids[0] == 100
