"""Pins of the oracle's block-scaled GEMV and of the per-row activation
quantisation used by the MMA path (CPU only)."""
from fractions import Fraction

import numpy as np
import pytest

from nvfp4_block_scaled_aq_gb300 import inputs
from test_oracle_formats import e2m1_table, e4m3_values_by_enumeration
from test_oracle_method import bf16_of, f32_of, unpack

E2M1 = {c: Fraction(v) for c, v in e2m1_table().items()}
E4M3 = e4m3_values_by_enumeration()


def exact_w_hat(packed, scales, g_dec):
    """Dequantised weight as exact Fractions, decoded with the test's own
    tables: w_hat = e2m1(q) * sd * g_dec."""
    q = unpack(packed)
    n, k = q.shape
    g = Fraction(float(g_dec))
    return [[E2M1[int(q[i, j])] * E4M3[int(scales[i, j // 16])] * g
             for j in range(k)] for i in range(n)]


def test_gemv_matches_exact_rational_sum(oracle_mod):
    """Brute force on a tiny problem: the exact sum of x * w_hat in rational
    arithmetic; the oracle's fp64 sum must agree to fp64 rounding."""
    n, k, m = 5, 48, 3
    W = inputs.bits_u16(inputs.weight(n, k, seed=21))
    x = inputs.bits_u16(inputs.tokens(m, k, seed=22))
    packed, scales, ge, gd = oracle_mod.quantize(W)
    y = oracle_mod.gemv(packed, scales, gd, x)
    wh = exact_w_hat(packed, scales, gd)
    xf = f32_of(x)
    for t in range(m):
        for i in range(n):
            ex = sum(Fraction(float(xf[t, j])) * wh[i][j] for j in range(k))
            scale = sum(abs(Fraction(float(xf[t, j])) * wh[i][j]) for j in range(k))
            assert abs(Fraction(y[t, i]) - ex) <= scale * Fraction(1, 2 ** 50)


def test_gemv_one_hot_returns_a_column(oracle_mod):
    n, k = 24, 64
    W = inputs.bits_u16(inputs.weight(n, k, seed=23))
    packed, scales, ge, gd = oracle_mod.quantize(W)
    wh = exact_w_hat(packed, scales, gd)
    for col in (0, 1, 15, 16, 63):
        x = np.zeros((1, k), np.uint16)
        x[0, col] = bf16_of([1.0])[0]
        y = oracle_mod.gemv(packed, scales, gd, x)[0]
        for i in range(n):
            assert Fraction(y[i]) == wh[i][col]


def test_gemv_constant_blocks_closed_form(oracle_mod):
    """x = 1 and every block constant: y = sum over blocks of 16*e2m1*sd*g_dec.
    With g_enc chosen so each block scale is exact, a block of value c
    quantises to code 6 (value 6) with sd = c/6*g_enc."""
    k = 64
    vals = np.array([[0.75, -1.5, 3.0, 0.375], [6.0, 6.0, -6.0, 1.5]])
    W = np.repeat(vals, 16, axis=1)
    packed, scales, ge, gd = oracle_mod.quantize(bf16_of(W))
    assert ge == 448.0  # amax 6
    x = np.tile(bf16_of([1.0]), (1, k))
    y = oracle_mod.gemv(packed, scales, gd, x)[0]
    # block c: t = c/6*448 is an exact E4M3 value, r = 448/t = 6/c, code 6,
    # so w_hat = 6 * (448 c / 6) * g_dec = 448 c g_dec (g_dec = fp32(6/2688))
    closed = 16.0 * 448.0 * float(gd) * vals.sum(axis=1)
    assert np.allclose(y, closed, rtol=1e-14, atol=0)


def test_gemv_rows_subset_and_m_invariance(oracle_mod):
    n, k, m = 40, 160, 5
    W = inputs.bits_u16(inputs.weight(n, k, seed=24))
    x = inputs.bits_u16(inputs.tokens(m, k, seed=25))
    packed, scales, ge, gd = oracle_mod.quantize(W)
    full = oracle_mod.gemv(packed, scales, gd, x)
    for t in range(m):
        assert np.array_equal(oracle_mod.gemv(packed, scales, gd, x[t:t + 1])[0], full[t])
    rows = np.array([39, 0, 7, 7, 20])
    assert np.array_equal(oracle_mod.gemv(packed, scales, gd, x, rows=rows),
                          full[:, rows])


def test_fused_equals_separate_when_scales_agree(oracle_mod):
    """Row-concatenating two weights (QKV or gate+up fusion) gives the
    concatenated outputs when both parts share one per-tensor scale: the
    quantisation of a row depends only on that row and g_enc."""
    k = 96
    A = inputs.bits_u16(inputs.weight(12, k, seed=26))
    B = inputs.bits_u16(inputs.weight(20, k, seed=27))
    F = np.concatenate([A, B])
    pf, sf, ge, gd = oracle_mod.quantize(F)
    pa, sa = oracle_mod.quantize_rows(A, ge)
    pb, sb = oracle_mod.quantize_rows(B, ge)
    assert np.array_equal(pf, np.concatenate([pa, pb]))
    assert np.array_equal(sf, np.concatenate([sa, sb]))


# --------------------------------------------------------- activations (R9)

def test_act_quant_is_per_row_weight_quant(oracle_mod):
    m, k = 4, 128
    x = inputs.bits_u16(inputs.tokens(m, k, seed=28))
    x[2] = bf16_of(np.linspace(-3, 3, k))
    xp, xs, xg = oracle_mod.quantize_act(x)
    for t in range(m):
        p, s, ge, gd = oracle_mod.quantize(x[t:t + 1])
        assert np.array_equal(xp[t], p[0]) and np.array_equal(xs[t], s[0])
        assert xg[t] == np.float32(gd)


def test_gemv_q_matches_exact_rational_sum(oracle_mod):
    n, k, m = 6, 64, 2
    W = inputs.bits_u16(inputs.weight(n, k, seed=29))
    x = inputs.bits_u16(inputs.tokens(m, k, seed=30))
    wp, ws, wge, wgd = oracle_mod.quantize(W)
    xp, xs, xg = oracle_mod.quantize_act(x)
    y = oracle_mod.gemv_q(wp, ws, wgd, xp, xs, xg)
    wh = exact_w_hat(wp, ws, wgd)
    for t in range(m):
        xh = exact_w_hat(xp[t:t + 1], xs[t:t + 1], xg[t])[0]
        for i in range(n):
            ex = sum(a * b for a, b in zip(xh, wh[i]))
            scale = sum(abs(a * b) for a, b in zip(xh, wh[i]))
            assert abs(Fraction(y[t, i]) - ex) <= scale * Fraction(1, 2 ** 50)


# ------------------------------------------------------------ bf16 GEMV pins

def test_gemv_bf16_matches_exact_rational_sum(oracle_mod):
    """Brute force on a tiny problem: the exact rational sum of x * w over
    bf16 values; the oracle's fp64 sum agrees to fp64 rounding."""
    n, k, m = 6, 40, 3
    W = inputs.bits_u16(inputs.weight(n, k, seed=61))
    x = inputs.bits_u16(inputs.tokens(m, k, seed=62))
    y = oracle_mod.gemv_bf16(W, x)
    wf, xf = f32_of(W), f32_of(x)
    for t in range(m):
        for i in range(n):
            terms = [Fraction(float(xf[t, j])) * Fraction(float(wf[i, j])) for j in range(k)]
            ex, scale = sum(terms), sum(abs(v) for v in terms)
            assert abs(Fraction(y[t, i]) - ex) <= scale * Fraction(1, 2 ** 50)


def test_gemv_bf16_one_hot_and_rows(oracle_mod):
    """A one-hot token returns the weight column exactly; `rows` selects rows."""
    n, k = 9, 24
    W = inputs.bits_u16(inputs.weight(n, k, seed=63))
    wf = f32_of(W)
    for col in (0, 7, 23):
        x = np.zeros((1, k), np.uint16)
        x[0, col] = bf16_of([1.0])[0]
        assert np.array_equal(oracle_mod.gemv_bf16(W, x)[0], wf[:, col].astype(np.float64))
    x = inputs.bits_u16(inputs.tokens(2, k, seed=64))
    rows = np.array([8, 0, 3])
    assert np.array_equal(oracle_mod.gemv_bf16(W, x, rows=rows), oracle_mod.gemv_bf16(W, x)[:, rows])


def test_gemv_bf16_is_the_matrix_product_of_the_decoded_values(oracle_mod):
    """Against numpy's fp64 matrix product of the decoded bf16 values (an
    independent summation): equal within the fp64 rounding of two orders."""
    n, k, m = 33, 200, 4
    W = inputs.bits_u16(inputs.weight(n, k, seed=65))
    x = inputs.bits_u16(inputs.tokens(m, k, seed=66))
    ref = f32_of(x).astype(np.float64) @ f32_of(W).astype(np.float64).T
    bound = (np.abs(f32_of(x)).astype(np.float64) @ np.abs(f32_of(W)).astype(np.float64).T) * 2e-15
    assert np.all(np.abs(oracle_mod.gemv_bf16(W, x) - ref) <= bound)
    # a transposed operand or a dropped term would not survive this
    assert not np.allclose(oracle_mod.gemv_bf16(W[:, ::-1].copy(), x), ref)


# ------------------------------------------------------- runtime low-rank pins

def lowrank_case(n, k, r, seed):
    W0 = inputs.bits_u16(inputs.weight(n, k, seed=seed))
    g = np.random.default_rng(seed)
    s = np.exp(0.1 * g.standard_normal(n)).astype(np.float32)
    U = inputs.bits_u16(inputs.weight(n, max(r, 1), seed=seed + 1, outliers=False))[:, :r]
    V = inputs.bits_u16(inputs.weight(k, max(r, 1), seed=seed + 2, outliers=False))[:, :r]
    return W0, s, U, V


def test_lowrank_matches_exact_rational_sum(oracle_mod):
    """Brute force: s*(x . w0_hat) + sum_r U[i,r] (V[:,r] . x) in rationals."""
    n, k, r, m = 4, 32, 3, 2
    W0, s, U, V = lowrank_case(n, k, r, 70)
    x = inputs.bits_u16(inputs.tokens(m, k, seed=71))
    packed, scales, ge, gd = oracle_mod.quantize(W0)
    y = oracle_mod.gemv_lowrank(packed, scales, gd, s, U, V, x)
    wh = exact_w_hat(packed, scales, gd)
    xf, uf, vf = f32_of(x), f32_of(U), f32_of(V)
    for t in range(m):
        X = [Fraction(float(xf[t, j])) for j in range(k)]
        proj = [sum(Fraction(float(vf[j, q])) * X[j] for j in range(k)) for q in range(r)]
        for i in range(n):
            base = sum(X[j] * wh[i][j] for j in range(k))
            ex = Fraction(float(s[i])) * base + sum(Fraction(float(uf[i, q])) * proj[q] for q in range(r))
            scale = abs(Fraction(float(s[i]))) * sum(abs(X[j] * wh[i][j]) for j in range(k)) + \
                sum(abs(Fraction(float(uf[i, q]))) * sum(abs(Fraction(float(vf[j, q])) * X[j])
                                                        for j in range(k)) for q in range(r))
            assert abs(Fraction(y[t, i]) - ex) <= scale * Fraction(1, 2 ** 48)


def test_lowrank_without_delta_is_the_scaled_gemv(oracle_mod):
    """r = 0: s = 1 gives the block GEMV bit for bit, s = 2^j scales it exactly."""
    n, k = 20, 96
    W0, s, U, V = lowrank_case(n, k, 0, 72)
    x = inputs.bits_u16(inputs.tokens(3, k, seed=73))
    packed, scales, ge, gd = oracle_mod.quantize(W0)
    plain = oracle_mod.gemv(packed, scales, gd, x)
    ones = np.ones(n, np.float32)
    assert np.array_equal(oracle_mod.gemv_lowrank(packed, scales, gd, ones, None, None, x), plain)
    pow2 = np.float32(2.0) ** np.arange(-3, n - 3, dtype=np.float32)
    assert np.array_equal(oracle_mod.gemv_lowrank(packed, scales, gd, pow2, None, None, x),
                          plain * pow2.astype(np.float64))


def test_lowrank_with_zero_block_is_the_rank_r_product(oracle_mod):
    """W0 = 0 quantises to all-zero nibbles: only (x V) U^T remains (checked
    against numpy's fp64 products, an independent summation)."""
    n, k, r = 24, 128, 4
    _, s, U, V = lowrank_case(n, k, r, 74)
    W0 = np.zeros((n, k), np.uint16)
    x = inputs.bits_u16(inputs.tokens(2, k, seed=75))
    packed, scales, ge, gd = oracle_mod.quantize(W0)
    y = oracle_mod.gemv_lowrank(packed, scales, gd, s, U, V, x)
    ref = (f32_of(x).astype(np.float64) @ f32_of(V).astype(np.float64)) @ f32_of(U).astype(np.float64).T
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)
    # U and V swapped roles (a transposed operand) would not agree
    assert not np.allclose(y, (f32_of(x).astype(np.float64) @ f32_of(V).astype(np.float64))
                           @ f32_of(U).astype(np.float64)[::-1].T)


# ------------------------------------------------- fused gate+up activation

def test_gelu_tanh_identities(oracle_mod):
    """gelu(z) - gelu(-z) = z (the tanh form is odd around z/2); gelu(0) = 0;
    within the tanh form's known distance (< 1e-3) of the exact z*Phi(z)."""
    import math
    assert oracle_mod.gelu_tanh(0.0) == 0.0
    for z in (-6.0, -3.1, -1.0, -0.25, 0.5, 1.0, 2.2, 5.0, 9.0):
        assert abs(oracle_mod.gelu_tanh(z) - oracle_mod.gelu_tanh(-z) - z) <= 1e-15 * max(1, abs(z))
        exact = 0.5 * z * (1.0 + math.erf(z / math.sqrt(2.0)))
        assert abs(oracle_mod.gelu_tanh(z) - exact) < 1e-3
    assert abs(oracle_mod.gelu_tanh(12.0) - 12.0) < 1e-12


def test_interleave_is_a_row_permutation(oracle_mod):
    f, k = 24, 16
    W = np.arange(2 * f * k, dtype=np.uint16).reshape(2 * f, k)
    Wi = oracle_mod.interleave_gate_up(W)
    assert sorted(Wi[:, 0].tolist()) == sorted(W[:, 0].tolist())
    for j in range(f):
        g, i = divmod(j, 8)
        assert np.array_equal(Wi[16 * g + i], W[j])          # gate row j
        assert np.array_equal(Wi[16 * g + 8 + i], W[f + j])  # up row j


def test_glu_is_gelu_of_gate_times_up(oracle_mod):
    """The fused form against the two plain GEMV rows of each column, with
    the activation from the erf definition (error bound of the tanh form)."""
    import math
    f, k, m = 32, 96, 2
    Wcat = inputs.bits_u16(inputs.weight(2 * f, k, seed=81))
    Wi = oracle_mod.interleave_gate_up(Wcat)
    x = inputs.bits_u16(inputs.tokens(m, k, seed=82))
    packed, scales, ge, gd = oracle_mod.quantize(Wi)
    h = oracle_mod.gemv_glu(packed, scales, gd, x)
    # the interleaved tensor's quantised rows are the concatenated tensor's
    pc, sc, gec, gdc = oracle_mod.quantize(Wcat)
    assert gd == gdc and np.array_equal(oracle_mod.interleave_gate_up(pc), packed)
    y = oracle_mod.gemv(pc, sc, gdc, x)   # [m, 2f] in concatenated order
    for t in range(m):
        for j in range(f):
            g, u = y[t, j], y[t, f + j]
            exact = 0.5 * g * (1.0 + math.erf(g / math.sqrt(2.0))) * u
            assert abs(h[t, j] - exact) <= 1e-3 * abs(u) + 1e-15
    cols = np.array([31, 0, 9])
    assert np.array_equal(oracle_mod.gemv_glu(packed, scales, gd, x, cols=cols), h[:, cols])


# ------------------------------------------------------ per-segment scales

def test_segments_compose_the_single_tensor_functions(oracle_mod):
    """One segment is the plain quantisation and GEMV; a segment that is an
    exact power-of-two multiple of another quantises to the same bytes with
    g_dec scaled by that power (the per-tensor scale follows its segment)."""
    n1, k = 32, 96
    A = inputs.bits_u16(inputs.weight(n1, k, seed=91))
    p1, s1, ge1, gd1 = oracle_mod.quantize(A)
    p, s, gd = oracle_mod.quantize_segments(A, [n1])
    assert np.array_equal(p, p1) and np.array_equal(s, s1) and gd[0] == np.float32(gd1)
    x = inputs.bits_u16(inputs.tokens(2, k, seed=92))
    assert np.array_equal(oracle_mod.gemv_segments(p, s, gd, [n1], x),
                          oracle_mod.gemv(p1, s1, gd1, x))
    B = bf16_of(f32_of(A) * np.float32(1024.0))   # exact: a power of two
    W = np.concatenate([A, B])
    p2, s2, gd2 = oracle_mod.quantize_segments(W, [n1, 2 * n1])
    assert np.array_equal(p2[:n1], p2[n1:]) and np.array_equal(s2[:n1], s2[n1:])
    assert gd2[1] == gd2[0] * np.float32(1024.0)
    # under one scale for the whole tensor the small segment's block scales
    # sit 2^10 lower in the E4M3 range (fewer bits left for it)
    pw, sw, gew, gdw = oracle_mod.quantize(W)
    assert np.array_equal(sw[n1:], s2[n1:]) and not np.array_equal(sw[:n1], s2[:n1])
