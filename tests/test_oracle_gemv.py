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
