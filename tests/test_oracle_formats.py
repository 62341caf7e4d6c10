"""Pins of the oracle's number formats against what the format definitions
and the pages fix (CPU only).

Each encoder is checked against a brute-force nearest-value search over the
finite value set -- a different method from the oracle's exponent/mantissa
decomposition -- so a wrong exponent bias, a dropped subnormal range, a
wrong tie rule or a lost sign fails here.
"""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def load_pairs(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


# -------------------------------------------------------- independent tables

def e2m1_table():
    """nibble -> value, from the golden grid file."""
    return {int(a, 16): float(b) for a, b in load_pairs("e2m1_grid.txt")}


def e4m3_values_by_enumeration():
    """code -> Fraction for every finite non-negative float8_e4m3fn code,
    built by walking the grid: 8 subnormal steps of 2^-9, then each binade
    [2^e, 2^(e+1)) for e = -6..8 split into 8 equal steps, stopping at 448."""
    vals = {}
    code = 0
    for m in range(8):                      # subnormals 0 .. 7 * 2^-9
        vals[code] = Fraction(m, 512)
        code += 1
    e = -6
    while code < 0x7F:
        base = Fraction(2) ** e
        for m in range(8):
            if code == 0x7F:
                break
            vals[code] = base + base * Fraction(m, 8)
            code += 1
        e += 1
    return vals


def nearest_even(x, table, even_of):
    """Brute force: the table entry nearest to x; on a tie the one whose
    code is even-mantissa (even_of(code) True)."""
    best = None
    for code, v in table.items():
        d = abs(x - v)
        if best is None or d < best[0] or (d == best[0] and even_of(code)
                                           and not even_of(best[1])):
            best = (d, code)
    return best[1]


# ------------------------------------------------------------------- E2M1

def test_e2m1_decode_matches_golden_grid(oracle_mod):
    tab = e2m1_table()
    codes = np.arange(16, dtype=np.uint8)
    got = oracle_mod.e2m1_decode(codes)
    for c in range(16):
        assert got[c] == tab[c]
        assert np.signbit(got[c]) == (c >= 8)  # 0x8 is -0


def test_e2m1_ties_golden(oracle_mod):
    for x, want in load_pairs("e2m1_ties.txt"):
        got = int(oracle_mod.e2m1_encode(np.array([float(x)], np.float32))[0])
        assert got == int(want, 16), (x, hex(got), want)


def _e2m1_brute(x):
    pos = {c: Fraction(v) for c, v in e2m1_table().items() if c < 8}
    a = abs(Fraction(float(x)))
    if a >= 6:
        mag = 7
    else:
        mag = nearest_even(a, pos, even_of=lambda c: c % 2 == 0)
    return mag | (8 if np.signbit(np.float32(x)) else 0)


def test_e2m1_encode_bruteforce_sweep(oracle_mod):
    # every multiple of 2^-8 in [-8, 8] (covers all midpoints exactly), the
    # fp32 neighbours of each midpoint, and random values
    grid = np.arange(-8 * 256, 8 * 256 + 1, dtype=np.float64) / 256.0
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)
    mids = np.concatenate([mids, -mids])
    nbrs = np.concatenate([np.nextafter(mids, np.float32(np.inf)),
                           np.nextafter(mids, np.float32(-np.inf))])
    rnd = np.random.default_rng(1).normal(0, 3, 4000).astype(np.float32)
    xs = np.concatenate([grid.astype(np.float32), mids, nbrs, rnd,
                         np.array([-0.0, 0.0, 1e30, -1e30, 1e-30], np.float32)])
    got = oracle_mod.e2m1_encode(xs)
    for x, g in zip(xs.tolist(), got.tolist()):
        assert g == _e2m1_brute(np.float32(x)), (x, g)


# ------------------------------------------------------------------- E4M3

def test_e4m3_decode_golden_points(oracle_mod):
    for code, val in load_pairs("e4m3_points.txt"):
        got = float(oracle_mod.e4m3_decode(np.array([int(code, 16)], np.uint8))[0])
        if val == "nan":
            assert np.isnan(got)
        else:
            assert got == float(val), (code, got, val)
            assert np.signbit(got) == val.startswith("-")


def test_e4m3_decode_matches_enumeration(oracle_mod):
    tab = e4m3_values_by_enumeration()
    assert len(tab) == 127 and tab[0x7E] == 448
    codes = np.arange(0x7F, dtype=np.uint8)
    got = oracle_mod.e4m3_decode(codes)
    for c in range(0x7F):
        assert Fraction(float(got[c])) == tab[c]
    neg = oracle_mod.e4m3_decode(codes | 0x80)
    assert np.array_equal(neg, -got)


def _e4m3_brute(t, tab):
    if t >= 448:
        return 0x7E
    return nearest_even(t, tab, even_of=lambda c: c % 2 == 0)


def test_e4m3_encode_bruteforce_sweep(oracle_mod):
    tab = e4m3_values_by_enumeration()
    vals = sorted(tab.values())
    mids = [(a + b) / 2 for a, b in zip(vals[:-1], vals[1:])]
    xs = [float(v) for v in vals] + [float(m) for m in mids]
    xs32 = np.array(xs, np.float32)
    xs32 = np.concatenate([
        xs32, np.nextafter(xs32, np.float32(np.inf)),
        np.nextafter(xs32, np.float32(0)),
        np.random.default_rng(2).uniform(0, 460, 3000).astype(np.float32),
        np.exp2(np.random.default_rng(3).uniform(-14, 9, 3000)).astype(np.float32),
        np.array([448.0, 449.0, 464.0, 1e9, 2.0 ** -10, 2.0 ** -11, 0.0],
                 np.float32)])
    got = oracle_mod.e4m3_encode(xs32)
    for x, g in zip(xs32.tolist(), got.tolist()):
        assert g == _e4m3_brute(Fraction(x), tab), (x, hex(g))
    # the midpoints are exactly representable in fp32: ties go to even codes
    for m in mids:
        g = int(oracle_mod.e4m3_encode(np.array([float(m)], np.float32))[0])
        assert g % 2 == 0
    # sign is kept; NaN maps to the NaN code
    assert oracle_mod.e4m3_encode(np.array([-1.0], np.float32))[0] == 0xB8
    assert oracle_mod.e4m3_encode(np.array([np.nan], np.float32))[0] == 0x7F


# ------------------------------------------------------------------- bf16

def test_bf16_rounding_matches_torch(oracle_mod):
    rng = np.random.default_rng(4)
    bits = rng.integers(0, 2 ** 32, 200000, dtype=np.uint64).astype(np.uint32)
    # plant exact halfway cases (low 16 bits = 0x8000) and near-halfway ones
    bits[:20000] = (bits[:20000] & 0xFFFF0000) | 0x8000
    bits[20000:40000] = (bits[20000:40000] & 0xFFFF0000) | 0x7FFF
    f = bits.view(np.float32)
    f = f[np.isfinite(f)]
    got = oracle_mod.f32_to_bf16_bits(f)
    want = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16)
    want = want.numpy().view(np.uint16)
    assert np.array_equal(got, want)


def test_bf16_to_f32_is_exact_widening(oracle_mod):
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f = oracle_mod.bf16_bits_to_f32(allbits)
    t = torch.from_numpy(allbits.view(np.int16).copy()).view(torch.bfloat16)
    want = t.to(torch.float32).numpy()
    same = (f.view(np.uint32) == want.view(np.uint32)) | (np.isnan(f) & np.isnan(want))
    assert same.all()
    fin = np.isfinite(f)
    back = oracle_mod.f32_to_bf16_bits(f[fin])
    assert np.array_equal(back, allbits[fin])
