"""Pins of the oracle's method steps (CPU only): reconstruction, per-tensor
scale, block quantisation, packing and the device scale layout.

Each check rests on something other than the oracle itself: the pages'
passthrough invariant, exact closed forms, torch's bf16 rounding (a library
routine), brute-force nearest-value searches, hand-worked layout offsets,
or the format's error bound.
"""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from nvfp4_block_scaled_aq_gb300 import inputs
from test_oracle_formats import (e2m1_table, e4m3_values_by_enumeration,
                                 load_pairs, nearest_even)


def bf16_of(values):
    """bf16 bit patterns of fp32/fp64 values via torch (round-to-nearest-even)."""
    t = torch.as_tensor(np.asarray(values, dtype=np.float64)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def f32_of(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


# ------------------------------------------------------------ reconstruct

def test_reconstruct_passthrough_every_bf16_pattern(oracle_mod):
    """AttnQuant docs, "Throughput", "Where the throughput comes from": at the
    passthrough setting the decomposition reconstructs the original weight
    bit-for-bit.  s = 1, U = V = 0 must return every non-NaN bf16 pattern,
    -0 and +-inf included, unchanged."""
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    allbits = allbits[~np.isnan(f32_of(allbits))]
    n, k = 8, allbits.size // 8
    W0 = allbits[: n * k].reshape(n, k)
    out = oracle_mod.reconstruct(W0, np.ones(n, np.float32),
                                 np.zeros((n, 4), np.uint16),
                                 np.zeros((k, 4), np.uint16))
    assert np.array_equal(out, W0)


def test_reconstruct_power_of_two_scale_is_exact(oracle_mod):
    rng = np.random.default_rng(5)
    W0 = bf16_of(rng.normal(0, 0.02, (16, 48)))
    for j in (-3, -1, 1, 4):
        s = np.full(16, 2.0 ** j, np.float32)
        out = oracle_mod.reconstruct(W0, s, np.zeros((16, 2), np.uint16),
                                     np.zeros((48, 2), np.uint16))
        assert np.array_equal(out, bf16_of(f32_of(W0).astype(np.float64) * 2.0 ** j))


def test_reconstruct_exact_integer_case(oracle_mod):
    """Small integers make every fp32 step exact, so the result is the exact
    s*W0 + U V^T rounded once to bf16.  n != k and r = 3 with distinct
    entries catch a transposed V, a swapped U/V or a dropped rank term."""
    rng = np.random.default_rng(6)
    n, k, r = 5, 7, 3
    W0i = rng.integers(-20, 21, (n, k))
    si = rng.integers(-4, 5, n)
    Ui = rng.integers(-9, 10, (n, r))
    Vi = rng.integers(-9, 10, (k, r))
    exact = si[:, None] * W0i + Ui @ Vi.T
    out = oracle_mod.reconstruct(bf16_of(W0i), si.astype(np.float32),
                                 bf16_of(Ui), bf16_of(Vi))
    assert np.array_equal(out, bf16_of(exact))


def test_reconstruct_random_within_one_rounding(oracle_mod):
    """Realistic theta: the oracle's W_eff is the exact value rounded to bf16
    except where fp32 double rounding moves a halfway case, so it is within
    one bf16 ulp everywhere and equal almost everywhere."""
    th = inputs.theta(64, 160, 4, seed=11)
    W0, U, V = (inputs.bits_u16(t) for t in (th.W0, th.U, th.V))
    s = th.s.numpy()
    out = oracle_mod.reconstruct(W0, s, U, V)
    exact = (s.astype(np.float64)[:, None] * f32_of(W0)
             + f32_of(U).astype(np.float64) @ f32_of(V).astype(np.float64).T)
    ref = bf16_of(exact)
    diff = np.abs(out.astype(np.int32) - ref.astype(np.int32))
    assert diff.max() <= 1
    assert (diff == 0).mean() > 0.999


# ----------------------------------------------------------- global scale

def test_amax_matches_numpy(oracle_mod):
    W = inputs.bits_u16(inputs.weight(33, 96, seed=3))
    assert oracle_mod.amax(W) == np.abs(f32_of(W)).max()
    W[5, 7] = 0x7FC0  # NaN
    assert np.isnan(oracle_mod.amax(W))


def test_global_scale_closed_forms(oracle_mod):
    assert oracle_mod.global_scales(2688.0) == (1.0, 1.0)
    assert oracle_mod.global_scales(0.0) == (1.0, 1.0)
    ge, gd = oracle_mod.global_scales(6.0)
    assert ge == 448.0 and gd == np.float32(6.0 / 2688.0)
    for bad in (np.inf, np.nan, -1.0, 1e-45):
        with pytest.raises(oracle_mod.OracleRangeError):
            oracle_mod.global_scales(bad)


# --------------------------------------------------------------- quantise

E2M1_POS = {c: Fraction(v) for c, v in e2m1_table().items() if c < 8}
E4M3 = e4m3_values_by_enumeration()


def brute_block(ws, g_enc):
    """One block by the definition, with the two encoders replaced by
    nearest-value searches over the value sets."""
    f = np.float32
    b = max(abs(f(w)) for w in ws)
    t = f(f(b) / f(6.0)) * f(g_enc)
    sf = 0x7E if t >= 448 else nearest_even(Fraction(float(t)), E4M3,
                                            lambda c: c % 2 == 0)
    sd = f(float(E4M3[sf]))
    if sd == 0:
        return sf, [0] * 16
    r = f(f(g_enc) / sd)
    q = []
    for w in ws:
        v = f(f(w) * r)
        a = abs(Fraction(float(v)))
        mag = 7 if a >= 6 else nearest_even(a, E2M1_POS, lambda c: c % 2 == 0)
        q.append(mag | (8 if np.signbit(v) else 0))
    return sf, q


def unpack(packed):
    lo = packed & 0xF
    hi = packed >> 4
    out = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,), np.uint8)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    return out


def nearest_even_vec(x, values, codes):
    """Vectorised brute force over a value table: for each x (fp32, >= 0)
    the code of the nearest value, ties to the even code.  Distances are
    taken in float64, where x and every table value are exact, so a tie is
    detected exactly."""
    d = np.abs(x.astype(np.float64)[:, None] - values[None, :])
    best = d.min(axis=1, keepdims=True)
    cand = d == best
    even = (codes % 2 == 0)[None, :]
    pick_even = cand & even
    use = np.where(pick_even.any(axis=1, keepdims=True), pick_even, cand)
    return codes[use.argmax(axis=1)]


E2M1_VALUES = np.array([float(E2M1_POS[c]) for c in range(8)])
E4M3_VALUES = np.array([float(E4M3[c]) for c in range(0x7F)])


def brute_blocks(blocks_f32, g_enc):
    """The block definition over many blocks at once, the two encoders
    replaced by the vectorised nearest-value search."""
    f = np.float32
    b = np.abs(blocks_f32).max(axis=1)
    t = (b / f(6.0)).astype(np.float32) * f(g_enc)
    sf = nearest_even_vec(np.minimum(t, f(448.0)), E4M3_VALUES,
                          np.arange(0x7F))
    sd = E4M3_VALUES[sf].astype(np.float32)
    r = np.where(sd == 0, f(0), f(g_enc) / np.where(sd == 0, f(1), sd))
    v = (blocks_f32 * r[:, None].astype(np.float32)).astype(np.float32)
    a = np.minimum(np.abs(v), f(6.0)).reshape(-1)
    mag = nearest_even_vec(a, E2M1_VALUES, np.arange(8)).reshape(v.shape)
    q = mag | np.where(np.signbit(v), 8, 0)
    q[sd == 0] = 0
    return sf, q


@pytest.mark.parametrize("g_enc", [2688.0, 1.0, 3.0e-3, 7.5e5])
def test_quantize_sweeps_every_bf16_value(oracle_mod, g_enc):
    """Every finite bf16 value of magnitude <= 1 sits in a block whose
    maximum is 1.0 (element 0), so it is quantised against a fixed scale;
    g_enc moves that scale through the normal, subnormal and saturated E4M3
    ranges.  Every element of every block is compared with the brute force;
    a seeded sample also goes through the scalar Fraction search."""
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = f32_of(allbits)
    allbits = allbits[np.isfinite(vals) & (np.abs(vals) <= 1.0)]
    per = 15
    nblk = -(-allbits.size // (per * 8)) * 8
    pad = np.zeros(nblk * per, np.uint16)
    pad[: allbits.size] = allbits
    blocks = np.concatenate([np.full((nblk, 1), 0x3F80, np.uint16),
                             pad.reshape(nblk, per)], axis=1)
    rows = blocks.reshape(-1, 16 * 8)
    packed, scales = oracle_mod.quantize_rows(rows, g_enc)
    q = unpack(packed).reshape(-1, 16)
    sc = scales.reshape(-1)
    sf, qb = brute_blocks(f32_of(blocks), g_enc)
    assert np.array_equal(sc, sf)
    assert np.array_equal(q, qb)
    for bi in np.random.default_rng(7).choice(nblk, 40, replace=False):
        sf1, q1 = brute_block(f32_of(blocks[bi]), g_enc)
        assert sc[bi] == sf1 and list(q[bi]) == q1


def test_quantize_all_bf16_magnitudes_one_block_each(oracle_mod):
    """Every finite bf16 value as the sole nonzero of its own block, with
    g_enc = 1: its scale and nibble follow the brute-force definition.  The
    block scale of a lone value w is E4M3(|w|/6) and its code is E2M1 of
    w * (1/sd), about +-6 whenever sd is a normal E4M3 value."""
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = f32_of(allbits)
    allbits = allbits[np.isfinite(vals)]
    blocks = np.zeros((allbits.size, 16), np.uint16)
    blocks[:, 3] = allbits
    packed, scales = oracle_mod.quantize_rows(blocks, 1.0)
    sf, qb = brute_blocks(f32_of(blocks), 1.0)
    assert np.array_equal(scales[:, 0], sf)
    assert np.array_equal(unpack(packed), qb)


def test_packing_order_low_nibble_is_even_element(oracle_mod):
    """Reading R6: byte i holds element 2i in its low nibble."""
    w = np.zeros((1, 32), np.float32)
    w[0, 0], w[0, 1] = 6.0, 0.5     # codes 0x7 and 0x1 at g_enc = 448/6 * 6
    w[0, 2], w[0, 3] = -1.0, 3.0    # codes 0xA and 0x5
    w[0, 16] = -6.0                 # second block: its max, code 0xF
    packed, scales = oracle_mod.quantize_rows(bf16_of(w), 448.0)
    # block 0: b = 6, t = 6/6*448 = 448 -> sd 448, r = 1 -> codes are exact
    assert scales[0, 0] == 0x7E and scales[0, 1] == 0x7E
    assert packed[0, 0] == 0x17 and packed[0, 1] == 0x5A
    assert packed[0, 8] == 0x0F


def test_zero_block_and_signed_zero(oracle_mod):
    """Reading R4: a zero scale zeroes its block (even -0); reading R5: in a
    nonzero block -0 and tiny negatives keep the sign (nibble 0x8)."""
    w = np.zeros((1, 32), np.float32)
    w[0, 1] = -0.0
    w[0, 16], w[0, 17], w[0, 18] = 1.0, -0.0, -1e-4
    packed, scales = oracle_mod.quantize_rows(bf16_of(w), 2688.0)
    q = unpack(packed)[0]
    assert scales[0, 0] == 0 and not q[:16].any()
    assert q[16] == 0x7 and q[17] == 0x8 and q[18] == 0x8


def test_quantize_error_bound(oracle_mod):
    """Round-to-nearest on the E2M1 grid: every element whose scaled value
    is inside the grid is within half a local grid step (times sd * g_dec)
    of the original; saturated ones are within the E4M3 rounding of the
    block scale."""
    W = inputs.bits_u16(inputs.weight(48, 256, seed=8))
    packed, scales, ge, gd = oracle_mod.quantize(W)
    wh = (oracle_mod.e2m1_decode(unpack(packed)).astype(np.float64)
          * np.repeat(oracle_mod.e4m3_decode(scales), 16, axis=1) * gd)
    w = f32_of(W).astype(np.float64)
    sd = np.repeat(oracle_mod.e4m3_decode(scales).astype(np.float64), 16, axis=1)
    a = np.abs(w) * ge / sd            # position on the E2M1 grid (approx.)
    step = np.where(a < 2, 0.5, np.where(a < 4, 1.0, 2.0))
    inside = a <= 6.0 * (1 - 1e-6)
    err = np.abs(w - wh)
    assert (err[inside] <= (0.5 * step * sd * gd)[inside] * (1 + 1e-5)).all()
    # saturated elements: the block max maps to 6*sd*gd within E4M3 rounding
    assert (err[~inside] <= (np.abs(w) / 16.0)[~inside] + 1e-12).all()
    # the tensor's largest element decodes exactly to +-amax*(1 +- 2^-4)
    i = np.unravel_index(np.abs(w).argmax(), w.shape)
    assert abs(abs(wh[i]) / abs(w[i]) - 1) <= 2 ** -4


# ------------------------------------------------------------ scale layout

def test_scale_layout_golden_offsets(oracle_mod):
    for row, block, k, off in load_pairs("scale_layout_offsets.txt"):
        assert oracle_mod.scale_layout_offset(int(row), int(block), int(k)) == int(off)


@pytest.mark.parametrize("n,k", [(16, 128), (1536, 1152), (37, 96), (1, 32),
                                 (5376, 4096), (17, 400)])
def test_scale_layout_is_a_bijection_with_zero_padding(oracle_mod, n, k):
    nblk = k // 16
    rows = np.repeat(np.arange(n), nblk)
    blks = np.tile(np.arange(nblk), n)
    offs = np.array([oracle_mod.scale_layout_offset(r, b, k)
                     for r, b in zip(rows[:20000], blks[:20000])])
    assert len(set(offs.tolist())) == offs.size
    total = oracle_mod.scale_layout_bytes(n, k)
    assert offs.max() < total
    assert total == -(-n // 16) * -(-k // 128) * 128
    canon = (np.arange(n * nblk) % 251 + 1).astype(np.uint8).reshape(n, nblk)
    dev = oracle_mod.scales_to_device_layout(canon, n, k)
    assert np.count_nonzero(dev) == n * nblk
    assert np.array_equal(dev[offs], canon.reshape(-1)[: offs.size])


def test_byte_accounting_matches_pages(oracle_mod):
    """AttnQuant docs, "Throughput", "What quantization actually saves":
    0.5625 B/element and 3.56x against bf16.  With N % 16 == 0 and
    K % 128 == 0 the device layout adds no padding, so the 31B-shaped stack
    (60 layers of the four projection shapes) is exactly 0.5625 B/element."""
    facts = dict(load_pairs("byte_accounting.txt"))
    bpe = float(facts["bytes_per_element"])
    assert round(2.0 / bpe, 2) == float(facts["bf16_over_nvfp4"])
    total = 0
    for n, k in inputs.LAYER_31B:
        b = n * k // 2 + oracle_mod.scale_layout_bytes(n, k)
        assert b == n * k * bpe
        total += b
    assert total * inputs.LAYERS_31B == 13_934_592_000
