"""GPU parity of the load-time kernels against the CPU oracle: quantised
bytes and scales bit-exact, reconstruction bit-exact."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import (DEV, assert_quantized_equal, bits, quantize_gpu, require_gpu,
                         weight_bytes)
from nvfp4_block_scaled_aq_gb300 import aq, inputs
from test_oracle_method import bf16_of, f32_of

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    require_gpu()
    aq.lib()


def to_dev(bits_np):
    return inputs.from_bits_u16(bits_np, device=DEV)


def test_quantize_fused_qkv_1b_shape_bit_exact():
    """Single fused-QKV projection of the Gemma-3-1B shape, [1536, 1152],
    N(0, 0.02^2) with 0.1% x20 outliers, seed 0."""
    W = inputs.weight(1536, 1152, seed=0, device=DEV)
    w = quantize_gpu(W)
    assert_quantized_equal(w, bits(W))
    assert aq.poll_device_status() == aq.OK


def _sweep_tensor(limit_bits, amax_bits):
    """Every finite bf16 value of magnitude <= the limit, 15 per block
    behind a block maximum equal to the limit, plus one row whose first
    element sets the tensor's amax."""
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    v = f32_of(allbits)
    lim = f32_of(np.array([limit_bits], np.uint16))[0]
    allbits = allbits[np.isfinite(v) & (np.abs(v) <= lim)]
    per, k = 15, 128
    nblk = -(-allbits.size // (per * 8)) * 8
    pad = np.zeros(nblk * per, np.uint16)
    pad[: allbits.size] = allbits
    blocks = np.concatenate([np.full((nblk, 1), limit_bits, np.uint16),
                             pad.reshape(nblk, per)], axis=1)
    rows = blocks.reshape(-1, k)
    extra = np.zeros((1, k), np.uint16)
    extra[0, 0] = amax_bits
    return np.concatenate([rows, extra])


@pytest.mark.parametrize("limit,amax", [(1.0, 1.0), (1.0, 2688.0), (1.0, 2.0 ** 15),
                                        (1.0, 2.0 ** 20), (2.0 ** -20, 2.0 ** -20),
                                        (6.0, 6.0)])
def test_quantize_every_bf16_value(limit, amax):
    """Every finite bf16 value through the GPU quantiser, against scales in
    the normal, subnormal, zero and saturated E4M3 ranges."""
    lb = bf16_of([limit])[0]
    ab = bf16_of([amax])[0]
    Wb = _sweep_tensor(lb, ab)
    w = quantize_gpu(to_dev(Wb))
    assert_quantized_equal(w, Wb)


def _adversarial():
    cases = {}
    k = 64
    z = np.zeros((3, k), np.float32)
    cases["zero_tensor"] = z.copy()
    one = z.copy()
    one[1, 37] = -0.0123
    cases["single_nonzero"] = one
    ties = z.copy()
    ties[0, :16] = [6, .25, .75, 1.25, 1.75, 2.5, 3.5, 5, -.25, -.75, -1.25, -1.75,
                    -2.5, -3.5, -5, 0]
    ties[1, :16] = [-6, .5, 1, 1.5, 2, 3, 4, 6, -0.0, 1e-3, -1e-3, 0, 0, 0, 0, 0]
    cases["exact_ties"] = ties
    sat = z.copy()
    sat[0, :16] = np.linspace(-6.3, 6.3, 16)
    sat[2, 16:32] = 6.0
    sat[2, 20] = 6.2
    cases["saturation"] = sat
    eq = z.copy()
    eq[:, 32:48] = 0.37
    eq[0, 0] = 5.0
    cases["all_equal_block"] = eq
    tiny = z.copy()
    tiny[0, 0] = 1.0
    tiny[1, :16] = [-0.0, 1e-9, -1e-9, 2e-7, -3e-7, 1e-5, -1e-6, 0, 0, 0, 0, 0, 0, 0, 0,
                    4e-7]
    cases["negative_zero_underflow"] = tiny
    return cases


@pytest.mark.parametrize("name", list(_adversarial().keys()))
def test_quantize_adversarial(name):
    Wb = bf16_of(_adversarial()[name])
    w = quantize_gpu(to_dev(Wb))
    assert_quantized_equal(w, Wb)
    assert aq.poll_device_status() == aq.OK


@pytest.mark.parametrize("n,k", [(1, 32), (37, 96), (16, 128), (5, 1184), (100, 2048),
                                 (1152, 6912), (16, 320000)])
def test_quantize_ragged_and_edge_shapes(n, k):
    """Plain quantisation on row counts and widths that end inside a tile;
    at k = 320000 (2500 tile columns, more than the warps the GPU holds at
    once) the amax and quantisation passes run as two launches."""
    W = inputs.weight(n, k, seed=n * 7 + k, device=DEV)
    w = quantize_gpu(W)
    assert_quantized_equal(w, bits(W))


@pytest.mark.parametrize("bad", [0x7F80, 0xFF80, 0x7FC1, 0x0001])
def test_quantize_out_of_range_amax_sets_status(bad):
    """inf, -inf, NaN, and the smallest subnormal (2688/amax overflows):
    outputs zero-filled, g_dec NaN, AQ_ERR_RANGE on the next poll."""
    Wb = bits(inputs.weight(32, 128, seed=3, device=DEV))
    if bad == 0x0001:
        Wb = np.zeros_like(Wb)
    Wb[5, 17] = bad
    with pytest.raises(oracle.OracleRangeError):
        oracle.quantize(Wb)
    w = quantize_gpu(to_dev(Wb))
    assert aq.poll_device_status() == aq.ERR_RANGE
    assert "amax" in aq.last_error()
    gp, gs, gd = weight_bytes(w)
    assert not gp.any() and not gs.any() and np.isnan(gd)
    assert aq.poll_device_status() == aq.OK  # polling clears the word


# ------------------------------------------------------------ reconstruction

@pytest.mark.parametrize("n,k", [(13824, 1152), (1152, 6912)])
def test_reconstruct_1b_mlp_theta_bit_exact(n, k):
    th = inputs.theta(n, k, 4, seed=n + k, device=DEV)
    W_eff = torch.empty((n, k), dtype=torch.bfloat16, device=DEV)
    aq.reconstruct(th.W0, th.s, th.U, th.V, W_eff)
    ref = oracle.reconstruct(bits(th.W0), th.s.cpu().numpy(), bits(th.U), bits(th.V))
    assert np.array_equal(bits(W_eff), ref)


def test_reconstruct_passthrough_every_bf16_pattern():
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    allbits = allbits[~np.isnan(f32_of(allbits))]
    n = 16
    k = (allbits.size // n) // 32 * 32
    W0 = to_dev(allbits[: n * k].reshape(n, k))
    s = torch.ones(n, device=DEV)
    U = torch.zeros((n, 4), dtype=torch.bfloat16, device=DEV)
    V = torch.zeros((k, 4), dtype=torch.bfloat16, device=DEV)
    W_eff = torch.empty_like(W0)
    aq.reconstruct(W0, s, U, V, W_eff)
    assert np.array_equal(bits(W_eff), bits(W0))


@pytest.mark.parametrize("r", [0, 1, 3, 4, 7])
def test_reconstruct_ranks(r):
    n, k = 40, 96
    th = inputs.theta(n, k, max(r, 1), seed=r + 1, device=DEV)
    U = th.U[:, :r].contiguous() if r else None
    V = th.V[:, :r].contiguous() if r else None
    W_eff = torch.empty((n, k), dtype=torch.bfloat16, device=DEV)
    aq.reconstruct(th.W0, th.s, U, V, W_eff)
    Ub = bits(U) if r else np.zeros((n, 0), np.uint16)
    Vb = bits(V) if r else np.zeros((k, 0), np.uint16)
    ref = oracle.reconstruct(bits(th.W0), th.s.cpu().numpy(), Ub, Vb)
    assert np.array_equal(bits(W_eff), ref)


@pytest.mark.parametrize("passthrough", [False, True])
@pytest.mark.parametrize("n,k,r", [(13824, 1152, 4), (1152, 6912, 4), (37, 96, 3)])
def test_fused_reconstruct_quantize_bit_exact(n, k, r, passthrough):
    """Theta -> NVFP4 in one pass equals the oracle's reconstruct then
    quantise; at passthrough it equals quantising W0 itself."""
    th = inputs.theta(n, k, r, seed=11 + n, device=DEV, passthrough=passthrough)
    w = aq.Nvfp4Weight.empty(n, k, device=DEV)
    ws = torch.zeros(aq.quantize_workspace_bytes(), dtype=torch.uint8, device=DEV)
    aq.reconstruct_quantize(th.W0, th.s, th.U, th.V, w, ws)
    W_eff = oracle.reconstruct(bits(th.W0), th.s.cpu().numpy(), bits(th.U), bits(th.V))
    if passthrough:
        assert np.array_equal(W_eff, bits(th.W0))
    assert_quantized_equal(w, W_eff)


@pytest.mark.parametrize("offset", [1, 4])
def test_rank4_v_alignment_paths_bit_exact(offset):
    """A rank-4 V that is only 2-byte aligned (a view one bf16 into a larger
    buffer) takes the generic rank path of the reconstruction and the fused
    reconstruct-and-quantise; one that is 8- but not 16-byte aligned (four
    bf16 in) takes the per-element rank-4 path instead of the one that stages
    V in shared memory.  Every path stays bit-exact with the oracle."""
    n, k, r = 48, 160, 4
    th = inputs.theta(n, k, r, seed=77, device=DEV)
    big = torch.empty(k * r + 8, dtype=torch.bfloat16, device=DEV)
    V = big[offset:offset + k * r].view(k, r)
    V.copy_(th.V)
    assert V.data_ptr() % 16 == 2 * offset
    ref = oracle.reconstruct(bits(th.W0), th.s.cpu().numpy(), bits(th.U), bits(th.V))
    W_eff = torch.empty((n, k), dtype=torch.bfloat16, device=DEV)
    aq.reconstruct(th.W0, th.s, th.U, V, W_eff)
    assert np.array_equal(bits(W_eff), ref)
    w = aq.Nvfp4Weight.empty(n, k, device=DEV)
    ws = torch.zeros(aq.quantize_workspace_bytes(), dtype=torch.uint8, device=DEV)
    aq.reconstruct_quantize(th.W0, th.s, th.U, V, w, ws)
    assert_quantized_equal(w, ref)
    assert aq.poll_device_status() == aq.OK


@pytest.mark.parametrize("which", ["U", "s"])
def test_rank4_u_s_alignment_fallback_bit_exact(which):
    """The rank-4 path that streams the tile's U rows and s values by TMA
    needs U and s 16-byte aligned; a U or an s view that is only naturally
    aligned takes the per-element rank path and stays bit-exact."""
    n, k, r = 48, 160, 4
    th = inputs.theta(n, k, r, seed=78, device=DEV)
    U, s = th.U, th.s
    if which == "U":
        big = torch.empty(n * r + 8, dtype=torch.bfloat16, device=DEV)
        U = big[1:1 + n * r].view(n, r)
        U.copy_(th.U)
        assert U.data_ptr() % 16 == 2
    else:
        big = torch.empty(n + 4, dtype=torch.float32, device=DEV)
        s = big[1:1 + n]
        s.copy_(th.s)
        assert s.data_ptr() % 16 == 4
    ref = oracle.reconstruct(bits(th.W0), th.s.cpu().numpy(), bits(th.U), bits(th.V))
    w = aq.Nvfp4Weight.empty(n, k, device=DEV)
    ws = torch.zeros(aq.quantize_workspace_bytes(), dtype=torch.uint8, device=DEV)
    aq.reconstruct_quantize(th.W0, s, U, th.V, w, ws)
    assert_quantized_equal(w, ref)
    assert aq.poll_device_status() == aq.OK


def _fused_r4(W0b, s, Ub, Vb):
    n, k = W0b.shape
    w = aq.Nvfp4Weight.empty(n, k, device=DEV)
    ws = torch.zeros(aq.quantize_workspace_bytes(), dtype=torch.uint8, device=DEV)
    aq.reconstruct_quantize(to_dev(W0b), torch.as_tensor(s, device=DEV), to_dev(Ub),
                            to_dev(Vb), w, ws)
    return w


@pytest.mark.parametrize("n,k", [(1, 32), (45, 160), (17, 4128), (300, 1152), (20, 40960),
                                 (16, 320000), (7680, 5376)])
def test_rank4_packed_path_ragged_shapes_bit_exact(n, k):
    """The rank-4 path with V 16-byte aligned on row counts that end inside a
    16-row tile and widths that end inside a 128-column tile column.  At
    k = 320000 there are more tile columns (2500) than warps the GPU holds
    at once, so the amax and quantisation passes run as two launches instead
    of one cooperative launch.  [7680, 5376] gives an 8-warp CTA's warp
    about nine row tiles, which takes the cooperative form without the W_eff
    hand-over, launched as one 16-warp CTA per SM (the smaller shapes take
    the hand-over with two 8-warp CTAs per SM)."""
    th = inputs.theta(n, k, 4, seed=n * 7 + k, device=DEV)
    assert th.V.data_ptr() % 16 == 0
    w = aq.Nvfp4Weight.empty(n, k, device=DEV)
    ws = torch.zeros(aq.quantize_workspace_bytes(), dtype=torch.uint8, device=DEV)
    aq.reconstruct_quantize(th.W0, th.s, th.U, th.V, w, ws)
    ref = oracle.reconstruct(bits(th.W0), th.s.cpu().numpy(), bits(th.U), bits(th.V))
    assert_quantized_equal(w, ref)
    assert aq.poll_device_status() == aq.OK


def test_rank4_31b_gate_up_full_size_sampled_rows_bit_exact():
    """The ~31B fused gate+up theta bundle [43008, 5376] at rank 4, in the
    launch form `bench.py --load-time` times (one cooperative launch of
    16-warp CTAs, one per SM).  The oracle rebuilds the whole W_eff for the
    per-tensor amax.  g_dec must match bit for bit.  So must the packed
    bytes and the device-layout scale bytes of 256 seeded rows; each
    (row, block) scale is located through the oracle's own layout
    function."""
    n, k = 43008, 5376
    th = inputs.theta(n, k, 4, seed=4300, device=DEV)
    w = aq.Nvfp4Weight.empty(n, k, device=DEV)
    ws = torch.zeros(aq.quantize_workspace_bytes(), dtype=torch.uint8, device=DEV)
    aq.reconstruct_quantize(th.W0, th.s, th.U, th.V, w, ws)
    assert aq.poll_device_status() == aq.OK
    W_eff = oracle.reconstruct(bits(th.W0), th.s.cpu().numpy(), bits(th.U), bits(th.V))
    ge, gd = oracle.global_scales(oracle.amax(W_eff))
    rows = np.sort(np.random.default_rng(4300).choice(n, 256, replace=False))
    packed, scales = oracle.quantize_rows(W_eff[rows], ge)
    gp, gs, ggd = weight_bytes(w)
    assert np.float32(ggd) == np.float32(gd), (ggd, gd)
    bad = np.argwhere(gp[rows] != packed)
    assert bad.size == 0, "packed differs at sampled (row index, byte) %s" % bad[:5].tolist()
    for i, r in enumerate(rows):
        got = np.array([gs[oracle.scale_layout_offset(int(r), b, k)] for b in range(k // 16)],
                       np.uint8)
        assert np.array_equal(got, scales[i]), "scales of row %d differ" % r


def test_rank4_zero_signs_and_exact_cancellation_bit_exact():
    """AttnQuant docs, landing page, "How it works": W_eff = s*W0 + U*V^T,
    with the rank term zero handled as s*W0 alone.  Rows built so that
    (a) s*w0 + delta cancels exactly (the result is +0), (b) delta is zero
    through an exact cancellation inside the rank sum, with s < 0 and signed
    zeros in W0 (the product's sign of zero must survive), (c) U = 0 with
    s = -0, +0 and negative s, (d) generic rows.  Every block also holds
    non-zero values, so a zero's sign shows in its nibble (0x0 or 0x8)."""
    rng = np.random.default_rng(5)
    n, k = 64, 256
    x = bf16_of(rng.normal(0, 0.05, k))            # shared row pattern
    W0 = np.tile(bf16_of(rng.normal(0, 0.05, k)), (n, 1))
    W0[:16, 0::2] = x[0::2]                         # (a) cancels with V[:, 0]
    zero_mask = rng.random((n, k)) < 0.3
    signs = np.where(rng.random((n, k)) < 0.5, 0x8000, 0x0000).astype(np.uint16)
    W0[16:48][zero_mask[16:48]] = signs[16:48][zero_mask[16:48]]
    W0[48:] = bf16_of(rng.normal(0, 0.05, (16, k)))
    V = np.zeros((k, 4), np.uint16)
    V[:, 0] = x ^ 0x8000                            # -x
    V[:, 1] = x                                     # v0 + v1 = 0 exactly
    V[:, 2] = bf16_of(rng.normal(0, 0.01, k))
    V[:, 3] = bf16_of(rng.normal(0, 0.01, k))
    one = bf16_of([1.0])[0]
    U = np.zeros((n, 4), np.uint16)
    U[:16, 0] = one                                 # (a) delta = -x_j
    U[16:32, 0] = one
    U[16:32, 1] = one                               # (b) delta = +0 by cancellation
    U[48:] = bf16_of(rng.normal(0, 0.01, (16, 4)))  # (d)
    s = np.exp(0.1 * rng.normal(size=n)).astype(np.float32)
    s[:16] = 1.0
    s[16:32] *= -1.5
    s[32:36] = -0.0                                 # (c)
    s[36:40] = 0.0
    s[40:48] *= -1.0
    w = _fused_r4(W0, s, U, V)
    ref = oracle.reconstruct(W0, s, U, V)
    assert np.all(ref[:16, 0::2] == 0)              # +0 from exact cancellation
    neg_zero = (ref[16:48] == 0x8000).sum()
    assert neg_zero > 100 and (ref[16:48] == 0).sum() > 100
    assert_quantized_equal(w, ref)
    assert aq.poll_device_status() == aq.OK


@pytest.mark.parametrize("case", ["inf_in_w0", "inf_from_rank_term", "nan_in_v"])
def test_rank4_non_finite_w_eff_sets_status(case):
    """A non-finite W_eff on the rank-4 path is caught like a non-finite
    weight: zero-filled outputs, NaN global scale, AQ_ERR_RANGE.  The rank
    term can overflow to inf from finite inputs (the product inside an fma is
    exact, so it cannot make a NaN); a NaN in one V entry makes one column of
    W_eff NaN, which the amax pass must propagate past every finite value."""
    rng = np.random.default_rng(9)
    n, k = 32, 256
    W0 = bf16_of(rng.normal(0, 0.02, (n, k)))
    U = bf16_of(rng.normal(0, 0.01, (n, 4)))
    V = bf16_of(rng.normal(0, 0.01, (k, 4)))
    s = np.ones(n, np.float32)
    if case == "inf_in_w0":
        W0[5, 77] = 0x7F80
    elif case == "inf_from_rank_term":
        big = bf16_of([3.0e38])[0]
        U[9] = [big, 0, 0, 0]
        V[130, 0] = big
    else:
        V[201, 2] = 0x7FC0
    w = _fused_r4(W0, s, U, V)
    assert aq.poll_device_status() == aq.ERR_RANGE
    gp, gs, gd = weight_bytes(w)
    assert not gp.any() and not gs.any() and np.isnan(gd)


def test_one_workspace_serves_every_path_and_is_left_zeroed():
    """A quantise workspace zero-filled once serves a sequence of calls on
    every path -- plain quantise, the cooperative rank-4 form, its two-launch
    form, the generic-rank form -- and each call leaves its words zero."""
    ws = torch.zeros(aq.quantize_workspace_bytes(), dtype=torch.uint8, device=DEV)
    cases = [("plain", 100, 2048, 0), ("r4", 300, 1152, 4), ("r4", 16, 320000, 4),
             ("generic", 37, 96, 3), ("r4", 45, 160, 4)]
    for i, (form, n, k, r) in enumerate(cases):
        th = inputs.theta(n, k, max(r, 1), seed=200 + i, device=DEV)
        w = aq.Nvfp4Weight.empty(n, k, device=DEV)
        if form == "plain":
            aq.quantize(th.W0, w, ws)
            ref = bits(th.W0)
        else:
            U = th.U[:, :r].contiguous()
            V = th.V[:, :r].contiguous()
            aq.reconstruct_quantize(th.W0, th.s, U, V, w, ws)
            ref = oracle.reconstruct(bits(th.W0), th.s.cpu().numpy(), bits(U), bits(V))
        torch.cuda.synchronize()
        assert not ws.any().item(), (form, n, k)
        assert_quantized_equal(w, ref)
        assert aq.poll_device_status() == aq.OK
