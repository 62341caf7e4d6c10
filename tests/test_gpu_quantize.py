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
                                 (1152, 6912)])
def test_quantize_ragged_and_edge_shapes(n, k):
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
    ws = torch.empty(aq.quantize_workspace_bytes(), dtype=torch.uint8, device=DEV)
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
    bf16 in) takes the per-element rank-4 path instead of the one that keeps
    V rows in registers.  Every path stays bit-exact with the oracle."""
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
    ws = torch.empty(aq.quantize_workspace_bytes(), dtype=torch.uint8, device=DEV)
    aq.reconstruct_quantize(th.W0, th.s, th.U, V, w, ws)
    assert_quantized_equal(w, ref)
    assert aq.poll_device_status() == aq.OK
