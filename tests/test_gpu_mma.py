"""GPU parity of the block-scaled MMA path: per-row activation quantisation
bit-exact against the oracle (reading R9), and the tcgen05 product of the
quantised weight and quantised activations within the GEMV tolerance of the
oracle's fp64 product of the same dequantised operands."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import DEV, assert_gemv_close, bits, gemv_gpu, quantize_gpu, require_gpu
from nvfp4_block_scaled_aq_gb300 import aq, inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    require_gpu()
    aq.lib()


def quantize_act_gpu(x):
    m, k = x.shape
    packed = torch.empty((m, k // 2), dtype=torch.uint8, device=DEV)
    scales = torch.empty((m, k // 16), dtype=torch.uint8, device=DEV)
    g_dec = torch.empty(m, dtype=torch.float32, device=DEV)
    aq.quantize_act(x, packed, scales, g_dec)
    torch.cuda.synchronize()
    return packed.cpu().numpy(), scales.cpu().numpy(), g_dec.cpu().numpy()


def mma_gpu(w, x, path=aq.PATH_MMA):
    return gemv_gpu(w, x, path=path)


# ------------------------------------------------------------ activations

@pytest.mark.parametrize("m,k", [(1, 1152), (3, 5376), (17, 6912), (64, 4096), (5, 32),
                                 (2, 21504)])
def test_activation_quantisation_bit_exact(m, k):
    x = inputs.tokens(m, k, seed=300 + m + k, device=DEV)
    gp, gs, gg = quantize_act_gpu(x)
    op, os_, og = oracle.quantize_act(bits(x))
    assert np.array_equal(gp, op)
    assert np.array_equal(gs, os_)
    assert np.array_equal(gg.view(np.uint32), og.view(np.uint32))
    assert aq.poll_device_status() == aq.OK


def test_activation_quantisation_special_rows():
    """A zero row (g_dec = 1, all zero), signed zeros, a one-hot row, rows
    near the top and the bottom of the bf16 range, and rows whose values
    sit on E2M1 rounding ties: every byte as the oracle."""
    k = 256
    x = torch.zeros((8, k), dtype=torch.float32)
    x[1, ::2] = -0.0
    x[2, 17] = 3.0
    x[3] = torch.linspace(-1e30, 1e30, k)
    x[4] = torch.linspace(-1e-30, 1e-30, k)
    x[5, :16] = torch.tensor([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0] * 2) / 6.0
    x[6] = torch.arange(k) * 0.5 - 64
    x[7] = torch.linspace(-448 * 6, 448 * 6, k)
    xb = x.to(torch.bfloat16).to(DEV)
    gp, gs, gg = quantize_act_gpu(xb)
    op, os_, og = oracle.quantize_act(bits(xb))
    assert np.array_equal(gp, op)
    assert np.array_equal(gs, os_)
    assert np.array_equal(gg.view(np.uint32), og.view(np.uint32))
    assert aq.poll_device_status() == aq.OK


def test_activation_quantisation_out_of_range_row():
    """A row with an infinite value: that row is zero-filled with a NaN
    g_dec and the status word reports AQ_ERR_RANGE; other rows are intact."""
    k = 128
    x = inputs.tokens(3, k, seed=310, device=DEV)
    x[1, 5] = float("inf")
    gp, gs, gg = quantize_act_gpu(x)
    assert aq.poll_device_status() == aq.ERR_RANGE
    assert not gp[1].any() and not gs[1].any() and np.isnan(gg[1])
    op, os_, og = oracle.quantize_act(bits(x[[0, 2]]))
    assert np.array_equal(gp[[0, 2]], op) and np.array_equal(gs[[0, 2]], os_)
    assert aq.poll_device_status() == aq.OK


# ------------------------------------------------------------ MMA product

def oracle_q(W, x, rows=None):
    packed, scales, ge, gd = oracle.quantize(bits(W) if torch.is_tensor(W) else W)
    xp, xs, xg = oracle.quantize_act(bits(x))
    if rows is not None:
        packed, scales = packed[rows], scales[rows]
    return oracle.gemv_q(packed, scales, gd, xp, xs, xg)


@pytest.mark.parametrize("n,k,m", [
    (1536, 1152, 1), (1536, 1152, 2), (1536, 1152, 16), (1536, 1152, 17), (1536, 1152, 64),
    (13824, 1152, 64), (1152, 6912, 32), (1152, 1024, 48), (37, 96, 5), (300, 160, 33),
    (16, 32, 1), (129, 2080, 64),
])
def test_mma_matches_oracle(n, k, m):
    W = inputs.weight(n, k, seed=400 + n + k, device=DEV)
    x = inputs.tokens(m, k, seed=500 + m, device=DEV)
    w = quantize_gpu(W)
    assert_gemv_close(mma_gpu(w, x), oracle_q(W, x), "mma n=%d k=%d m=%d" % (n, k, m))
    assert aq.poll_device_status() == aq.OK


def test_mma_is_independent_of_m_and_deterministic():
    n, k = 1152, 6912
    w = quantize_gpu(inputs.weight(n, k, seed=41, device=DEV))
    x = inputs.tokens(64, k, seed=42, device=DEV)
    y64 = mma_gpu(w, x)
    assert torch.equal(mma_gpu(w, x), y64)
    for m in (1, 2, 15, 16, 17, 33, 63):
        assert torch.equal(mma_gpu(w, x[:m].contiguous()), y64[:m]), m
    for t in (0, 31, 63):
        assert torch.equal(mma_gpu(w, x[t:t + 1].contiguous())[0], y64[t])


def test_auto_path_uses_the_mma_path_above_sixteen_tokens():
    n, k = 1536, 1152
    w = quantize_gpu(inputs.weight(n, k, seed=43, device=DEV))
    x = inputs.tokens(24, k, seed=44, device=DEV)
    assert torch.equal(gemv_gpu(w, x, path=aq.PATH_AUTO), mma_gpu(w, x))


@pytest.mark.parametrize("proj", [2, 3])
@pytest.mark.parametrize("m", [1, 64])
def test_31b_mlp_shapes_sampled_parity(proj, m):
    """The batch-sweep weights (~31B-shaped fused gate+up and down) at full
    size: 512 seeded rows against the oracle."""
    n, k = inputs.LAYER_31B[proj]
    W = inputs.weight(n, k, seed=inputs.seed_of(0, 0, proj), device=DEV)
    x = inputs.tokens(m, k, seed=inputs.seed_of(1, 0, proj) + m, device=DEV)
    w = quantize_gpu(W)
    y = mma_gpu(w, x)
    Wb = bits(W)
    del W
    ge, gd = oracle.global_scales(oracle.amax(Wb))
    rows = np.sort(np.random.default_rng(proj + m).choice(n, 512, replace=False))
    packed_r, scales_r = oracle.quantize_rows(Wb[rows], ge)
    xp, xs, xg = oracle.quantize_act(bits(x))
    y_ref = oracle.gemv_q(packed_r, scales_r, gd, xp, xs, xg)
    assert_gemv_close(y[:, rows], y_ref, "31B proj %d m=%d" % (proj, m))
