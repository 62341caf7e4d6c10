"""GPU parity of the block-scaled GEMV against the oracle's fp64 sum of the
same dequantised values, plus the invariants the method fixes."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import (DEV, KERNELS, assert_gemv_close, assert_quantized_equal, bits,
                         gemv_gpu, quantize_gpu, require_gpu, weight_bytes)
from nvfp4_block_scaled_aq_gb300 import aq, inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    require_gpu()
    aq.lib()


def oracle_y(W, x):
    packed, scales, ge, gd = oracle.quantize(bits(W))
    return oracle.gemv(packed, scales, gd, bits(x))


@pytest.mark.parametrize("n,k,m", [
    (1536, 1152, 1),      # fused QKV, 1B shape
    (1152, 1024, 1),      # o_proj, 1B shape
    (13824, 1152, 1),     # fused gate+up, 1B shape
    (1152, 6912, 1),      # down, 1B shape (long K: split-K)
    (1536, 1152, 2), (1536, 1152, 3), (1536, 1152, 8), (1536, 1152, 9),
    (1536, 1152, 16), (1152, 6912, 16),
    (37, 96, 1), (37, 96, 5), (1, 32, 1), (16, 128, 2), (100, 1184, 4),
    (65, 4096, 1), (300, 160, 7),
])
def test_gemv_matches_oracle(n, k, m):
    """Both kernels, and the automatic choice, within tolerance."""
    W = inputs.weight(n, k, seed=1000 + n + k, device=DEV)
    x = inputs.tokens(m, k, seed=2000 + m, device=DEV)
    w = quantize_gpu(W)
    y_ref = oracle_y(W, x)
    assert_gemv_close(gemv_gpu(w, x), y_ref, "auto n=%d k=%d m=%d" % (n, k, m))
    for name, (path, max_m) in KERNELS.items():
        if m <= max_m:
            assert_gemv_close(gemv_gpu(w, x, path=path), y_ref,
                              "%s n=%d k=%d m=%d" % (name, n, k, m))
    assert aq.poll_device_status() == aq.OK


def test_gemv_fused_qkv_config_exact_rounding_rate():
    """[1536, 1152], seed 0, one token: within tolerance everywhere, and the
    bf16 output is the correctly rounded oracle value for nearly all rows
    (fp32 accumulation differs from fp64 only in the last bits)."""
    W = inputs.weight(1536, 1152, seed=0, device=DEV)
    x = inputs.tokens(1, 1152, seed=0, device=DEV)
    y = gemv_gpu(quantize_gpu(W), x)
    y_ref = oracle_y(W, x)
    assert_gemv_close(y, y_ref)
    ref_bf16 = torch.from_numpy(y_ref).to(torch.bfloat16)
    exact = (y.cpu() == ref_bf16).float().mean().item()
    assert exact > 0.98, exact


@pytest.mark.parametrize("kernel", sorted(KERNELS))
@pytest.mark.parametrize("n,k", [(1152, 6912), (13824, 1152)])
def test_gemv_is_independent_of_m(kernel, n, k):
    """On each kernel, each token's output is bit-identical whatever else
    is in the batch, for batches of two or more.  A single token on the
    register-decode kernel takes its one-token form (block sums on the MMA's
    n dimension, a different fp32 summation order): it is held to the
    oracle instead, like every other output."""
    path, max_m = KERNELS[kernel]
    W = inputs.weight(n, k, seed=5, device=DEV)
    w = quantize_gpu(W)
    x = inputs.tokens(max_m, k, seed=6, device=DEV)
    y_all = gemv_gpu(w, x, path=path)
    one_token_form = kernel == "regdecode"
    for m in sorted({1, 2, 3, 8, 9, max_m}):
        if m <= max_m and not (m == 1 and one_token_form):
            ym = gemv_gpu(w, x[:m].contiguous(), path=path)
            assert torch.equal(ym, y_all[:m]), m
    ts = sorted({0, max_m // 2, max_m - 1})
    singles = torch.stack([gemv_gpu(w, x[t:t + 1].contiguous(), path=path)[0] for t in ts])
    if one_token_form:
        assert_gemv_close(singles, oracle_y(W, x[ts]), "single tokens")
        assert_gemv_close(y_all[ts], oracle_y(W, x[ts]), "batched")
    else:
        assert torch.equal(singles, y_all[ts])


def test_gemv_is_deterministic_and_workspace_rearms():
    n, k = 5376, 4096
    w = quantize_gpu(inputs.weight(n, k, seed=8, device=DEV))
    x = inputs.tokens(2, k, seed=9, device=DEV)
    ws = torch.zeros(aq.gemv_workspace_bytes(n, k, 2), dtype=torch.uint8, device=DEV)
    ys = [gemv_gpu(w, x, ws) for _ in range(4)]
    for y in ys[1:]:
        assert torch.equal(y, ys[0])


def test_one_workspace_serves_interleaved_shapes():
    """Calls of different shapes share one zeroed workspace in any order."""
    shapes = [(1536, 1152), (1152, 6912), (13824, 1152), (1152, 1024)]
    ws_bytes = max(aq.gemv_workspace_bytes(n, k, 1) for n, k in shapes)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=DEV)
    cases = []
    for i, (n, k) in enumerate(shapes):
        w = quantize_gpu(inputs.weight(n, k, seed=40 + i, device=DEV))
        x = inputs.tokens(1, k, seed=50 + i, device=DEV)
        cases.append((w, x, gemv_gpu(w, x)))
    for order in ([0, 1, 2, 3], [3, 1, 0, 2, 1, 3, 2, 0]):
        for i in order:
            w, x, want = cases[i]
            assert torch.equal(gemv_gpu(w, x, ws), want), i


@pytest.mark.parametrize("kernel", sorted(KERNELS))
def test_gemv_power_of_two_input_scaling_is_exact(kernel):
    """Scaling x by 2^j scales y by 2^j exactly: both kernels normalise the
    activations by powers of two and undo them exactly."""
    path = KERNELS[kernel][0]
    n, k = 300, 2048
    w = quantize_gpu(inputs.weight(n, k, seed=12, device=DEV))
    x = inputs.tokens(1, k, seed=13, device=DEV)
    y = gemv_gpu(w, x, path=path).float()
    for j in (-90, -20, 7, 60):
        yj = gemv_gpu(w, (x.float() * 2.0 ** j).to(torch.bfloat16), path=path).float()
        assert torch.equal(yj, y * 2.0 ** j), j


@pytest.mark.parametrize("kernel", sorted(KERNELS))
def test_gemv_wide_dynamic_range_activations(kernel):
    n, k = 128, 1024
    W = inputs.weight(n, k, seed=14, device=DEV)
    x = inputs.tokens(1, k, seed=15, device=DEV).float()
    x[0, ::7] *= 1e12
    x[0, 3::11] *= 1e-12
    x = x.to(torch.bfloat16)
    y = gemv_gpu(quantize_gpu(W), x, path=KERNELS[kernel][0])
    assert_gemv_close(y, oracle_y(W, x))


def test_gemv_one_hot_tokens_return_columns():
    """One-hot tokens give back columns of w_hat (bit-exact on the
    register-decode kernel, whose f16 path is exact here; within tolerance
    on the tcgen05 kernel, whose six-term activation sum is exact to about
    2^-19)."""
    n, k = 64, 256
    W = inputs.weight(n, k, seed=16, device=DEV)
    w = quantize_gpu(W)
    packed, scales, ge, gd = oracle.quantize(bits(W))
    cols = [0, 1, 31, 32, 127, 128, 255]
    x = torch.zeros((len(cols), k), dtype=torch.bfloat16, device=DEV)
    for t, c in enumerate(cols):
        x[t, c] = 1.0
    y_ref = oracle.gemv(packed, scales, gd, bits(x))
    y = gemv_gpu(w, x, path=aq.PATH_GEMV_REGDECODE)
    assert torch.equal(y.cpu(), torch.from_numpy(y_ref).to(torch.bfloat16))
    for t0 in range(0, len(cols), 5):
        xt = x[t0:t0 + 5].contiguous()
        assert_gemv_close(gemv_gpu(w, xt, path=aq.PATH_GEMV_TCGEN05), y_ref[t0:t0 + 5])


def test_passthrough_gemv_equals_plain_gemv_bit_exact():
    n, k = 13824, 1152
    th = inputs.theta(n, k, 4, seed=17, device=DEV, passthrough=True)
    w_theta = aq.Nvfp4Weight.empty(n, k, device=DEV)
    ws = torch.zeros(aq.quantize_workspace_bytes(), dtype=torch.uint8, device=DEV)
    aq.reconstruct_quantize(th.W0, th.s, th.U, th.V, w_theta, ws)
    w_plain = quantize_gpu(th.W0)
    x = inputs.tokens(1, k, seed=18, device=DEV)
    assert torch.equal(gemv_gpu(w_theta, x), gemv_gpu(w_plain, x))


def test_fused_projection_equals_its_parts():
    """A fused gate+up weight read once gives the rows of its parts: the
    first part's rows form a valid weight view (its row count is a
    multiple of 16), evaluated on the same quantised bytes."""
    k, na, nb = 1152, 6912, 6912
    W = inputs.weight(na + nb, k, seed=19, device=DEV)
    w = quantize_gpu(W)
    x = inputs.tokens(1, k, seed=20, device=DEV)
    y = gemv_gpu(w, x)
    sb = aq.scale_bytes(na, k)
    part = aq.Nvfp4Weight(na, k, w.packed[: na * k // 2], w.scales[:sb], w.global_scale)
    yp = gemv_gpu(part, x)
    y_ref = oracle_y(W, x)
    assert_gemv_close(yp, y_ref[:, :na])
    assert_gemv_close(y[:, :na], y_ref[:, :na])


def test_gemv_rejects_a_too_small_workspace():
    w = quantize_gpu(inputs.weight(64, 256, seed=21, device=DEV))
    x = inputs.tokens(1, 256, seed=22, device=DEV)
    y = torch.empty((1, 64), dtype=torch.bfloat16, device=DEV)
    small = torch.zeros(8, dtype=torch.uint8, device=DEV)
    with pytest.raises(aq.AqError) as e:
        aq.gemv(w, x, y, small)
    assert e.value.status == aq.ERR_WORKSPACE


# ------------------------------------------------------------ full size

@pytest.mark.parametrize("proj", range(4))
def test_31b_shapes_sampled_parity(proj):
    """One layer of the ~31B-shaped stack at full size, in the launch
    configuration the benchmark times: all bytes of 512 seeded rows
    bit-exact and their GEMV outputs within tolerance."""
    n, k = inputs.LAYER_31B[proj]
    W = inputs.weight(n, k, seed=inputs.seed_of(0, 0, proj), device=DEV)
    x = inputs.tokens(1, k, seed=inputs.seed_of(1, 0, proj), device=DEV)
    w = quantize_gpu(W)
    y = gemv_gpu(w, x)
    Wb = bits(W)
    del W
    ge, gd = oracle.global_scales(oracle.amax(Wb))
    rows = np.sort(np.random.default_rng(proj).choice(n, 512, replace=False))
    packed_r, scales_r = oracle.quantize_rows(Wb[rows], ge)
    gp, gs, ggd = weight_bytes(w)
    assert np.float32(ggd) == np.float32(gd)
    assert np.array_equal(gp[rows], packed_r)
    offs = np.array([[oracle.scale_layout_offset(r, b, k) for b in range(k // 16)]
                     for r in rows[:64]])
    assert np.array_equal(gs[offs], scales_r[:64])
    y_ref = oracle.gemv(packed_r, scales_r, gd, bits(x))
    assert_gemv_close(y[:, rows], y_ref, "31B proj %d" % proj)
