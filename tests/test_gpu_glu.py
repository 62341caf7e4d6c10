"""GPU parity of the fused gate+up activation (aq_gemv_glu_nvfp4:
h = gelu(gate) * up from an 8-row interleaved fused weight) against the
oracle, within the GEMV tolerance; the interleave kernel bit for bit
against the permutation; m-invariance; the full-size ~31B gate+up."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import DEV, assert_gemv_close, bits, quantize_gpu, require_gpu
from nvfp4_block_scaled_aq_gb300 import aq, inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    require_gpu()
    aq.lib()


def interleaved(Wcat):
    out = torch.empty_like(Wcat)
    aq.interleave_gate_up(Wcat, out)
    torch.cuda.synchronize()
    return out


def glu_gpu(w, x, flags=0):
    m = x.shape[0]
    ws = torch.zeros(aq.gemv_workspace_bytes(w.n, w.k, m), dtype=torch.uint8, device=DEV)
    h = torch.full((m, w.n // 2), float("nan"), dtype=torch.bfloat16, device=DEV)
    aq.gemv_glu(w, x, h, ws, flags=flags)
    torch.cuda.synchronize()
    return h


def test_interleave_matches_the_permutation():
    f, k = 200, 136
    Wcat = inputs.weight(2 * f, k, seed=9001, device=DEV)
    got = bits(interleaved(Wcat))
    assert np.array_equal(got, oracle.interleave_gate_up(bits(Wcat)))


@pytest.mark.parametrize("f,k,m", [
    (6912, 1152, 1),      # 1B gate+up
    (64, 96, 1), (8, 32, 3), (200, 1056, 5), (136, 2080, 9), (520, 4096, 16),
])
def test_glu_matches_oracle(f, k, m):
    Wcat = inputs.weight(2 * f, k, seed=9100 + f + k, device=DEV)
    x = inputs.tokens(m, k, seed=9200 + m, device=DEV)
    Wi = interleaved(Wcat)
    w = quantize_gpu(Wi)
    packed, scales, ge, gd = oracle.quantize(bits(Wi))
    h_ref = oracle.gemv_glu(packed, scales, gd, bits(x))
    assert_gemv_close(glu_gpu(w, x), h_ref, "glu f=%d k=%d m=%d" % (f, k, m))
    assert aq.poll_device_status() == aq.OK


def test_glu_is_independent_of_m():
    """Bit-identical per token for batches of two or more; one token (the
    one-token kernel form) within tolerance of the oracle."""
    f, k = 520, 4096
    Wi = interleaved(inputs.weight(2 * f, k, seed=9301, device=DEV))
    w = quantize_gpu(Wi)
    x = inputs.tokens(16, k, seed=9302, device=DEV)
    h16 = glu_gpu(w, x)
    assert torch.equal(glu_gpu(w, x), h16)
    for m in (2, 3, 9):
        assert torch.equal(glu_gpu(w, x[:m].contiguous(), flags=aq.STEP_PDL), h16[:m]), m
    packed, scales, ge, gd = oracle.quantize(bits(Wi))
    h_ref = oracle.gemv_glu(packed, scales, gd, bits(x[:1]))
    assert_gemv_close(glu_gpu(w, x[:1].contiguous(), flags=aq.STEP_PDL), h_ref, "one token")


def test_glu_31b_gate_up_sampled_parity():
    """The ~31B fused gate+up [43008, 5376] interleaved, m = 1: 512 seeded
    output columns against the oracle."""
    n, k = inputs.LAYER_31B[2]
    Wi = interleaved(inputs.weight(n, k, seed=inputs.seed_of(0, 0, 2), device=DEV))
    x = inputs.tokens(1, k, seed=9401, device=DEV)
    w = quantize_gpu(Wi)
    h = glu_gpu(w, x)
    Wb = bits(Wi)
    del Wi
    ge, gd = oracle.global_scales(oracle.amax(Wb))
    cols = np.sort(np.random.default_rng(9402).choice(n // 2, 512, replace=False))
    gate = (cols // 8) * 16 + cols % 8
    # the selected rows, arranged as an interleaved weight of their own:
    # groups of 8 gate rows followed by their 8 up rows
    rows = np.concatenate([np.concatenate([gate[q:q + 8], gate[q:q + 8] + 8])
                           for q in range(0, cols.size, 8)])
    packed_r, scales_r = oracle.quantize_rows(Wb[rows], ge)
    h_ref = oracle.gemv_glu(packed_r, scales_r, gd, bits(x))
    assert_gemv_close(h[:, cols], h_ref, "glu 31B")
