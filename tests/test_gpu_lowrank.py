"""GPU parity of the runtime low-rank GEMV y = s*(W0_hat x) + U(V^T x)
(aq_gemv_lowrank_nvfp4) against the oracle, within the GEMV tolerance; the
r = 0, s = 1 case against the plain GEMV bit for bit; one W0 shared by the
bundles of a band; m-invariance."""
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


def bundle(n, k, r, seed):
    """s = exp(0.1 z) fp32, U and V ~ N(0, 0.01^2) bf16 (the theta recipe)."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    s = torch.exp(0.1 * torch.randn(n, generator=g)).to(torch.float32).to(DEV)
    U = (0.01 * torch.randn((n, r), generator=g)).to(torch.bfloat16).to(DEV) if r else None
    V = (0.01 * torch.randn((k, r), generator=g)).to(torch.bfloat16).to(DEV) if r else None
    return s, U, V


def lowrank_gpu(w0, s, U, V, x, flags=0):
    r = 0 if U is None else U.shape[1]
    m = x.shape[0]
    ws = torch.zeros(aq.gemv_lowrank_workspace_bytes(w0.n, w0.k, m, r), dtype=torch.uint8,
                     device=DEV)
    y = torch.full((m, w0.n), float("nan"), dtype=torch.bfloat16, device=DEV)
    aq.gemv_lowrank(w0, s, U, V, x, y, ws, flags=flags)
    torch.cuda.synchronize()
    return y


def oracle_lowrank(W0, s, U, V, x):
    packed, scales, ge, gd = oracle.quantize(bits(W0))
    r = 0 if U is None else U.shape[1]
    return oracle.gemv_lowrank(packed, scales, gd, s.cpu().numpy(),
                               bits(U) if r else None, bits(V) if r else None, bits(x))


@pytest.mark.parametrize("n,k,r,m", [
    (1536, 1152, 4, 1), (13824, 1152, 4, 1), (1152, 6912, 4, 1),   # 1B shapes, rank 4
    (37, 96, 1, 1), (300, 160, 16, 7), (129, 2080, 4, 16), (65, 4096, 0, 3), (16, 32, 2, 9),
])
def test_lowrank_matches_oracle(n, k, r, m):
    W0 = inputs.weight(n, k, seed=8000 + n + k, device=DEV)
    s, U, V = bundle(n, k, r, 8100 + r)
    x = inputs.tokens(m, k, seed=8200 + m, device=DEV)
    w0 = quantize_gpu(W0)
    y = lowrank_gpu(w0, s, U, V, x)
    assert_gemv_close(y, oracle_lowrank(W0, s, U, V, x), "lowrank n=%d k=%d r=%d m=%d" % (n, k, r, m))
    assert aq.poll_device_status() == aq.OK


@pytest.mark.parametrize("m", [1, 5, 16])
def test_lowrank_without_delta_equals_the_gemv(m):
    n, k = 1152, 6912
    w0 = quantize_gpu(inputs.weight(n, k, seed=8301, device=DEV))
    x = inputs.tokens(m, k, seed=8302, device=DEV)
    ones = torch.ones(n, dtype=torch.float32, device=DEV)
    assert torch.equal(lowrank_gpu(w0, ones, None, None, x),
                       gemv_gpu(w0, x, path=aq.PATH_GEMV_REGDECODE))


def test_lowrank_band_shares_one_block_and_is_independent_of_m():
    """Three bundles of one band share W0; each matches the oracle, and so
    does each token's single-token call (the one-token kernel form)."""
    n, k, r = 1536, 1152, 4
    W0 = inputs.weight(n, k, seed=8401, device=DEV)
    w0 = quantize_gpu(W0)
    x = inputs.tokens(6, k, seed=8402, device=DEV)
    for layer in range(3):
        s, U, V = bundle(n, k, r, 8410 + layer)
        y = lowrank_gpu(w0, s, U, V, x)
        y_ref = oracle_lowrank(W0, s, U, V, x)
        assert_gemv_close(y, y_ref, "band layer %d" % layer)
        for t in (0, 5):
            y1 = lowrank_gpu(w0, s, U, V, x[t:t + 1].contiguous(), flags=aq.STEP_PDL)
            assert_gemv_close(y1, y_ref[t:t + 1], "band layer %d token %d" % (layer, t))
        assert torch.equal(lowrank_gpu(w0, s, U, V, x[2:5].contiguous()), y[2:5])
