"""GPU parity of the bf16 GEMV (aq_gemv_bf16, the unquantised lm_head and
attention families) against the oracle's fp64 product, within the GEMV
tolerance; m-invariance and determinism; the full-size 31B lm_head on
sampled rows; one workspace shared with the NVFP4 GEMV."""
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


def bf16_gpu(W, x, ws=None, flags=0):
    n, k = W.shape
    m = x.shape[0]
    if ws is None:
        ws = torch.zeros(aq.gemv_bf16_workspace_bytes(n, k, m), dtype=torch.uint8, device=DEV)
    y = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device=DEV)
    aq.gemv_bf16(W, x, y, ws, flags=flags)
    torch.cuda.synchronize()
    return y


@pytest.mark.parametrize("n,k,m", [
    (1536, 1152, 1),     # fused QKV, 1B shape, left in bf16
    (1152, 1024, 1),     # o_proj, 1B shape
    (8192, 5376, 1),     # fused QKV, 31B shape
    (5376, 4096, 2),     # o_proj, 31B shape
    (37, 96, 1), (1, 8, 1), (16, 24, 3), (100, 1000, 4), (300, 160, 7),
    (129, 2056, 9), (65, 4104, 12), (1152, 6912, 16), (257, 64, 8),
])
def test_bf16_gemv_matches_oracle(n, k, m):
    W = inputs.weight(n, k, seed=7000 + n + k, device=DEV, outliers=False)
    x = inputs.tokens(m, k, seed=7100 + m, device=DEV)
    y = bf16_gpu(W, x)
    assert_gemv_close(y, oracle.gemv_bf16(bits(W), bits(x)), "bf16 n=%d k=%d m=%d" % (n, k, m))
    assert aq.poll_device_status() == aq.OK


def test_bf16_gemv_one_hot_is_exact():
    """A one-hot token returns the weight column bit for bit."""
    n, k = 300, 1000
    W = inputs.weight(n, k, seed=7201, device=DEV)
    for col in (0, 63, 64, 999):
        x = torch.zeros((1, k), dtype=torch.bfloat16, device=DEV)
        x[0, col] = 1.0
        assert torch.equal(bf16_gpu(W, x)[0], W[:, col])


@pytest.mark.parametrize("n,k", [(1152, 6912), (8192, 5376), (100, 1000)])
def test_bf16_gemv_is_independent_of_m_and_deterministic(n, k):
    W = inputs.weight(n, k, seed=7301, device=DEV)
    x = inputs.tokens(16, k, seed=7302, device=DEV)
    y16 = bf16_gpu(W, x)
    assert torch.equal(bf16_gpu(W, x), y16)
    for m in (1, 2, 3, 8, 9, 15):
        assert torch.equal(bf16_gpu(W, x[:m].contiguous()), y16[:m]), m
    assert torch.equal(bf16_gpu(W, x[5:6].contiguous(), flags=aq.STEP_PDL)[0], y16[5])


def test_bf16_lm_head_31b_sampled_parity():
    """The full-size ~31B tied lm_head [262144, 5376] at m = 1 in the launch
    configuration the bench times: 512 seeded rows against the oracle."""
    n, k = inputs.LM_HEAD_31B
    W = inputs.weight(n, k, seed=7401, device=DEV, outliers=False)
    x = inputs.tokens(1, k, seed=7402, device=DEV)
    y = bf16_gpu(W, x)
    rows = np.sort(np.random.default_rng(7403).choice(n, 512, replace=False))
    Wr = bits(W[torch.from_numpy(rows).to(DEV)])
    del W
    assert_gemv_close(y[:, rows], oracle.gemv_bf16(Wr, bits(x)), "lm_head 31B")
    assert aq.poll_device_status() == aq.OK


def test_bf16_and_nvfp4_share_one_workspace():
    """The two GEMVs leave the workspace as the other needs it."""
    shapes = [(8192, 5376), (5376, 21504)]
    Ws = [inputs.weight(n, k, seed=7500 + i, device=DEV) for i, (n, k) in enumerate(shapes)]
    qs = [quantize_gpu(W) for W in Ws]
    size = max(max(aq.gemv_bf16_workspace_bytes(n, k, 16), aq.gemv_workspace_bytes(n, k, 16))
               for n, k in shapes)
    shared = torch.zeros(size, dtype=torch.uint8, device=DEV)
    for i, (j, m, kind) in enumerate([(0, 1, "bf16"), (1, 3, "nvfp4"), (1, 1, "bf16"),
                                      (0, 12, "bf16"), (0, 1, "nvfp4"), (1, 2, "bf16")]):
        n, k = shapes[j]
        x = inputs.tokens(m, k, seed=7600 + i, device=DEV)
        if kind == "bf16":
            got, ref = bf16_gpu(Ws[j], x, ws=shared), bf16_gpu(Ws[j], x)
        else:
            got = gemv_gpu(qs[j], x, ws=shared, path=aq.PATH_GEMV_REGDECODE)
            ref = gemv_gpu(qs[j], x, path=aq.PATH_GEMV_REGDECODE)
        torch.cuda.synchronize()
        assert torch.equal(got, ref), (i, kind, j, m)
        assert aq.poll_device_status() == aq.OK
    assert not shared[: 12 << 20].any()
