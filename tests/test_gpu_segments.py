"""GPU parity of per-segment tensor scales (aq_quantize_nvfp4_segments,
aq_gemv_nvfp4_segments): every byte and each segment's g_dec as the oracle
quantising the segments on their own; the GEMV within the tolerance of the
oracle's per-segment product; one segment equal to the plain calls."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import (DEV, assert_gemv_close, bits, canonical_scales, gemv_gpu, quantize_gpu,
                         require_gpu)
from nvfp4_block_scaled_aq_gb300 import aq, inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    require_gpu()
    aq.lib()


def quantize_segments_gpu(W, seg_end):
    n, k = W.shape
    w = aq.Nvfp4Weight.empty(n, k, device=DEV, nscales=len(seg_end))
    ws = torch.zeros(aq.quantize_workspace_bytes(), dtype=torch.uint8, device=DEV)
    aq.quantize_segments(W, seg_end, w, ws)
    torch.cuda.synchronize()
    return w


def gemv_segments_gpu(w, seg_end, x, flags=0):
    m = x.shape[0]
    ws = torch.zeros(aq.gemv_workspace_bytes(w.n, w.k, m), dtype=torch.uint8, device=DEV)
    y = torch.full((m, w.n), float("nan"), dtype=torch.bfloat16, device=DEV)
    aq.gemv_segments(w, seg_end, x, y, ws, flags=flags)
    torch.cuda.synchronize()
    return y


def qkv_like(seg_end, k, seed):
    """Segments with very different ranges (x1, x64, x1/8), like q, k, v."""
    parts, start = [], 0
    for s, end in enumerate(seg_end):
        W = inputs.weight(end - start, k, seed=seed + s, device=DEV)
        parts.append((W.float() * (1.0, 64.0, 0.125, 4.0)[s % 4]).to(torch.bfloat16))
        start = end
    return torch.cat(parts)


@pytest.mark.parametrize("seg_end,k", [
    ([64, 96, 128], 256), ([16, 32, 48, 64, 80, 96, 112, 120], 64), ([300], 160),
    ([4096, 6144, 8192], 5376),   # the ~31B fused QKV split q / k / v
])
def test_segment_quantisation_bit_exact(seg_end, k):
    W = qkv_like(seg_end, k, 9500)
    w = quantize_segments_gpu(W, seg_end)
    packed, scales, gdec = oracle.quantize_segments(bits(W), seg_end)
    assert np.array_equal(w.packed.cpu().numpy().reshape(w.n, k // 2), packed)
    assert np.array_equal(canonical_scales(w), scales)
    assert np.array_equal(w.global_scale.cpu().numpy().view(np.uint32), gdec.view(np.uint32))


@pytest.mark.parametrize("seg_end,k,m", [
    ([64, 96, 128], 256, 1), ([16, 32, 48, 64, 80, 96, 112, 120], 64, 3), ([4096, 6144, 8192], 5376, 1),
    ([1536, 1920, 2304], 1152, 9),
])
def test_segment_gemv_matches_oracle(seg_end, k, m):
    W = qkv_like(seg_end, k, 9600)
    x = inputs.tokens(m, k, seed=9700 + m, device=DEV)
    w = quantize_segments_gpu(W, seg_end)
    packed, scales, gdec = oracle.quantize_segments(bits(W), seg_end)
    y_ref = oracle.gemv_segments(packed, scales, gdec, seg_end, bits(x))
    assert_gemv_close(gemv_segments_gpu(w, seg_end, x), y_ref, "segments %s m=%d" % (seg_end, m))
    assert aq.poll_device_status() == aq.OK


def test_one_segment_is_the_plain_path_and_m_invariant():
    n, k = 1536, 1152
    W = inputs.weight(n, k, seed=9801, device=DEV)
    x = inputs.tokens(12, k, seed=9802, device=DEV)
    w1 = quantize_segments_gpu(W, [n])
    w = quantize_gpu(W)
    assert torch.equal(w1.packed, w.packed) and torch.equal(w1.scales, w.scales)
    assert torch.equal(w1.global_scale, w.global_scale)
    y = gemv_segments_gpu(w1, [n], x)
    assert torch.equal(y, gemv_gpu(w, x, path=aq.PATH_GEMV_REGDECODE))
    seg = [512, 1024, 1536]
    w3 = quantize_segments_gpu(qkv_like(seg, k, 9803), seg)
    y3 = gemv_segments_gpu(w3, seg, x)
    for m in (2, 5):
        assert torch.equal(gemv_segments_gpu(w3, seg, x[:m].contiguous(), flags=aq.STEP_PDL),
                           y3[:m])
    # one token: the one-token kernel form, held to the oracle
    W3 = qkv_like(seg, k, 9803)
    packed, scales, gdec = oracle.quantize_segments(bits(W3), seg)
    assert_gemv_close(gemv_segments_gpu(w3, seg, x[:1].contiguous(), flags=aq.STEP_PDL),
                      oracle.gemv_segments(packed, scales, gdec, seg, bits(x[:1])), "one token")
