"""Helpers of the GPU parity tests: run the CUDA path through the C ABI and
compare with the CPU oracle on the same seeded inputs."""
import numpy as np
import torch

import oracle
from nvfp4_block_scaled_aq_gb300 import aq, inputs

DEV = torch.device("cuda:0")

# GEMV acceptance (reading R10): |y - y_ref| <= REL * max(|y_ref|, FLOOR *
# rms(y_ref)) + half a bf16 ulp of the output.  REL is the stated 2e-3 on
# the fp32-accumulated value; the bf16 output rounding adds up to half an
# ulp (2^-8 relative, which alone would exceed 2e-3).
REL = 2e-3
FLOOR = 1e-2


def require_gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(DEV)


def quantize_gpu(W):
    n, k = W.shape
    w = aq.Nvfp4Weight.empty(n, k, device=W.device)
    ws = torch.zeros(aq.quantize_workspace_bytes(), dtype=torch.uint8, device=W.device)
    aq.quantize(W, w, ws)
    return w


def gemv_gpu(w, x, ws=None, path=None):
    m = x.shape[0]
    if ws is None:
        ws = torch.zeros(aq.gemv_workspace_bytes(w.n, w.k, m), dtype=torch.uint8,
                         device=x.device)
    y = torch.empty((m, w.n), dtype=torch.bfloat16, device=x.device)
    aq.gemv(w, x, y, ws, path=aq.PATH_AUTO if path is None else path)
    return y


# The two GEMV kernels: the tcgen05 one serves 1..5 tokens.
KERNELS = {"tcgen05": (aq.PATH_GEMV_TCGEN05, 5), "regdecode": (aq.PATH_GEMV_REGDECODE, 16)}


def weight_bytes(w):
    """(packed [n, k/2], device-layout scales, g_dec) copied to the host."""
    torch.cuda.synchronize()
    return (w.packed.cpu().numpy().reshape(w.n, w.k // 2), w.scales.cpu().numpy(),
            float(w.global_scale.cpu().numpy()[0]))


def canonical_scales(w):
    canon = torch.empty(w.n * (w.k // 16), dtype=torch.uint8, device=w.packed.device)
    aq.scales_to_canonical(w, canon)
    return canon.cpu().numpy().reshape(w.n, w.k // 16)


def assert_quantized_equal(w, W_bits):
    """GPU bytes == oracle bytes for the whole tensor."""
    packed, scales, ge, gd = oracle.quantize(W_bits)
    gp, gs, ggd = weight_bytes(w)
    n, k = W_bits.shape
    bad = np.argwhere(gp != packed)
    assert bad.size == 0, "packed differs at %s (gpu %s, oracle %s)" % (
        bad[:5].tolist(), gp[tuple(bad[0])], packed[tuple(bad[0])])
    dev_layout = oracle.scales_to_device_layout(scales, n, k)
    assert np.array_equal(gs, dev_layout), "device-layout scales differ"
    assert np.array_equal(canonical_scales(w), scales), "canonical scales differ"
    assert np.float32(ggd) == np.float32(gd), (ggd, gd)
    return packed, scales, ge, gd


def bf16_half_ulp(v):
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.exp2(e - 8), 0.0)


def gemv_errors(y_gpu, y_ref):
    """Normalised errors |y - y_ref| / tolerance (<= 1 passes)."""
    yg = y_gpu.float().cpu().numpy().astype(np.float64) if torch.is_tensor(y_gpu) \
        else np.asarray(y_gpu, np.float64)
    rms = np.sqrt(np.mean(y_ref ** 2)) if y_ref.size else 0.0
    tol = REL * np.maximum(np.abs(y_ref), FLOOR * rms) + \
        bf16_half_ulp(np.maximum(np.abs(y_ref), np.abs(yg)))
    tol = np.where(tol > 0, tol, 1e-300)
    return np.abs(yg - y_ref) / tol


def bf16_round(v):
    """fp64 -> nearest bf16 value (ties to even), as fp64; no double
    rounding through fp32."""
    v = np.asarray(v, np.float64)
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    ulp = np.exp2(e - 7)
    return np.where(a > 0, np.round(v / ulp) * ulp, 0.0)


# Second GEMV check: the output within one bf16 ulp of the correctly rounded
# oracle value on at least ULP_RATE of the outputs.  Outputs in deep
# cancellation (|y_ref| < 2^-10 rms(y_ref)) are left out: there one bf16 ulp
# of the output is as small as the fp32 accumulation's own rounding over
# thousands of terms, and the R10 floor already governs them.
ULP_RATE = 0.999


def ulp_agreement(y_gpu, y_ref):
    """(fraction within one bf16 ulp, outputs counted)."""
    yg = y_gpu.float().cpu().numpy().astype(np.float64) if torch.is_tensor(y_gpu) \
        else np.asarray(y_gpu, np.float64)
    y_ref = np.asarray(y_ref, np.float64)
    if y_ref.size == 0:
        return 1.0, 0
    rms = np.sqrt(np.mean(y_ref ** 2))
    keep = np.abs(y_ref) >= np.exp2(-10) * rms
    q = bf16_round(y_ref)
    aq_ = np.abs(q)
    ulp = np.where(aq_ > 0, np.exp2(np.floor(np.log2(np.where(aq_ > 0, aq_, 1.0))) - 7), 0.0)
    ok = np.abs(yg - q) <= ulp
    n = int(keep.sum())
    return (float(ok[keep].mean()) if n else 1.0), n


def assert_gemv_close(y_gpu, y_ref, what=""):
    err = gemv_errors(y_gpu, y_ref)
    worst = np.unravel_index(np.argmax(err), err.shape) if err.size else None
    assert err.size == 0 or err.max() <= 1.0, "%s: max normalised error %.3f at %s" % (
        what, err.max(), worst)
    rate, n = ulp_agreement(y_gpu, y_ref)
    assert rate >= ULP_RATE, "%s: %.5f of %d outputs within one bf16 ulp (need %.3f)" % (
        what, rate, n, ULP_RATE)
    return float(err.max()) if err.size else 0.0


def bits(t):
    return inputs.bits_u16(t)
