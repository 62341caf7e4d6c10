"""Python face of the CPU oracle (ctypes over oracle/libaq_oracle.so).

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference
legs may import this package.  It shares no code with the CUDA library and
never imports it.  Arrays are numpy; bf16 values are carried as their
uint16 bit patterns.  The arithmetic lives in aq_oracle.c, which cites the
passage each function follows.
"""
import ctypes as C

import numpy as np

from . import build_oracle

_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = C.CDLL(build_oracle.build())
        _declare(_lib)
    return _lib


_p = C.c_void_p
_i64 = C.c_int64


def _declare(L):
    L.aqo_bf16_to_f32.argtypes = [C.c_uint16]
    L.aqo_bf16_to_f32.restype = C.c_float
    L.aqo_f32_to_bf16_rne.argtypes = [C.c_float]
    L.aqo_f32_to_bf16_rne.restype = C.c_uint16
    L.aqo_e4m3_decode.argtypes = [C.c_uint8]
    L.aqo_e4m3_decode.restype = C.c_float
    L.aqo_e4m3_encode_satfinite.argtypes = [C.c_float]
    L.aqo_e4m3_encode_satfinite.restype = C.c_uint8
    L.aqo_e2m1_decode.argtypes = [C.c_uint8]
    L.aqo_e2m1_decode.restype = C.c_float
    L.aqo_e2m1_encode_satfinite.argtypes = [C.c_float]
    L.aqo_e2m1_encode_satfinite.restype = C.c_uint8
    L.aqo_reconstruct.argtypes = [_p, _p, _p, _p, _i64, _i64, _i64, _p]
    L.aqo_reconstruct.restype = None
    L.aqo_amax_bf16.argtypes = [_p, _i64]
    L.aqo_amax_bf16.restype = C.c_float
    L.aqo_global_scales.argtypes = [C.c_float, C.POINTER(C.c_float),
                                    C.POINTER(C.c_float)]
    L.aqo_global_scales.restype = C.c_int
    L.aqo_quantize_rows.argtypes = [_p, _i64, _i64, C.c_float, _p, _p]
    L.aqo_quantize_rows.restype = None
    L.aqo_scale_layout_bytes.argtypes = [_i64, _i64]
    L.aqo_scale_layout_bytes.restype = _i64
    L.aqo_scale_layout_offset.argtypes = [_i64, _i64, _i64]
    L.aqo_scale_layout_offset.restype = _i64
    L.aqo_scales_to_device_layout.argtypes = [_p, _i64, _i64, _p]
    L.aqo_scales_to_device_layout.restype = None
    L.aqo_gemv.argtypes = [_p, _p, C.c_float, _p, _i64, _i64, _i64, _p, _i64, _p]
    L.aqo_gemv.restype = None
    L.aqo_quantize_act.argtypes = [_p, _i64, _i64, _p, _p, _p]
    L.aqo_quantize_act.restype = C.c_int
    L.aqo_gemv_q.argtypes = [_p, _p, C.c_float, _p, _p, _p, _i64, _i64, _i64,
                             _p, _i64, _p]
    L.aqo_gemv_q.restype = None
    L.aqo_gemv_bf16.argtypes = [_p, _p, _i64, _i64, _i64, _p, _i64, _p]
    L.aqo_gemv_bf16.restype = None
    L.aqo_gelu_tanh.argtypes = [C.c_double]
    L.aqo_gelu_tanh.restype = C.c_double
    L.aqo_gemv_glu.argtypes = [_p, _p, C.c_float, _p, _i64, _i64, _i64, _p, _i64, _p]
    L.aqo_gemv_glu.restype = None
    L.aqo_gemv_lowrank.argtypes = [_p, _p, C.c_float, _p, _p, _p, _i64, _p, _i64, _i64, _i64,
                                   _p, _i64, _p]
    L.aqo_gemv_lowrank.restype = None
    for name, tin, tout in (("aqo_bf16_round_array", np.float32, np.uint16),
                            ("aqo_e4m3_encode_array", np.float32, np.uint8),
                            ("aqo_e4m3_decode_array", np.uint8, np.float32),
                            ("aqo_e2m1_encode_array", np.float32, np.uint8),
                            ("aqo_e2m1_decode_array", np.uint8, np.float32)):
        fn = getattr(L, name)
        fn.argtypes = [_p, _i64, _p]
        fn.restype = None


RANGE_ERROR = 4


class OracleRangeError(ValueError):
    """amax non-finite, or so small that 2688/amax overflows."""


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data


# ------------------------------------------------------------ conversions

def bf16_bits_to_f32(bits):
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16_bits(values):
    v, pv = _c(values, np.float32)
    out = np.empty(v.shape, np.uint16)
    lib().aqo_bf16_round_array(pv, v.size, out.ctypes.data)
    return out


def e4m3_encode(values):
    v, pv = _c(values, np.float32)
    out = np.empty(v.shape, np.uint8)
    lib().aqo_e4m3_encode_array(pv, v.size, out.ctypes.data)
    return out


def e4m3_decode(codes):
    c, pc = _c(codes, np.uint8)
    out = np.empty(c.shape, np.float32)
    lib().aqo_e4m3_decode_array(pc, c.size, out.ctypes.data)
    return out


def e2m1_encode(values):
    v, pv = _c(values, np.float32)
    out = np.empty(v.shape, np.uint8)
    lib().aqo_e2m1_encode_array(pv, v.size, out.ctypes.data)
    return out


def e2m1_decode(nibbles):
    c, pc = _c(nibbles, np.uint8)
    out = np.empty(c.shape, np.float32)
    lib().aqo_e2m1_decode_array(pc, c.size, out.ctypes.data)
    return out


# ------------------------------------------------------------ the method

def reconstruct(W0, s, U, V):
    """W_eff bits [n,k] from W0 bits [n,k], s fp32 [n], U bits [n,r], V bits [k,r]."""
    W0, p0 = _c(W0, np.uint16)
    s, ps = _c(s, np.float32)
    U, pu = _c(U, np.uint16)
    V, pv = _c(V, np.uint16)
    n, k = W0.shape
    r = U.shape[1] if U.ndim == 2 else 0
    assert s.shape == (n,) and U.shape[0] == n and V.shape[0] == k
    assert r == 0 or V.shape[1] == r
    out = np.empty((n, k), np.uint16)
    lib().aqo_reconstruct(p0, ps, pu, pv, n, k, r, out.ctypes.data)
    return out


def amax(W):
    W, pw = _c(W, np.uint16)
    return float(lib().aqo_amax_bf16(pw, W.size))


def global_scales(a):
    """(g_enc, g_dec) as Python floats holding fp32 values."""
    ge, gd = C.c_float(), C.c_float()
    st = lib().aqo_global_scales(C.c_float(a), C.byref(ge), C.byref(gd))
    if st != 0:
        raise OracleRangeError("amax %r out of range" % a)
    return ge.value, gd.value


def quantize_rows(W, g_enc):
    """Quantise the rows of W bits [rows, k]: (packed [rows,k/2], scales [rows,k/16])."""
    W, pw = _c(W, np.uint16)
    rows, k = W.shape
    assert k % 16 == 0
    packed = np.empty((rows, k // 2), np.uint8)
    scales = np.empty((rows, k // 16), np.uint8)
    lib().aqo_quantize_rows(pw, rows, k, C.c_float(g_enc), packed.ctypes.data,
                            scales.ctypes.data)
    return packed, scales


def quantize(W):
    """Whole-tensor NVFP4 quantisation: (packed, canonical scales, g_enc, g_dec)."""
    ge, gd = global_scales(amax(W))
    packed, scales = quantize_rows(W, ge)
    return packed, scales, ge, gd


def scale_layout_bytes(n, k):
    return int(lib().aqo_scale_layout_bytes(n, k))


def scale_layout_offset(row, block, k):
    return int(lib().aqo_scale_layout_offset(row, block, k))


def scales_to_device_layout(canon, n, k):
    c, pc = _c(canon, np.uint8)
    assert c.shape == (n, k // 16)
    out = np.empty(scale_layout_bytes(n, k), np.uint8)
    lib().aqo_scales_to_device_layout(pc, n, k, out.ctypes.data)
    return out


def gemv(packed, scales, g_dec, x, rows=None):
    """fp64 y [m, nrows] = x [m,k] (bf16 bits) times dequantised weight rows."""
    packed, pp = _c(packed, np.uint8)
    scales, ps = _c(scales, np.uint8)
    x, px = _c(np.atleast_2d(x), np.uint16)
    n = packed.shape[0]
    m, k = x.shape
    assert packed.shape == (n, k // 2) and scales.shape == (n, k // 16)
    if rows is None:
        nrows, prow = n, None
    else:
        rows, prow = _c(rows, np.int64)
        nrows = rows.size
        assert rows.min(initial=0) >= 0 and rows.max(initial=0) < max(n, 1)
    y = np.empty((m, nrows), np.float64)
    lib().aqo_gemv(pp, ps, C.c_float(g_dec), px, m, n, k, prow, nrows,
                   y.ctypes.data)
    return y


def gemv_bf16(W, x, rows=None):
    """fp64 y [m, nrows] = x [m,k] times bf16 weight rows W [n,k] (both bf16 bits)."""
    W, pw = _c(W, np.uint16)
    x, px = _c(np.atleast_2d(x), np.uint16)
    n, k = W.shape
    m = x.shape[0]
    assert x.shape[1] == k
    if rows is None:
        nrows, prow = n, None
    else:
        rows, prow = _c(rows, np.int64)
        nrows = rows.size
        assert rows.min(initial=0) >= 0 and rows.max(initial=0) < max(n, 1)
    y = np.empty((m, nrows), np.float64)
    lib().aqo_gemv_bf16(pw, px, m, n, k, prow, nrows, y.ctypes.data)
    return y


def gemv_lowrank(packed, scales, g_dec, s, U, V, x, rows=None):
    """fp64 y [m, nrows] = s * (x w0_hat^T) + (x V) U^T for a quantised W0
    (packed, canonical scales, g_dec), s fp32 [n], U bits [n,r], V bits [k,r]."""
    packed, pp = _c(packed, np.uint8)
    scales, ps = _c(scales, np.uint8)
    s, pscale = _c(s, np.float32)
    x, px = _c(np.atleast_2d(x), np.uint16)
    n = packed.shape[0]
    m, k = x.shape
    r = 0 if U is None or np.asarray(U).size == 0 else np.asarray(U).size // n
    U, pu = _c(np.asarray(U if r else np.zeros((n, 1))).reshape(n, max(r, 1)), np.uint16)
    V, pv = _c(np.asarray(V if r else np.zeros((k, 1))).reshape(k, max(r, 1)), np.uint16)
    assert packed.shape == (n, k // 2) and scales.shape == (n, k // 16) and s.shape == (n,)
    if rows is None:
        nrows, prow = n, None
    else:
        rows, prow = _c(rows, np.int64)
        nrows = rows.size
        assert rows.min(initial=0) >= 0 and rows.max(initial=0) < max(n, 1)
    y = np.empty((m, nrows), np.float64)
    lib().aqo_gemv_lowrank(pp, ps, C.c_float(g_dec), pscale, pu if r else None,
                           pv if r else None, r, px, m, n, k, prow, nrows, y.ctypes.data)
    return y


def gelu_tanh(z):
    return float(lib().aqo_gelu_tanh(float(z)))


def interleave_gate_up(W):
    """Rows of the row-concatenated [gate; up] W [2f, k] in the 8-row
    interleaved order of the fused-activation GEMV (an index permutation)."""
    W = np.asarray(W)
    f = W.shape[0] // 2
    order = np.empty(2 * f, np.int64)
    for r in range(2 * f):
        g, i = divmod(r, 16)
        order[r] = g * 8 + i if i < 8 else f + g * 8 + (i - 8)
    return W[order]


def gemv_glu(packed, scales, g_dec, x, cols=None):
    """fp64 h [m, ncols] = gelu(y_gate) * y_up for an 8-row interleaved weight."""
    packed, pp = _c(packed, np.uint8)
    scales, ps = _c(scales, np.uint8)
    x, px = _c(np.atleast_2d(x), np.uint16)
    n = packed.shape[0]
    m, k = x.shape
    assert n % 16 == 0 and packed.shape == (n, k // 2) and scales.shape == (n, k // 16)
    if cols is None:
        ncols, pc = n // 2, None
    else:
        cols, pc = _c(cols, np.int64)
        ncols = cols.size
        assert cols.min(initial=0) >= 0 and cols.max(initial=0) < max(n // 2, 1)
    h = np.empty((m, ncols), np.float64)
    lib().aqo_gemv_glu(pp, ps, C.c_float(g_dec), px, m, n, k, pc, ncols, h.ctypes.data)
    return h


def quantize_segments(W, seg_end):
    """Per-segment quantisation: each row segment [seg_end[s-1], seg_end[s])
    of W bits through quantize() on its own.  Returns (packed [n,k/2],
    canonical scales [n,k/16], g_dec per segment as float32 [nseg])."""
    W = np.asarray(W)
    parts, start = [], 0
    for end in seg_end:
        parts.append(quantize(W[start:end]))
        start = end
    packed = np.concatenate([p[0] for p in parts])
    scales = np.concatenate([p[1] for p in parts])
    gdec = np.array([p[3] for p in parts], np.float32)
    return packed, scales, gdec


def gemv_segments(packed, scales, gdec, seg_end, x):
    """fp64 y [m, n]: each segment's rows through gemv() with its own g_dec."""
    ys, start = [], 0
    for s, end in enumerate(seg_end):
        ys.append(gemv(packed[start:end], scales[start:end], float(gdec[s]), x))
        start = end
    return np.concatenate(ys, axis=1)


def quantize_act(x):
    """Per-row activation quantisation: (packed [m,k/2], scales [m,k/16], g_dec [m])."""
    x, px = _c(np.atleast_2d(x), np.uint16)
    m, k = x.shape
    packed = np.empty((m, k // 2), np.uint8)
    scales = np.empty((m, k // 16), np.uint8)
    gdec = np.empty(m, np.float32)
    st = lib().aqo_quantize_act(px, m, k, packed.ctypes.data,
                                scales.ctypes.data, gdec.ctypes.data)
    if st != 0:
        raise OracleRangeError("activation row amax out of range")
    return packed, scales, gdec


def gemv_q(w_packed, w_scales, w_gdec, x_packed, x_scales, x_gdec, rows=None):
    """fp64 y [m, nrows] from a quantised weight and quantised activations."""
    wp, pwp = _c(w_packed, np.uint8)
    ws, pws = _c(w_scales, np.uint8)
    xp, pxp = _c(np.atleast_2d(x_packed), np.uint8)
    xs, pxs = _c(np.atleast_2d(x_scales), np.uint8)
    xg, pxg = _c(np.atleast_1d(x_gdec), np.float32)
    n, half_k = wp.shape
    k = half_k * 2
    m = xp.shape[0]
    if rows is None:
        nrows, prow = n, None
    else:
        rows, prow = _c(rows, np.int64)
        nrows = rows.size
    y = np.empty((m, nrows), np.float64)
    lib().aqo_gemv_q(pwp, pws, C.c_float(w_gdec), pxp, pxs, pxg, m, n, k, prow,
                     nrows, y.ctypes.data)
    return y
