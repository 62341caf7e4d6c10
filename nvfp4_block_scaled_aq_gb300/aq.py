"""ctypes binding of libaq.so, the C-ABI declared in include/aq.h.

Argument marshalling only: every step of the computation runs in the
library's CUDA kernels.  PyTorch supplies device memory (``data_ptr()``)
and streams (``cuda_stream``); nothing here computes on tensor values.
The library is loaded on first use and a missing build raises
``AqLibraryMissing`` -- there is no fallback.
"""
import ctypes as C
import os
from dataclasses import dataclass

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libaq.so")

# aq_status
OK = 0
ERR_INVALID_ARG = 1
ERR_SHAPE = 2
ERR_ALIGNMENT = 3
ERR_RANGE = 4
ERR_UNSUPPORTED = 5
ERR_TIMEOUT = 6
ERR_CUDA = 7
ERR_WORKSPACE = 8
STATUS_NAMES = {0: "AQ_OK", 1: "AQ_ERR_INVALID_ARG", 2: "AQ_ERR_SHAPE",
                3: "AQ_ERR_ALIGNMENT", 4: "AQ_ERR_RANGE", 5: "AQ_ERR_UNSUPPORTED",
                6: "AQ_ERR_TIMEOUT", 7: "AQ_ERR_CUDA", 8: "AQ_ERR_WORKSPACE"}

PATH_AUTO, PATH_GEMV, PATH_MMA, PATH_GEMV_REGDECODE, PATH_GEMV_TCGEN05 = 0, 1, 2, 3, 4
STEP_PDL = 1
STEP_REGDECODE = 2
STEP_TCGEN05 = 4
STEP_MMA = 8
MAX_M = 16
MAX_M_MMA = 64
NOALLOC_MAX_SCRATCH = 32 << 20  # AQ_GEMV_NOALLOC_MAX_SCRATCH


class AqLibraryMissing(RuntimeError):
    pass


class AqError(RuntimeError):
    def __init__(self, status, message):
        super().__init__("%s: %s" % (STATUS_NAMES.get(status, status), message))
        self.status = status


class Nvfp4WeightC(C.Structure):
    _fields_ = [("n", C.c_int32), ("k", C.c_int32), ("packed", C.c_void_p),
                ("scales", C.c_void_p), ("global_scale", C.c_void_p)]


_lib = None
_p = C.c_void_p
_i32 = C.c_int32
_sz = C.c_size_t


def lib():
    """The loaded library (raises AqLibraryMissing if it was never built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise AqLibraryMissing(
                "libaq.so is not built; run nvfp4_block_scaled_aq_gb300/build.py "
                "(or __graft_entry__.build())")
        L = C.CDLL(LIB_PATH)
        _declare(L)
        _lib = L
    return _lib


def _declare(L):
    W = C.POINTER(Nvfp4WeightC)
    sigs = {
        "aq_version": ([], _i32),
        "aq_last_error": ([], C.c_char_p),
        "aq_packed_bytes": ([_i32, _i32], _sz),
        "aq_scale_bytes": ([_i32, _i32], _sz),
        "aq_reconstruct": ([_p, _p, _p, _p, _i32, _i32, _i32, _p, _p], C.c_int),
        "aq_quantize_workspace_bytes": ([], _sz),
        "aq_quantize_nvfp4": ([_p, _i32, _i32, W, _p, _sz, _p], C.c_int),
        "aq_reconstruct_quantize_nvfp4": ([_p, _p, _p, _p, _i32, _i32, _i32, W, _p,
                                           _sz, _p], C.c_int),
        "aq_gemv_workspace_bytes": ([_i32, _i32, _i32], _sz),
        "aq_gemv_nvfp4": ([W, _p, _i32, _p, C.c_int, _p, _sz, _p], C.c_int),
        "aq_gemv_nvfp4_noalloc": ([W, _p, _i32, _p, C.c_int, _p], C.c_int),
        "aq_gemv_bf16_workspace_bytes": ([_i32, _i32, _i32], _sz),
        "aq_gemv_lowrank_workspace_bytes": ([_i32, _i32, _i32, _i32], _sz),
        "aq_interleave_gate_up": ([_p, _i32, _i32, _p, _p], C.c_int),
        "aq_selftest_timeout": ([C.c_uint32, _p], C.c_int),
        "aq_quantize_nvfp4_segments": ([_p, _i32, _i32, _i32, C.POINTER(_i32), W, _p, _sz, _p],
                                       C.c_int),
        "aq_gemv_nvfp4_segments": ([W, _i32, C.POINTER(_i32), _p, _i32, _p, C.c_uint32, _p, _sz,
                                    _p], C.c_int),
        "aq_gemv_glu_nvfp4": ([W, _p, _i32, _p, C.c_uint32, _p, _sz, _p], C.c_int),
        "aq_gemv_lowrank_nvfp4": ([W, _p, _p, _p, _i32, _p, _i32, _p, C.c_uint32, _p, _sz, _p],
                                  C.c_int),
        "aq_gemv_bf16": ([_p, _i32, _i32, _p, _i32, _p, C.c_uint32, _p, _sz, _p], C.c_int),
        "aq_quantize_act_nvfp4": ([_p, _i32, _i32, _p, _p, _p, _p], C.c_int),
        "aq_decode_step_weights": ([W, _i32, C.POINTER(_p), C.POINTER(_p), _i32,
                                    C.c_uint32, _p, _sz, _p], C.c_int),
        "aq_scales_to_canonical": ([W, _p, _p], C.c_int),
        "aq_step_plan_bytes": ([_i32], _sz),
        "aq_step_plan_create": ([W, _i32, C.POINTER(_p), C.POINTER(_p), _i32, _p, _sz,
                                 C.POINTER(_sz)], C.c_int),
        "aq_step_run": ([_p, _i32, _p, _sz, _p], C.c_int),
        "aq_poll_device_status": ([_p], C.c_int),
    }
    for name, (args, res) in sigs.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = res


def last_error() -> str:
    return lib().aq_last_error().decode()


def check(status):
    if status != OK:
        raise AqError(status, last_error())
    return status


def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream)


# ------------------------------------------------------------ weights

@dataclass
class Nvfp4Weight:
    """Device buffers of one NVFP4 weight [n, k] (allocated by torch)."""
    n: int
    k: int
    packed: "object"        # uint8 [n*k/2]
    scales: "object"        # uint8 [aq_scale_bytes(n, k)]
    global_scale: "object"  # float32 [1]

    @classmethod
    def empty(cls, n, k, device="cuda", nscales=1):
        import torch
        pb = lib().aq_packed_bytes(n, k)
        sb = lib().aq_scale_bytes(n, k)
        if pb == 0 or sb == 0:
            raise AqError(ERR_SHAPE, "unsupported weight shape [%d, %d]" % (n, k))
        return cls(n, k, torch.empty(pb, dtype=torch.uint8, device=device),
                   torch.empty(sb, dtype=torch.uint8, device=device),
                   torch.empty(nscales, dtype=torch.float32, device=device))

    def c(self):
        return Nvfp4WeightC(self.n, self.k, self.packed.data_ptr(),
                            self.scales.data_ptr(), self.global_scale.data_ptr())

    @property
    def nbytes(self):
        return self.packed.numel() + self.scales.numel()


def packed_bytes(n, k):
    return int(lib().aq_packed_bytes(n, k))


def scale_bytes(n, k):
    return int(lib().aq_scale_bytes(n, k))


# ------------------------------------------------------------ calls

def reconstruct(W0, s, U, V, W_eff, stream=None):
    n, k = W0.shape
    r = 0 if U is None else U.shape[1]
    check(lib().aq_reconstruct(_ptr(W0), _ptr(s), _ptr(U), _ptr(V), n, k, r,
                               _ptr(W_eff), _stream(stream)))


def quantize_workspace_bytes():
    return int(lib().aq_quantize_workspace_bytes())


def quantize(W, out: Nvfp4Weight, workspace, stream=None):
    n, k = W.shape
    wc = out.c()
    check(lib().aq_quantize_nvfp4(_ptr(W), n, k, C.byref(wc), _ptr(workspace),
                                  workspace.numel() * workspace.element_size(),
                                  _stream(stream)))


def reconstruct_quantize(W0, s, U, V, out: Nvfp4Weight, workspace, stream=None):
    n, k = W0.shape
    r = 0 if U is None else U.shape[1]
    wc = out.c()
    check(lib().aq_reconstruct_quantize_nvfp4(
        _ptr(W0), _ptr(s), _ptr(U), _ptr(V), n, k, r, C.byref(wc), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def gemv_workspace_bytes(n, k, m=1):
    b = int(lib().aq_gemv_workspace_bytes(n, k, m))
    if b == 0:
        raise AqError(ERR_SHAPE, last_error() or "bad GEMV shape")
    return b


def gemv(w: Nvfp4Weight, x, y, workspace, path=PATH_AUTO, stream=None):
    m = x.shape[0]
    wc = w.c()
    check(lib().aq_gemv_nvfp4(C.byref(wc), _ptr(x), m, _ptr(y), path, _ptr(workspace),
                              workspace.numel() * workspace.element_size(),
                              _stream(stream)))


def gemv_bf16_workspace_bytes(n, k, m=1):
    b = int(lib().aq_gemv_bf16_workspace_bytes(n, k, m))
    if b == 0:
        raise AqError(ERR_SHAPE, last_error() or "bad bf16 GEMV shape")
    return b


def gemv_bf16(W, x, y, workspace, flags=0, stream=None):
    """y [m, n] = x [m, k] W [n, k]^T for a bf16 weight (aq_gemv_bf16)."""
    n, k = W.shape
    check(lib().aq_gemv_bf16(_ptr(W), n, k, _ptr(x), x.shape[0], _ptr(y), flags,
                             _ptr(workspace), workspace.numel() * workspace.element_size(),
                             _stream(stream)))


def interleave_gate_up(W, out, stream=None):
    """Row-concatenated [gate; up] bf16 W [2f, k] -> the 8-row interleaved
    order of the fused-activation GEMV (aq_interleave_gate_up)."""
    check(lib().aq_interleave_gate_up(_ptr(W), W.shape[0] // 2, W.shape[1], _ptr(out),
                                      _stream(stream)))


def gemv_glu(w: "Nvfp4Weight", x, h, workspace, flags=0, stream=None):
    """h [m, n/2] = gelu(gate) * up of an interleaved fused weight (aq_gemv_glu_nvfp4)."""
    wc = w.c()
    check(lib().aq_gemv_glu_nvfp4(C.byref(wc), _ptr(x), x.shape[0], _ptr(h), flags,
                                  _ptr(workspace), workspace.numel() * workspace.element_size(),
                                  _stream(stream)))


def selftest_timeout(polls=4096, stream=None):
    """Run the bounded-wait failure path once (aq_selftest_timeout)."""
    check(lib().aq_selftest_timeout(polls, _stream(stream)))


MAX_SEGMENTS = 8  # AQ_MAX_SEGMENTS


def _seg_array(seg_end):
    return (_i32 * len(seg_end))(*[int(e) for e in seg_end])


def quantize_segments(W, seg_end, out: "Nvfp4Weight", workspace, stream=None):
    """Each row segment of W quantised on its own (aq_quantize_nvfp4_segments);
    out.global_scale holds one g_dec per segment."""
    n, k = W.shape
    wc = out.c()
    check(lib().aq_quantize_nvfp4_segments(_ptr(W), n, k, len(seg_end), _seg_array(seg_end),
                                           C.byref(wc), _ptr(workspace),
                                           workspace.numel() * workspace.element_size(),
                                           _stream(stream)))


def gemv_segments(w: "Nvfp4Weight", seg_end, x, y, workspace, flags=0, stream=None):
    """y = bf16(g_dec[segment(row)] * acc) (aq_gemv_nvfp4_segments)."""
    wc = w.c()
    check(lib().aq_gemv_nvfp4_segments(C.byref(wc), len(seg_end), _seg_array(seg_end), _ptr(x),
                                       x.shape[0], _ptr(y), flags, _ptr(workspace),
                                       workspace.numel() * workspace.element_size(),
                                       _stream(stream)))


LOWRANK_MAX_R = 16  # AQ_LOWRANK_MAX_R


def gemv_lowrank_workspace_bytes(n, k, m=1, r=0):
    b = int(lib().aq_gemv_lowrank_workspace_bytes(n, k, m, r))
    if b == 0:
        raise AqError(ERR_SHAPE, last_error() or "bad low-rank GEMV shape")
    return b


def gemv_lowrank(w0: "Nvfp4Weight", s, U, V, x, y, workspace, flags=0, stream=None):
    """y = s * (W0_hat x) + U (V^T x) (aq_gemv_lowrank_nvfp4); U [n, r] and
    V [k, r] bf16, or None when r = 0."""
    r = 0 if U is None else U.shape[1]
    wc = w0.c()
    check(lib().aq_gemv_lowrank_nvfp4(C.byref(wc), _ptr(s), _ptr(U), _ptr(V), r, _ptr(x),
                                      x.shape[0], _ptr(y), flags, _ptr(workspace),
                                      workspace.numel() * workspace.element_size(),
                                      _stream(stream)))


def quantize_act(x, packed, scales, g_dec, stream=None):
    """Per-row NVFP4 quantisation of activations x [m, k] (canonical scales)."""
    m, k = x.shape
    check(lib().aq_quantize_act_nvfp4(_ptr(x), m, k, _ptr(packed), _ptr(scales), _ptr(g_dec),
                                      _stream(stream)))


def gemv_noalloc(w: Nvfp4Weight, x, y, path=PATH_AUTO, stream=None):
    """aq_gemv_nvfp4 with the library's own fixed scratch (no workspace)."""
    m = x.shape[0]
    wc = w.c()
    check(lib().aq_gemv_nvfp4_noalloc(C.byref(wc), _ptr(x), m, _ptr(y), path,
                                      _stream(stream)))


class StepArgs:
    """Host arrays of one decode step (kept alive while the step is reused)."""

    def __init__(self, weights, xs, ys):
        n = len(weights)
        assert len(xs) == n and len(ys) == n
        self.n = n
        self.w = (Nvfp4WeightC * n)(*[w.c() for w in weights])
        self.x = (C.c_void_p * n)(*[t.data_ptr() for t in xs])
        self.y = (C.c_void_p * n)(*[t.data_ptr() for t in ys])
        self.m = xs[0].shape[0] if n else 1


def decode_step(args: StepArgs, workspace, flags=STEP_PDL, stream=None):
    check(lib().aq_decode_step_weights(args.w, args.n, args.x, args.y, args.m, flags,
                                       _ptr(workspace),
                                       workspace.numel() * workspace.element_size(),
                                       _stream(stream)))


class StepPlan:
    """A persistent decode-step plan: device buffer written once by
    aq_step_plan_create.  Keeps the weights and activation buffers it
    points to alive."""

    def __init__(self, weights, xs, ys):
        import torch
        self.args = StepArgs(weights, xs, ys)
        self.keep = (list(weights), list(xs), list(ys))
        self.m = self.args.m
        nbytes = int(lib().aq_step_plan_bytes(self.args.n))
        if nbytes == 0:
            raise AqError(ERR_INVALID_ARG, "bad projection count")
        self.buf = torch.empty(nbytes, dtype=torch.uint8, device=xs[0].device)
        ws = C.c_size_t(0)
        check(lib().aq_step_plan_create(self.args.w, self.args.n, self.args.x, self.args.y,
                                        self.m, _ptr(self.buf), nbytes, C.byref(ws)))
        self.workspace_bytes = int(ws.value)

    def workspace(self):
        import torch
        return torch.zeros(self.workspace_bytes, dtype=torch.uint8, device=self.buf.device)


def step_run(plan: StepPlan, workspace, m=None, stream=None):
    check(lib().aq_step_run(_ptr(plan.buf), plan.m if m is None else m, _ptr(workspace),
                            workspace.numel() * workspace.element_size(), _stream(stream)))


def scales_to_canonical(w: Nvfp4Weight, canon, stream=None):
    wc = w.c()
    check(lib().aq_scales_to_canonical(C.byref(wc), _ptr(canon), _stream(stream)))


def poll_device_status(stream=None):
    """Synchronises the stream; returns the aq_status code (does not raise)."""
    return lib().aq_poll_device_status(_stream(stream))
