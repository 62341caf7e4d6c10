// api.cu -- the extern "C" entry points of libaq.so declared in
// include/aq.h: host-side validation, per-device set-up, the device status
// word and the thread-local error message.  Every check runs before any
// launch; a failed check launches nothing.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "aq_internal.cuh"

namespace aq {

// The device status word (one per device that loads the library).
__device__ unsigned g_device_status = 0;

namespace {

thread_local char t_err[512] = "";

constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];
std::once_flag g_dev_once[kMaxDevices];
aq_status g_dev_state[kMaxDevices];

}  // namespace

aq_status set_error(aq_status st, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_err, sizeof t_err, fmt, ap);
  va_end(ap);
  return st;
}

aq_status cuda_error(cudaError_t e, const char *what) {
  return set_error(AQ_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e),
                   cudaGetErrorString(e));
}

const DeviceInfo *device_info() {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    cuda_error(e, "cudaGetDevice");
    return nullptr;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    set_error(AQ_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
    return nullptr;
  }
  std::call_once(g_dev_once[dev], [dev] {
    DeviceInfo &d = g_dev[dev];
    d.ordinal = dev;
    g_dev_state[dev] = AQ_OK;
    cudaDeviceProp prop;
    cudaError_t err = cudaGetDeviceProperties(&prop, dev);
    if (err != cudaSuccess) {
      g_dev_state[dev] = AQ_ERR_CUDA;
      return;
    }
    d.sms = prop.multiProcessorCount;
    d.cc_major = prop.major;
    d.cc_minor = prop.minor;
    d.smem_optin = prop.sharedMemPerBlockOptin;
    if (prop.major != 10 || prop.minor != 3) {
      g_dev_state[dev] = AQ_ERR_UNSUPPORTED;
      return;
    }
    void *p = nullptr;
    err = cudaGetSymbolAddress(&p, g_device_status);
    if (err != cudaSuccess) {
      g_dev_state[dev] = AQ_ERR_CUDA;
      return;
    }
    d.status = static_cast<unsigned *>(p);
  });
  switch (g_dev_state[dev]) {
    case AQ_OK:
      return &g_dev[dev];
    case AQ_ERR_UNSUPPORTED:
      set_error(AQ_ERR_UNSUPPORTED,
                "device %d is sm_%d%d; this library is built for sm_103a (GB300) only", dev,
                g_dev[dev].cc_major, g_dev[dev].cc_minor);
      return nullptr;
    default:
      set_error(AQ_ERR_CUDA, "could not set up device %d", dev);
      return nullptr;
  }
}

}  // namespace aq

using namespace aq;

namespace {

constexpr int32_t kMaxN = 1 << 24;
constexpr int32_t kMaxK = 1 << 20;
constexpr int32_t kMaxR = 64;

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

aq_status check_nk(int32_t n, int32_t k) {
  if (n < 1 || n > kMaxN)
    return set_error(AQ_ERR_SHAPE, "n = %d outside [1, %d]", n, kMaxN);
  if (k < 32 || k > kMaxK || k % 32 != 0)
    return set_error(AQ_ERR_SHAPE, "k = %d must be a multiple of 32 in [32, %d]", k, kMaxK);
  return AQ_OK;
}

aq_status check_theta(const uint16_t *W0, const float *s, const uint16_t *U,
                      const uint16_t *V, int32_t n, int32_t k, int32_t r) {
  aq_status st = check_nk(n, k);
  if (st != AQ_OK) return st;
  if (r < 0 || r > kMaxR) return set_error(AQ_ERR_SHAPE, "r = %d outside [0, %d]", r, kMaxR);
  if (!W0 || !s) return set_error(AQ_ERR_INVALID_ARG, "W0 and s must not be NULL");
  if (r > 0 && (!U || !V)) return set_error(AQ_ERR_INVALID_ARG, "U and V must not be NULL when r > 0");
  if (!aligned(W0, 16)) return set_error(AQ_ERR_ALIGNMENT, "W0 must be 16-byte aligned");
  if (!aligned(s, 4) || (r > 0 && (!aligned(U, 2) || !aligned(V, 2))))
    return set_error(AQ_ERR_ALIGNMENT, "s, U, V must be naturally aligned");
  return AQ_OK;
}

aq_status check_weight(const aq_nvfp4_weight *w, const char *what) {
  if (!w) return set_error(AQ_ERR_INVALID_ARG, "%s: weight descriptor is NULL", what);
  aq_status st = check_nk(w->n, w->k);
  if (st != AQ_OK) return st;
  if (!w->packed || !w->scales || !w->global_scale)
    return set_error(AQ_ERR_INVALID_ARG, "%s: weight pointers must not be NULL", what);
  if (!aligned(w->packed, 16) || !aligned(w->scales, 16) || !aligned(w->global_scale, 4))
    return set_error(AQ_ERR_ALIGNMENT, "%s: packed and scales must be 16-byte aligned", what);
  return AQ_OK;
}

aq_status check_ws(void *ws, size_t have, size_t need, const char *what) {
  if (need == 0) return AQ_OK;
  if (!ws) return set_error(AQ_ERR_WORKSPACE, "%s: workspace is NULL", what);
  if (!aligned(ws, 256)) return set_error(AQ_ERR_WORKSPACE, "%s: workspace must be 256-byte aligned", what);
  if (have < need)
    return set_error(AQ_ERR_WORKSPACE, "%s: workspace of %zu bytes, %zu needed", what, have, need);
  return AQ_OK;
}

aq_status launched(cudaError_t e, const char *what) {
  return e == cudaSuccess ? AQ_OK : cuda_error(e, what);
}

aq_status quantize_common(const uint16_t *W, const float *s, const uint16_t *U,
                          const uint16_t *V, int32_t n, int32_t k, int32_t r, bool fused,
                          const aq_nvfp4_weight *out, void *ws, size_t ws_bytes,
                          aq_stream_t stream) {
  const char *what = fused ? "aq_reconstruct_quantize_nvfp4" : "aq_quantize_nvfp4";
  aq_status st = fused ? check_theta(W, s, U, V, n, k, r) : check_nk(n, k);
  if (st != AQ_OK) return st;
  if (!fused && !W) return set_error(AQ_ERR_INVALID_ARG, "%s: W is NULL", what);
  if (!fused && !aligned(W, 16)) return set_error(AQ_ERR_ALIGNMENT, "%s: W must be 16-byte aligned", what);
  if ((st = check_weight(out, what)) != AQ_OK) return st;
  if (out->n != n || out->k != k)
    return set_error(AQ_ERR_SHAPE, "%s: out is [%d, %d], input is [%d, %d]", what, out->n,
                     out->k, n, k);
  if ((st = check_ws(ws, ws_bytes, aq_quantize_workspace_bytes(), what)) != AQ_OK) return st;
  const DeviceInfo *dev = device_info();
  if (!dev) return AQ_ERR_UNSUPPORTED;
  return launched(launch_quantize(W, s, U, V, r, fused, n, k, *out, ws, *dev,
                                  reinterpret_cast<cudaStream_t>(stream)),
                  what);
}

}  // namespace

extern "C" {

int32_t aq_version(void) { return 100; }

const char *aq_last_error(void) { return t_err; }

size_t aq_packed_bytes(int32_t n, int32_t k) {
  if (n < 1 || n > kMaxN || k < 32 || k > kMaxK || k % 32) return 0;
  return size_t(n) * size_t(k) / 2;
}

size_t aq_scale_bytes(int32_t n, int32_t k) {
  if (n < 1 || n > kMaxN || k < 32 || k > kMaxK || k % 32) return 0;
  return size_t(ceil_div(n, kTileRows) * ceil_div(k, kTileCols) * 128);
}

aq_status aq_reconstruct(const uint16_t *W0, const float *s, const uint16_t *U,
                         const uint16_t *V, int32_t n, int32_t k, int32_t r, uint16_t *W_eff,
                         aq_stream_t stream) {
  aq_status st = check_theta(W0, s, U, V, n, k, r);
  if (st != AQ_OK) return st;
  if (!W_eff) return set_error(AQ_ERR_INVALID_ARG, "aq_reconstruct: W_eff is NULL");
  if (!aligned(W_eff, 16)) return set_error(AQ_ERR_ALIGNMENT, "aq_reconstruct: W_eff must be 16-byte aligned");
  if (!device_info()) return AQ_ERR_UNSUPPORTED;
  return launched(launch_reconstruct(W0, s, U, V, n, k, r, W_eff,
                                     reinterpret_cast<cudaStream_t>(stream)),
                  "aq_reconstruct");
}

size_t aq_quantize_workspace_bytes(void) { return 256; }

aq_status aq_quantize_nvfp4(const uint16_t *W, int32_t n, int32_t k, const aq_nvfp4_weight *out,
                            void *workspace, size_t workspace_bytes, aq_stream_t stream) {
  return quantize_common(W, nullptr, nullptr, nullptr, n, k, 0, false, out, workspace,
                         workspace_bytes, stream);
}

aq_status aq_reconstruct_quantize_nvfp4(const uint16_t *W0, const float *s, const uint16_t *U,
                                        const uint16_t *V, int32_t n, int32_t k, int32_t r,
                                        const aq_nvfp4_weight *out, void *workspace,
                                        size_t workspace_bytes, aq_stream_t stream) {
  return quantize_common(W0, s, U, V, n, k, r, true, out, workspace, workspace_bytes, stream);
}

aq_status aq_quantize_act_nvfp4(const uint16_t *x, int32_t m, int32_t k, uint8_t *packed,
                                uint8_t *scales, float *g_dec, aq_stream_t stream) {
  const char *what = "aq_quantize_act_nvfp4";
  if (m < 1 || m > (1 << 20))
    return set_error(AQ_ERR_SHAPE, "%s: m = %d outside [1, 2^20]", what, m);
  aq_status s = check_nk(1, k);
  if (s != AQ_OK) return s;
  if (!x || !packed || !scales || !g_dec)
    return set_error(AQ_ERR_INVALID_ARG, "%s: pointers must not be NULL", what);
  if (!aligned(x, 16) || !aligned(packed, 16) || !aligned(g_dec, 4))
    return set_error(AQ_ERR_ALIGNMENT, "%s: x and packed must be 16-byte aligned, g_dec 4-byte",
                     what);
  const DeviceInfo *dev = device_info();
  if (!dev) return AQ_ERR_UNSUPPORTED;
  return launched(launch_act_quant(x, m, k, packed, scales, k / 16, g_dec, *dev,
                                   reinterpret_cast<cudaStream_t>(stream)),
                  what);
}

// Enough for every path that serves m tokens.
static size_t workspace_for(int32_t n, int32_t k, int32_t m, const DeviceInfo &dev) {
  size_t b = gemv_workspace_bytes(n, k, dev);
  if (m <= AQ_MAX_M_MMA) {
    const size_t mb = mma_workspace(n, k, m, dev).bytes;
    if (mb > b) b = mb;
  }
  return b;
}

size_t aq_gemv_workspace_bytes(int32_t n, int32_t k, int32_t m) {
  if (check_nk(n, k) != AQ_OK || m < 1 || m > AQ_MAX_M_MMA) return 0;
  const DeviceInfo *dev = device_info();
  if (!dev) return 0;
  return workspace_for(n, k, m, *dev);
}

// Host-only checks of one GEMV call (no device query).
aq_status gemv_args(const aq_nvfp4_weight *w, const uint16_t *x, int32_t m,
                           const uint16_t *y, aq_path path, const char *what) {
  aq_status s = check_weight(w, what);
  if (s != AQ_OK) return s;
  if (path != AQ_PATH_AUTO && path != AQ_PATH_GEMV && path != AQ_PATH_MMA &&
      path != AQ_PATH_GEMV_REGDECODE && path != AQ_PATH_GEMV_TCGEN05)
    return set_error(AQ_ERR_INVALID_ARG, "%s: unknown path %d", what, int(path));
  const int32_t max_m = (path == AQ_PATH_MMA || path == AQ_PATH_AUTO) ? AQ_MAX_M_MMA : AQ_MAX_M;
  if (m < 1 || m > max_m)
    return set_error(AQ_ERR_SHAPE, "%s: m = %d outside [1, %d] for this path", what, m, max_m);
  if (!x || !y) return set_error(AQ_ERR_INVALID_ARG, "%s: x and y must not be NULL", what);
  if (!aligned(x, 16) || !aligned(y, 16))
    return set_error(AQ_ERR_ALIGNMENT, "%s: x and y must be 16-byte aligned", what);
  return AQ_OK;
}

aq_status aq_gemv_nvfp4(const aq_nvfp4_weight *w, const uint16_t *x, int32_t m, uint16_t *y,
                        aq_path path, void *workspace, size_t workspace_bytes,
                        aq_stream_t stream) {
  const char *what = "aq_gemv_nvfp4";
  aq_status s = gemv_args(w, x, m, y, path, what);
  if (s != AQ_OK) return s;
  const DeviceInfo *dev = device_info();
  if (!dev) return AQ_ERR_UNSUPPORTED;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (path == AQ_PATH_MMA || (path == AQ_PATH_AUTO && m > AQ_MAX_M)) {
    if (!mma_eligible(w->n, w->k, m, *dev))
      return set_error(AQ_ERR_UNSUPPORTED, "%s: the MMA path does not serve m = %d", what, m);
    if ((s = check_ws(workspace, workspace_bytes, mma_workspace(w->n, w->k, m, *dev).bytes, what)) != AQ_OK)
      return s;
    return launched(launch_mma(*w, x, m, y, workspace, false, *dev, st), what);
  }
  if ((s = check_ws(workspace, workspace_bytes, gemv_workspace_bytes(w->n, w->k, *dev), what)) != AQ_OK)
    return s;
  if (path == AQ_PATH_GEMV_REGDECODE)
    return launched(launch_gemv_regdecode(*w, x, m, y, workspace, false, *dev, st), what);
  if (path == AQ_PATH_GEMV_TCGEN05) {
    if (!tc_eligible(w->n, w->k, m, *dev))
      return set_error(AQ_ERR_UNSUPPORTED,
                       "%s: the tcgen05 kernel does not serve [%d, %d] with m = %d", what, w->n,
                       w->k, m);
    return launched(launch_gemv_tc(*w, x, m, y, workspace, false, *dev, st), what);
  }
  return launched(launch_gemv(*w, x, m, y, workspace, false, *dev, st), what);
}

// bf16 weight shape: rows of whole 16-byte vectors.
static aq_status check_bf16_nk(int32_t n, int32_t k) {
  if (n < 1 || n > kMaxN)
    return set_error(AQ_ERR_SHAPE, "n = %d outside [1, %d]", n, kMaxN);
  if (k < 8 || k > kMaxK || k % 8 != 0)
    return set_error(AQ_ERR_SHAPE, "k = %d must be a multiple of 8 in [8, %d]", k, kMaxK);
  return AQ_OK;
}

size_t aq_gemv_bf16_workspace_bytes(int32_t n, int32_t k, int32_t m) {
  if (check_bf16_nk(n, k) != AQ_OK || m < 1 || m > AQ_MAX_M) return 0;
  const DeviceInfo *dev = device_info();
  if (!dev) return 0;
  return gemv_bf16_workspace_bytes(n, k, *dev);
}

aq_status aq_gemv_bf16(const uint16_t *w, int32_t n, int32_t k, const uint16_t *x, int32_t m,
                       uint16_t *y, uint32_t flags, void *workspace, size_t workspace_bytes,
                       aq_stream_t stream) {
  const char *what = "aq_gemv_bf16";
  aq_status s = check_bf16_nk(n, k);
  if (s != AQ_OK) return s;
  if (m < 1 || m > AQ_MAX_M)
    return set_error(AQ_ERR_SHAPE, "%s: m = %d outside [1, %d]", what, m, AQ_MAX_M);
  if (flags & ~AQ_STEP_PDL) return set_error(AQ_ERR_INVALID_ARG, "%s: unknown flags 0x%x", what, flags);
  if (!w || !x || !y) return set_error(AQ_ERR_INVALID_ARG, "%s: w, x and y must not be NULL", what);
  if (!aligned(w, 16) || !aligned(x, 16) || !aligned(y, 16))
    return set_error(AQ_ERR_ALIGNMENT, "%s: w, x and y must be 16-byte aligned", what);
  const DeviceInfo *dev = device_info();
  if (!dev) return AQ_ERR_UNSUPPORTED;
  if ((s = check_ws(workspace, workspace_bytes, gemv_bf16_workspace_bytes(n, k, *dev), what)) != AQ_OK)
    return s;
  return launched(launch_gemv_bf16(w, n, k, x, m, y, workspace, (flags & AQ_STEP_PDL) != 0, *dev,
                                   reinterpret_cast<cudaStream_t>(stream)),
                  what);
}

static aq_status check_segments(int32_t n, int32_t nseg, const int32_t *seg_end,
                                const char *what) {
  if (nseg < 1 || nseg > AQ_MAX_SEGMENTS)
    return set_error(AQ_ERR_SHAPE, "%s: nseg = %d outside [1, %d]", what, nseg, AQ_MAX_SEGMENTS);
  if (!seg_end) return set_error(AQ_ERR_INVALID_ARG, "%s: seg_end is NULL", what);
  int32_t prev = 0;
  for (int32_t s = 0; s < nseg; ++s) {
    if (seg_end[s] <= prev)
      return set_error(AQ_ERR_SHAPE, "%s: seg_end must increase (segment %d)", what, s);
    if (prev % 16 != 0)
      return set_error(AQ_ERR_SHAPE, "%s: segment %d starts at row %d, not a multiple of 16", what,
                       s, prev);
    prev = seg_end[s];
  }
  if (prev != n)
    return set_error(AQ_ERR_SHAPE, "%s: the last segment ends at %d, not n = %d", what, prev, n);
  return AQ_OK;
}

aq_status aq_quantize_nvfp4_segments(const uint16_t *W, int32_t n, int32_t k, int32_t nseg,
                                     const int32_t *seg_end, const aq_nvfp4_weight *out,
                                     void *workspace, size_t workspace_bytes, aq_stream_t stream) {
  const char *what = "aq_quantize_nvfp4_segments";
  aq_status st = check_nk(n, k);
  if (st != AQ_OK) return st;
  if ((st = check_segments(n, nseg, seg_end, what)) != AQ_OK) return st;
  if ((st = check_weight(out, what)) != AQ_OK) return st;
  if (out->n != n || out->k != k)
    return set_error(AQ_ERR_SHAPE, "%s: out is [%d, %d], input is [%d, %d]", what, out->n,
                     out->k, n, k);
  if (!W) return set_error(AQ_ERR_INVALID_ARG, "%s: W is NULL", what);
  const int64_t tile_bytes = int64_t(ceil_div(k, kTileCols)) * 128;  // scales of 16 rows
  int32_t start = 0;
  for (int32_t s = 0; s < nseg; ++s) {
    aq_nvfp4_weight sub = *out;
    sub.n = seg_end[s] - start;
    sub.packed = out->packed + int64_t(start) * (k / 2);
    sub.scales = out->scales + int64_t(start / 16) * tile_bytes;
    sub.global_scale = out->global_scale + s;
    st = quantize_common(W + int64_t(start) * k, nullptr, nullptr, nullptr, sub.n, k, 0, false,
                         &sub, workspace, workspace_bytes, stream);
    if (st != AQ_OK) return st;
    start = seg_end[s];
  }
  return AQ_OK;
}

aq_status aq_gemv_nvfp4_segments(const aq_nvfp4_weight *w, int32_t nseg, const int32_t *seg_end,
                                 const uint16_t *x, int32_t m, uint16_t *y, uint32_t flags,
                                 void *workspace, size_t workspace_bytes, aq_stream_t stream) {
  const char *what = "aq_gemv_nvfp4_segments";
  aq_status st = gemv_args(w, x, m, y, AQ_PATH_GEMV_REGDECODE, what);
  if (st != AQ_OK) return st;
  if ((st = check_segments(w->n, nseg, seg_end, what)) != AQ_OK) return st;
  if (flags & ~AQ_STEP_PDL) return set_error(AQ_ERR_INVALID_ARG, "%s: unknown flags 0x%x", what, flags);
  const DeviceInfo *dev = device_info();
  if (!dev) return AQ_ERR_UNSUPPORTED;
  if ((st = check_ws(workspace, workspace_bytes, gemv_workspace_bytes(w->n, w->k, *dev), what)) !=
      AQ_OK)
    return st;
  return launched(launch_gemv_regdecode(*w, x, m, y, workspace, (flags & AQ_STEP_PDL) != 0, *dev,
                                        reinterpret_cast<cudaStream_t>(stream), nullptr, nullptr,
                                        false, nseg, seg_end),
                  what);
}

aq_status aq_selftest_timeout(uint32_t polls, aq_stream_t stream) {
  const char *what = "aq_selftest_timeout";
  if (polls < 1 || polls > (1u << 20))
    return set_error(AQ_ERR_INVALID_ARG, "%s: polls = %u outside [1, 2^20]", what, polls);
  const DeviceInfo *dev = device_info();
  if (!dev) return AQ_ERR_UNSUPPORTED;
  return launched(launch_selftest_wait(polls, *dev, reinterpret_cast<cudaStream_t>(stream)), what);
}

aq_status aq_interleave_gate_up(const uint16_t *w, int32_t f, int32_t k, uint16_t *out,
                                aq_stream_t stream) {
  const char *what = "aq_interleave_gate_up";
  if (f < 8 || f % 8 != 0 || f > kMaxN / 2)
    return set_error(AQ_ERR_SHAPE, "%s: f = %d must be a multiple of 8 in [8, %d]", what, f, kMaxN / 2);
  if (k < 8 || k > kMaxK || k % 8 != 0)
    return set_error(AQ_ERR_SHAPE, "%s: k = %d must be a multiple of 8 in [8, %d]", what, k, kMaxK);
  if (!w || !out) return set_error(AQ_ERR_INVALID_ARG, "%s: w and out must not be NULL", what);
  if (!aligned(w, 16) || !aligned(out, 16))
    return set_error(AQ_ERR_ALIGNMENT, "%s: w and out must be 16-byte aligned", what);
  return launched(launch_interleave_gate_up(w, f, k, out, reinterpret_cast<cudaStream_t>(stream)),
                  what);
}

aq_status aq_gemv_glu_nvfp4(const aq_nvfp4_weight *w, const uint16_t *x, int32_t m, uint16_t *h,
                            uint32_t flags, void *workspace, size_t workspace_bytes,
                            aq_stream_t stream) {
  const char *what = "aq_gemv_glu_nvfp4";
  aq_status st = gemv_args(w, x, m, h, AQ_PATH_GEMV_REGDECODE, what);
  if (st != AQ_OK) return st;
  if (w->n % 16 != 0)
    return set_error(AQ_ERR_SHAPE, "%s: n = %d must be a multiple of 16 (gate/up row pairs)", what,
                     w->n);
  if (flags & ~AQ_STEP_PDL) return set_error(AQ_ERR_INVALID_ARG, "%s: unknown flags 0x%x", what, flags);
  const DeviceInfo *dev = device_info();
  if (!dev) return AQ_ERR_UNSUPPORTED;
  if ((st = check_ws(workspace, workspace_bytes, gemv_workspace_bytes(w->n, w->k, *dev), what)) !=
      AQ_OK)
    return st;
  return launched(launch_gemv_regdecode(*w, x, m, h, workspace, (flags & AQ_STEP_PDL) != 0, *dev,
                                        reinterpret_cast<cudaStream_t>(stream), nullptr, nullptr,
                                        true),
                  what);
}

size_t aq_gemv_lowrank_workspace_bytes(int32_t n, int32_t k, int32_t m, int32_t r) {
  if (check_nk(n, k) != AQ_OK || m < 1 || m > AQ_MAX_M || r < 0 || r > AQ_LOWRANK_MAX_R) return 0;
  const DeviceInfo *dev = device_info();
  if (!dev) return 0;
  return gemv_lowrank_workspace_bytes(n, k, m, r, *dev);
}

aq_status aq_gemv_lowrank_nvfp4(const aq_nvfp4_weight *w0, const float *s, const uint16_t *U,
                                const uint16_t *V, int32_t r, const uint16_t *x, int32_t m,
                                uint16_t *y, uint32_t flags, void *workspace,
                                size_t workspace_bytes, aq_stream_t stream) {
  const char *what = "aq_gemv_lowrank_nvfp4";
  aq_status st = gemv_args(w0, x, m, y, AQ_PATH_GEMV_REGDECODE, what);
  if (st != AQ_OK) return st;
  if (r < 0 || r > AQ_LOWRANK_MAX_R)
    return set_error(AQ_ERR_SHAPE, "%s: r = %d outside [0, %d]", what, r, AQ_LOWRANK_MAX_R);
  if (flags & ~AQ_STEP_PDL) return set_error(AQ_ERR_INVALID_ARG, "%s: unknown flags 0x%x", what, flags);
  if (!s) return set_error(AQ_ERR_INVALID_ARG, "%s: s must not be NULL", what);
  if (r > 0 && (!U || !V))
    return set_error(AQ_ERR_INVALID_ARG, "%s: U and V must not be NULL when r > 0", what);
  if (!aligned(s, 4) || (r > 0 && (!aligned(U, 2) || !aligned(V, 2))))
    return set_error(AQ_ERR_ALIGNMENT, "%s: s, U, V must be naturally aligned", what);
  const DeviceInfo *dev = device_info();
  if (!dev) return AQ_ERR_UNSUPPORTED;
  if ((st = check_ws(workspace, workspace_bytes,
                     gemv_lowrank_workspace_bytes(w0->n, w0->k, m, r, *dev), what)) != AQ_OK)
    return st;
  return launched(launch_gemv_lowrank(*w0, s, U, V, r, x, m, y, workspace,
                                      (flags & AQ_STEP_PDL) != 0, *dev,
                                      reinterpret_cast<cudaStream_t>(stream)),
                  what);
}

aq_status aq_decode_step_weights(const aq_nvfp4_weight *w, int32_t n_proj,
                                 const uint16_t *const *x, uint16_t *const *y, int32_t m,
                                 uint32_t flags, void *workspace, size_t workspace_bytes,
                                 aq_stream_t stream) {
  const char *what = "aq_decode_step_weights";
  if (n_proj < 0) return set_error(AQ_ERR_INVALID_ARG, "%s: n_proj < 0", what);
  if (n_proj == 0) return AQ_OK;
  if (!w || !x || !y) return set_error(AQ_ERR_INVALID_ARG, "%s: w, x, y must not be NULL", what);
  if (flags & ~(AQ_STEP_PDL | AQ_STEP_REGDECODE | AQ_STEP_TCGEN05 | AQ_STEP_MMA))
    return set_error(AQ_ERR_INVALID_ARG, "%s: unknown flags 0x%x", what, flags);
  const uint32_t kernels = flags & (AQ_STEP_REGDECODE | AQ_STEP_TCGEN05 | AQ_STEP_MMA);
  if (kernels & (kernels - 1))
    return set_error(AQ_ERR_INVALID_ARG, "%s: at most one kernel flag", what);
  // Validate every projection before the first launch.
  for (int32_t p = 0; p < n_proj; ++p) {
    aq_status s = gemv_args(&w[p], x[p], m, y[p],
                            (flags & AQ_STEP_MMA) ? AQ_PATH_MMA : AQ_PATH_GEMV, what);
    if (s != AQ_OK) {
      char msg[sizeof t_err];
      std::strncpy(msg, t_err, sizeof msg - 1);
      msg[sizeof msg - 1] = 0;
      return set_error(s, "projection %d: %s", p, msg);
    }
  }
  const DeviceInfo *dev = device_info();
  if (!dev) return AQ_ERR_UNSUPPORTED;
  for (int32_t p = 0; p < n_proj; ++p) {
    const size_t need = (flags & AQ_STEP_MMA) ? mma_workspace(w[p].n, w[p].k, m, *dev).bytes
                                              : gemv_workspace_bytes(w[p].n, w[p].k, *dev);
    aq_status s = check_ws(workspace, workspace_bytes, need, what);
    if (s != AQ_OK) return s;
    if ((flags & AQ_STEP_MMA) && !mma_eligible(w[p].n, w[p].k, m, *dev))
      return set_error(AQ_ERR_UNSUPPORTED, "%s: projection %d: the MMA path does not serve m = %d",
                       what, p, m);
  }
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const bool pdl = (flags & AQ_STEP_PDL) != 0;
  for (int32_t p = 0; p < n_proj; ++p) {
    // the register-decode kernel pulls the next projection's first weight
    // units into L2 while its own launch drains
    const aq_nvfp4_weight *next = p + 1 < n_proj ? &w[p + 1] : nullptr;
    cudaError_t e;
    if (flags & AQ_STEP_MMA)
      e = launch_mma(w[p], x[p], m, y[p], workspace, pdl, *dev, st);
    else if (flags & AQ_STEP_REGDECODE)
      e = launch_gemv_regdecode(w[p], x[p], m, y[p], workspace, pdl, *dev, st, next);
    else if ((flags & AQ_STEP_TCGEN05) && tc_eligible(w[p].n, w[p].k, m, *dev))
      e = launch_gemv_tc(w[p], x[p], m, y[p], workspace, pdl, *dev, st);
    else
      e = launch_gemv(w[p], x[p], m, y[p], workspace, pdl, *dev, st, next);
    if (e != cudaSuccess) return cuda_error(e, what);
  }
  return AQ_OK;
}

size_t aq_step_plan_bytes(int32_t n_proj) {
  if (n_proj < 1 || n_proj > (1 << 20)) return 0;
  return step_plan_bytes(n_proj);
}

aq_status aq_step_plan_create(const aq_nvfp4_weight *w, int32_t n_proj, const uint16_t *const *x,
                              uint16_t *const *y, int32_t m, void *plan, size_t plan_bytes,
                              size_t *workspace_bytes) {
  const char *what = "aq_step_plan_create";
  if (n_proj < 1 || n_proj > (1 << 20))
    return set_error(AQ_ERR_INVALID_ARG, "%s: n_proj = %d outside [1, 2^20]", what, n_proj);
  if (!w || !x || !y || !plan)
    return set_error(AQ_ERR_INVALID_ARG, "%s: w, x, y and plan must not be NULL", what);
  if (!aligned(plan, 128)) return set_error(AQ_ERR_ALIGNMENT, "%s: plan must be 128-byte aligned", what);
  for (int32_t p = 0; p < n_proj; ++p) {
    aq_status s = gemv_args(&w[p], x[p], m, y[p], AQ_PATH_GEMV, what);
    if (s != AQ_OK) {
      char msg[sizeof t_err];
      std::strncpy(msg, t_err, sizeof msg - 1);
      msg[sizeof msg - 1] = 0;
      return set_error(s, "projection %d: %s", p, msg);
    }
  }
  const DeviceInfo *dev = device_info();
  if (!dev) return AQ_ERR_UNSUPPORTED;
  return step_plan_create(w, n_proj, x, y, m, plan, plan_bytes, workspace_bytes, *dev);
}

aq_status aq_step_run(const void *plan, int32_t m, void *workspace, size_t workspace_bytes,
                      aq_stream_t stream) {
  const char *what = "aq_step_run";
  if (!plan || !workspace)
    return set_error(AQ_ERR_INVALID_ARG, "%s: plan and workspace must not be NULL", what);
  if (!aligned(plan, 128)) return set_error(AQ_ERR_ALIGNMENT, "%s: plan must be 128-byte aligned", what);
  if (!aligned(workspace, 256))
    return set_error(AQ_ERR_WORKSPACE, "%s: workspace must be 256-byte aligned", what);
  if (m < 1 || m > AQ_MAX_M)
    return set_error(AQ_ERR_SHAPE, "%s: m = %d outside [1, %d]", what, m, AQ_MAX_M);
  const DeviceInfo *dev = device_info();
  if (!dev) return AQ_ERR_UNSUPPORTED;
  return launched(launch_step(plan, m, workspace, workspace_bytes, *dev,
                              reinterpret_cast<cudaStream_t>(stream)),
                  what);
}

aq_status aq_scales_to_canonical(const aq_nvfp4_weight *w, uint8_t *canon, aq_stream_t stream) {
  aq_status s = check_weight(w, "aq_scales_to_canonical");
  if (s != AQ_OK) return s;
  if (!canon) return set_error(AQ_ERR_INVALID_ARG, "aq_scales_to_canonical: canon is NULL");
  if (!device_info()) return AQ_ERR_UNSUPPORTED;
  return launched(launch_scales_to_canonical(*w, canon, reinterpret_cast<cudaStream_t>(stream)),
                  "aq_scales_to_canonical");
}

aq_status aq_poll_device_status(aq_stream_t stream) {
  const DeviceInfo *dev = device_info();
  if (!dev) return AQ_ERR_UNSUPPORTED;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_error(e, "aq_poll_device_status: stream");
  unsigned word = 0;
  e = cudaMemcpy(&word, dev->status, sizeof word, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_error(e, "aq_poll_device_status: read");
  if (word != 0) {
    const unsigned zero = 0;
    e = cudaMemcpy(dev->status, &zero, sizeof zero, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_error(e, "aq_poll_device_status: clear");
  }
  switch (word) {
    case kDevOk:
      return AQ_OK;
    case kDevRange:
      return set_error(AQ_ERR_RANGE, "per-tensor amax was non-finite or too small to scale");
    case kDevTimeout:
      return set_error(AQ_ERR_TIMEOUT, "a bounded device-side wait gave up; re-zero GEMV workspaces");
    case kDevBadPlan:
      return set_error(AQ_ERR_INVALID_ARG,
                       "aq_step_run: plan, m, grid or workspace size do not match the plan");
    default:
      return set_error(AQ_ERR_CUDA, "unknown device status %u", word);
  }
}

}  // extern "C"
