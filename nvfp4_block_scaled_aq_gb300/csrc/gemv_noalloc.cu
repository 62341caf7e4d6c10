// gemv_noalloc.cu -- aq_gemv_nvfp4_noalloc: the block-scaled GEMV of
// aq_gemv_nvfp4 for callers that cannot hand the library a workspace.
//
// Who needs it: code that has no device allocator of its own to call -- a
// plugin or kernel library loaded into a host program that owns all device
// memory and forbids cudaMalloc after start-up (cudaMalloc can synchronise
// the whole device, which a latency-bound decode loop cannot afford), or a
// foreign-language binding that can pass tensors but not create them.  Such
// callers pass only the weight, x and y; the split-K scratch of the GEMV
// (tickets + partial sums) lives in one fixed array of this library in
// device memory, which every GPU that loads the library holds until the
// process exits.
//
// The array is shared by every call on a device and keeps what the last
// call left in it.  Calls whose kernels overlap on the GPU (two streams, or
// two host threads) race on it; callers must order them.
#include <cstring>
#include <mutex>

#include "gemv_core.cuh"

namespace aq {
namespace {

// Scratch of the no-allocation GEMV: AQ_GEMV_NOALLOC_MAX_SCRATCH bytes per
// device.  In host code the name is only a handle for cudaGetSymbolAddress.
__device__ __align__(256) uint8_t g_noalloc_scratch[AQ_GEMV_NOALLOC_MAX_SCRATCH];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
uint8_t *g_scratch[kMaxDevices];  // device address of g_noalloc_scratch, per device
bool g_ready[kMaxDevices];

// First call on a device (that device current): resolve the array's device
// address and zero it once.  Synchronous: the first call on each device
// must not be made while a stream is being captured.  The address is kept
// for the life of the process; a cudaDeviceReset reloads the module at a
// new address, so the call must not be used across a device reset.
aq_status scratch_for(const DeviceInfo &dev, uint8_t **out) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (dev.ordinal < 0 || dev.ordinal >= kMaxDevices)
    return set_error(AQ_ERR_UNSUPPORTED, "aq_gemv_nvfp4_noalloc: device ordinal %d out of range",
                     dev.ordinal);
  if (!g_ready[dev.ordinal]) {
    void *p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_error(e, "aq_gemv_nvfp4_noalloc: cudaGetSymbolAddress");
    e = cudaMemset(p, 0, AQ_GEMV_NOALLOC_MAX_SCRATCH);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_error(e, "aq_gemv_nvfp4_noalloc: clearing the scratch");
    g_scratch[dev.ordinal] = static_cast<uint8_t *>(p);
    g_ready[dev.ordinal] = true;
  }
  *out = g_scratch[dev.ordinal];
  return AQ_OK;
}

}  // namespace
}  // namespace aq

using namespace aq;

aq_status aq_gemv_nvfp4_noalloc(const aq_nvfp4_weight *w, const uint16_t *x, int32_t m,
                                uint16_t *y, aq_path path, aq_stream_t stream) {
  const char *what = "aq_gemv_nvfp4_noalloc";
  aq_status s = gemv_args(w, x, m, y, path, what);
  if (s != AQ_OK) return s;
  if (path == AQ_PATH_GEMV_TCGEN05 || path == AQ_PATH_MMA || m > AQ_MAX_M)
    return set_error(AQ_ERR_UNSUPPORTED,
                     "%s: runs the register-decode kernel only (m <= %d, no MMA or tcgen05 path)",
                     what, AQ_MAX_M);
  const DeviceInfo *dev = device_info();
  if (!dev) return AQ_ERR_UNSUPPORTED;
  // only the register-decode kernel runs here, so only its scratch counts
  const size_t need = gemv_regdecode_workspace_bytes(w->n, w->k, *dev);
  if (need > AQ_GEMV_NOALLOC_MAX_SCRATCH)
    return set_error(AQ_ERR_WORKSPACE,
                     "%s: a [%d, %d] weight needs %zu bytes of scratch on this device, more than "
                     "the %zu-byte static scratch; call aq_gemv_nvfp4 with a workspace instead",
                     what, w->n, w->k, need, size_t(AQ_GEMV_NOALLOC_MAX_SCRATCH));
  uint8_t *scratch = nullptr;
  if ((s = scratch_for(*dev, &scratch)) != AQ_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // The split-K tickets and the encoded partials of the zero region must
  // start at zero.  A completed call leaves them zero, but one that gave up
  // on a bounded wait may not, so the part of both that this weight uses is
  // cleared on the stream before every launch; the plain partials after
  // them are always written before they are read.
  const GemvPlan plan = plan_gemv(w->n, w->k, *dev, kGemvRG);
  const size_t tickets = size_t(plan.row_blocks) * kGemvRG * sizeof(uint32_t);
  cudaError_t e = cudaMemsetAsync(scratch, 0, tickets, st);
  if (e == cudaSuccess && core::direct_partials_fit<kGemvRG>(plan.row_blocks, plan.max_contrib, m))
    e = cudaMemsetAsync(scratch + core::kTicketBytes, 0,
                        size_t(plan.row_blocks) * (plan.max_contrib - 1) * m * (16 * kGemvRG) * 4,
                        st);
  if (e != cudaSuccess) return cuda_error(e, what);
  e = launch_gemv_uncached(*w, x, m, y, scratch, *dev, st);
  return e == cudaSuccess ? AQ_OK : cuda_error(e, what);
}
