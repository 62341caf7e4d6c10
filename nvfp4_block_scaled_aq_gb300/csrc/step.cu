// step.cu -- the whole weight stream of one decode step in one persistent
// kernel (aq_step_plan_create / aq_step_run).
//
// AttnQuant docs, "GPU acceleration", "CUDA graph capture": a batch-1
// decode step issues hundreds of kernel dispatches, and replaying the step
// as one unit removes their launch cost; "Q/K/V fusion": one weight read per
// fused projection.  Here the step is one cooperative launch:
//  * the producer warp of every CTA streams the weights of all projections
//    back to back (weights never depend on earlier outputs), so HBM never
//    waits for a projection boundary while the shared-memory ring has room;
//  * the consumer warps take the projections in order.  Before reading x of
//    projection p they wait until projection p-1's completion counter holds
//    one arrival from every CTA that worked on p-1, and once their own
//    outputs of p are written they add their arrival to p's counter.  So
//    projection p reads x only after every output of p-1 is written -- the
//    stream-order semantics of per-projection launches -- without launch
//    gaps and without a grid-wide barrier that the producers would join;
//  * each projection uses the partition and kernel form of the
//    single-projection launch (the balanced stream-K grid, the one-token
//    form for m = 1), so every output equals aq_gemv_nvfp4 on the
//    register-decode kernel bit for bit.
//
// The plan (device memory, written once by aq_step_plan_create) holds a
// header and, per projection, the two tensor maps, the pointers and the
// stream-K partition.  The workspace holds the GEMV scratch, then one
// counter per projection (128 bytes apart) and an exit counter; the last
// CTA to leave puts every counter back to zero for the next run.
#include <cstring>
#include <mutex>
#include <vector>

#include "gemv_core.cuh"

namespace aq {

using namespace core;

namespace {

constexpr int32_t kPlanMagic = 0x41515355;  // "AQSU"
constexpr int kHeaderBytes = 128;
constexpr int kStepXCapBytes = 24 * 1024;  // activation buffer of the step kernel
constexpr int kCounterStride = 32;         // u32 words between counters (128 bytes)

struct StepHeader {
  int32_t magic;
  int32_t n_proj;
  int32_t m;
  int32_t stages;
  int32_t x_cap;       // f16 capacity of the activation buffer
  int32_t grid;        // CTAs of the launch (two per SM)
  int64_t ws_required;
  int64_t partial_off;
  int64_t counter_off; // n_proj counters, then the exit counter
};
static_assert(sizeof(StepHeader) <= kHeaderBytes, "header too large");

struct alignas(128) StepProj {
  CUtensorMap tm_w;    // tensor maps must be 64-byte aligned
  CUtensorMap tm_s;
  const float *g_dec;
  const uint16_t *x;
  uint16_t *y;
  int64_t total;
  int32_t n, k, units, max_contrib, grid;
  int32_t direct;      // split-K partials through the zero region
};

__device__ __forceinline__ Proj to_proj(const StepProj &s) {
  Proj p{};
  p.tm_w = &s.tm_w;
  p.tm_s = &s.tm_s;
  p.g_dec = s.g_dec;
  p.x = s.x;
  p.y = s.y;
  p.total = s.total;
  p.n = s.n;
  p.k = s.k;
  p.units = s.units;
  p.max_contrib = s.max_contrib;
  p.grid = s.grid;
  p.direct = s.direct;
  p.scale_box = 1;
  p.nx_w = p.nx_s = nullptr;
  p.nx_total = 0;
  p.nx_units = p.nx_grid = p.nx_pf = 0;
  return p;
}

constexpr int RG = kGemvRG;  // the single-projection launch's geometry
using G = Geo<RG>;

template <int NT, bool BD>
__global__ void __launch_bounds__(G::kThreads, G::kCtasPerSm)
    step_kernel(const uint8_t *__restrict__ plan, uint8_t *ws, uint64_t ws_bytes, int m,
                unsigned *status) {
  const StepHeader h = *reinterpret_cast<const StepHeader *>(plan);
  const StepProj *projs = reinterpret_cast<const StepProj *>(plan + kHeaderBytes);
  if (h.magic != kPlanMagic || int64_t(ws_bytes) < h.ws_required || int(gridDim.x) != h.grid ||
      h.m != m || h.stages < kMinStages || h.stages > G::kMaxStages) {
    if (blockIdx.x == 0 && threadIdx.x == 0) raise_status(status, kDevBadPlan);
    return;
  }
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const SmemView sv = carve<RG>(smem_raw, h.stages);
  Ctrl &ct = *sv.ct;
  volatile int *aborted = &ct.aborted;
  if (threadIdx.x == 0) init_ring<RG>(ct, h.stages);
  __syncthreads();

  Run r{};
  r.tickets = reinterpret_cast<uint32_t *>(ws);
  r.zero = reinterpret_cast<uint32_t *>(ws + kTicketBytes);
  r.partial = reinterpret_cast<float *>(ws + h.partial_off);
  r.status = status;
  r.m = h.m;
  r.stages = h.stages;
  r.x_cap = h.x_cap;
  RingPos pos;

  if ((threadIdx.x >> 5) == G::kW) {  // producer warp: every projection, back to back
    if ((threadIdx.x & 31) == 0) {
      for (int p = 0; p < h.n_proj; ++p)
        if (!produce<RG>(to_proj(projs[p]), sv.base, ct, h.stages, pos, aborted, status)) break;
      drain(ct, h.stages, pos.count);
    }
    return;
  }
  unsigned *counters = reinterpret_cast<unsigned *>(ws + h.counter_off);
  for (int p = 0; p < h.n_proj; ++p) {
    if (*aborted) break;
    const Proj P = to_proj(projs[p]);
    Dep dep;
    if (p > 0) {
      dep.kind = kDepCounter;
      dep.ctr = counters + size_t(p - 1) * kCounterStride;
      dep.target = unsigned(projs[p - 1].grid);
    }
    if (int64_t(blockIdx.x) < P.grid) {
      consume<NT, kEpiPlain, BD, RG>(P, r, sv.base, ct, sv.xs, pos, aborted, dep);
      arrive_counter<RG>(counters + size_t(p) * kCounterStride);
    }
  }
  // Exit: the last CTA out (every other CTA has passed all of its waits)
  // returns the counters to zero for the next run on this workspace.
  consumer_sync<RG>();
  if (threadIdx.x == 0) {
    unsigned *exit_ctr = counters + size_t(h.n_proj) * kCounterStride;
    __threadfence();
    if (atomicAdd(exit_ctr, 1u) == gridDim.x - 1) {
      __threadfence();
      for (int p = 0; p < h.n_proj; ++p) counters[size_t(p) * kCounterStride] = 0;
      *exit_ctr = 0;
      __threadfence();
    }
  }
}

template <int NT, bool BD>
cudaError_t set_step_smem_attr(int device) {
  static bool done[64] = {};
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (device >= 0 && device < 64 && done[device]) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(step_kernel<NT, BD>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       G::kSmemBudget);
  if (e == cudaSuccess && device >= 0 && device < 64) done[device] = true;
  return e;
}

template <int NT, bool BD>
cudaError_t launch_step_form(const cudaLaunchConfig_t &cfg, const uint8_t *pl, uint8_t *w,
                             size_t ws_bytes, int m, const DeviceInfo &dev) {
  cudaError_t e = set_step_smem_attr<NT, BD>(dev.ordinal);
  if (e != cudaSuccess) return e;
  return cudaLaunchKernelEx(&cfg, step_kernel<NT, BD>, pl, w, uint64_t(ws_bytes), m, dev.status);
}

}  // namespace

size_t step_plan_bytes(int n_proj) {
  return size_t(kHeaderBytes) + size_t(n_proj) * sizeof(StepProj);
}

// Host side of aq_step_plan_create (arguments already validated).
aq_status step_plan_create(const aq_nvfp4_weight *w, int n_proj, const uint16_t *const *x,
                           uint16_t *const *y, int m, void *plan, size_t plan_bytes,
                           size_t *ws_bytes, const DeviceInfo &dev) {
  const int64_t G_launch = int64_t(dev.sms) * G::kCtasPerSm;
  std::vector<uint8_t> buf(step_plan_bytes(n_proj), 0);
  StepHeader h = {};
  h.magic = kPlanMagic;
  h.n_proj = n_proj;
  h.m = m;
  h.grid = int(G_launch);
  int64_t x_need = int64_t(m) * x_stride_chunk(m);
  int64_t partial_max = 0;
  for (int i = 0; i < n_proj; ++i) {
    StepProj sp;
    std::memset(&sp, 0, sizeof sp);
    if (!encode_maps(w[i], &sp.tm_w, &sp.tm_s, RG))
      return set_error(AQ_ERR_CUDA, "aq_step_plan_create: tensor map encoding failed (projection %d)", i);
    // the partition of the single-projection launch (same grid, same
    // contributors), so each output is that launch's bit for bit
    const GemvPlan gp = plan_gemv(w[i].n, w[i].k, dev, RG);
    sp.g_dec = w[i].global_scale;
    sp.x = x[i];
    sp.y = y[i];
    sp.total = gp.total;
    sp.n = w[i].n;
    sp.k = w[i].k;
    sp.units = int32_t(gp.units);
    sp.grid = gp.grid;
    sp.max_contrib = gp.max_contrib;
    sp.direct = direct_partials_fit<RG>(gp.row_blocks, gp.max_contrib, m) ? 1 : 0;
    const int64_t longest = ceil_div(sp.total, sp.grid);
    const int64_t need = int64_t(m) * x_stride_full(x_slots(longest, int(gp.units)));
    if (need * 2 <= kStepXCapBytes && need > x_need) x_need = need;
    const int64_t pb = gp.row_blocks * gp.max_contrib * G::kRB * 16 * int64_t(sizeof(float));
    if (pb > partial_max) partial_max = pb;
    std::memcpy(buf.data() + kHeaderBytes + size_t(i) * sizeof(StepProj), &sp, sizeof sp);
  }
  h.x_cap = int32_t(x_need);
  h.stages = stages_for(h.x_cap, RG);
  if (h.stages < kMinStages)
    return set_error(AQ_ERR_SHAPE, "aq_step_plan_create: activations of m = %d leave no room for the ring", m);
  h.partial_off = int64_t(kRestOffset);
  h.counter_off = int64_t(kRestOffset) + (partial_max + 255) / 256 * 256;
  h.ws_required = h.counter_off + int64_t(n_proj + 1) * kCounterStride * 4;
  std::memcpy(buf.data(), &h, sizeof h);
  if (plan_bytes < buf.size())
    return set_error(AQ_ERR_INVALID_ARG, "aq_step_plan_create: plan of %zu bytes, %zu needed",
                     plan_bytes, buf.size());
  cudaError_t e = cudaMemcpy(plan, buf.data(), buf.size(), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_error(e, "aq_step_plan_create: upload");
  if (ws_bytes) *ws_bytes = size_t(h.ws_required);
  return AQ_OK;
}

cudaError_t launch_step(const void *plan, int m, void *ws, size_t ws_bytes, const DeviceInfo &dev,
                        cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(dev.sms * G::kCtasPerSm);
  cfg.blockDim = dim3(G::kThreads);
  cfg.dynamicSmemBytes = G::kSmemBudget;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const uint8_t *pl = static_cast<const uint8_t *>(plan);
  uint8_t *w = static_cast<uint8_t *>(ws);
  if (m == 1) return launch_step_form<1, true>(cfg, pl, w, ws_bytes, m, dev);
  if (m <= 8) return launch_step_form<1, false>(cfg, pl, w, ws_bytes, m, dev);
  return launch_step_form<2, false>(cfg, pl, w, ws_bytes, m, dev);
}

}  // namespace aq
