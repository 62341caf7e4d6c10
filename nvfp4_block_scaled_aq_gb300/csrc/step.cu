// step.cu -- the whole weight stream of one decode step in one persistent
// kernel (aq_step_plan_create / aq_step_run).
//
// AttnQuant docs, "GPU acceleration", "CUDA graph capture": a batch-1
// decode step issues hundreds of kernel dispatches, and replaying the step
// as one unit removes their launch cost; "Q/K/V fusion": one weight read per
// fused projection.  Here the step is one cooperative launch: the producer
// warp of every CTA streams the weights of all projections back to back
// (weights never depend on earlier outputs), while the consumer warps take
// the projections in order and pass a grid-wide barrier before reading each
// projection's activations, so projection p+1 reads x only after every
// output of projection p is written -- the stream-order semantics of the
// per-projection launches, without their launch gaps.  The shared-memory
// ring keeps HBM busy across each barrier.
//
// The plan (device memory, written once by aq_step_plan_create) holds a
// header and, per projection, the two tensor maps, the pointers and the
// stream-K partition.
#include <cstring>
#include <mutex>
#include <vector>

#include "gemv_core.cuh"

namespace aq {

using namespace core;

namespace {

constexpr int32_t kPlanMagic = 0x41515354;  // "AQST"
constexpr int kHeaderBytes = 128;
constexpr int kStepXCapBytes = 24 * 1024;  // activation buffer of the step kernel
constexpr unsigned kBarrierSpin = 1u << 22;

struct StepHeader {
  int32_t magic;
  int32_t n_proj;
  int32_t m;
  int32_t stages;
  int32_t x_cap;       // f16 capacity of the activation buffer
  int32_t grid;
  int64_t ws_required;
  int64_t partial_off;
  int64_t barrier_off;
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

// Grid-wide barrier of the consumer warps (generation counter; the last CTA
// to arrive re-arms the count and bumps the generation).  Bounded: a wait
// that gives up records AQ_ERR_TIMEOUT and marks the CTA aborted.
__device__ __forceinline__ void grid_barrier(unsigned *bar, unsigned nblocks,
                                             volatile int *aborted, unsigned *status) {
  consumer_sync();
  if (threadIdx.x == 0 && !*aborted) {
    volatile unsigned *gen = bar + 1;
    const unsigned gen0 = *gen;
    __threadfence();
    const unsigned arrived = atomicAdd(bar, 1u);
    if (arrived == nblocks - 1) {
      atomicExch(bar, 0u);
      __threadfence();
      atomicAdd(bar + 1, 1u);
    } else {
      unsigned it = 0;
      while (*gen == gen0) {
        if (++it > kBarrierSpin) {
          *aborted = 1;
          raise_status(status, kDevTimeout);
          break;
        }
        __nanosleep(64);
      }
    }
    __threadfence();
  }
  consumer_sync();
}

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

// Projection s with the L2 prefetch of projection n's first units.
__device__ __forceinline__ Proj with_next(Proj p, const StepProj &n) {
  p.nx_w = &n.tm_w;
  p.nx_s = &n.tm_s;
  p.nx_total = n.total;
  p.nx_units = n.units;
  p.nx_grid = n.grid;
  p.nx_pf = kPrefetchUnits;
  return p;
}

template <int NT>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    step_kernel(const uint8_t *__restrict__ plan, uint8_t *ws, uint64_t ws_bytes, int m,
                unsigned *status) {
  const StepHeader h = *reinterpret_cast<const StepHeader *>(plan);
  const StepProj *projs = reinterpret_cast<const StepProj *>(plan + kHeaderBytes);
  if (h.magic != kPlanMagic || int64_t(ws_bytes) < h.ws_required || int(gridDim.x) != h.grid ||
      h.m != m || h.stages < kMinStages || h.stages > kMaxStages) {
    if (blockIdx.x == 0 && threadIdx.x == 0) raise_status(status, kDevBadPlan);
    return;
  }
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const SmemView sv = carve(smem_raw, h.stages);
  Ctrl &ct = *sv.ct;
  volatile int *aborted = &ct.aborted;
  if (threadIdx.x == 0) init_ring(ct, h.stages);
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

  if ((threadIdx.x >> 5) == kW) {  // producer warp: every projection, back to back
    if ((threadIdx.x & 31) == 0) {
      for (int p = 0; p < h.n_proj; ++p) {
        if (!produce(to_proj(projs[p]), sv.base, ct, h.stages, pos, aborted, status)) break;
        if (p + 1 < h.n_proj) prefetch_next(with_next(to_proj(projs[p]), projs[p + 1]));
      }
      drain(ct, h.stages, pos.count);
    }
    return;
  }
  unsigned *bar = reinterpret_cast<unsigned *>(ws + h.barrier_off);
  for (int p = 0; p < h.n_proj; ++p) {
    if (p > 0) grid_barrier(bar, gridDim.x, aborted, status);
    if (*aborted) break;
    consume<NT>(to_proj(projs[p]), r, sv.base, ct, sv.xs, pos, aborted);
  }
}

template <int NT>
cudaError_t set_step_smem_attr(int device) {
  static bool done[64] = {};
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (device >= 0 && device < 64 && done[device]) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(step_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSmemBudget);
  if (e == cudaSuccess && device >= 0 && device < 64) done[device] = true;
  return e;
}

}  // namespace

size_t step_plan_bytes(int n_proj) {
  return size_t(kHeaderBytes) + size_t(n_proj) * sizeof(StepProj);
}

// Host side of aq_step_plan_create (arguments already validated).
aq_status step_plan_create(const aq_nvfp4_weight *w, int n_proj, const uint16_t *const *x,
                           uint16_t *const *y, int m, void *plan, size_t plan_bytes,
                           size_t *ws_bytes, const DeviceInfo &dev) {
  const int64_t G_launch = int64_t(dev.sms) * kCtasPerSm;
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
    if (!encode_maps(w[i], &sp.tm_w, &sp.tm_s))
      return set_error(AQ_ERR_CUDA, "aq_step_plan_create: tensor map encoding failed (projection %d)", i);
    const int64_t row_blocks = ceil_div(w[i].n, kRB);
    const int64_t units = ceil_div(ceil_div(w[i].k, kTileCols), kKT);
    sp.g_dec = w[i].global_scale;
    sp.x = x[i];
    sp.y = y[i];
    sp.total = row_blocks * units;
    sp.n = w[i].n;
    sp.k = w[i].k;
    sp.units = int32_t(units);
    // each projection is spread over min(launch grid, units) CTAs so every
    // participating CTA owns at least one unit
    const int64_t G = sp.total < G_launch ? sp.total : G_launch;
    sp.grid = int32_t(G);
    int worst = 1;
    for (int64_t rb = 0; rb < row_blocks; ++rb) {
      const int64_t u0 = rb * units, u1 = u0 + units - 1;
      const int c = int(owner_of(u1, sp.total, G) - owner_of(u0, sp.total, G) + 1);
      if (c > worst) worst = c;
    }
    sp.max_contrib = worst;
    sp.direct = direct_partials_fit(row_blocks, worst, m) ? 1 : 0;
    const int64_t longest = ceil_div(sp.total, G);
    const int64_t need = int64_t(m) * x_stride_full(x_slots(longest, int(units)));
    if (need * 2 <= kStepXCapBytes && need > x_need) x_need = need;
    const int64_t pb = row_blocks * worst * kRB * 16 * int64_t(sizeof(float));
    if (pb > partial_max) partial_max = pb;
    std::memcpy(buf.data() + kHeaderBytes + size_t(i) * sizeof(StepProj), &sp, sizeof sp);
  }
  h.x_cap = int32_t(x_need);
  h.stages = stages_for(h.x_cap);
  if (h.stages < kMinStages)
    return set_error(AQ_ERR_SHAPE, "aq_step_plan_create: activations of m = %d leave no room for the ring", m);
  h.partial_off = int64_t(kRestOffset);
  h.barrier_off = int64_t(kRestOffset) + (partial_max + 255) / 256 * 256;
  h.ws_required = h.barrier_off + 256;
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
  cfg.gridDim = dim3(dev.sms * kCtasPerSm);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBudget;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const uint8_t *pl = static_cast<const uint8_t *>(plan);
  uint8_t *w = static_cast<uint8_t *>(ws);
  cudaError_t e;
  if (m <= 8) {
    if ((e = set_step_smem_attr<1>(dev.ordinal)) != cudaSuccess) return e;
    e = cudaLaunchKernelEx(&cfg, step_kernel<1>, pl, w, uint64_t(ws_bytes), m, dev.status);
  } else {
    if ((e = set_step_smem_attr<2>(dev.ordinal)) != cudaSuccess) return e;
    e = cudaLaunchKernelEx(&cfg, step_kernel<2>, pl, w, uint64_t(ws_bytes), m, dev.status);
  }
  return e;
}

}  // namespace aq
