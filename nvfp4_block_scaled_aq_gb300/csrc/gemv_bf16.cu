// gemv_bf16.cu -- y = x W^T for a weight kept in bf16: the projections the
// method leaves unquantised (the tied lm_head / embedding, and the attention
// projections when they are excluded from quantisation).
//
// AttnQuant docs, "GPU acceleration", "Where GPU time goes": besides the
// NVFP4 MLP the decode step streams bf16 attention projections and the bf16
// tied lm_head, measured there at 57 % and 65 % of peak bandwidth;
// "NVFP4 quantization": the bf16 embedding / lm_head is 2.82 GB of the 31B
// model's weights (262144 x 5376).
//
// The kernel is the register-decode GEMV's streaming skeleton without the
// decode: the same persistent two-CTA-per-SM grid, stream-K ranges of work
// units, TMA ring (one 128-byte x 128-row box per unit: 128 rows x 64 bf16
// columns, 128-byte swizzle), programmatic dependent launch and split-K
// epilogue (finish_rows, shared with the NVFP4 kernel).  The weights are
// the A operand of mma.sync m16n8k16 bf16 as they sit in shared memory, the
// activations (bf16, copied to shared memory once per CTA or per chunk) the
// B operand; fp32 accumulation, no scaling.
//
// Fragment layout: lane (g, c) loads the 16-byte chunks c and c + 4 of its
// two fragment rows, i.e. columns 8c .. 8c+7 and 32 + 8c .. 32 + 8c+7 of
// the unit.  MMA step s takes from chunk c (s < 2) or c + 4 (s >= 2) the
// pairs 4(s & 1) and 4(s & 1) + 2 as its k-slots 2c, 2c+1 and 2c+8, 2c+9;
// the activations follow the same map, so each step sums 16 distinct
// columns and the four steps cover the unit's 64 columns once.
#include <mutex>

#include "gemv_core.cuh"

namespace aq {

using namespace core;

namespace {

constexpr int kBfUnitK = 64;  // bf16 columns of one unit (one 128-byte box row)

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Activations of units [s0, s0 + ns) of the CTA's staged slots (slot s is
// unit (uk_first + s) mod units) into xs: token-major, `stride` bf16 per
// token, columns past k as zero.  Called by all consumer threads.
__device__ __forceinline__ void stage_x_bf16(const Proj &p, int m, uint16_t *xs, int stride,
                                             int uk_first, int s0, int ns, int units) {
  const int per_tok = ns * (kBfUnitK / 8);  // 16-byte vectors per token
  for (int idx = threadIdx.x; idx < m * per_tok; idx += kW * 32) {
    const int tok = idx / per_tok, v = idx - tok * per_tok;
    const int s = v / (kBfUnitK / 8), within = (v % (kBfUnitK / 8)) * 8;
    const int uk = (uk_first + s0 + s) % units;
    const int kk = uk * kBfUnitK + within;
    uint4 q = make_uint4(0, 0, 0, 0);
    if (kk < p.k) q = __ldg(reinterpret_cast<const uint4 *>(p.x + int64_t(tok) * p.k + kk));
    *reinterpret_cast<uint4 *>(xs + tok * stride + s * kBfUnitK + within) = q;
  }
}

template <int NT>
__device__ __forceinline__ void consume_bf16(const Proj &p, const Run &r, uint8_t *base, Ctrl &ct,
                                             uint16_t *xs, RingPos &pos,
                                             volatile int *aborted) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int rg = warp;
  const int64_t grid = p.grid;
  if (int64_t(blockIdx.x) >= grid) return;
  const int64_t u_begin = range_begin(blockIdx.x, p.total, grid);
  const int64_t u_end = range_begin(blockIdx.x + 1, p.total, grid);
  if (u_begin >= u_end) return;
  const int S = r.stages, m = r.m, units = p.units;

  // Stored rows sg and sg + 8 of the row group (sg = sigma(g), as in the
  // NVFP4 kernel, so each quarter-warp's chunks fill all 32 banks).
  const int sg = (g >> 1) | ((g & 1) << 2);
  const int row_lo = (rg * 16 + sg) * kUnitCols, row_hi = (rg * 16 + sg + 8) * kUnitCols;
  const int off_lo0 = row_lo + ((c ^ sg) << 4), off_lo1 = row_lo + (((c + 4) ^ sg) << 4);
  const int off_hi0 = row_hi + ((c ^ sg) << 4), off_hi1 = row_hi + (((c + 4) ^ sg) << 4);

  // Activations: every unit the range touches when they fit, else chunks.
  const int64_t L = u_end - u_begin;
  const bool all_units = L >= units;
  const int uk_first = all_units ? 0 : int(u_begin % units);
  const int slots = x_slots(L, units);
  const int stride_full = slots * kBfUnitK + 8;  // +8: tokens start in different banks
  const bool full = m * stride_full <= r.x_cap;
  int chunk = (r.x_cap / m - 8) / kBfUnitK;
  chunk = chunk < 1 ? 1 : chunk;
  const int stride = full ? stride_full : chunk * kBfUnitK + 8;
  if (full) {
    stage_x_bf16(p, m, xs, stride, uk_first, 0, slots, units);
    consumer_sync();
  }

  int64_t u = u_begin;
  while (u < u_end) {
    const int64_t rb = u / units;
    const int uk0 = int(u - rb * units);
    const int uk1 = int(uk0 + (u_end - u) < units ? uk0 + (u_end - u) : units);

    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[nt][i] = 0.0f;

    const int step_units = full ? (uk1 - uk0) : chunk;
    for (int cu0 = uk0; cu0 < uk1; cu0 += step_units) {
      const int cu1 = min(uk1, cu0 + step_units);
      if (!full) {
        consumer_sync();  // earlier readers of the staging buffer are done
        stage_x_bf16(p, m, xs, stride, cu0, 0, cu1 - cu0, units);
        consumer_sync();
      }
      int slot = full ? (cu0 - uk_first + units) % units : 0;
      for (int uk = cu0; uk < cu1; ++uk, ++slot, pos.advance(S)) {
        const int st = pos.st;
        uint4 w0 = make_uint4(0, 0, 0, 0), w1 = w0, w2 = w0, w3 = w0;
        const bool ok = !*aborted && mbar_wait(&ct.full[st], pos.phase, aborted);
        if (ok) {
          const uint8_t *stage = base + st * kStageBytes;
          w0 = *reinterpret_cast<const uint4 *>(stage + off_lo0);
          w1 = *reinterpret_cast<const uint4 *>(stage + off_lo1);
          w2 = *reinterpret_cast<const uint4 *>(stage + off_hi0);
          w3 = *reinterpret_cast<const uint4 *>(stage + off_hi1);
        } else if (lane == 0 && !*aborted) {
          *aborted = 1;
          raise_status(r.status, kDevTimeout);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&ct.empty[st]);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const uint16_t *px = xs + min(nt * 8 + g, m - 1) * stride + slot * kBfUnitK + 8 * c;
          const uint4 xa = *reinterpret_cast<const uint4 *>(px);
          const uint4 xb = *reinterpret_cast<const uint4 *>(px + 32);
          mma_bf16(acc[nt], w0.x, w2.x, w0.y, w2.y, xa.x, xa.y);
          mma_bf16(acc[nt], w0.z, w2.z, w0.w, w2.w, xa.z, xa.w);
          mma_bf16(acc[nt], w1.x, w3.x, w1.y, w3.y, xb.x, xb.y);
          mma_bf16(acc[nt], w1.z, w3.z, w1.w, w3.w, xb.z, xb.w);
        }
      }
    }
    finish_rows<NT>(p, r, rb, uk0 == 0 && uk1 == units, acc, 1.0f, rg, sg, lane, aborted);
    u += uk1 - uk0;
  }
}

template <int NT>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    gemv_bf16_kernel(const __grid_constant__ CUtensorMap tm_w, Proj p, const Run r) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const SmemView sv = carve(smem_raw, r.stages);
  Ctrl &ct = *sv.ct;
  volatile int *aborted = &ct.aborted;
  p.tm_w = &tm_w;
  if (threadIdx.x == 0) {
    init_ring(ct, r.stages);
    pdl_launch_dependents();
  }
  __syncthreads();
  RingPos pos;
  if ((threadIdx.x >> 5) == kW) {  // producer warp
    if ((threadIdx.x & 31) == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_w)) : "memory");
      produce(p, sv.base, ct, r.stages, pos, aborted, r.status);
      drain(ct, r.stages, pos.count);
    }
    return;
  }
  pdl_wait();  // x and the workspace may come from the previous kernel
  consume_bf16<NT>(p, r, sv.base, ct, sv.xs, pos, aborted);
}

template <int NT>
cudaError_t set_bf16_smem_attr(int device) {
  static bool done[64] = {};
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (device >= 0 && device < 64 && done[device]) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(gemv_bf16_kernel<NT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBudget);
  if (e == cudaSuccess && device >= 0 && device < 64) done[device] = true;
  return e;
}

// Activation buffer (bf16 halves) of one launch: every unit the longest CTA
// range touches when that fits in 48 KiB, else chunks of as many units as
// fit in 8 KiB.
int bf16_x_cap(const GemvPlan &p, int m) {
  const int64_t longest = ceil_div(p.total, p.grid);
  const int full = m * (x_slots(longest, int(p.units)) * kBfUnitK + 8);
  if (full * 2 <= 48 * 1024) return full;
  int chunk = (8 * 1024 / 2 / m - 8) / kBfUnitK;
  chunk = chunk < 1 ? 1 : chunk;
  return m * (chunk * kBfUnitK + 8);
}

}  // namespace

GemvPlan plan_gemv_bf16(int n, int k, const DeviceInfo &dev) {
  GemvPlan p;
  p.row_blocks = ceil_div(n, kRB);
  p.units = ceil_div(k, kBfUnitK);
  p.k_tiles = p.units;
  p.total = p.row_blocks * p.units;
  // Two persistent CTAs per SM; the grid depends on (n, k) and the SM
  // count only, never on m.
  int64_t g = int64_t(dev.sms) * kCtasPerSm;
  if (g > p.total) g = p.total;
  if (g < 1) g = 1;
  p.grid = int(g);
  int worst = 1;
  for (int64_t rb = 0; rb < p.row_blocks; ++rb) {
    const int64_t u0 = rb * p.units, u1 = u0 + p.units - 1;
    const int c = int(owner_of(u1, p.total, g) - owner_of(u0, p.total, g) + 1);
    if (c > worst) worst = c;
  }
  p.max_contrib = worst;
  return p;
}

size_t gemv_bf16_workspace_bytes(int n, int k, const DeviceInfo &dev) {
  const GemvPlan p = plan_gemv_bf16(n, k, dev);
  return kRestOffset + size_t(p.row_blocks) * p.max_contrib * kRB * 16 * sizeof(float);
}

cudaError_t launch_gemv_bf16(const uint16_t *w, int n, int k, const uint16_t *x, int m,
                             uint16_t *y, void *ws, bool pdl, const DeviceInfo &dev,
                             cudaStream_t st) {
  const GemvPlan plan = plan_gemv_bf16(n, k, dev);
  CUtensorMap tm_w;
  if (!encode_bf16_map(w, n, k, &tm_w)) return cudaErrorInvalidValue;

  Run r{};
  uint8_t *wsb = static_cast<uint8_t *>(ws);
  r.tickets = reinterpret_cast<uint32_t *>(wsb);
  r.zero = reinterpret_cast<uint32_t *>(wsb + kTicketBytes);
  r.partial = reinterpret_cast<float *>(wsb + kRestOffset);
  r.status = dev.status;
  r.m = m;
  r.x_cap = bf16_x_cap(plan, m);
  r.stages = stages_for(r.x_cap, 8);
  if (r.stages < kMinStages) return cudaErrorInvalidConfiguration;

  Proj p{};
  p.x = x;
  p.y = y;
  p.total = plan.total;
  p.n = n;
  p.k = k;
  p.units = int(plan.units);
  p.max_contrib = plan.max_contrib;
  p.grid = plan.grid;
  p.direct = direct_partials_fit(plan.row_blocks, plan.max_contrib, m) ? 1 : 0;
  p.scale_box = 0;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(plan.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem_bytes(r.stages, r.x_cap, 8);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  cudaError_t e;
  if (m <= 8) {
    if ((e = set_bf16_smem_attr<1>(dev.ordinal)) != cudaSuccess) return e;
    e = cudaLaunchKernelEx(&cfg, gemv_bf16_kernel<1>, tm_w, p, r);
  } else {
    if ((e = set_bf16_smem_attr<2>(dev.ordinal)) != cudaSuccess) return e;
    e = cudaLaunchKernelEx(&cfg, gemv_bf16_kernel<2>, tm_w, p, r);
  }
  return e;
}

}  // namespace aq
