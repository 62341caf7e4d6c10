// mma_gemm.cu -- the block-scaled MMA path: y = bf16( g_dec_w * g_dec_x[t] *
// sum_j sd_w[i, j] * sd_x[t, j] * sum_{k in block j} e2m1(q_w[i, k]) * e2m1(q_x[t, k]) )
// for 1..64 tokens whose activations were quantised to NVFP4 per row
// (AttnQuant docs, "Throughput", per-kernel profile: the NVFP4 MLP GEMMs of
// the serving stack consume fp4 weights directly and quantise the
// activations; "GPU acceleration", "NVFP4 quantization").
//
// Both operands reach the tensor core as they are stored: per 128 x 256
// unit, TMA brings the weight nibbles (16 KB, 128-byte swizzle), the weight
// scale tile (2 KB), the activation nibbles (N x 128 B, N = tokens rounded
// up to 16, rows past m read as zero) and the activation scales (N x 16 B).
// Four scale warps rearrange both scale sets into tcgen05.cp atoms; one
// lane of the MMA warp copies them into tensor memory and issues the four
// kind::mxf4nvf4 MMAs (M = 128, K = 64) of the unit into an fp32
// accumulator; four epilogue warps scale by g_dec_w * g_dec_x[t], round to
// bf16, and combine split-K partials deterministically (contributor 0
// reduces each row quarter once the others have published; partials added
// in contributor order).  Two persistent CTAs per
// SM, stream-K ranges of units exactly as the register-decode GEMV.  Every wait is
// bounded.
#include <cudaTypedefs.h>

#include <mutex>

#include "gemv_core.cuh"
#include "tc_ptx.cuh"

namespace aq {

using namespace core;

namespace {

constexpr int kMmaThreads = 320;  // producer, MMA, 4 scale warps, 4 epilogue warps
constexpr int kMmaMaxStages = 8;
constexpr int kMmaMinStages = 3;
// Two CTAs per SM: two independent TMA streams per SM keep HBM far busier
// than one (pure streaming of these boxes: ~6.3 TB/s with two, ~4.4 with
// one, whatever the depth).
constexpr int kMmaSmem = 113 * 1024;
constexpr int kWarpEpi = 6;
// tensor memory: accumulators 2 x 64 columns, weight-scale sets 2 x 16,
// activation-scale sets 2 x 16 (alternate units; copies and MMAs run in
// issue order)
constexpr int kAccCols = 64;
constexpr int kSfaCol = 2 * kAccCols;
constexpr int kSfbCol = kSfaCol + 32;
constexpr uint32_t kMmaTmemCols = 256;

__host__ __device__ __forceinline__ int mma_n(int m) { return (m + 15) / 16 * 16; }
// Stage layout for N activation rows.
__host__ __device__ __forceinline__ int st_b(int) { return kStageBytes; }
__host__ __device__ __forceinline__ int st_sfb(int n) { return kStageBytes + n * 128; }
__host__ __device__ __forceinline__ int st_atoms(int n) {
  return (kStageBytes + n * 128 + n * 16 + 127) / 128 * 128;
}
__host__ __device__ __forceinline__ int st_bytes(int n) {
  return (st_atoms(n) + 4096 + 1023) / 1024 * 1024;
}
__host__ __device__ __forceinline__ int tx_bytes(int n) { return kStageBytes + n * 128 + n * 16; }

struct MmaCtrl {
  uint64_t full[kMmaMaxStages];
  uint64_t empty[kMmaMaxStages];
  uint64_t sfready[kMmaMaxStages];
  uint64_t accfull[2];
  uint64_t accempty[2];
  uint64_t mma_done;
  uint32_t tmem;
  int aborted;
};
constexpr int kMmaCtrlBytes = (int(sizeof(MmaCtrl)) + 127) / 128 * 128;

__host__ __device__ __forceinline__ int mma_stages(int n) {
  const int s = (kMmaSmem - 1024 - kMmaCtrlBytes) / st_bytes(n);
  return s > kMmaMaxStages ? kMmaMaxStages : s;
}

// Activations and their scales as the kernel sees them.
struct ActQ {
  const float *g_dec;  // [m]
  int m;
  int slots;           // partial-sum token slots per row (>= m, multiple of 16)
};

__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, unsigned parity, volatile int *aborted,
                                              unsigned *status) {
  if (mbar_wait(bar, parity, aborted)) return true;
  if (!*aborted) {
    *aborted = 1;
    raise_status(status, kDevTimeout);
  }
  return false;
}

__global__ void __launch_bounds__(kMmaThreads, 2)
    mma_gemm_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_s,
                    const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_xs,
                    Proj p, const Run r, const ActQ a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *ring = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = r.stages, m = a.m, units = p.units;
  const int N = mma_n(m);
  const int SB = st_bytes(N);
  const int64_t grid = p.grid;
  const int64_t u_begin = range_begin(blockIdx.x, p.total, grid);
  const int64_t u_end = range_begin(blockIdx.x + 1, p.total, grid);
  MmaCtrl &ct = *reinterpret_cast<MmaCtrl *>(ring + S * SB);
  volatile int *aborted = &ct.aborted;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&ct.full[s], 1);
      mbar_init(&ct.empty[s], 1);
      mbar_init(&ct.sfready[s], 4);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&ct.accfull[b], 1);
      mbar_init(&ct.accempty[b], 4);
    }
    mbar_init(&ct.mma_done, 1);
    ct.aborted = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    pdl_launch_dependents();
  }
  if (warp == 1) tcx::tmem_alloc(&ct.tmem, kMmaTmemCols);
  tcx::fence_before_sync();
  __syncthreads();
  tcx::fence_after_sync();
  const uint32_t tmem = ct.tmem;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      // The weight nibbles and scales of the first ring stages do not depend
      // on the previous kernel (the activation quantisation): they are
      // issued before the dependent-launch wait, the activation boxes of
      // those stages after it.
      const int64_t pre = u_end - u_begin < S ? u_end - u_begin : S;
      for (int64_t i = 0; i < pre; ++i) {
        const int64_t u = u_begin + i, rb = u / units;
        const int uk = int(u - rb * units);
        uint8_t *stage = ring + i * SB;
        mbar_expect_tx(&ct.full[i], tx_bytes(N));
        tma_load_2d(stage, &tm_w, uk * kUnitCols, int(rb * kRB), &ct.full[i]);
        tma_load_2d(stage + kPackedStage, &tm_s, uk * kKT * 128, int(rb * kRG), &ct.full[i]);
      }
      pdl_wait();
      RingPos pos;
      for (int64_t i = 0; i < pre; ++i, pos.advance(S)) {
        const int64_t u = u_begin + i, rb = u / units;
        const int uk = int(u - rb * units);
        uint8_t *stage = ring + i * SB;
        (void)rb;
        tma_load_2d(stage + st_b(N), &tm_x, uk * kUnitCols, 0, &ct.full[i]);
        tma_load_2d(stage + st_sfb(N), &tm_xs, uk * 16, 0, &ct.full[i]);
      }
      for (int64_t u = u_begin + pre; u < u_end; ++u, pos.advance(S)) {
        const int st = pos.st;
        if (pos.wrapped && !wait_or_abort(&ct.empty[st], pos.phase ^ 1u, aborted, r.status)) break;
        if (*aborted) break;
        const int64_t rb = u / units;
        const int uk = int(u - rb * units);
        uint8_t *stage = ring + st * SB;
        mbar_expect_tx(&ct.full[st], tx_bytes(N));
        tma_load_2d(stage, &tm_w, uk * kUnitCols, int(rb * kRB), &ct.full[st]);
        tma_load_2d(stage + kPackedStage, &tm_s, uk * kKT * 128, int(rb * kRG), &ct.full[st]);
        tma_load_2d(stage + st_b(N), &tm_x, uk * kUnitCols, 0, &ct.full[st]);
        tma_load_2d(stage + st_sfb(N), &tm_xs, uk * 16, 0, &ct.full[st]);
      }
      int never = 0;
      for (int64_t j = pos.count > S ? pos.count - S : 0; j < pos.count; ++j)
        mbar_wait(&ct.full[j % S], unsigned(j / S) & 1u, &never);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue
    const bool leader = lane == 0;
    const uint32_t idesc = tcx::idesc_nvf4(N);
    const uint32_t ring_a = tcx::smem_addr(ring);
    RingPos pos;
    int uses[2] = {0, 0};
    int buf = 0;
    bool ok = true;
    int64_t u = u_begin;
    while (u < u_end && ok) {
      const int64_t rb = u / units;
      const int uk0 = int(u - rb * units);
      const int uk1 = int(uk0 + (u_end - u) < units ? uk0 + (u_end - u) : units);
      if (uses[buf] > 0)
        ok = __all_sync(0xFFFFFFFFu, wait_or_abort(&ct.accempty[buf], unsigned(uses[buf] - 1) & 1u,
                                                    aborted, r.status));
      if (!ok) break;
      for (int uk = uk0; uk < uk1; ++uk, pos.advance(S)) {
        const int st = pos.st;
        ok = __all_sync(0xFFFFFFFFu, wait_or_abort(&ct.full[st], pos.phase, aborted, r.status) &&
                                         wait_or_abort(&ct.sfready[st], pos.phase, aborted, r.status));
        if (!ok) break;
        tcx::fence_after_sync();
        const uint32_t stage_a = ring_a + st * SB;
        const uint32_t atoms = stage_a + st_atoms(N);
        const uint32_t sfa = tmem + kSfaCol + uint32_t(pos.count & 1) * 16;
        const uint32_t sfb = tmem + kSfbCol + uint32_t(pos.count & 1) * 16;
        if (leader) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            tcx::cp_atom(sfa + 4 * j, tcx::desc_atom(atoms + 512 * j));
            tcx::cp_atom(sfb + 4 * j, tcx::desc_atom(atoms + 2048 + 512 * j));
          }
#pragma unroll
          for (int j = 0; j < 4; ++j)
            tcx::mma_nvf4(tmem + buf * kAccCols, tcx::desc_k_sw128(stage_a + 32 * j),
                          tcx::desc_k_sw128(stage_a + st_b(N) + 32 * j), idesc, sfa + 4 * j,
                          sfb + 4 * j, uk > uk0 || j > 0);
          tcx::commit_to(&ct.empty[st]);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (leader) tcx::commit_to(&ct.accfull[buf]);
      __syncwarp();
      ++uses[buf];
      buf ^= 1;
      u += uk1 - uk0;
    }
    if (leader) {
      tcx::commit_to(&ct.mma_done);
      int never = 0;
      mbar_wait(&ct.mma_done, 0, &never);
    }
    __syncwarp();
  } else if (warp < kWarpEpi) {
    // ------------------------------------------------------------ scales
    // Thread t: weight row t's 16 scale bytes from the tile layout into its
    // words of the four weight atoms; and up to two activation scale words
    // (row n, k-step j) into the four activation atoms.  No barrier spans
    // the warps.
    const int t = threadIdx.x - 64;  // 0..127
    const int rt = t >> 4, h = (t >> 3) & 1, g = t & 7;
    RingPos pos;
    for (int64_t u = u_begin; u < u_end && !*aborted; ++u, pos.advance(S)) {
      const int st = pos.st;
      if (!wait_or_abort(&ct.full[st], pos.phase, aborted, r.status)) break;
      uint8_t *stage = ring + st * SB;
      uint8_t *atoms = stage + st_atoms(N);
      uint32_t wa[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int off = kPackedStage + rt * 256 + (j >> 1) * 128 + (4 * g + 2 * (j & 1)) * 4 + 2 * h;
        const uint32_t lo = *reinterpret_cast<const uint16_t *>(stage + off);
        const uint32_t hi = *reinterpret_cast<const uint16_t *>(stage + off + 4);
        wa[j] = lo | (hi << 16);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j)
        *reinterpret_cast<uint32_t *>(atoms + 512 * j + (t & 31) * 16 + (t >> 5) * 4) = wa[j];
      const uint8_t *sbox = stage + st_sfb(N);
      for (int idx = t; idx < N * 4; idx += 128) {
        const int n = idx >> 2, j = idx & 3;
        *reinterpret_cast<uint32_t *>(atoms + 2048 + 512 * j + (n & 31) * 16 + (n >> 5) * 4) =
            *reinterpret_cast<const uint32_t *>(sbox + n * 16 + 4 * j);
      }
      tcx::fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ct.sfready[st]);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    pdl_wait();  // outputs and the workspace may be in use by the previous kernel
    const float gdw = __ldg(p.g_dec);
    const int q = warp & 3;
    const uint32_t lane_base = tmem + (uint32_t(q * 32) << 16);
    const int row_local = q * 32 + lane;
    int uses[2] = {0, 0};
    int buf = 0;
    int64_t u = u_begin;
    while (u < u_end) {
      const int64_t rb = u / units;
      const int uk0 = int(u - rb * units);
      const int uk1 = int(uk0 + (u_end - u) < units ? uk0 + (u_end - u) : units);
      const bool ok = wait_or_abort(&ct.accfull[buf], unsigned(uses[buf]) & 1u, aborted, r.status);
      tcx::fence_after_sync();
      const bool complete = (uk0 == 0 && uk1 == units);
      const int64_t unit0 = rb * units;
      const int64_t own_lo = owner_of(unit0, p.total, grid);
      const int contrib = int(owner_of(unit0 + units - 1, p.total, grid) - own_lo + 1);
      const int jj = int(blockIdx.x - own_lo);
      const int64_t row = rb * kRB + row_local;
      // Partials are token-major ([row block][contributor][token][128
      // rows]) so a warp's 32 rows of one token are one coalesced 128-byte
      // store, and each 32-row quarter has its own ticket: the warp that
      // takes the quarter's last ticket adds the contributors' partials of
      // those 32 rows, in contributor order.  The accumulator is read 16
      // tokens at a time.
      float *mine = r.partial + (rb * p.max_contrib + jj) * int64_t(a.slots) * kRB + row_local;
      for (int c0 = 0; c0 < N; c0 += 16) {
        uint32_t h16[16];
        tcx::ld_x16(lane_base + buf * kAccCols + c0, h16);
        tcx::wait_ld();
        if (!ok) continue;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int tok = c0 + i;
          if (tok >= m) break;
          const float v = __uint_as_float(h16[i]);
          if (complete) {
            if (row < p.n)
              p.y[int64_t(tok) * p.n + row] =
                  f32_to_bf16_rn(__fmul_rn(__fmul_rn(v, __ldg(a.g_dec + tok)), gdw));
          } else {
            mine[tok * kRB] = v;
          }
        }
      }
      tcx::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ct.accempty[buf]);
      ++uses[buf];
      buf ^= 1;
      if (!ok) break;
      if (!complete) {
        // Contributor 0 (whose range ends in this row block, so usually the
        // last to finish it) reduces each 32-row quarter once the others
        // have published their partials with a release-add that nobody
        // waits on; it adds every contributor's partials (its own
        // included) in contributor order.
        __syncwarp();  // the warp's partial stores precede lane 0's release
        uint32_t *flag = r.tickets + rb * 4 + q;
        if (jj != 0) {
          if (lane == 0)
            asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(flag) : "memory");
        } else {
          bool ready = true;
          if (lane == 0) {
            const unsigned want = unsigned(contrib - 1);
            for (unsigned it = 0;; ++it) {
              unsigned seen;
              asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(seen) : "l"(flag) : "memory");
              if (seen >= want) break;
              if (it >= kSpinLimit || *aborted) {
                ready = false;
                break;
              }
              __nanosleep(32);
            }
            if (!ready && !*aborted) {
              *aborted = 1;
              raise_status(r.status, kDevTimeout);
            }
          }
          ready = __shfl_sync(0xFFFFFFFFu, ready, 0);
          __syncwarp();  // every lane's loads below follow lane 0's acquire
          if (ready && row < p.n) {
            // contributor by contributor, all tokens' loads in flight at once
            const float *base = r.partial + rb * p.max_contrib * int64_t(a.slots) * kRB + row_local;
            const int64_t cstride = int64_t(a.slots) * kRB;
            for (int t0 = 0; t0 < m; t0 += 16) {
              float acc[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) acc[i] = 0.0f;
              for (int c = 0; c < contrib; ++c) {
                float v[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                  v[i] = t0 + i < m ? __ldcg(base + c * cstride + (t0 + i) * kRB) : 0.0f;
#pragma unroll
                for (int i = 0; i < 16; ++i) acc[i] = __fadd_rn(acc[i], v[i]);
              }
#pragma unroll
              for (int i = 0; i < 16; ++i)
                if (t0 + i < m)
                  p.y[int64_t(t0 + i) * p.n + row] =
                      f32_to_bf16_rn(__fmul_rn(__fmul_rn(acc[i], __ldg(a.g_dec + t0 + i)), gdw));
            }
          }
          __syncwarp();
          if (ready && lane == 0) *flag = 0;
        }
      }
      u += uk1 - uk0;
    }
  }
  tcx::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tcx::fence_after_sync();
    tcx::tmem_dealloc(tmem, kMmaTmemCols);
  }
}

bool g_attr_done[64];
std::mutex g_attr_mu;

cudaError_t set_attr(int device) {
  std::lock_guard<std::mutex> lock(g_attr_mu);
  if (device >= 0 && device < 64 && g_attr_done[device]) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(mma_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMmaSmem);
  if (e == cudaSuccess && device >= 0 && device < 64) g_attr_done[device] = true;
  return e;
}

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

}  // namespace

// Workspace of the MMA path for m tokens: tickets, partials with
// mma_n(m) >= 16 token slots, then the quantised activations (packed,
// scales, g_dec), each 256-byte aligned.
MmaWorkspace mma_workspace(int n, int k, int m, const DeviceInfo &dev) {
  const GemvPlan p = plan_gemv(n, k, dev, 8);
  MmaWorkspace w;
  w.slots = mma_n(m) < 16 ? 16 : mma_n(m);
  w.scale_pitch = (k / 16 + 15) / 16 * 16;
  w.partial_off = kRestOffset;
  w.xq_off = align256(w.partial_off + size_t(p.row_blocks) * p.max_contrib * kRB * w.slots * 4);
  w.xs_off = align256(w.xq_off + size_t(m) * (k / 2));
  w.xg_off = align256(w.xs_off + size_t(m) * w.scale_pitch);
  w.bytes = align256(w.xg_off + size_t(m) * 4);
  return w;
}

bool mma_eligible(int n, int k, int m, const DeviceInfo &dev) {
  (void)n;
  (void)k;
  (void)dev;
  return m >= 1 && m <= 64 && mma_stages(mma_n(m)) >= kMmaMinStages;
}

// a7 then a8 on one stream: quantise x into the workspace, then the MMA.
cudaError_t launch_mma(const aq_nvfp4_weight &w, const uint16_t *x, int m, uint16_t *y, void *ws,
                       bool pdl, const DeviceInfo &dev, cudaStream_t st) {
  const MmaWorkspace lay = mma_workspace(w.n, w.k, m, dev);
  uint8_t *wsb = static_cast<uint8_t *>(ws);
  uint8_t *xq = wsb + lay.xq_off;
  uint8_t *xs = wsb + lay.xs_off;
  float *xg = reinterpret_cast<float *>(wsb + lay.xg_off);
  // Both kernels are launched as programmatic dependents.  The activation
  // quantisation waits for whatever precedes it before it reads x or writes
  // the workspace, so that is safe after any kernel (one that never lets
  // dependents start early simply finishes first), and it lets the MMA
  // kernel start streaming weights while the previous kernel drains and x
  // is quantised; the MMA kernel waits for the quantisation before it reads
  // the quantised activations or touches the workspace.
  (void)pdl;
  cudaError_t e = launch_act_quant(x, m, w.k, xq, xs, lay.scale_pitch, xg, dev, st, true);
  if (e != cudaSuccess) return e;

  const GemvPlan plan = plan_gemv(w.n, w.k, dev, 8);
  const int N = mma_n(m);
  CUtensorMap tm_w, tm_s, tm_x, tm_xs;
  if (!encode_maps(w, &tm_w, &tm_s, 8)) return cudaErrorInvalidValue;
  if (!encode_act_maps(xq, xs, m, w.k, lay.scale_pitch, N, &tm_x, &tm_xs))
    return cudaErrorInvalidValue;
  Run r{};
  r.tickets = reinterpret_cast<uint32_t *>(wsb);
  r.partial = reinterpret_cast<float *>(wsb + lay.partial_off);
  r.status = dev.status;
  r.m = m;
  r.stages = mma_stages(N);
  r.x_cap = 0;
  if (r.stages < kMmaMinStages) return cudaErrorInvalidConfiguration;
  Proj p{};
  p.tm_w = nullptr;
  p.tm_s = nullptr;
  p.g_dec = w.global_scale;
  p.x = x;
  p.y = y;
  p.total = plan.total;
  p.n = w.n;
  p.k = w.k;
  p.units = int(plan.units);
  p.max_contrib = plan.max_contrib;
  p.grid = plan.grid;
  ActQ a;
  a.g_dec = xg;
  a.m = m;
  a.slots = lay.slots;

  if ((e = set_attr(dev.ordinal)) != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(plan.grid);
  cfg.blockDim = dim3(kMmaThreads);
  cfg.dynamicSmemBytes = kMmaSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mma_gemm_kernel, tm_w, tm_s, tm_x, tm_xs, p, r, a);
}

}  // namespace aq
