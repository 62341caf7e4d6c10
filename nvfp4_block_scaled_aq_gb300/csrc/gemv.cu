// gemv.cu -- block-scaled NVFP4 GEMV for batch-1 / small-batch decode:
// y[t, i] = bf16( g_dec * sum_j sd[i, j] * sum_{k in block j} x[t, k] * e2m1(q[i, k]) )
// (Weightless docs, "GPU and cache acceleration", "Future work": a GEMV
// that dequantises the 4-bit weights in registers and streams them at full
// HBM bandwidth; AttnQuant docs, "Throughput", per-kernel MLP analysis: a
// skinny `down` projection needs split-K to fill the machine.)
//
// Design for sm_103a:
//  * Work unit = (row block of 16*W rows, k tile of 128 columns).  The
//    units are laid out row-block-major and cut into `grid` equal
//    contiguous ranges, one per persistent CTA (stream-K), so every CTA
//    streams the same number of weight bytes whatever the shape.
//  * One producer warp streams each unit's packed nibbles (16*W x 64 B)
//    and scale words (W x 128 B) into an S-stage shared-memory ring with
//    2-D TMA copies completing on mbarriers; it starts before the
//    programmatic-dependent-launch wait, so weights of the next projection
//    are in flight while the previous kernel drains.
//  * W consumer warps, one 16-row group each.  Lane 4g+c owns rows g and
//    g+8 and columns [32c, 32c+32) of a tile: one 16-byte read per row and
//    one 32-bit scale word.  Nibbles become f16 pairs with the hardware
//    e2m1x2 conversion, are multiplied by their E4M3 block scale (exact in
//    f16: at most 6 significant bits, within [2^-10, 2688]), and feed
//    mma.sync m16n8k16 with fp32 accumulation; the token activations are
//    the B operand, so 1..16 tokens share every decoded weight fragment.
//    The column order inside the MMA's k16 step is a permutation of the
//    tile's columns applied identically to weights and activations.
//  * Activations are staged per segment into shared memory as f16 after an
//    exact power-of-two rescale that puts the segment's largest |x| in
//    [2^14, 2^15); bf16 values keep all 8 significand bits in f16 there
//    (only values 2^29 below the maximum round), and the partial sum is
//    scaled back exactly.
//  * Split-K across CTAs is deterministic: each contributor writes its fp32
//    partial to the workspace, the last to arrive (atomic ticket per row
//    block) adds the partials in contributor order and writes bf16 y, then
//    re-arms the ticket.  The partition depends only on (n, k) and the SM
//    count, never on m, so each token's result is independent of m.
//  * Every mbarrier wait is bounded; a wait that gives up records
//    AQ_ERR_TIMEOUT in the device status word and the CTA winds down.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>
#include <unordered_map>

#include "aq_internal.cuh"

namespace aq {
namespace {

// Geometry of one work unit: a row block of kRB = 16 * kRG rows by kKT
// k-tiles of 128 columns.  Consumer warp w owns row group (w % kRG) of the
// block and k-tile (w / kRG) of the unit; the kKT warps of one row group
// add their sums in a fixed order at the end of a segment.
#ifndef AQ_GEMV_STAGES
#define AQ_GEMV_STAGES 6
#endif
#ifndef AQ_GEMV_CTAS_PER_SM
#define AQ_GEMV_CTAS_PER_SM 2
#endif
constexpr int kRG = 4;                          // row groups per row block
constexpr int kKT = 2;                          // k-tiles per unit
constexpr int kRB = 16 * kRG;                   // rows per row block
constexpr int kW = kRG * kKT;                   // consumer warps
constexpr int kStages = AQ_GEMV_STAGES;         // TMA ring depth
constexpr int kThreads = (kW + 1) * 32;
constexpr int kUnitCols = 64 * kKT;             // packed bytes per row per unit
constexpr int kPackedStage = kRB * kUnitCols;   // 8 KiB, 128-byte swizzled rows
constexpr int kScaleStage = kRG * 128 * kKT;    // scale words of the unit
constexpr int kStageBytes = kPackedStage + kScaleStage;
constexpr int kXChunkBudget = 16;               // m * units staged at once
constexpr int kTileHalves = 160;                // f16 per staged 128-column tile (padded)
constexpr unsigned kSpinLimit = 1u << 22;
static_assert(kStageBytes % 1024 == 0, "128-byte swizzle needs 1 KiB-aligned stages");
static_assert(kUnitCols == 128, "the swizzle pattern below assumes 128-byte rows");

struct Smem {
  alignas(1024) uint8_t stage[kStages][kStageBytes];
  alignas(8) uint64_t full[kStages];
  uint64_t empty[kStages];
  float red[kRG][32][2][4];  // k-tile 1 sums handed to k-tile 0 warps
  uint32_t xmax[16];
  int shift[16];
  int flag;
  int aborted;
};
// activation staging follows the struct (dynamic, 16-byte aligned)

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Bounded wait for the phase with the given parity; false on give-up.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, unsigned parity,
                                          volatile int *aborted) {
  const uint32_t addr = smem_u32(bar);
  for (unsigned it = 0; it < kSpinLimit; ++it) {
    uint32_t done;
    asm volatile(
        "{ .reg .pred p;\n"
        "  mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "  selp.u32 %0, 1, 0, p; }"
        : "=r"(done)
        : "r"(addr), "r"(parity)
        : "memory");
    if (done) return true;
    if ((it & 1023u) == 1023u && *aborted) return false;
  }
  return false;
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y,
                                            uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// Consumer-warps-only barrier (the producer warp never joins it).
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kW * 32) : "memory");
}

// v * 2^e exactly (two steps keep each factor a normal fp32).
__device__ __forceinline__ float mul_pow2(float v, int e) {
  int e1 = e > 126 ? 126 : (e < -126 ? -126 : e);
  int e2 = e - e1;
  v = __fmul_rn(v, __int_as_float((e1 + 127) << 23));
  if (e2 != 0) v = __fmul_rn(v, __int_as_float((max(min(e2, 126), -126) + 127) << 23));
  return v;
}

// Stream-K partition helpers.
__device__ __host__ __forceinline__ int64_t range_begin(int64_t i, int64_t total, int64_t grid) {
  return (i * total) / grid;
}
__device__ __host__ __forceinline__ int64_t owner_of(int64_t u, int64_t total, int64_t grid) {
  return ((u + 1) * grid - 1) / total;
}

struct GemvArgs {
  const float *g_dec;
  const uint16_t *x;
  uint16_t *y;
  float *partial;      // [row_blocks][max_contrib][kRB][16]
  uint32_t *tickets;   // [row_blocks]
  unsigned *status;
  int64_t total;       // row_blocks * units (work units of the launch)
  int n, k, m;
  int k_tiles;         // ceil(k / 128)
  int units;           // units per row block = ceil(k_tiles / kKT)
  int max_contrib;
  int chunk_units;     // units whose activations are staged at once
  int x_stride;        // f16 elements per staged token row
};

}  // namespace

namespace {

// One k-tile of one warp: decode the lane's two 16-byte nibble runs (rows g
// and g+8, columns 32c..32c+31 of the tile), scale them by their block
// scales in f16, and accumulate 8 m16n8k16 products per n8 block of tokens.
// Even and odd k16 steps go to separate accumulators for latency overlap.
template <int NT>
__device__ __forceinline__ void tile_mma(float (&acc)[2][NT][4], const uint4 wlo,
                                         const uint4 whi, uint32_t sw,
                                         const uint32_t (&xr)[NT][16]) {
  const uint32_t s01 = e4m3x2_to_f16x2(uint16_t(sw & 0xFFFFu));
  const uint32_t s23 = e4m3x2_to_f16x2(uint16_t(sw >> 16));
  const uint32_t sa0 = __byte_perm(s01, 0, 0x1010), sa1 = __byte_perm(s01, 0, 0x3232);
  const uint32_t sb0 = __byte_perm(s23, 0, 0x1010), sb1 = __byte_perm(s23, 0, 0x3232);
  const uint32_t lo[4] = {wlo.x, wlo.y, wlo.z, wlo.w};
  const uint32_t hi[4] = {whi.x, whi.y, whi.z, whi.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t fl[4], fh[4];
    e2m1x8_to_f16x2x4(lo[q], fl);
    e2m1x8_to_f16x2x4(hi[q], fh);
    const uint32_t sa = q < 2 ? sa0 : sa1, sb = q < 2 ? sb0 : sb1;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t A[4] = {hmul2(fl[2 * h], sa), hmul2(fh[2 * h], sb),
                             hmul2(fl[2 * h + 1], sa), hmul2(fh[2 * h + 1], sb)};
      const int s = 2 * q + h;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma_16816(acc[h][nt], A, xr[nt][2 * s], xr[nt][2 * s + 1]);
    }
  }
}

template <int NT>
__global__ void __launch_bounds__(kThreads)
    gemv_kernel(const __grid_constant__ CUtensorMap tm_w,
                const __grid_constant__ CUtensorMap tm_s, const GemvArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // The 128-byte swizzle of the weight stages needs a 1 KiB-aligned base.
  uint8_t *smem_base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Smem &sm = *reinterpret_cast<Smem *>(smem_base);
  uint16_t *xs = reinterpret_cast<uint16_t *>(smem_base + sizeof(Smem));
  volatile int *aborted = &sm.aborted;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t grid = gridDim.x;
  const int64_t u_begin = range_begin(blockIdx.x, a.total, grid);
  const int64_t u_end = range_begin(blockIdx.x + 1, a.total, grid);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], kW);
    }
    sm.aborted = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    pdl_launch_dependents();
  }
  __syncthreads();

  // ------------------------------------------------------------ producer
  if (warp == kW) {
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_w)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_s)) : "memory");
      int64_t issued = 0;
      for (int64_t j = 0; u_begin + j < u_end; ++j) {
        const int st = int(j % kStages);
        if (j >= kStages &&
            !mbar_wait(&sm.empty[st], unsigned((j / kStages) - 1) & 1u, aborted)) {
          if (!*aborted) {
            *aborted = 1;
            raise_status(a.status, kDevTimeout);
          }
          break;
        }
        if (*aborted) break;
        const int64_t u = u_begin + j;
        const int64_t rb = u / a.units;
        const int uk = int(u - rb * a.units);
        mbar_expect_tx(&sm.full[st], kStageBytes);
        tma_load_2d(sm.stage[st], &tm_w, uk * kUnitCols, int(rb * kRB), &sm.full[st]);
        tma_load_2d(sm.stage[st] + kPackedStage, &tm_s, uk * kScaleStage / kRG, int(rb * kRG),
                    &sm.full[st]);
        issued = j + 1;
      }
      // No copy may still be landing in shared memory when the CTA exits:
      // wait (bounded) for the last phase of every stage that was filled.
      int never = 0;
      for (int64_t j = issued > kStages ? issued - kStages : 0; j < issued; ++j)
        mbar_wait(&sm.full[j % kStages], unsigned(j / kStages) & 1u, &never);
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  const int g = lane >> 2, c = lane & 3;
  const int rg = warp % kRG, kt = warp / kRG;
  // 128-byte swizzle: logical 16-byte chunk ch of row r sits at ch ^ (r & 7).
  const int off_lo = (rg * 16 + g) * kUnitCols + (((kt * 4 + c) ^ (g & 7)) << 4);
  const int off_hi = (rg * 16 + g + 8) * kUnitCols + (((kt * 4 + c) ^ ((g + 8) & 7)) << 4);
  const int off_sc = kPackedStage + (rg * kKT + kt) * 128 + lane * 4;
  pdl_wait();  // x and the workspace may come from the previous kernel
  const float gd = __ldg(a.g_dec);
  int64_t j = 0;
  int64_t u = u_begin;
  while (u < u_end) {
    const int64_t rb = u / a.units;
    const int uk0 = int(u - rb * a.units);
    const int uk1 = int(uk0 + (u_end - u) < a.units ? uk0 + (u_end - u) : a.units);

    // -- per-token exponent of this segment's activations
    if (threadIdx.x < 16) sm.xmax[threadIdx.x] = 0;
    consumer_sync();
    {
      const int k0 = uk0 * kUnitCols * 2, k1 = min(uk1 * kUnitCols * 2, a.k);
      const int nvec = (k1 - k0) / 8;
      for (int tok = 0; tok < a.m; ++tok) {
        const uint4 *xv = reinterpret_cast<const uint4 *>(a.x + int64_t(tok) * a.k + k0);
        uint32_t mx = 0;
        for (int v = threadIdx.x; v < nvec; v += kW * 32) {
          const uint4 q = __ldg(xv + v);
          mx = __vmaxu2(mx, q.x & 0x7FFF7FFFu);
          mx = __vmaxu2(mx, q.y & 0x7FFF7FFFu);
          mx = __vmaxu2(mx, q.z & 0x7FFF7FFFu);
          mx = __vmaxu2(mx, q.w & 0x7FFF7FFFu);
        }
        mx = max(mx & 0xFFFFu, mx >> 16);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
        if (lane == 0 && mx != 0) atomicMax(&sm.xmax[tok], mx);
      }
    }
    consumer_sync();
    if (threadIdx.x < a.m) {
      const uint32_t b = sm.xmax[threadIdx.x];
      int sh = 0;
      if (b != 0 && b < 0x7F80u) sh = 14 - ilogbf(__uint_as_float(b << 16));
      sm.shift[threadIdx.x] = sh;
    }

    float acc[2][NT][4];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[h][nt][i] = 0.0f;

    for (int cu0 = uk0; cu0 < uk1; cu0 += a.chunk_units) {
      const int cu1 = min(uk1, cu0 + a.chunk_units);
      consumer_sync();  // earlier readers of the staging buffer are done
      // -- stage x[:, k-tiles of units cu0..cu1) as scaled f16 (zero past k)
      {
        const int nv = (cu1 - cu0) * kKT * 16;  // 8-element vectors per token
        const int kbase = cu0 * kKT * 128;
        for (int idx = threadIdx.x; idx < a.m * nv; idx += kW * 32) {
          const int tok = idx / nv, v = idx - tok * nv;
          const int e = v * 8, kk = kbase + e;
          uint4 q = make_uint4(0, 0, 0, 0);
          if (kk < a.k)
            q = __ldg(reinterpret_cast<const uint4 *>(a.x + int64_t(tok) * a.k + kk));
          const int sh = sm.shift[tok];
          uint4 h;
          h.x = f32x2_to_f16x2(mul_pow2(bf16_hi(q.x), sh), mul_pow2(bf16_lo(q.x), sh));
          h.y = f32x2_to_f16x2(mul_pow2(bf16_hi(q.y), sh), mul_pow2(bf16_lo(q.y), sh));
          h.z = f32x2_to_f16x2(mul_pow2(bf16_hi(q.z), sh), mul_pow2(bf16_lo(q.z), sh));
          h.w = f32x2_to_f16x2(mul_pow2(bf16_hi(q.w), sh), mul_pow2(bf16_lo(q.w), sh));
          const int off = tok * a.x_stride + (e >> 7) * kTileHalves + ((e >> 5) & 3) * 40 +
                          (e & 31);
          *reinterpret_cast<uint4 *>(xs + off) = h;
        }
      }
      consumer_sync();

      for (int uk = cu0; uk < cu1; ++uk, ++j) {
        const int st = int(j % kStages);
        uint4 wlo = make_uint4(0, 0, 0, 0), whi = make_uint4(0, 0, 0, 0);
        uint32_t sw = 0;
        const bool ok = !*aborted &&
                        mbar_wait(&sm.full[st], unsigned(j / kStages) & 1u, aborted);
        if (ok) {
          const uint8_t *base = sm.stage[st];
          wlo = *reinterpret_cast<const uint4 *>(base + off_lo);
          whi = *reinterpret_cast<const uint4 *>(base + off_hi);
          sw = *reinterpret_cast<const uint32_t *>(base + off_sc);
        } else if (lane == 0 && !*aborted) {
          *aborted = 1;
          raise_status(a.status, kDevTimeout);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[st]);

        // -- activations of this warp's k-tile for each n8 block of tokens
        const int tl = (uk - cu0) * kKT + kt;
        uint32_t xr[NT][16];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const int tok = min(nt * 8 + g, a.m - 1);
          const uint4 *p =
              reinterpret_cast<const uint4 *>(xs + tok * a.x_stride + tl * kTileHalves + 40 * c);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint4 v = p[q];
            xr[nt][4 * q + 0] = v.x;
            xr[nt][4 * q + 1] = v.y;
            xr[nt][4 * q + 2] = v.z;
            xr[nt][4 * q + 3] = v.w;
          }
        }
        tile_mma<NT>(acc, wlo, whi, sw, xr);
      }
    }

    // -- fold: even/odd accumulators, then k-tile 1 warps into k-tile 0 warps
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[0][nt][i] = __fadd_rn(acc[0][nt][i], acc[1][nt][i]);
    if (kt == 1) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) sm.red[rg][lane][nt][i] = acc[0][nt][i];
    }
    consumer_sync();
    if (kt == 0) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i)
          acc[0][nt][i] = __fadd_rn(acc[0][nt][i], sm.red[rg][lane][nt][i]);
    }

    // -- epilogue: k-tile-0 warps hold rows g, g+8 x tokens nt*8 + 2c + {0,1}
    const bool complete = (uk0 == 0 && uk1 == a.units);
    const int64_t unit0 = rb * a.units;
    const int64_t own_lo = owner_of(unit0, a.total, grid);
    const int contrib = int(owner_of(unit0 + a.units - 1, a.total, grid) - own_lo + 1);
    const int jj = int(blockIdx.x - own_lo);
    if (kt == 0) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int token = nt * 8 + 2 * c + (i & 1);
          const int row_local = rg * 16 + g + 8 * (i >> 1);
          if (token >= a.m) continue;
          const float p = mul_pow2(acc[0][nt][i], -sm.shift[token]);
          if (complete) {
            const int64_t row = rb * kRB + row_local;
            if (row < a.n) a.y[int64_t(token) * a.n + row] = f32_to_bf16_rn(__fmul_rn(p, gd));
          } else {
            a.partial[((rb * a.max_contrib + jj) * kRB + row_local) * 16 + token] = p;
          }
        }
    }
    if (!complete) {
      __threadfence();
      consumer_sync();
      if (threadIdx.x == 0) {
        const unsigned ticket = atomicAdd(&a.tickets[rb], 1u);
        sm.flag = (ticket == unsigned(contrib - 1));
      }
      consumer_sync();
      if (sm.flag) {
        __threadfence();
        for (int idx = threadIdx.x; idx < kRB * a.m; idx += kW * 32) {
          const int row_local = idx / a.m, token = idx - row_local * a.m;
          const int64_t row = rb * kRB + row_local;
          if (row >= a.n) continue;
          float s = 0.0f;
          for (int q = 0; q < contrib; ++q)
            s = __fadd_rn(s, __ldcg(a.partial + ((rb * a.max_contrib + q) * kRB + row_local) * 16 +
                                    token));
          a.y[int64_t(token) * a.n + row] = f32_to_bf16_rn(__fmul_rn(s, gd));
        }
        if (threadIdx.x == 0) a.tickets[rb] = 0;
      }
    }
    u += uk1 - uk0;
  }
}

}  // namespace

// ------------------------------------------------------------------ host

namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool encoder() {
  std::call_once(g_encode_once, [] {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

// 2-D uint8 tensor [rows, cols] with a row pitch of `pitch` bytes, copied
// in boxes of box_cols x box_rows; out-of-range box parts read as zero.
bool make_map(CUtensorMap *map, const void *base, uint64_t cols, uint64_t rows,
              uint64_t pitch, uint32_t box_cols, uint32_t box_rows, bool swizzle128) {
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {pitch};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Encoded tensor maps are a pure function of (base, shape, box), so an
// exact-key cache can never return a stale map; it saves the encode on
// every launch of a decode step.
struct MapKey {
  uintptr_t base;
  uint64_t cols, rows;
  uint32_t box_rows;
  bool operator==(const MapKey &o) const {
    return base == o.base && cols == o.cols && rows == o.rows && box_rows == o.box_rows;
  }
};
struct MapKeyHash {
  size_t operator()(const MapKey &k) const {
    return std::hash<uintptr_t>()(k.base) ^ (std::hash<uint64_t>()(k.cols * 1000003u + k.rows) << 1) ^
           k.box_rows;
  }
};
std::mutex g_map_mu;
std::unordered_map<MapKey, CUtensorMap, MapKeyHash> g_maps;

bool cached_map(CUtensorMap *map, const void *base, uint64_t cols, uint64_t rows,
                uint32_t box_cols, uint32_t box_rows, bool swizzle128) {
  const MapKey key{reinterpret_cast<uintptr_t>(base), cols, rows,
                   box_rows * 2u + (swizzle128 ? 1u : 0u)};
  {
    std::lock_guard<std::mutex> lock(g_map_mu);
    auto it = g_maps.find(key);
    if (it != g_maps.end()) {
      *map = it->second;
      return true;
    }
  }
  if (!make_map(map, base, cols, rows, cols, box_cols, box_rows, swizzle128)) return false;
  std::lock_guard<std::mutex> lock(g_map_mu);
  if (g_maps.size() > 65536) g_maps.clear();
  g_maps.emplace(key, *map);
  return true;
}

int chunk_units_for(int m) { return kXChunkBudget / m < 1 ? 1 : kXChunkBudget / m; }

int x_stride_for(int m) { return chunk_units_for(m) * kKT * kTileHalves + 8; }

size_t smem_bytes_for(int m) { return 1024 + sizeof(Smem) + size_t(m) * x_stride_for(m) * 2; }

template <int NT>
cudaError_t set_smem_attr(int device) {
  // Largest dynamic shared memory any m <= 16 needs, set once per device.
  static bool done[64] = {};
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (device >= 0 && device < 64 && done[device]) return cudaSuccess;
  size_t worst = 0;
  for (int m = 1; m <= AQ_MAX_M; ++m) worst = smem_bytes_for(m) > worst ? smem_bytes_for(m) : worst;
  cudaError_t e = cudaFuncSetAttribute(gemv_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(worst));
  if (e == cudaSuccess && device >= 0 && device < 64) done[device] = true;
  return e;
}

}  // namespace

GemvPlan plan_gemv(int n, int k, const DeviceInfo &dev) {
  GemvPlan p;
  p.row_blocks = ceil_div(n, kRB);
  p.k_tiles = ceil_div(k, kTileCols);
  p.units = ceil_div(p.k_tiles, kKT);
  p.total = p.row_blocks * p.units;
  // Two resident CTAs per SM keep ~100 KiB of weights in flight per SM and
  // leave room for one CTA of the next projection to start early under
  // programmatic dependent launch.  Tiny projections get one unit per CTA.
  int64_t g = int64_t(dev.sms) * AQ_GEMV_CTAS_PER_SM;
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

// Workspace layout: a ticket region of fixed size at the start (one 32-bit
// ticket per row block of the largest legal n), then the fp32 partials.
// The fixed offset keeps the tickets of every shape clear of the partials
// of every other shape, so one zeroed workspace serves calls of any shape.
constexpr size_t kTicketBytes = size_t(((1 << 24) + kRB - 1) / kRB) * 4;

size_t gemv_workspace_bytes(int n, int k, const DeviceInfo &dev) {
  const GemvPlan p = plan_gemv(n, k, dev);
  return kTicketBytes + size_t(p.row_blocks) * p.max_contrib * kRB * 16 * sizeof(float);
}

cudaError_t launch_gemv(const aq_nvfp4_weight &w, const uint16_t *x, int m, uint16_t *y,
                        void *ws, bool pdl, const DeviceInfo &dev, cudaStream_t st) {
  if (!encoder()) return cudaErrorNotSupported;
  const GemvPlan p = plan_gemv(w.n, w.k, dev);
  CUtensorMap tm_w, tm_s;
  if (!cached_map(&tm_w, w.packed, uint64_t(w.k) / 2, uint64_t(w.n), kUnitCols, kRB, true))
    return cudaErrorInvalidValue;
  const uint64_t srow = uint64_t(p.k_tiles) * 128;
  if (!cached_map(&tm_s, w.scales, srow, uint64_t(ceil_div(w.n, kTileRows)), kScaleStage / kRG,
                  kRG, false))
    return cudaErrorInvalidValue;

  GemvArgs a;
  a.g_dec = w.global_scale;
  a.x = x;
  a.y = y;
  uint8_t *base = static_cast<uint8_t *>(ws);
  a.tickets = reinterpret_cast<uint32_t *>(base);
  a.partial = reinterpret_cast<float *>(base + kTicketBytes);
  a.status = dev.status;
  a.total = p.total;
  a.n = w.n;
  a.k = w.k;
  a.m = m;
  a.k_tiles = int(p.k_tiles);
  a.units = int(p.units);
  a.max_contrib = p.max_contrib;
  a.chunk_units = chunk_units_for(m);
  a.x_stride = x_stride_for(m);

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem_bytes_for(m);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  cudaError_t e;
  if (m <= 8) {
    if ((e = set_smem_attr<1>(dev.ordinal)) != cudaSuccess) return e;
    e = cudaLaunchKernelEx(&cfg, gemv_kernel<1>, tm_w, tm_s, a);
  } else {
    if ((e = set_smem_attr<2>(dev.ordinal)) != cudaSuccess) return e;
    e = cudaLaunchKernelEx(&cfg, gemv_kernel<2>, tm_w, tm_s, a);
  }
  return e;
}

}  // namespace aq
