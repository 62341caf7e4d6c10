// gemv.cu -- block-scaled NVFP4 GEMV for batch-1 / small-batch decode:
// y[t, i] = bf16( g_dec * sum_j sd[i, j] * sum_{k in block j} x[t, k] * e2m1(q[i, k]) )
// (Weightless docs, "GPU and cache acceleration", "Future work": a GEMV
// that dequantises the 4-bit weights in registers and streams them at full
// HBM bandwidth; AttnQuant docs, "Throughput", per-kernel MLP analysis: a
// skinny `down` projection needs split-K to fill the machine.)
//
// Design for sm_103a:
//  * Work unit = a row block of 128 rows by 2 k-tiles of 128 columns: one
//    16 KiB TMA box of packed nibbles (128-byte swizzle) plus one 2 KiB box
//    of scale words.  Tall boxes keep HBM efficient even though each CTA
//    streams its own contiguous range of units.
//  * Units are laid out row-block-major and cut into equal contiguous
//    ranges, one per persistent CTA (stream-K), two CTAs per SM, so every
//    CTA streams the same number of bytes whatever the shape.
//  * One producer warp streams units into a ring of 2..6 stages (as many as
//    the shared-memory budget allows after the activations); it runs ahead
//    of the programmatic-dependent-launch wait, so the next projection's
//    weights are in flight while the previous kernel drains.
//  * Eight consumer warps, one 16-row group each.  Lane 4g+c owns rows g
//    and g+8 and columns [32c, 32c+32) of each of the unit's two k-tiles:
//    16 bytes of nibbles per row per tile and one 32-bit scale word.
//    Nibbles become f16 pairs with the hardware e2m1x2 conversion, are
//    multiplied by their E4M3 block scale (exact in f16: at most 6
//    significant bits, within [2^-10, 2688]), and feed mma.sync m16n8k16
//    with fp32 accumulation; the two k-tiles use two independent
//    accumulators whose MMAs are interleaved.  Token activations are the B
//    operand, so 1..16 tokens share every decoded weight fragment.  The
//    column order inside an MMA k16 step is a permutation of the tile's
//    columns applied identically to weights and activations.
//  * Activations are staged in shared memory as f16 after an exact
//    power-of-two rescale that puts each token's largest |x| (over the whole
//    row) in [2^14, 2^15); bf16 values keep all 8 significand bits in f16
//    there (only values 2^29 below the maximum round), and the partial sums
//    are scaled back exactly.  When they fit they are staged once per CTA;
//    otherwise a few units at a time.
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

constexpr int kRG = 8;                          // row groups (consumer warps) per CTA
constexpr int kKT = 2;                          // k-tiles per unit
constexpr int kRB = 16 * kRG;                   // rows per row block
constexpr int kW = kRG;                         // consumer warps
constexpr int kThreads = (kW + 1) * 32;
constexpr int kUnitCols = 64 * kKT;             // packed bytes per row per unit (128)
constexpr int kPackedStage = kRB * kUnitCols;   // 16 KiB, 128-byte swizzled rows
constexpr int kScaleStage = kRG * 128 * kKT;    // 2 KiB of scale words
constexpr int kStageBytes = kPackedStage + kScaleStage;
constexpr int kMaxStages = 6;
constexpr int kMinStages = 2;
constexpr int kCtasPerSm = 2;
// Two CTAs per SM: each may use up to this much dynamic shared memory.
constexpr int kSmemBudget = 113 * 1024;
constexpr int kXChunkBudget = 16;               // m * units staged at once (chunked mode)
constexpr int kXFullBytes = 48 * 1024;          // activations staged once when they fit
constexpr int kTileHalves = 128;                // f16 per staged 128-column tile
constexpr unsigned kSpinLimit = 1u << 22;
static_assert(kStageBytes % 1024 == 0, "128-byte swizzle needs 1 KiB-aligned stages");
static_assert(kUnitCols == 128, "the swizzle pattern below assumes 128-byte rows");

// Control block that follows the ring in shared memory.
struct Ctrl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint32_t xmax[16];
  int shift[16];
  int flag;
  int aborted;
};
constexpr int kCtrlBytes = (int(sizeof(Ctrl)) + 15) / 16 * 16;

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

// Offset (in f16) of the 8 activations starting at column e of a staged
// token row: tile e/128, 32-column chunk c, 8-column sub-block q.  Chunks
// 2 and 3 store their sub-blocks in XOR-2 order so the four chunks a warp
// reads at once fall in distinct shared-memory banks.
__device__ __forceinline__ int x_off(int e) {
  const int c = (e >> 5) & 3, q = (e >> 3) & 3;
  return (e >> 7) * kTileHalves + c * 32 + ((q ^ (c & 2)) << 3);
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
  int units;           // units per row block = ceil(ceil(k / 128) / kKT)
  int max_contrib;
  int stages;          // ring depth
  int chunk_units;     // units whose activations are staged at once (chunked mode)
  int x_stride;        // f16 elements per staged token row
  int x_full;          // 1: all activations staged once at kernel start
};

}  // namespace

namespace {

// D += A * B with A 16x16 f16 (row), B 16x8 f16 (col), fp32 accumulate.
// Not volatile: the compiler may interleave independent MMA chains.
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// One unit of one warp: both k-tiles, MMAs of the two tiles interleaved.
// wlo/whi: the lane's 16 nibble bytes of rows g / g+8 per tile; sw: the
// lane's scale word per tile (rows g, g+8 x blocks 2c, 2c+1); xr: the
// lane's 32 activations per tile and n8 block of tokens, as f16 pairs.
template <int NT>
__device__ __forceinline__ void unit_mma(float (&acc)[2][NT][4], const uint4 (&wlo)[2],
                                         const uint4 (&whi)[2], const uint32_t (&sw)[2],
                                         const uint32_t (&xr)[2][NT][16]) {
  uint32_t sa[2][2], sb[2][2];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const uint32_t s01 = e4m3x2_to_f16x2(uint16_t(sw[t] & 0xFFFFu));
    const uint32_t s23 = e4m3x2_to_f16x2(uint16_t(sw[t] >> 16));
    sa[t][0] = __byte_perm(s01, 0, 0x1010);
    sa[t][1] = __byte_perm(s01, 0, 0x3232);
    sb[t][0] = __byte_perm(s23, 0, 0x1010);
    sb[t][1] = __byte_perm(s23, 0, 0x3232);
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t fl[2][4], fh[2][4];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const uint32_t lo = q == 0 ? wlo[t].x : q == 1 ? wlo[t].y : q == 2 ? wlo[t].z : wlo[t].w;
      const uint32_t hi = q == 0 ? whi[t].x : q == 1 ? whi[t].y : q == 2 ? whi[t].z : whi[t].w;
      e2m1x8_to_f16x2x4(lo, fl[t]);
      e2m1x8_to_f16x2x4(hi, fh[t]);
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int s = 2 * q + h;
      uint32_t A[2][4];
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        A[t][0] = hmul2(fl[t][2 * h], sa[t][q >> 1]);
        A[t][1] = hmul2(fh[t][2 * h], sb[t][q >> 1]);
        A[t][2] = hmul2(fl[t][2 * h + 1], sa[t][q >> 1]);
        A[t][3] = hmul2(fh[t][2 * h + 1], sb[t][q >> 1]);
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int t = 0; t < 2; ++t) mma_f16(acc[t][nt], A[t], xr[t][nt][2 * s], xr[t][nt][2 * s + 1]);
    }
  }
}

// Stage x[:, columns e0 .. e0 + nv*8) of every token into xs as scaled f16
// (zero past k); element e0 + e goes to offset x_off(e).
__device__ __forceinline__ void stage_x(const GemvArgs &a, const int *shift, uint16_t *xs, int e0,
                                        int nv) {
  for (int idx = threadIdx.x; idx < a.m * nv; idx += kW * 32) {
    const int tok = idx / nv, v = idx - tok * nv;
    const int e = v * 8, kk = e0 + e;
    uint4 q = make_uint4(0, 0, 0, 0);
    if (kk < a.k) q = __ldg(reinterpret_cast<const uint4 *>(a.x + int64_t(tok) * a.k + kk));
    const int sh = shift[tok];
    uint4 h;
    h.x = f32x2_to_f16x2(mul_pow2(bf16_hi(q.x), sh), mul_pow2(bf16_lo(q.x), sh));
    h.y = f32x2_to_f16x2(mul_pow2(bf16_hi(q.y), sh), mul_pow2(bf16_lo(q.y), sh));
    h.z = f32x2_to_f16x2(mul_pow2(bf16_hi(q.z), sh), mul_pow2(bf16_lo(q.z), sh));
    h.w = f32x2_to_f16x2(mul_pow2(bf16_hi(q.w), sh), mul_pow2(bf16_lo(q.w), sh));
    *reinterpret_cast<uint4 *>(xs + tok * a.x_stride + x_off(e)) = h;
  }
}

template <int NT>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    gemv_kernel(const __grid_constant__ CUtensorMap tm_w,
                const __grid_constant__ CUtensorMap tm_s, const GemvArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // The 128-byte swizzle of the weight stages needs a 1 KiB-aligned base.
  uint8_t *base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Ctrl &ct = *reinterpret_cast<Ctrl *>(base + a.stages * kStageBytes);
  uint16_t *xs = reinterpret_cast<uint16_t *>(base + a.stages * kStageBytes + kCtrlBytes);
  volatile int *aborted = &ct.aborted;
  const int S = a.stages;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t grid = gridDim.x;
  const int64_t u_begin = range_begin(blockIdx.x, a.total, grid);
  const int64_t u_end = range_begin(blockIdx.x + 1, a.total, grid);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&ct.full[s], 1);
      mbar_init(&ct.empty[s], kW);
    }
    ct.aborted = 0;
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
        const int st = int(j % S);
        if (j >= S && !mbar_wait(&ct.empty[st], unsigned((j / S) - 1) & 1u, aborted)) {
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
        uint8_t *stage = base + st * kStageBytes;
        mbar_expect_tx(&ct.full[st], kStageBytes);
        tma_load_2d(stage, &tm_w, uk * kUnitCols, int(rb * kRB), &ct.full[st]);
        tma_load_2d(stage + kPackedStage, &tm_s, uk * kKT * 128, int(rb * kRG), &ct.full[st]);
        issued = j + 1;
      }
      // No copy may still be landing in shared memory when the CTA exits:
      // wait (bounded) for the last phase of every stage that was filled.
      int never = 0;
      for (int64_t j = issued > S ? issued - S : 0; j < issued; ++j)
        mbar_wait(&ct.full[j % S], unsigned(j / S) & 1u, &never);
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  const int g = lane >> 2, c = lane & 3;
  const int rg = warp;
  // 128-byte swizzle: logical 16-byte chunk ch of box row r sits at ch ^ (r & 7);
  // rows rg*16 + g and rg*16 + g + 8 both have r & 7 == g.
  int off_lo[2], off_hi[2], off_sc[2];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    off_lo[t] = (rg * 16 + g) * kUnitCols + (((t * 4 + c) ^ g) << 4);
    off_hi[t] = (rg * 16 + g + 8) * kUnitCols + (((t * 4 + c) ^ g) << 4);
    off_sc[t] = kPackedStage + rg * (kKT * 128) + t * 128 + lane * 4;
  }
  pdl_wait();  // x and the workspace may come from the previous kernel
  const float gd = __ldg(a.g_dec);

  // -- per-token power-of-two shift from the largest |x| of the whole row
  //    (independent of the partition and of m); in full mode the raw bf16
  //    activations land in shared memory on the same pass and are converted
  //    in place afterwards.
  if (threadIdx.x < 16) ct.xmax[threadIdx.x] = 0;
  consumer_sync();
  {
    const int nv = a.units * kKT * 16;  // 8-element vectors per token (padded tiles)
    for (int tok = 0; tok < a.m; ++tok) {
      const uint16_t *xrow = a.x + int64_t(tok) * a.k;
      uint32_t mx = 0;
      for (int v = threadIdx.x; v < nv; v += kW * 32) {
        const int e = v * 8;
        uint4 q = make_uint4(0, 0, 0, 0);
        if (e < a.k) q = __ldg(reinterpret_cast<const uint4 *>(xrow + e));
        mx = __vmaxu2(mx, q.x & 0x7FFF7FFFu);
        mx = __vmaxu2(mx, q.y & 0x7FFF7FFFu);
        mx = __vmaxu2(mx, q.z & 0x7FFF7FFFu);
        mx = __vmaxu2(mx, q.w & 0x7FFF7FFFu);
        if (a.x_full) *reinterpret_cast<uint4 *>(xs + tok * a.x_stride + x_off(e)) = q;
      }
      mx = max(mx & 0xFFFFu, mx >> 16);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
      if (lane == 0 && mx != 0) atomicMax(&ct.xmax[tok], mx);
    }
  }
  consumer_sync();
  if (threadIdx.x < a.m) {
    const uint32_t b = ct.xmax[threadIdx.x];
    int sh = 0;
    if (b != 0 && b < 0x7F80u) sh = 14 - ilogbf(__uint_as_float(b << 16));
    ct.shift[threadIdx.x] = sh;
  }
  consumer_sync();
  if (a.x_full) {
    const int nv = a.units * kKT * 16;
    for (int tok = 0; tok < a.m; ++tok) {
      const int sh = ct.shift[tok];
      for (int v = threadIdx.x; v < nv; v += kW * 32) {
        uint4 *p = reinterpret_cast<uint4 *>(xs + tok * a.x_stride + x_off(v * 8));
        const uint4 q = *p;  // written by this same thread above
        uint4 h;
        h.x = f32x2_to_f16x2(mul_pow2(bf16_hi(q.x), sh), mul_pow2(bf16_lo(q.x), sh));
        h.y = f32x2_to_f16x2(mul_pow2(bf16_hi(q.y), sh), mul_pow2(bf16_lo(q.y), sh));
        h.z = f32x2_to_f16x2(mul_pow2(bf16_hi(q.z), sh), mul_pow2(bf16_lo(q.z), sh));
        h.w = f32x2_to_f16x2(mul_pow2(bf16_hi(q.w), sh), mul_pow2(bf16_lo(q.w), sh));
        *p = h;
      }
    }
    consumer_sync();
  }

  int64_t j = 0;
  int64_t u = u_begin;
  while (u < u_end) {
    const int64_t rb = u / a.units;
    const int uk0 = int(u - rb * a.units);
    const int uk1 = int(uk0 + (u_end - u) < a.units ? uk0 + (u_end - u) : a.units);

    float acc[2][NT][4];
#pragma unroll
    for (int t = 0; t < 2; ++t)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[t][nt][i] = 0.0f;

    const int step_units = a.x_full ? (uk1 - uk0) : a.chunk_units;
    for (int cu0 = uk0; cu0 < uk1; cu0 += step_units) {
      const int cu1 = min(uk1, cu0 + step_units);
      if (!a.x_full) {
        consumer_sync();  // earlier readers of the staging buffer are done
        stage_x(a, ct.shift, xs, cu0 * kKT * 128, (cu1 - cu0) * kKT * 16);
        consumer_sync();
      }
      const int tile0 = a.x_full ? 0 : cu0 * kKT;  // first k-tile held in xs

      for (int uk = cu0; uk < cu1; ++uk, ++j) {
        const int st = int(j % S);
        uint4 wlo[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
        uint4 whi[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
        uint32_t sw[2] = {0, 0};
        const bool ok = !*aborted && mbar_wait(&ct.full[st], unsigned(j / S) & 1u, aborted);
        if (ok) {
          const uint8_t *stage = base + st * kStageBytes;
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            wlo[t] = *reinterpret_cast<const uint4 *>(stage + off_lo[t]);
            whi[t] = *reinterpret_cast<const uint4 *>(stage + off_hi[t]);
            sw[t] = *reinterpret_cast<const uint32_t *>(stage + off_sc[t]);
          }
        } else if (lane == 0 && !*aborted) {
          *aborted = 1;
          raise_status(a.status, kDevTimeout);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&ct.empty[st]);

        // -- activations of the unit's two k-tiles for each n8 block of tokens
        uint32_t xr[2][NT][16];
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const int tl = uk * kKT + t - tile0;
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const int tok = min(nt * 8 + g, a.m - 1);
            const uint4 *p = reinterpret_cast<const uint4 *>(xs + tok * a.x_stride +
                                                             tl * kTileHalves + 32 * c);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const uint4 v = p[q ^ (c & 2)];
              xr[t][nt][4 * q + 0] = v.x;
              xr[t][nt][4 * q + 1] = v.y;
              xr[t][nt][4 * q + 2] = v.z;
              xr[t][nt][4 * q + 3] = v.w;
            }
          }
        }
        unit_mma<NT>(acc, wlo, whi, sw, xr);
      }
    }

    // -- epilogue: this warp holds rows g, g+8 x tokens nt*8 + 2c + {0,1};
    //    the two k-tile accumulators are added in a fixed order
    const bool complete = (uk0 == 0 && uk1 == a.units);
    const int64_t unit0 = rb * a.units;
    const int64_t own_lo = owner_of(unit0, a.total, grid);
    const int contrib = int(owner_of(unit0 + a.units - 1, a.total, grid) - own_lo + 1);
    const int jj = int(blockIdx.x - own_lo);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int token = nt * 8 + 2 * c + (i & 1);
        const int row_local = rg * 16 + g + 8 * (i >> 1);
        if (token >= a.m) continue;
        const float p = mul_pow2(__fadd_rn(acc[0][nt][i], acc[1][nt][i]), -ct.shift[token]);
        if (complete) {
          const int64_t row = rb * kRB + row_local;
          if (row < a.n) a.y[int64_t(token) * a.n + row] = f32_to_bf16_rn(__fmul_rn(p, gd));
        } else {
          a.partial[((rb * a.max_contrib + jj) * kRB + row_local) * 16 + token] = p;
        }
      }
    if (!complete) {
      // the barrier orders every warp's partial stores before thread 0's
      // gpu-scope fence, which publishes them with the ticket increment
      consumer_sync();
      if (threadIdx.x == 0) {
        __threadfence();
        const unsigned ticket = atomicAdd(&a.tickets[rb], 1u);
        __threadfence();
        ct.flag = (ticket == unsigned(contrib - 1));
      }
      consumer_sync();
      if (ct.flag) {
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

// 2-D uint8 tensor [rows, cols] (row pitch = cols bytes), copied in boxes
// of box_cols x box_rows; out-of-range parts of a box read as zero.
bool make_map(CUtensorMap *map, const void *base, uint64_t cols, uint64_t rows,
              uint32_t box_cols, uint32_t box_rows, bool swizzle128) {
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols};
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
  uint32_t box;
  bool operator==(const MapKey &o) const {
    return base == o.base && cols == o.cols && rows == o.rows && box == o.box;
  }
};
struct MapKeyHash {
  size_t operator()(const MapKey &k) const {
    return std::hash<uintptr_t>()(k.base) ^ (std::hash<uint64_t>()(k.cols * 1000003u + k.rows) << 1) ^
           k.box;
  }
};
std::mutex g_map_mu;
std::unordered_map<MapKey, CUtensorMap, MapKeyHash> g_maps;

bool cached_map(CUtensorMap *map, const void *base, uint64_t cols, uint64_t rows,
                uint32_t box_cols, uint32_t box_rows, bool swizzle128) {
  const MapKey key{reinterpret_cast<uintptr_t>(base), cols, rows,
                   (box_cols << 16) ^ (box_rows << 1) ^ (swizzle128 ? 1u : 0u)};
  {
    std::lock_guard<std::mutex> lock(g_map_mu);
    auto it = g_maps.find(key);
    if (it != g_maps.end()) {
      *map = it->second;
      return true;
    }
  }
  if (!make_map(map, base, cols, rows, box_cols, box_rows, swizzle128)) return false;
  std::lock_guard<std::mutex> lock(g_map_mu);
  if (g_maps.size() > 65536) g_maps.clear();
  g_maps.emplace(key, *map);
  return true;
}

int chunk_units_for(int m) { return kXChunkBudget / m < 1 ? 1 : kXChunkBudget / m; }

// Activation staging and ring depth of a launch.  All padded k-tiles are
// staged once (full mode) when m rows of them fit in kXFullBytes, else
// chunk_units units at a time; the ring gets what remains of the budget.
struct Layout {
  bool x_full;
  int x_stride;  // f16 per staged token row (+8 spreads tokens over banks)
  int stages;
  size_t smem;   // dynamic shared memory bytes
};
Layout layout_for(int64_t units, int m) {
  Layout L;
  const int full_stride = int(units * kKT * kTileHalves + 8);
  L.x_full = size_t(m) * full_stride * 2 <= size_t(kXFullBytes);
  L.x_stride = L.x_full ? full_stride : chunk_units_for(m) * kKT * kTileHalves + 8;
  const size_t x_bytes = size_t(m) * L.x_stride * 2;
  const size_t fixed = 1024 + kCtrlBytes + x_bytes;
  int st = int((size_t(kSmemBudget) - fixed) / kStageBytes);
  L.stages = st > kMaxStages ? kMaxStages : st;
  L.smem = fixed + size_t(L.stages) * kStageBytes;
  return L;
}

template <int NT>
cudaError_t set_smem_attr(int device) {
  static bool done[64] = {};
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (device >= 0 && device < 64 && done[device]) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(gemv_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSmemBudget);
  if (e == cudaSuccess && device >= 0 && device < 64) done[device] = true;
  return e;
}

// Ticket region of fixed size at the start of the workspace (one 32-bit
// ticket per row block of the largest legal n), then the fp32 partials.
// The fixed offset keeps the tickets of every shape clear of the partials
// of every other shape, so one zeroed workspace serves calls of any shape.
constexpr size_t kTicketBytes = size_t(((1 << 24) + kRB - 1) / kRB) * 4;

}  // namespace

GemvPlan plan_gemv(int n, int k, const DeviceInfo &dev) {
  GemvPlan p;
  p.row_blocks = ceil_div(n, kRB);
  p.k_tiles = ceil_div(k, kTileCols);
  p.units = ceil_div(p.k_tiles, kKT);
  p.total = p.row_blocks * p.units;
  // Two persistent CTAs per SM (the shared-memory budget of each CTA is set
  // so both are resident); tiny projections get one unit per CTA.  The
  // grid depends only on (n, k) and the SM count, never on m.
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

size_t gemv_workspace_bytes(int n, int k, const DeviceInfo &dev) {
  const GemvPlan p = plan_gemv(n, k, dev);
  return kTicketBytes + size_t(p.row_blocks) * p.max_contrib * kRB * 16 * sizeof(float);
}

cudaError_t launch_gemv(const aq_nvfp4_weight &w, const uint16_t *x, int m, uint16_t *y,
                        void *ws, bool pdl, const DeviceInfo &dev, cudaStream_t st) {
  if (!encoder()) return cudaErrorNotSupported;
  const GemvPlan p = plan_gemv(w.n, w.k, dev);
  const Layout L = layout_for(p.units, m);
  if (L.stages < kMinStages) return cudaErrorInvalidConfiguration;
  CUtensorMap tm_w, tm_s;
  if (!cached_map(&tm_w, w.packed, uint64_t(w.k) / 2, uint64_t(w.n), kUnitCols, kRB, true))
    return cudaErrorInvalidValue;
  const uint64_t srow = uint64_t(p.k_tiles) * 128;
  if (!cached_map(&tm_s, w.scales, srow, uint64_t(ceil_div(w.n, kTileRows)), kKT * 128, kRG,
                  false))
    return cudaErrorInvalidValue;

  GemvArgs a;
  a.g_dec = w.global_scale;
  a.x = x;
  a.y = y;
  uint8_t *wsb = static_cast<uint8_t *>(ws);
  a.tickets = reinterpret_cast<uint32_t *>(wsb);
  a.partial = reinterpret_cast<float *>(wsb + kTicketBytes);
  a.status = dev.status;
  a.total = p.total;
  a.n = w.n;
  a.k = w.k;
  a.m = m;
  a.units = int(p.units);
  a.max_contrib = p.max_contrib;
  a.stages = L.stages;
  a.chunk_units = chunk_units_for(m);
  a.x_stride = L.x_stride;
  a.x_full = L.x_full ? 1 : 0;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = L.smem;
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
