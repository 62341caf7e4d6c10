// gemv_core.cuh -- device code shared by the single-projection GEMV kernel
// (gemv.cu) and the persistent decode-step kernel (step.cu): the TMA ring,
// the producer loop, and the consumer loop that dequantises NVFP4 weights
// in registers and accumulates with mma.sync.
//
// Method: Weightless docs, "GPU and cache acceleration", "Future work" (a
// GEMV that dequantises 4-bit weights in registers and streams at full HBM
// bandwidth); AttnQuant docs, "Throughput", per-kernel MLP analysis
// (split-K for skinny projections).  Design notes are in gemv.cu.
#pragma once

#include <cuda.h>

#include "aq_internal.cuh"

namespace aq {
namespace core {

constexpr int kRG = 8;                          // row groups (consumer warps) per CTA
constexpr int kKT = 2;                          // k-tiles per unit
constexpr int kRB = 16 * kRG;                   // rows per row block (128)
constexpr int kW = kRG;                         // consumer warps
constexpr int kThreads = (kW + 1) * 32;
constexpr int kUnitCols = 64 * kKT;             // packed bytes per row per unit (128)
constexpr int kUnitK = 128 * kKT;               // k columns per unit (256)
constexpr int kPackedStage = kRB * kUnitCols;   // 16 KiB, 128-byte swizzled rows
constexpr int kScaleStage = kRG * 128 * kKT;    // 2 KiB of scale words
constexpr int kStageBytes = kPackedStage + kScaleStage;
constexpr int kMaxStages = 6;
constexpr int kMinStages = 2;
constexpr int kCtasPerSm = 2;
constexpr int kSmemBudget = 113 * 1024;         // per CTA, so two fit on an SM
constexpr int kXChunkBudget = 64;               // m * units staged at once (chunked mode)
constexpr int kTileHalves = 128;                // f16 per staged 128-column tile
constexpr unsigned kSpinLimit = 1u << 22;
// Layout of every GEMV workspace:
//  [0, kTicketBytes)          32-bit tickets, eight per row block of the
//                             largest legal n (one per 16-row group of the
//                             register-decode kernel, or per 32-row quarter
//                             of the tcgen05 kernels);
//  [kTicketBytes, kRestOffset) the zero region: encoded split-K partials of
//                             the register-decode kernel, a word of zero
//                             meaning "not written yet";
//  [kRestOffset, ...)         the other kernels' partials and buffers.
// The first two regions are zero between calls: every kernel that writes
// there puts zeros back before it completes.
constexpr size_t kTicketBytes = size_t(((1 << 24) + kRB - 1) / kRB) * kTicketsPerRowBlock * 4;
constexpr size_t kZeroBytes = size_t(8) << 20;
constexpr size_t kRestOffset = kTicketBytes + kZeroBytes;
static_assert(kTicketsPerRowBlock == kRG, "one ticket per row group");
static_assert(kStageBytes % 1024 == 0, "128-byte swizzle needs 1 KiB-aligned stages");

// Geometry of the register-decode kernels for RG row groups (consumer warps)
// per CTA.  RG = 8: 128-row units of 18 KiB, two CTAs per SM (the constants
// above).  RG = 16: 256-row units of 36 KiB, one CTA per SM with sixteen
// consumer warps and one producer warp on one shared ring -- the SM's
// warps then finish a projection together (two CTAs on an SM do not: the
// warp schedulers favour the older one), the SM stages the activations
// once, and one 2-D copy moves 32 KiB.  Ticket words: RG per row block of
// 16 RG rows, so kTicketBytes serves both.
template <int RG>
struct Geo {
  static constexpr int kRG = RG;
  static constexpr int kRB = 16 * RG;
  static constexpr int kW = RG;
  static constexpr int kThreads = (RG + 1) * 32;
  static constexpr int kCtasPerSm = RG == 8 ? 2 : 1;
  static constexpr int kPackedStage = kRB * kUnitCols;
  static constexpr int kScaleStage = RG * 128 * kKT;
  static constexpr int kStageBytes = kPackedStage + kScaleStage;
  static constexpr int kSmemBudget = RG == 8 ? 113 * 1024 : 227 * 1024;
  // Deeper rings stream HBM more slowly (measured with these boxes: two
  // CTAs per SM peak at 3-4 stages of 18 KiB, one CTA per SM at 4 of 36 KiB).
  static constexpr int kMaxStages = RG == 8 ? 6 : 4;
  static_assert(RG == 8 || RG == 16, "8 or 16 row groups");
  static_assert(kStageBytes % 1024 == 0, "128-byte swizzle needs 1 KiB-aligned stages");
  static_assert(kMaxStages <= 6, "Ctrl holds six barrier pairs");
};
static_assert(kUnitCols == 128, "the swizzle pattern assumes 128-byte rows");

// Control block that follows the ring in shared memory.
struct Ctrl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint4 zero;               // 16 zero bytes: B operand of the one-token form
  uint32_t xmax[32];       // per token, or per (token, warp) for m <= 2
  int shift[16];
  int flag;
  int aborted;
};
constexpr int kCtrlBytes = (int(sizeof(Ctrl)) + 15) / 16 * 16;

// Position in the ring, advanced once per unit (no division on the hot
// path): stage index, parity of the current pass over the ring, and
// whether the ring has been through one full pass.
struct RingPos {
  int st = 0;
  unsigned phase = 0;
  bool wrapped = false;
  int64_t count = 0;  // units passed so far
  __host__ __device__ __forceinline__ void advance(int S) {
    ++count;
    if (++st == S) {
      st = 0;
      phase ^= 1u;
      wrapped = true;
    }
  }
};

// One projection as the kernels see it.
struct Proj {
  const CUtensorMap *tm_w;  // packed nibbles [n, k/2], box 128 B x 128 rows, 128B swizzle
  const CUtensorMap *tm_s;  // scale words [ceil(n/16), ceil(k/128)*128], box 256 B x 8 rows
  const float *g_dec;
  const uint16_t *x;        // [m, k] bf16
  uint16_t *y;              // [m, n] bf16
  int64_t total;            // row_blocks * units
  int n, k;
  int units;                // units per row block
  int max_contrib;          // most CTAs sharing a row block
  int grid;                 // CTAs that share this projection (<= total); the
                            // rest of the launch sits it out
  // The projection that runs next on the stream, whose first weight units
  // this CTA pulls into L2 once its own loads are issued (nx_pf = 0: none).
  const CUtensorMap *nx_w;
  const CUtensorMap *nx_s;
  int64_t nx_total;
  int nx_units;
  int nx_grid;
  int nx_pf;                // units per CTA to prefetch
  int direct;               // split-K partials go to the zero region, see
                            // direct_partials_fit()
  int scale_box;            // 1: each unit also loads its scale box (NVFP4);
                            // 0: the unit is the 16 KiB weight box only (bf16)
  // Runtime low-rank form (lr_s != nullptr): y = s * (g_dec * acc) + U t,
  // s fp32 [n], U bf16 [n, lr_r], t = V^T x fp32 [m, lr_r] (written by the
  // launch before this one on the stream).
  const float *lr_s;
  const uint16_t *lr_u;
  const float *lr_t;
  int lr_r;
  // Per-segment tensor scales: rows [seg_end[s-1], seg_end[s]) use
  // g_dec[s] (g_dec then points to nseg floats).
  int nseg;
  int seg_end[AQ_MAX_SEGMENTS];
};

// The reducer of a split row block can poll the partials themselves when
// they are stored encoded in the zero region: [row_blocks][max_contrib - 1]
// [m][rows per row block] words of ~bits(partial) (never zero: no fp32 operation yields
// the all-ones NaN), which it reads, adds and puts back to zero.  Used for
// m <= 8 (the one-n8-block kernel, where its registers are free) when the
// words fit the region; the sums are the same either way.
template <int RG = 8>
__host__ __device__ __forceinline__ bool direct_partials_fit(int64_t row_blocks, int max_contrib,
                                                             int m) {
  return m <= 8 && max_contrib <= 16 &&
         size_t(row_blocks) * size_t(max_contrib - 1) * size_t(m) * Geo<RG>::kRB * 4 <= kZeroBytes;
}

// Units of the next projection each CTA prefetches into L2 once its own
// loads are issued (4 x 18 KiB on each of 304 CTAs, 22 MB).  Measured on the
// decode-step chain: 4 gains ~1.5 %, deeper prefetch competes with the
// running launch's own loads and loses.
constexpr int kPrefetchUnits = 4;

// Per-launch state.
struct Run {
  float *partial;           // [row_blocks][max_contrib][kRB][16]
  uint32_t *tickets;        // [row_blocks][kRG]
  uint32_t *zero;           // the zero region (encoded partials)
  unsigned *status;
  int m;
  int stages;
  int x_cap;                // f16 capacity of the activation staging buffer
};

__host__ __device__ __forceinline__ int64_t range_begin(int64_t i, int64_t total, int64_t grid) {
  return (i * total) / grid;
}
__host__ __device__ __forceinline__ int64_t owner_of(int64_t u, int64_t total, int64_t grid) {
  return ((u + 1) * grid - 1) / total;
}

// The CTAs whose ranges meet row block rb (contrib of them) and the index
// jj of this CTA among them (0: the one whose range ends in rb).
__device__ __forceinline__ void row_block_share(const Proj &p, int64_t rb, int &contrib, int &jj) {
  const int64_t unit0 = rb * p.units;
  const int64_t own_lo = owner_of(unit0, p.total, p.grid);
  contrib = int(owner_of(unit0 + p.units - 1, p.total, p.grid) - own_lo + 1);
  jj = int(blockIdx.x - own_lo);
}

// Activations a CTA stages for its unit range [u_begin, u_end): the
// `slots` distinct units of k it touches (all units if the range is at
// least a row block long), each 256 columns, per token.
__host__ __device__ __forceinline__ int x_slots(int64_t range, int units) {
  return range >= units ? units : int(range);
}
__host__ __device__ __forceinline__ int x_stride_full(int slots) {
  return slots * 2 * kTileHalves + 8;  // +8 f16 spreads tokens over banks
}
__host__ __device__ __forceinline__ int chunk_units_for(int m) {
  return kXChunkBudget / m < 1 ? 1 : kXChunkBudget / m;
}
__host__ __device__ __forceinline__ int x_stride_chunk(int m) {
  return chunk_units_for(m) * 2 * kTileHalves + 8;
}

#ifdef __CUDACC__

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

// Bounded wait for the phase with the given parity (at most `limit` polls);
// false on give-up.
__device__ __forceinline__ bool mbar_wait_n(uint64_t *bar, unsigned parity,
                                            volatile int *aborted, unsigned limit) {
  const uint32_t addr = smem_u32(bar);
  for (unsigned it = 0; it < limit; ++it) {
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
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, unsigned parity,
                                          volatile int *aborted) {
  return mbar_wait_n(bar, parity, aborted, kSpinLimit);
}

// Epilogue kinds of the register-decode kernel.
constexpr int kEpiPlain = 0;    // y = bf16(g_dec * acc)
constexpr int kEpiLowRank = 1;  // y = bf16(s * (g_dec * acc) + U t)
constexpr int kEpiGlu = 2;      // h = bf16(gelu(gate) * up), rows paired in 8-row groups
constexpr int kEpiSegments = 3; // y = bf16(g_dec[segment(row)] * acc)

// GELU in its tanh form, fp32: 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))).
__device__ __forceinline__ float gelu_tanh(float x) {
  const float u = __fmul_rn(0.7978845608028654f,
                            __fmaf_rn(__fmul_rn(0.044715f, x), __fmul_rn(x, x), x));
  return __fmul_rn(__fmul_rn(0.5f, x), __fadd_rn(1.0f, tanhf(u)));
}

// Output value of one (row, token) before the bf16 rounding: g_dec * v, or
// in the runtime low-rank form s[row] * (g_dec * v) + sum_q U[row, q] *
// t[token, q], one fp32 multiply and then fused multiply-adds in q order.
// Plain loads: t comes from the previous kernel on the stream.
template <int EPI>
__device__ __forceinline__ float out_value(const Proj &p, int64_t row, int token, float v,
                                           float gd) {
  if (EPI == kEpiSegments) {
    int s = 0;
#pragma unroll
    for (int q = 0; q + 1 < AQ_MAX_SEGMENTS; ++q) s += (q + 1 < p.nseg && row >= p.seg_end[q]);
    gd = p.g_dec[s];
  }
  float z = __fmul_rn(v, gd);
  if (EPI == kEpiLowRank) {
    z = __fmul_rn(p.lr_s[row], z);
    for (int q = 0; q < p.lr_r; ++q)
      z = __fmaf_rn(__uint_as_float(uint32_t(p.lr_u[row * p.lr_r + q]) << 16),
                    p.lr_t[token * p.lr_r + q], z);
  }
  return z;
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y,
                                            uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// The same copy with an L2 eviction-priority hint (a policy made by
// createpolicy): the weight stream is read once per step, so its lines go
// in at evict_first and leave L2 to what is read again soon -- the
// activations, the split-K partials and the next projection's prefetched
// first units.
__device__ __forceinline__ void tma_load_2d_hint(void *dst, const CUtensorMap *map, int x, int y,
                                                 uint64_t *bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Consumer-warps-only barrier (the producer warp never joins it).
template <int RG = 8>
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(Geo<RG>::kW * 32) : "memory");
}

// What the consumers wait for before they read x (the weights never wait):
// nothing, the previous kernel on the stream (programmatic dependent
// launch), or, inside one persistent launch, a completion counter that
// every CTA of the previous projection bumps once its outputs are written.
struct Dep {
  int kind = 0;                  // kDepNone, kDepPdl or kDepCounter
  const unsigned *ctr = nullptr;
  unsigned target = 0;           // CTAs of the previous projection
};
constexpr int kDepNone = 0;
constexpr int kDepPdl = 1;
constexpr int kDepCounter = 2;

// Consumer thread 0 polls the counter (acquire, bounded) until it reaches
// the target; the barrier then releases every consumer thread after it.
template <int RG = 8>
__device__ __forceinline__ void wait_counter(const Dep &d, volatile int *aborted,
                                             unsigned *status) {
  if (threadIdx.x == 0) {
    for (unsigned it = 0;; ++it) {
      unsigned v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(d.ctr) : "memory");
      if (v >= d.target) break;
      if (it >= kSpinLimit || *aborted) {
        if (!*aborted) {
          *aborted = 1;
          raise_status(status, kDevTimeout);
        }
        break;
      }
      __nanosleep(20);
    }
  }
  consumer_sync<RG>();
}

// Every consumer's writes of a projection precede one release-add by
// consumer thread 0 (the barrier orders them; release is cumulative).
template <int RG = 8>
__device__ __forceinline__ void arrive_counter(unsigned *ctr) {
  consumer_sync<RG>();
  if (threadIdx.x == 0)
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(ctr) : "memory");
}

// v * 2^e exactly (two steps keep each factor a normal fp32).
__device__ __forceinline__ float mul_pow2(float v, int e) {
  int e1 = e > 126 ? 126 : (e < -126 ? -126 : e);
  int e2 = e - e1;
  v = __fmul_rn(v, __int_as_float((e1 + 127) << 23));
  if (e2 != 0) v = __fmul_rn(v, __int_as_float((max(min(e2, 126), -126) + 127) << 23));
  return v;
}

// Offset (in f16) of the 8 activations starting at staged column e: tile
// e/128, 32-column chunk c, 8-column sub-block q.  Chunks 2 and 3 store
// their sub-blocks in XOR-2 order so the four chunks a warp reads at once
// fall in distinct shared-memory banks.
__device__ __forceinline__ int x_off(int e) {
  const int c = (e >> 5) & 3, q = (e >> 3) & 3;
  return (e >> 7) * kTileHalves + c * 32 + ((q ^ (c & 2)) << 3);
}

__device__ __forceinline__ uint4 scale_to_f16(uint4 q, int sh) {
  uint4 h;
  h.x = f32x2_to_f16x2(mul_pow2(bf16_hi(q.x), sh), mul_pow2(bf16_lo(q.x), sh));
  h.y = f32x2_to_f16x2(mul_pow2(bf16_hi(q.y), sh), mul_pow2(bf16_lo(q.y), sh));
  h.z = f32x2_to_f16x2(mul_pow2(bf16_hi(q.z), sh), mul_pow2(bf16_lo(q.z), sh));
  h.w = f32x2_to_f16x2(mul_pow2(bf16_hi(q.w), sh), mul_pow2(bf16_lo(q.w), sh));
  return h;
}

__device__ __forceinline__ uint32_t absmax8(uint32_t mx, uint4 q) {
  mx = __vmaxu2(mx, q.x & 0x7FFF7FFFu);
  mx = __vmaxu2(mx, q.y & 0x7FFF7FFFu);
  mx = __vmaxu2(mx, q.z & 0x7FFF7FFFu);
  mx = __vmaxu2(mx, q.w & 0x7FFF7FFFu);
  return mx;
}

// D += A * B with A 16x16 f16 (row), B 16x8 f16 (col), fp32 accumulate.
// Not volatile: the compiler may interleave independent MMA chains.
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// D = A * B with a zero accumulator (the first MMA of a chain).
__device__ __forceinline__ void mma_f16_first(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%10, %10, %10, %10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.0f));
}

// 16 bytes from shared memory.  Volatile: never moved across the barriers
// that publish the staged activations.
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

// One unit of one warp for a single token, with the MMA's n dimension spent
// on blocks instead of tokens.  In k-tile t, MMA i (i = 0..7) takes element
// pair (2i, 2i+1) of each of the tile's eight 16-element blocks: MMA column
// pair (2c, 2c+1) carries block 2c and pair (2c+8, 2c+9) block 2c+1 of the
// lane's 32 columns, and the activation operand is block-diagonal, B[k, j] =
// x[k] when column k lies in block j and 0 otherwise.  After the eight MMAs
// D[row, j] is the unscaled dot product of block j, and the lane holds rows
// sg, sg+8 x blocks 2c, 2c+1 -- exactly the four blocks of its scale word --
// so each block scale costs one fp32 multiply-add instead of an f16
// multiply per weight pair.
// acc[0][0][i]: running sums over both tiles of (row sg, block 2c),
// (sg, 2c+1), (sg+8, 2c), (sg+8, 2c+1) of each tile.  xb[b][i]: the lane's B registers for column
// pair (2c, 2c+1) (b = 0) or (2c+8, 2c+9) (b = 1) of MMA i: block 2c + b of
// the token when the lane's MMA column g is 2c + b, else zero.
// The B registers of tile t are loaded from xb_addr[b][qq] + tb[t] * xb_step[b]
// just before the tile's MMAs.
__device__ __forceinline__ void unit_mma_bd(float (&acc)[2][1][4], const uint4 (&wlo)[2],
                                            const uint4 (&whi)[2], const uint32_t (&sw)[2],
                                            const uint32_t (&xb_addr)[2][2],
                                            const uint32_t (&xb_step)[2], const uint32_t (&tb)[2]) {
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    uint32_t xb[2][8];
#pragma unroll
    for (int b = 0; b < 2; ++b)
#pragma unroll
      for (int qq = 0; qq < 2; ++qq) {
        const uint4 v = lds128(xb_addr[b][qq] + tb[t] * xb_step[b]);
        xb[b][4 * qq + 0] = v.x;
        xb[b][4 * qq + 1] = v.y;
        xb[b][4 * qq + 2] = v.z;
        xb[b][4 * qq + 3] = v.w;
      }
    float d[4];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      uint32_t fl[4], fh[4], gl[4], gh[4];
      e2m1x8_to_f16x2x4(hh ? wlo[t].y : wlo[t].x, fl);  // row sg, block 2c
      e2m1x8_to_f16x2x4(hh ? whi[t].y : whi[t].x, fh);  // row sg+8, block 2c
      e2m1x8_to_f16x2x4(hh ? wlo[t].w : wlo[t].z, gl);  // row sg, block 2c+1
      e2m1x8_to_f16x2x4(hh ? whi[t].w : whi[t].z, gh);  // row sg+8, block 2c+1
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t A[4] = {fl[j], fh[j], gl[j], gh[j]};
        if (hh == 0 && j == 0)
          mma_f16_first(d, A, xb[0][0], xb[1][0]);
        else
          mma_f16(d, A, xb[0][4 * hh + j], xb[1][4 * hh + j]);
      }
    }
    const uint32_t s01 = e4m3x2_to_f16x2(uint16_t(sw[t] & 0xFFFFu));
    const uint32_t s23 = e4m3x2_to_f16x2(uint16_t(sw[t] >> 16));
    acc[0][0][0] = __fmaf_rn(d[0], f16_lo_to_f32(s01), acc[0][0][0]);
    acc[0][0][1] = __fmaf_rn(d[1], f16_hi_to_f32(s01), acc[0][0][1]);
    acc[0][0][2] = __fmaf_rn(d[2], f16_lo_to_f32(s23), acc[0][0][2]);
    acc[0][0][3] = __fmaf_rn(d[3], f16_hi_to_f32(s23), acc[0][0][3]);
  }
}

// One unit of one warp: both k-tiles, MMAs of the two tiles interleaved.
// wlo/whi: the lane's 16 nibble bytes of fragment rows g / g+8 per tile; sw: the
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

// Producer: stream this CTA's units of projection p into the ring.  j
// numbers the units this CTA handles across every projection of the launch,
// in the same order the consumers take them.  Returns false after a
// bounded wait gave up (the CTA is then aborting).
template <int RG = 8>
__device__ __forceinline__ bool produce(const Proj &p, uint8_t *base, Ctrl &ct, int S,
                                        RingPos &pos, volatile int *aborted, unsigned *status) {
  const int64_t grid = p.grid;
  if (int64_t(blockIdx.x) >= grid) return true;
  const int64_t u_begin = range_begin(blockIdx.x, p.total, grid);
  const int64_t u_end = range_begin(blockIdx.x + 1, p.total, grid);
  int64_t rb = u_begin / p.units;  // row block and k-unit of u, advanced
  int uk = int(u_begin - rb * p.units);  // without a division per unit
  const uint64_t policy = l2_evict_first_policy();
  for (int64_t u = u_begin; u < u_end; ++u, pos.advance(S)) {
    const int st = pos.st;
    // the stage was last filled one pass ago: wait for its release
    if (pos.wrapped && !mbar_wait(&ct.empty[st], pos.phase ^ 1u, aborted)) {
      if (!*aborted) {
        *aborted = 1;
        raise_status(status, kDevTimeout);
      }
      return false;
    }
    if (*aborted) return false;
    uint8_t *stage = base + st * Geo<RG>::kStageBytes;
    mbar_expect_tx(&ct.full[st], p.scale_box ? Geo<RG>::kStageBytes : Geo<RG>::kPackedStage);
    tma_load_2d_hint(stage, p.tm_w, uk * kUnitCols, int(rb * Geo<RG>::kRB), &ct.full[st], policy);
    if (p.scale_box)
      tma_load_2d_hint(stage + Geo<RG>::kPackedStage, p.tm_s, uk * kKT * 128, int(rb * Geo<RG>::kRG), &ct.full[st],
                       policy);
    if (++uk == p.units) {
      uk = 0;
      ++rb;
    }
  }
  return true;
}

// L2 prefetch of the first units of the next projection that the CTA with
// this index will load (same partition rule as produce()).  Weights never
// depend on earlier results, so this may run at any time; it reads nothing
// into the computation.  Issued by the producer lane after its own loads.
template <int RG = 8>
__device__ __forceinline__ void prefetch_next(const Proj &p) {
  if (p.nx_pf <= 0 || int64_t(blockIdx.x) >= p.nx_grid) return;
  const int64_t u_begin = range_begin(blockIdx.x, p.nx_total, p.nx_grid);
  int64_t u_end = range_begin(blockIdx.x + 1, p.nx_total, p.nx_grid);
  if (u_end > u_begin + p.nx_pf) u_end = u_begin + p.nx_pf;
  for (int64_t u = u_begin; u < u_end; ++u) {
    const int64_t rb = u / p.nx_units;
    const int uk = int(u - rb * p.nx_units);
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(p.nx_w)),
                 "r"(uk * kUnitCols), "r"(int(rb * Geo<RG>::kRB))
                 : "memory");
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(p.nx_s)),
                 "r"(uk * kKT * 128), "r"(int(rb * Geo<RG>::kRG))
                 : "memory");
  }
}

// No copy may still be landing in shared memory when the CTA exits: wait
// (bounded) for the last phase of every stage that was filled.  `issued`
// counts the units whose copies were started.
__device__ __forceinline__ void drain(Ctrl &ct, int S, int64_t issued) {
  int never = 0;
  for (int64_t j = issued > S ? issued - S : 0; j < issued; ++j)
    mbar_wait(&ct.full[j % S], unsigned(j / S) & 1u, &never);
}

// Pull the activation lines this CTA will stage into L2 ahead of the wait
// for the previous kernel (or projection): a prefetch reads nothing into the
// computation, and L2 stays coherent with any later write to x, so it is
// safe before the wait and takes the HBM latency off the staging after it.
template <int RG = 8>
__device__ __forceinline__ void prefetch_x_l2(const Proj &p, int m) {
  const int64_t grid = p.grid;
  if (int64_t(blockIdx.x) >= grid) return;
  const int64_t u_begin = range_begin(blockIdx.x, p.total, grid);
  const int64_t u_end = range_begin(blockIdx.x + 1, p.total, grid);
  if (u_begin >= u_end) return;
  const int units = p.units;
  const int64_t L = u_end - u_begin;
  const bool all_units = L >= units;
  const int uk_begin = int(u_begin % units);
  const int slots = x_slots(L, units);
  const int lines = m * slots * 4;  // 128-byte lines (64 bf16) per 256-column slot
  for (int i = threadIdx.x; i < lines; i += Geo<RG>::kW * 32) {
    const int tok = i / (slots * 4), rem = i - tok * slots * 4;
    const int s = rem >> 2, q = rem & 3;
    const int uk = all_units ? s : (uk_begin + s) % units;
    const int kk = uk * kUnitK + q * 64;
    if (kk < p.k)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(p.x + int64_t(tok) * p.k + kk));
  }
}

// The end of one row block's share of a CTA for one warp: vown[nt][i] is
// the warp's fp32 sum (before g_dec) for fragment rows sg, sg + 8 (i >> 1)
// and tokens nt*8 + 2c + (i & 1).  A row block wholly inside the CTA's range
// is written as bf16(g_dec * v).  Split row blocks: contributor 0 (the CTA
// whose range ends in this row block, so usually among the last to finish
// it) reduces, keeping its own partial in registers and adding the others'
// in contributor order; no barrier spans the warps, and no other
// contributor waits.
// contrib / jj: the CTAs sharing the row block and this CTA's index among
// them, when the caller has them already (contrib == 0: work them out).
template <int NT, int EPI = kEpiPlain, int RG = 8>
__device__ __forceinline__ void finish_rows(const Proj &p, const Run &r, int64_t rb, bool complete,
                                            const float (&vown)[NT][4], float gd, int rg, int sg,
                                            int lane, volatile int *aborted, int contrib = 0,
                                            int jj = 0) {
  const int units = p.units, m = r.m, c = lane & 3;
  if (contrib == 0) row_block_share(p, rb, contrib, jj);
  //  * direct: the others store ~bits(partial) to the zero region and
  //    leave; the reducer polls those words (bounded) until none is zero,
  //    then puts the zeros back.
  //  * otherwise: the others store plain partials and publish them with
  //    one release-add per (row block, row group); the reducer waits
  //    (bounded) for the count, reads the partials and clears the count.
  const bool reducer = !complete && jj == 0;
  const bool direct = NT == 1 && p.direct;
  const int64_t zrow = (rb * (p.max_contrib - 1) - 1) * m;  // + (j * m + token) * rows + row
  float fin[NT][4];  // final values before rounding (GLU: stored in pairs at the end)
  bool have = complete;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int token = nt * 8 + 2 * c + (i & 1);
      const int row_local = rg * 16 + sg + 8 * (i >> 1);
      const int64_t row = rb * Geo<RG>::kRB + row_local;
      const float v = vown[nt][i];
      if (token >= m || row >= p.n) continue;
      if (complete) {
        if (EPI == kEpiGlu)
          fin[nt][i] = out_value<EPI>(p, row, token, v, gd);
        else
          p.y[int64_t(token) * p.n + row] = f32_to_bf16_rn(out_value<EPI>(p, row, token, v, gd));
      } else if (!reducer) {
        if (direct)
          asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(
                           r.zero + (zrow + int64_t(jj) * m + token) * Geo<RG>::kRB + row_local),
                       "r"(~__float_as_uint(v))
                       : "memory");
        else
          r.partial[((rb * p.max_contrib + jj) * Geo<RG>::kRB + row_local) * 16 + token] = v;
      }
    }
  if (!complete && !reducer && !direct) {
    __syncwarp();  // the warp's partial stores precede lane 0's release
    if (lane == 0)
      asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(r.tickets + rb * Geo<RG>::kRG + rg)
                   : "memory");
  } else if (reducer && direct) {
    // Rows sg and sg + 8 of one token: every other contributor's word of
    // both is loaded before any is used, so one round trip serves the pair
    // when the partials are there already.
    bool ok = true;
    const int64_t qs = int64_t(m) * Geo<RG>::kRB;  // word of contributor q: at + q * qs
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        const int token = nt * 8 + 2 * c + b;
        if (!ok || token >= m) continue;
        const int rl0 = rg * 16 + sg, rl1 = rl0 + 8;
        const bool v0 = rb * Geo<RG>::kRB + rl0 < p.n, v1 = rb * Geo<RG>::kRB + rl1 < p.n;
        const int64_t at0 = (zrow + token) * Geo<RG>::kRB + rl0, at1 = at0 + 8;
        uint32_t w0[16], w1[16];
#pragma unroll
        for (int q = 1; q < 16; ++q) {
          w0[q] = 1u;
          w1[q] = 1u;
          if (q < contrib && v0)
            asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(w0[q]) : "l"(r.zero + (at0 + q * qs)) : "memory");
          if (q < contrib && v1)
            asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(w1[q]) : "l"(r.zero + (at1 + q * qs)) : "memory");
        }
        for (unsigned it = 0;; ++it) {
          bool all = true;
#pragma unroll
          for (int q = 1; q < 16; ++q) all = all && w0[q] != 0u && w1[q] != 0u;
          if (all) break;
          if (it >= kSpinLimit || *aborted) {
            ok = false;
            break;
          }
          __nanosleep(32);
#pragma unroll
          for (int q = 1; q < 16; ++q) {
            if (q < contrib && w0[q] == 0u)
              asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(w0[q]) : "l"(r.zero + (at0 + q * qs)) : "memory");
            if (q < contrib && w1[q] == 0u)
              asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(w1[q]) : "l"(r.zero + (at1 + q * qs)) : "memory");
          }
        }
        if (!ok) continue;
        float s0 = __fadd_rn(0.0f, vown[nt][b]), s1 = __fadd_rn(0.0f, vown[nt][b + 2]);
#pragma unroll
        for (int q = 1; q < 16; ++q)
          if (q < contrib) {
            s0 = __fadd_rn(s0, __uint_as_float(~w0[q]));
            s1 = __fadd_rn(s1, __uint_as_float(~w1[q]));
            if (v0)
              asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(r.zero + (at0 + q * qs)), "r"(0u) : "memory");
            if (v1)
              asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(r.zero + (at1 + q * qs)), "r"(0u) : "memory");
          }
        const int64_t row0 = rb * Geo<RG>::kRB + rl0, row1 = row0 + 8;
        if (EPI == kEpiGlu) {
          fin[nt][b] = out_value<EPI>(p, row0, token, s0, gd);
          fin[nt][b + 2] = out_value<EPI>(p, row1, token, s1, gd);
        } else {
          if (v0) p.y[int64_t(token) * p.n + row0] = f32_to_bf16_rn(out_value<EPI>(p, row0, token, s0, gd));
          if (v1) p.y[int64_t(token) * p.n + row1] = f32_to_bf16_rn(out_value<EPI>(p, row1, token, s1, gd));
        }
      }
    have = ok;
    if (!ok && !*aborted) {
      *aborted = 1;
      raise_status(r.status, kDevTimeout);
    }
  } else if (reducer) {
    uint32_t *flag = r.tickets + rb * Geo<RG>::kRG + rg;
    bool ok = true;
    if (lane == 0) {
      const unsigned want = unsigned(contrib - 1);
      unsigned seen = 0;
      for (unsigned it = 0;; ++it) {
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(seen) : "l"(flag) : "memory");
        if (seen >= want) break;
        if (it >= kSpinLimit || *aborted) {
          ok = false;
          break;
        }
        __nanosleep(32);
      }
      if (!ok && !*aborted) {
        *aborted = 1;
        raise_status(r.status, kDevTimeout);
      }
    }
    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    __syncwarp();  // every lane's loads below follow lane 0's acquire
    if (ok) {
      const int64_t qs = int64_t(Geo<RG>::kRB) * 16;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int token = nt * 8 + 2 * c + (i & 1);
          const int row_local = rg * 16 + sg + 8 * (i >> 1);
          const int64_t row = rb * Geo<RG>::kRB + row_local;
          if (token >= m || row >= p.n) continue;
          const float *src = r.partial + (rb * p.max_contrib * Geo<RG>::kRB + row_local) * 16 + token;
          float s = __fadd_rn(0.0f, vown[nt][i]);
          if (contrib <= 16) {
            float v[16];
#pragma unroll
            for (int q = 1; q < 16; ++q) v[q] = q < contrib ? __ldcg(src + q * qs) : 0.0f;
#pragma unroll
            for (int q = 1; q < 16; ++q)
              if (q < contrib) s = __fadd_rn(s, v[q]);
          } else {
            // sixteen loads in flight at a time, added in contributor order
            for (int q0 = 1; q0 < contrib; q0 += 16) {
              float v[16];
#pragma unroll
              for (int j = 0; j < 16; ++j) v[j] = q0 + j < contrib ? __ldcg(src + (q0 + j) * qs) : 0.0f;
#pragma unroll
              for (int j = 0; j < 16; ++j)
                if (q0 + j < contrib) s = __fadd_rn(s, v[j]);
            }
          }
          if (EPI == kEpiGlu)
            fin[nt][i] = out_value<EPI>(p, row, token, s, gd);
          else
            p.y[int64_t(token) * p.n + row] = f32_to_bf16_rn(out_value<EPI>(p, row, token, s, gd));
        }
      __syncwarp();
      if (lane == 0) *flag = 0;
    }
    have = ok;
  }
  if (EPI == kEpiGlu && have) {
    // rows sg (gate) and sg + 8 (up) of the row group pair up: output column
    // j = rb * 64 + rg * 8 + sg of h [m, n / 2]
    const int64_t j = rb * (Geo<RG>::kRB / 2) + rg * 8 + sg;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int token = nt * 8 + 2 * c + i;
        if (token >= m || 2 * j >= p.n) continue;
        p.y[int64_t(token) * (p.n / 2) + j] =
            f32_to_bf16_rn(__fmul_rn(gelu_tanh(fin[nt][i]), fin[nt][i + 2]));
      }
  }
}

// Consumers: the whole of this CTA's share of projection p -- activation
// staging, the unit loop, and the split-K epilogue.  Called by the RG
// consumer warps only.
// dep: what to wait for before reading x (the previous kernel on the
// stream, or the previous projection's completion counter), done once
// everything that does not read its results is worked out.
// BD: one token (NT == 1, m == 1) in the block-diagonal form of unit_mma_bd.
template <int NT, int EPI = kEpiPlain, bool BD = false, int RG = 8>
__device__ __forceinline__ void consume(const Proj &p, const Run &r, uint8_t *base, Ctrl &ct,
                                        uint16_t *xs, RingPos &pos, volatile int *aborted,
                                        const Dep &dep = Dep()) {
  static_assert(!BD || NT == 1, "the block-diagonal form serves one token");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int rg = warp;
  const int64_t grid = p.grid;
  if (int64_t(blockIdx.x) >= grid) return;
  const int64_t u_begin = range_begin(blockIdx.x, p.total, grid);
  const int64_t u_end = range_begin(blockIdx.x + 1, p.total, grid);
  if (u_begin >= u_end) return;
  const int S = r.stages, m = r.m, units = p.units;

  // 128-byte swizzle: logical 16-byte chunk ch of box row r sits at ch ^ (r & 7).
  // Fragment row g of the MMA holds stored row sg = sigma(g) (and sg + 8):
  // the eight lanes of each quarter-warp then read rows sg and sg ^ 4,
  // whose swizzled chunks fill all 32 banks once -- with sg = g the rows g
  // and g + 1 would share banks.  The rows are relabelled in the epilogue.
  const int sg = (g >> 1) | ((g & 1) << 2);
  int off_lo[2], off_hi[2], off_sc[2];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    off_lo[t] = (rg * 16 + sg) * kUnitCols + (((t * 4 + c) ^ sg) << 4);
    off_hi[t] = (rg * 16 + sg + 8) * kUnitCols + (((t * 4 + c) ^ sg) << 4);
    off_sc[t] = Geo<RG>::kPackedStage + rg * (kKT * 128) + t * 128 + (4 * sg + c) * 4;
  }

  // -- which k-units this CTA touches: all of them when its range covers a
  //    row block, else the L consecutive units (mod units) from uk_begin
  const int64_t L = u_end - u_begin;
  const bool all_units = L >= units;
  const int64_t rb0 = u_begin / units;
  const int uk_begin = int(u_begin - rb0 * units);
  const int slots = x_slots(L, units);
  const bool full = int64_t(m) * x_stride_full(slots) <= r.x_cap;
  const int stride = full ? x_stride_full(slots) : x_stride_chunk(m);
  // Only the first and the last row block of the range can be shared with
  // other CTAs: their contributor counts and this CTA's index among them.
  int contrib0, jj0, contrib1, jj1;
  row_block_share(p, rb0, contrib0, jj0);
  row_block_share(p, (u_end - 1) / units, contrib1, jj1);

  // -- per-token power-of-two shift from the largest |x| over the staged
  //    columns (a function of the token's own data and the partition only,
  //    never of m).
  const int nv_all = slots * (kUnitK / 8);  // 16-byte vectors per token
  const int per = (nv_all + Geo<RG>::kW * 32 - 1) / (Geo<RG>::kW * 32);
  constexpr int kV = 4;
  const bool in_regs = NT == 1 && full && m <= 2 && m * per <= 4;
  int kk_of[kV];  // column of each register-staged vector (-1: none)
#pragma unroll
  for (int j = 0; j < kV; ++j) {
    const int tok = j / per, v = threadIdx.x + (j - tok * per) * Geo<RG>::kW * 32;
    kk_of[j] = -1;
    if (in_regs && tok < m && v < nv_all) {
      const int s = v / (kUnitK / 8), within = (v % (kUnitK / 8)) * 8;
      const int uk = all_units ? s : (uk_begin + s) % units;
      const int kk = uk * kUnitK + within;
      if (kk < p.k) kk_of[j] = kk;
    }
  }
  if (dep.kind == kDepPdl)
    pdl_wait();
  else if (dep.kind == kDepCounter)
    wait_counter<RG>(dep, aborted, r.status);
  if (in_regs) {
    // Few vectors per thread: they stay in registers from the load to the
    // f16 store.  Each warp leaves its maximum per token in xmax[tok * RG +
    // warp]; after one barrier every thread derives the shift itself.
    uint4 q[kV];
    uint32_t mx0 = 0, mx1 = 0;
#pragma unroll
    for (int j = 0; j < kV; ++j) {
      const int tok = j / per;
      q[j] = make_uint4(0, 0, 0, 0);
      if (kk_of[j] >= 0)
        q[j] = __ldg(reinterpret_cast<const uint4 *>(p.x + int64_t(tok) * p.k + kk_of[j]));
    }
#pragma unroll
    for (int j = 0; j < kV; ++j) {
      if (j / per == 0) mx0 = absmax8(mx0, q[j]);
      else mx1 = absmax8(mx1, q[j]);
    }
    mx0 = max(mx0 & 0xFFFFu, mx0 >> 16);
    mx1 = max(mx1 & 0xFFFFu, mx1 >> 16);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      mx0 = max(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, o));
      mx1 = max(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, o));
    }
    if (lane == 0) {
      ct.xmax[warp] = mx0;
      if (m == 2) ct.xmax[Geo<RG>::kW + warp] = mx1;
    }
    consumer_sync<RG>();
    int sh[2] = {0, 0};
#pragma unroll
    for (int tok = 0; tok < 2; ++tok) {
      if (tok >= m) break;
      uint32_t b = 0;
#pragma unroll
      for (int w2 = 0; w2 < Geo<RG>::kW; ++w2) b = max(b, ct.xmax[tok * RG + w2]);
      if (b != 0 && b < 0x7F80u) sh[tok] = 14 - ilogbf(__uint_as_float(b << 16));
      if (threadIdx.x == tok) ct.shift[tok] = sh[tok];
    }
#pragma unroll
    for (int j = 0; j < kV; ++j) {
      const int tok = j / per, v = threadIdx.x + (j - tok * per) * Geo<RG>::kW * 32;
      if (tok < m && v < nv_all)
        *reinterpret_cast<uint4 *>(xs + tok * stride + x_off(v * 8)) =
            scale_to_f16(q[j], tok == 0 ? sh[0] : sh[1]);
    }
    consumer_sync<RG>();
  } else {
    // In full mode the raw bf16 values land in shared memory on the same
    // pass and are converted in place afterwards.
    if (threadIdx.x < 16) ct.xmax[threadIdx.x] = 0;
    consumer_sync<RG>();
    {
      const int nv = nv_all;
      for (int tok = 0; tok < m; ++tok) {
        const uint16_t *xrow = p.x + int64_t(tok) * p.k;
        uint32_t mx = 0;
        // four vectors per thread per round, every load issued before any
        // shared-memory store (the stores go through generic pointers, which
        // would otherwise keep each load waiting for the previous store)
        constexpr int kV = 4;
        for (int v0 = threadIdx.x; v0 < nv; v0 += kV * Geo<RG>::kW * 32) {
          uint4 q[kV];
#pragma unroll
          for (int i = 0; i < kV; ++i) {
            const int v = v0 + i * Geo<RG>::kW * 32;
            const int s = v / (kUnitK / 8), within = (v % (kUnitK / 8)) * 8;
            const int uk = all_units ? s : (uk_begin + s) % units;
            const int kk = uk * kUnitK + within;
            q[i] = make_uint4(0, 0, 0, 0);
            if (v < nv && kk < p.k) q[i] = __ldg(reinterpret_cast<const uint4 *>(xrow + kk));
          }
#pragma unroll
          for (int i = 0; i < kV; ++i) {
            const int v = v0 + i * Geo<RG>::kW * 32;
            if (v >= nv) break;
            mx = absmax8(mx, q[i]);
            if (full) *reinterpret_cast<uint4 *>(xs + tok * stride + x_off(v * 8)) = q[i];
          }
        }
        mx = max(mx & 0xFFFFu, mx >> 16);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
        if (lane == 0 && mx != 0) atomicMax(&ct.xmax[tok], mx);
      }
    }
    consumer_sync<RG>();
    if (threadIdx.x < m) {
      const uint32_t b = ct.xmax[threadIdx.x];
      int sh = 0;
      if (b != 0 && b < 0x7F80u) sh = 14 - ilogbf(__uint_as_float(b << 16));
      ct.shift[threadIdx.x] = sh;
    }
    consumer_sync<RG>();
    if (full) {
      const int nv = nv_all;
      for (int tok = 0; tok < m; ++tok) {
        const int sh = ct.shift[tok];
        for (int v = threadIdx.x; v < nv; v += Geo<RG>::kW * 32) {
          uint4 *q = reinterpret_cast<uint4 *>(xs + tok * stride + x_off(v * 8));
          *q = scale_to_f16(*q, sh);  // written by this same thread above
        }
      }
      consumer_sync<RG>();
    }
  }
  const float gd = __ldg(p.g_dec);

  // block-diagonal B operand: a lane whose MMA column g is block 2c + b of
  // its columns loads that block's two staged sub-blocks (address
  // xb_addr[b][qq] + the tile's offset); every other load of the lane reads
  // the 16 zero bytes of the control block (the tile offset times zero)
  uint32_t xb_addr[2][2], xb_step[2];
  if constexpr (BD) {
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      const bool act = g == 2 * c + b;
      xb_step[b] = act ? 1u : 0u;
#pragma unroll
      for (int qq = 0; qq < 2; ++qq)
        xb_addr[b][qq] = act ? smem_u32(xs) + 64 * c + 16 * ((2 * b + qq) ^ (c & 2))
                             : smem_u32(&ct.zero);
    }
  }

  int64_t u = u_begin, rb = rb0;
  int uk0 = uk_begin;
  while (u < u_end) {
    const int uk1 = int(uk0 + (u_end - u) < units ? uk0 + (u_end - u) : units);

    float acc[2][NT][4];
#pragma unroll
    for (int t = 0; t < 2; ++t)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[t][nt][i] = 0.0f;

    const int step_units = full ? (uk1 - uk0) : chunk_units_for(m);
    for (int cu0 = uk0; cu0 < uk1; cu0 += step_units) {
      const int cu1 = min(uk1, cu0 + step_units);
      if (!full) {
        consumer_sync<RG>();  // earlier readers of the staging buffer are done
        // four vectors per thread per round, all loaded before any is
        // converted and stored (a store through a generic pointer would
        // otherwise hold the next load back until it completes)
        const int nv = (cu1 - cu0) * (kUnitK / 8);
        constexpr int kCV = 4;
        constexpr int kStep = Geo<RG>::kW * 32;
        for (int base = threadIdx.x; base < m * nv; base += kCV * kStep) {
          uint4 q[kCV];
#pragma unroll
          for (int i = 0; i < kCV; ++i) {
            const int idx = base + i * kStep;
            const int tok = idx / nv, v = idx - tok * nv;
            const int kk = cu0 * kUnitK + v * 8;
            q[i] = make_uint4(0, 0, 0, 0);
            if (idx < m * nv && kk < p.k)
              q[i] = __ldg(reinterpret_cast<const uint4 *>(p.x + int64_t(tok) * p.k + kk));
          }
#pragma unroll
          for (int i = 0; i < kCV; ++i) {
            const int idx = base + i * kStep;
            if (idx >= m * nv) break;
            const int tok = idx / nv, v = idx - tok * nv;
            *reinterpret_cast<uint4 *>(xs + tok * stride + x_off(v * 8)) =
                scale_to_f16(q[i], ct.shift[tok]);
          }
        }
        consumer_sync<RG>();
      }

      // staged slot of unit cu0 (slots follow units, wrapping at `units`)
      int slot = full ? (all_units ? cu0 : (cu0 >= uk_begin ? cu0 - uk_begin : cu0 + units - uk_begin))
                      : 0;
      for (int uk = cu0; uk < cu1; ++uk, ++slot, pos.advance(S)) {
        const int st = pos.st;
        uint4 wlo[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
        uint4 whi[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
        uint32_t sw[2] = {0, 0};
        const bool ok = !*aborted && mbar_wait(&ct.full[st], pos.phase, aborted);
        if (ok) {
          const uint8_t *stage = base + st * Geo<RG>::kStageBytes;
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            wlo[t] = *reinterpret_cast<const uint4 *>(stage + off_lo[t]);
            whi[t] = *reinterpret_cast<const uint4 *>(stage + off_hi[t]);
            sw[t] = *reinterpret_cast<const uint32_t *>(stage + off_sc[t]);
          }
        } else if (lane == 0 && !*aborted) {
          *aborted = 1;
          raise_status(r.status, kDevTimeout);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&ct.empty[st]);

        if constexpr (BD) {
          const uint32_t tb[2] = {uint32_t(slot * kKT) * (kTileHalves * 2),
                                  uint32_t(slot * kKT + 1) * (kTileHalves * 2)};
          unit_mma_bd(acc, wlo, whi, sw, xb_addr, xb_step, tb);
          continue;
        }

        // -- activations of the unit's two k-tiles for each n8 block of tokens
        uint32_t xr[2][NT][16];
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const int tl = slot * kKT + t;
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const int tok = min(nt * 8 + g, m - 1);
            const uint4 *px =
                reinterpret_cast<const uint4 *>(xs + tok * stride + tl * kTileHalves + 32 * c);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const uint4 v = px[q ^ (c & 2)];
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

    // -- epilogue: this warp holds rows sg, sg+8 x tokens nt*8 + 2c + {0,1};
    //    the two k-tile accumulators are added in a fixed order
    const bool complete = (uk0 == 0 && uk1 == units);
    float v[NT][4];
    if constexpr (BD) {
      // rows sg and sg+8: the lane's two block columns, then the four lanes
      // of the quad (all four end with the same sums)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float rs = __fadd_rn(acc[0][0][2 * h], acc[0][0][2 * h + 1]);
        rs = __fadd_rn(rs, __shfl_xor_sync(0xFFFFFFFFu, rs, 1));
        rs = __fadd_rn(rs, __shfl_xor_sync(0xFFFFFFFFu, rs, 2));
        v[0][2 * h] = mul_pow2(rs, -ct.shift[0]);
        v[0][2 * h + 1] = 0.0f;  // token 1: not present
      }
    } else {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int token = nt * 8 + 2 * c + (i & 1);
          v[nt][i] = mul_pow2(__fadd_rn(acc[0][nt][i], acc[1][nt][i]), -ct.shift[min(token, 15)]);
        }
    }
    // (two token blocks: the shares are worked out again, which keeps
    // their registers free through the unit loop)
    finish_rows<NT, EPI, RG>(p, r, rb, complete, v, gd, rg, sg, lane, aborted,
                         NT > 1 ? 0 : complete ? 1 : (rb == rb0 ? contrib0 : contrib1),
                         complete ? 0 : (rb == rb0 ? jj0 : jj1));
    u += uk1 - uk0;
    ++rb;
    uk0 = 0;
  }
}

// Shared-memory carve-up: ring (1 KiB aligned), control block, activations.
struct SmemView {
  uint8_t *base;
  Ctrl *ct;
  uint16_t *xs;
};
template <int RG = 8>
__device__ __forceinline__ SmemView carve(uint8_t *raw, int stages) {
  SmemView v;
  v.base = raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
  v.ct = reinterpret_cast<Ctrl *>(v.base + stages * Geo<RG>::kStageBytes);
  v.xs = reinterpret_cast<uint16_t *>(v.base + stages * Geo<RG>::kStageBytes + kCtrlBytes);
  return v;
}

template <int RG = 8>
__device__ __forceinline__ void init_ring(Ctrl &ct, int S) {
  for (int s = 0; s < S; ++s) {
    mbar_init(&ct.full[s], 1);
    mbar_init(&ct.empty[s], Geo<RG>::kW);
  }
  ct.aborted = 0;
  ct.zero = make_uint4(0, 0, 0, 0);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

#endif  // __CUDACC__

// Host-side helpers shared by the launchers.
size_t smem_bytes(int stages, int x_cap_halves, int rg);
int stages_for(int x_cap_halves, int rg);
bool encode_maps(const aq_nvfp4_weight &w, CUtensorMap *tm_w, CUtensorMap *tm_s, int rg);
bool encode_bf16_map(const uint16_t *w, int n, int k, CUtensorMap *tm);
bool encode_bf16_rows_map(const uint16_t *w, int n, int k, int box_rows, CUtensorMap *tm);
bool encode_bytes_1d(const void *base, uint64_t bytes, uint32_t box, CUtensorMap *tm);

}  // namespace core
}  // namespace aq
