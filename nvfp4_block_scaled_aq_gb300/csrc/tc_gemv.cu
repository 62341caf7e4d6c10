// tc_gemv.cu -- the block-scaled NVFP4 GEMV on the tcgen05 tensor cores.
// y[t, i] = bf16( g_dec * sum_j sd[i, j] * sum_{k in block j} x[t, k] * e2m1(q[i, k]) )
// for 1..5 tokens (AttnQuant docs, "GPU acceleration", "NVFP4 quantization":
// packed nibbles plus E4M3 block scales; Weightless docs, "GPU and cache
// acceleration", "Future work": a 4-bit GEMV that streams the weights at
// HBM bandwidth).
//
// Why the tensor core's block-scaled fp4 MMA: it consumes the packed
// nibbles and their E4M3 scales straight from shared memory, so the weight
// stream needs no per-element decode on the CUDA cores (the decode is what
// bounds the register-decode kernel in gemv.cu).  The operation is an
// fp4 x fp4 product, so the bf16 activations are given to it as an exact
// short sum of NVFP4 terms (below), not rounded to one fp4 value.
//
// Activations as NVFP4 terms.  For each token the CTA takes the largest |x|
// over the columns it touches, xmax, and sets G_1 = 2^(ilogb(xmax) - 6) and
// G_t = G_1 * 2^(-3(t-1)).  Each 16-column block is split greedily into
// kTerms terms: with r the block's residual (x at first), term t has the
// E4M3 block scale s_t = E4M3(max|r| / 6 / G_t) (nearest even, saturating),
// nibbles q_t = E2M1(r / (s_t G_t)) (nearest even, saturating), and the
// residual becomes r - q_t s_t G_t (every product exact).  Each term
// shrinks the residual about six-fold, so after 6 terms it is below about
// 2^-19 of the token's largest |x| (checked on the CPU against fp64 over
// N(0,1) rows: GEMV error ~1e-5 relative, far inside the 2e-3 tolerance).  The terms of
// token t are the B-operand columns 6t .. 6t+5 (N = 16 for <= 2 tokens, 32
// for <= 5); the epilogue forms y = g_dec * sum_t G_t * D[:, col], where D
// is the fp32 accumulator in tensor memory.  Results depend only on the
// token's own data and the (n, k)-fixed partition: never on m.
//
// CTA (one per SM, persistent, stream-K ranges of 128 x 256 units exactly
// as the register-decode kernel, 227 KB shared memory), 14 warps:
//  * warp 0: TMA producer into a ring of 3..8 stages (16 KB nibbles with
//    128-byte swizzle + 2 KB scale tiles per stage), ahead of the PDL wait.
//  * warp 1: allocates tensor memory; one lane issues 4 MMAs (K = 64 each)
//    per unit (k-step j into chain j of one of two accumulator sets), commits each stage back to the
//    producer and each finished row block to the epilogue.
//  * warps 2..5: per unit, move the weight scales of the stage (and the
//    activation-term scales of the unit's k range) from shared memory into
//    tensor memory in the MMA's scale layout.
//  * warps 6..9: epilogue -- read the accumulator, combine the terms, write
//    y or the split-K partial (same deterministic ticket scheme as gemv.cu).
//  * warps 10..13 help stage: warps 2..13 first stage the activation terms
//    of the CTA's k range.
// Every wait is bounded; a wait that gives up records AQ_ERR_TIMEOUT and
// the CTA winds down, waiting (bounded) for its copies and MMAs, and frees
// its tensor memory.
#include <cudaTypedefs.h>

#include <climits>
#include <mutex>

#include "gemv_core.cuh"
#include "tc_ptx.cuh"

namespace aq {

using namespace core;

namespace {

constexpr int kTerms = 6;
constexpr int kTcMaxTokens = 5;
constexpr int kTcThreads = 448;
constexpr int kWarpMma = 1, kWarpEpi = 6;  // scale warps 2..5, staging-only warps 10..13
constexpr int kStagers = 384;              // warps 2..13 stage the activation terms
constexpr int kTcMaxStages = 12;
constexpr int kTcMinStages = 3;
constexpr int kTcSmem = 227 * 1024;
constexpr int kDCols = 32;   // tensor-memory columns per accumulator
// A ring stage: the 16 KB nibble box and the 2 KB scale box (both by TMA),
// then the four 512-byte copy atoms of the weight scales (by the scale
// warps).
constexpr int kTcStageBytes = kStageBytes + 2048;
constexpr int kBoxOff = kPackedStage;
constexpr int kSfaOff = kStageBytes;
// Tensor memory: two accumulators (columns 0..63), two weight-scale sets
// used by alternate units (64..95; copies and MMAs run in issue order, so a
// set is rewritten only after the MMAs that read it), then the activation-
// term scales of every staged slot, 16 columns per slot, written once per
// launch.
constexpr int kSfaCol = 64;
constexpr int kSfbCol = 96;
constexpr int kTcMaxSlots = (512 - kSfbCol) / 16;
static_assert(kTcStageBytes % 1024 == 0, "stages stay 1 KiB aligned");

struct TcCtrl {
  uint64_t full[kTcMaxStages];
  uint64_t empty[kTcMaxStages];
  uint64_t sfready[kTcMaxStages];
  uint64_t accfull[2];
  uint64_t accempty[2];
  uint64_t mma_done;
  uint32_t tmem;
  uint32_t xmax[8];
  int e1[8];
  int flag;
  int aborted;
};
constexpr int kTcCtrlBytes = (int(sizeof(TcCtrl)) + 127) / 128 * 128;

__host__ __device__ __forceinline__ int tc_n(int m) { return m <= 2 ? 16 : 32; }
__host__ __device__ __forceinline__ int tc_b_bytes(int slots, int n) {
  return slots * n * 128 + slots * 4 * n * 4;  // nibble tiles + scale words
}
__host__ __device__ __forceinline__ int tc_stages(int slots, int n) {
  const int room = kTcSmem - 1024 - kTcCtrlBytes - tc_b_bytes(slots, n);
  const int s = room / kTcStageBytes;
  return s > kTcMaxStages ? kTcMaxStages : s;
}
constexpr uint32_t kTmemCols = 512;
static_assert(kSfbCol + 16 * kTcMaxSlots <= int(kTmemCols), "tensor-memory budget");

__device__ __forceinline__ void bar_named(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, unsigned parity, volatile int *aborted,
                                              unsigned *status) {
  if (mbar_wait(bar, parity, aborted)) return true;
  if (!*aborted) {
    *aborted = 1;
    raise_status(status, kDevTimeout);
  }
  return false;
}

// One E2M1 pair (a byte) -> f16x2 (exact), the low nibble in the low half.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t r;
  asm("{ .reg .b8 b;\n"
      "  cvt.u8.u32 b, %1;\n"
      "  cvt.rn.f16x2.e2m1x2 %0, b; }"
      : "=r"(r)
      : "r"(byte));
  return r;
}

// 2^e as fp32 for e in [-126, 127]; 0 below.
__device__ __forceinline__ float pow2f(int e) {
  return e < -126 ? 0.0f : __int_as_float((e > 127 ? 127 + 127 : e + 127) << 23);
}

// Split one 16-column block of one token into kTerms NVFP4 terms; write the
// nibbles of term t into B row `row0 + t` of the slot's tile and its scale
// byte into the slot's scale words.
__device__ __forceinline__ void decompose_block(float (&r)[16], int e1, uint8_t *tile,
                                                uint8_t *sfw, int row0, int blk, int N) {
#pragma unroll 1
  for (int t = 0; t < kTerms; ++t) {
    const int e = e1 - 3 * t;
    if (e < -126) break;
    float am = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) am = fmaxf(am, fabsf(r[i]));
    if (am == 0.0f) break;
    const float tsc = __fmul_rn(__fmul_rn(am, 1.0f / 6.0f), pow2f(-e));
    const uint32_t code = f32x2_to_e4m3x2(0.0f, tsc) & 0xFFu;
    if (code == 0) continue;
    const float sd = __fmul_rn(f16_lo_to_f32(e4m3x2_to_f16x2(uint16_t(code))), pow2f(e));
    // any reciprocal will do: the residual below is formed from the nibble
    // actually chosen, so the terms still add up to x
    float inv;
    asm("rcp.approx.f32 %0, %1;" : "=f"(inv) : "f"(sd));
    uint32_t packed[2] = {0, 0};
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
      const uint32_t byte = f32x2_to_e2m1x2(__fmul_rn(r[i + 1], inv), __fmul_rn(r[i], inv));
      packed[i >> 3] |= byte << (4 * (i & 7));
      const uint32_t h2 = e2m1x2_to_f16x2(byte);
      const float d0 = f16_lo_to_f32(h2);
      const float d1 = f16_lo_to_f32(h2 >> 16);
      r[i] = __fsub_rn(r[i], __fmul_rn(d0, sd));
      r[i + 1] = __fsub_rn(r[i + 1], __fmul_rn(d1, sd));
    }
    const int row = row0 + t;
    const int chunk = blk >> 1, half = blk & 1;
    uint8_t *dst = tile + (row >> 3) * 1024 + (row & 7) * 128 + ((chunk ^ (row & 7)) << 4) + half * 8;
    *reinterpret_cast<uint2 *>(dst) = make_uint2(packed[0], packed[1]);
    sfw[((blk >> 2) * N + row) * 4 + (blk & 3)] = uint8_t(code);
  }
}

// Block idx of the staging (token-major, then slot, then block in slot):
// its 16 bf16 values as fp32 (zeros past k), folding |x| into mx[token].
__device__ __forceinline__ void load_block(const Proj &p, int idx, int nb, bool all_units,
                                           int uk_begin, int units, float (&v)[16],
                                           uint32_t (&mx)[kTcMaxTokens]) {
  const int tok = idx / nb, b = idx - tok * nb, s = b >> 4;
  const int uk = all_units ? s : (uk_begin + s) % units;
  const int kk = uk * kUnitK + (b & 15) * 16;
  uint4 q0 = make_uint4(0, 0, 0, 0), q1 = q0;
  if (kk < p.k) {
    const uint4 *src = reinterpret_cast<const uint4 *>(p.x + int64_t(tok) * p.k + kk);
    q0 = __ldg(src);
    q1 = __ldg(src + 1);
  }
  const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
  uint32_t am = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    v[2 * i] = bf16_lo(w[i]);
    v[2 * i + 1] = bf16_hi(w[i]);
    am = max(am, max(__float_as_uint(fabsf(v[2 * i])), __float_as_uint(fabsf(v[2 * i + 1]))));
  }
#pragma unroll
  for (int t = 0; t < kTcMaxTokens; ++t)
    if (t == tok) mx[t] = max(mx[t], am);
}

__device__ __forceinline__ void stage_block(float (&v)[16], int idx, int nb, const int *e1s,
                                            uint8_t *btile, uint8_t *bscale, int N, int k,
                                            bool all_units, int uk_begin, int units) {
  const int tok = idx / nb, b = idx - tok * nb, s = b >> 4;
  const int uk = all_units ? s : (uk_begin + s) % units;
  const int e1 = e1s[tok];
  if (uk * kUnitK + (b & 15) * 16 >= k || e1 == INT_MIN / 2) return;
  decompose_block(v, e1, btile + s * N * 128, bscale + s * 4 * N * 4, tok * kTerms, b & 15, N);
}

__global__ void __launch_bounds__(kTcThreads, 1)
    tc_gemv_kernel(const __grid_constant__ CUtensorMap tm_w,
                   const __grid_constant__ CUtensorMap tm_s, Proj p, const Run r) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = r.stages, m = r.m, units = p.units;
  const int N = tc_n(m);
  const int64_t grid = p.grid;
  const int64_t u_begin = range_begin(blockIdx.x, p.total, grid);
  const int64_t u_end = range_begin(blockIdx.x + 1, p.total, grid);
  const int64_t L = u_end - u_begin;
  const bool all_units = L >= units;
  const int uk_begin = int(u_begin % units);
  const int slots = x_slots(L, units);

  uint8_t *ring = base;
  uint8_t *btile = base + S * kTcStageBytes;                // [slots][N rows][128 B]
  uint8_t *bscale = btile + slots * N * 128;                // [slots][4 k-steps][N] words
  TcCtrl &ct = *reinterpret_cast<TcCtrl *>(bscale + slots * 4 * N * 4);
  volatile int *aborted = &ct.aborted;
  p.tm_w = &tm_w;
  p.tm_s = &tm_s;
  const uint32_t cols = kTmemCols;

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
    for (int t = 0; t < 8; ++t) ct.xmax[t] = 0;
    ct.aborted = 0;
    ct.flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    pdl_launch_dependents();
  }
  if (warp == kWarpMma) tcx::tmem_alloc(&ct.tmem, cols);
  tcx::fence_before_sync();
  __syncthreads();
  tcx::fence_after_sync();
  const uint32_t tmem = ct.tmem;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_w)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_s)) : "memory");
      RingPos pos;
      for (int64_t u = u_begin; u < u_end; ++u, pos.advance(S)) {
        const int st = pos.st;
        if (pos.wrapped && !wait_or_abort(&ct.empty[st], pos.phase ^ 1u, aborted, r.status)) break;
        if (*aborted) break;
        const int64_t rb = u / units;
        const int uk = int(u - rb * units);
        uint8_t *stage = ring + st * kTcStageBytes;
        mbar_expect_tx(&ct.full[st], kStageBytes);
        tma_load_2d(stage, p.tm_w, uk * kUnitCols, int(rb * kRB), &ct.full[st]);
        tma_load_2d(stage + kBoxOff, p.tm_s, uk * kKT * 128, int(rb * kRG), &ct.full[st]);
      }
      // no copy may still be landing when the CTA exits
      int never = 0;
      for (int64_t j = pos.count > S ? pos.count - S : 0; j < pos.count; ++j)
        mbar_wait(&ct.full[j % S], unsigned(j / S) & 1u, &never);
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issue
    bar_named(2, kStagers + 32);  // activation terms staged
    // The whole warp runs the loop (waits included) and stays converged;
    // one lane issues the copies, MMAs and commits.
    tcx::fence_after_sync();
    const bool leader = lane == 0;
    const uint32_t idesc = tcx::idesc_nvf4(N);
    const uint32_t ring_a = tcx::smem_addr(ring), b_a = tcx::smem_addr(btile);
    RingPos pos;
    int uses[2] = {0, 0};
    int buf = 0;
    bool ok = !*aborted;
    int64_t u = u_begin;
    while (u < u_end && ok) {
      const int64_t rb = u / units;
      const int uk0 = int(u - rb * units);
      const int uk1 = int(uk0 + (u_end - u) < units ? uk0 + (u_end - u) : units);
      if (uses[buf] > 0)
        ok = __all_sync(0xFFFFFFFFu, wait_or_abort(&ct.accempty[buf], unsigned(uses[buf] - 1) & 1u,
                                                    aborted, r.status));
      if (!ok) break;
      int slot = all_units ? uk0 : (uk0 >= uk_begin ? uk0 - uk_begin : uk0 + units - uk_begin);
      for (int uk = uk0; uk < uk1; ++uk, ++slot, pos.advance(S)) {
        const int st = pos.st;
        ok = __all_sync(0xFFFFFFFFu, wait_or_abort(&ct.full[st], pos.phase, aborted, r.status) &&
                                         wait_or_abort(&ct.sfready[st], pos.phase, aborted, r.status));
        if (!ok) break;
        tcx::fence_after_sync();
        const uint32_t stage_a = ring_a + st * kTcStageBytes;
        const uint32_t sfa = tmem + kSfaCol + uint32_t(pos.count & 1) * 16;
        const uint32_t sfb = tmem + kSfbCol + slot * 16;
        if (leader) {
#pragma unroll
          for (int j = 0; j < 4; ++j) tcx::cp_atom(sfa + 4 * j, tcx::desc_atom(stage_a + kSfaOff + 512 * j));
#pragma unroll
          for (int j = 0; j < 4; ++j)
            tcx::mma_nvf4(tmem + buf * kDCols, tcx::desc_k_sw128(stage_a + 32 * j),
                          tcx::desc_k_sw128(b_a + slot * N * 128 + 32 * j), idesc, sfa + 4 * j,
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
  } else {
    // ------------------------------------------------------------ warps 2..13
    const int tid = threadIdx.x - 64;  // 0..383
    pdl_wait();                         // x and the workspace may come from the previous kernel
    for (int i = tid; i < slots * 4 * N; i += kStagers) reinterpret_cast<uint32_t *>(bscale)[i] = 0;
    const int nb = slots * 16;  // 16-column blocks per token
    const int nblk = m * nb;
    // Up to two blocks per thread stay in registers between the passes;
    // larger stagings read x twice (the second time from L2).
    const bool in_regs = nblk <= 2 * kStagers;
    float v0[16], v1[16];
    uint32_t mx[kTcMaxTokens] = {0, 0, 0, 0, 0};
    if (in_regs) {
      if (tid < nblk) load_block(p, tid, nb, all_units, uk_begin, units, v0, mx);
      if (tid + kStagers < nblk) load_block(p, tid + kStagers, nb, all_units, uk_begin, units, v1, mx);
    } else {
      for (int idx = tid; idx < nblk; idx += kStagers) load_block(p, idx, nb, all_units, uk_begin, units, v0, mx);
    }
#pragma unroll
    for (int t = 0; t < kTcMaxTokens; ++t) {
      const uint32_t v = __reduce_max_sync(0xFFFFFFFFu, mx[t]);
      if (lane == 0 && v != 0 && t < m) atomicMax(&ct.xmax[t], v);
    }
    bar_named(1, kStagers);
    if (tid < m) {
      const uint32_t b = ct.xmax[tid];  // fp32 bits of the largest |x|
      // non-finite activations give no terms (the rows come out as 0)
      ct.e1[tid] = (b == 0 || b >= 0x7F800000u) ? INT_MIN / 2 : ilogbf(__uint_as_float(b)) - 6;
    }
    bar_named(1, kStagers);
    if (in_regs) {
      if (tid < nblk) stage_block(v0, tid, nb, ct.e1, btile, bscale, N, p.k, all_units, uk_begin, units);
      if (tid + kStagers < nblk)
        stage_block(v1, tid + kStagers, nb, ct.e1, btile, bscale, N, p.k, all_units, uk_begin, units);
    } else {
      for (int idx = tid; idx < nblk; idx += kStagers) {
        uint32_t unused[kTcMaxTokens] = {0, 0, 0, 0, 0};
        load_block(p, idx, nb, all_units, uk_begin, units, v0, unused);
        stage_block(v0, idx, nb, ct.e1, btile, bscale, N, p.k, all_units, uk_begin, units);
      }
    }
    tcx::fence_async_smem();
    bar_named(1, kStagers);
    if (warp < kWarpEpi) {
      // Activation-term scales of every slot into tensor memory, once: B
      // row n's word of k-step j at column kSfbCol + 16 slot + 4 j, lane
      // n % 32 of every quarter (one warp per quarter; rows n < N <= 32).
      const uint32_t lb = tmem + (uint32_t((warp & 3) * 32) << 16) + kSfbCol;
      const uint32_t *bw = reinterpret_cast<const uint32_t *>(bscale);
      for (int sl = 0; sl < slots; ++sl) {
        uint32_t v[16];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          v[4 * j] = lane < N ? bw[(sl * 4 + j) * N + lane] : 0u;
          v[4 * j + 1] = 0u;
          v[4 * j + 2] = 0u;
          v[4 * j + 3] = 0u;
        }
        tcx::st_x16(lb + 16 * sl, v);
      }
      tcx::wait_st();
    }
    tcx::fence_before_sync();
    bar_named(2, kStagers + 32);  // with the MMA warp
    const float gd = __ldg(p.g_dec);
    const int q = warp & 3;                       // tensor-memory lane quarter
    const uint32_t lane_base = tmem + (uint32_t(q * 32) << 16);

    if (warp < kWarpEpi) {
      // ---------------------------------------------------------- scales
      // Thread t of the four scale warps owns weight row t of the unit: it
      // gathers the row's 16 scale bytes from the tile layout and writes
      // them as its words of the four copy atoms (one per 64-column
      // k-step).  No barrier spans the warps.
      const int t = threadIdx.x - 64;  // 0..127
      const int rt = t >> 4, h = (t >> 3) & 1, g = t & 7;
      RingPos pos;
      for (int64_t u = u_begin; u < u_end && !*aborted; ++u, pos.advance(S)) {
        const int st = pos.st;
        const int64_t rb = u / units;
        const int uk = int(u - rb * units);
        if (!wait_or_abort(&ct.full[st], pos.phase, aborted, r.status)) break;
        uint8_t *stage = ring + st * kTcStageBytes;
        uint32_t wa[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int off = kBoxOff + rt * 256 + (j >> 1) * 128 + (4 * g + 2 * (j & 1)) * 4 + 2 * h;
          const uint32_t lo = *reinterpret_cast<const uint16_t *>(stage + off);
          const uint32_t hi = *reinterpret_cast<const uint16_t *>(stage + off + 4);
          wa[j] = lo | (hi << 16);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
          *reinterpret_cast<uint32_t *>(stage + kSfaOff + 512 * j + (t & 31) * 16 + (t >> 5) * 4) = wa[j];
        tcx::fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ct.sfready[st]);
      }
    } else if (warp < kWarpEpi + 4) {
      // ---------------------------------------------------------- epilogue
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
        float d[32];
        {
          uint32_t h0[16], h1[16];
          tcx::ld_x16(lane_base + buf * kDCols, h0);
          if (N > 16) tcx::ld_x16(lane_base + buf * kDCols + 16, h1);
          tcx::wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            d[i] = __uint_as_float(h0[i]);
            d[16 + i] = N > 16 ? __uint_as_float(h1[i]) : 0.0f;
          }
        }
        tcx::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ct.accempty[buf]);
        ++uses[buf];
        buf ^= 1;
        if (!ok) break;

        const bool complete = (uk0 == 0 && uk1 == units);
        const int64_t unit0 = rb * units;
        const int64_t own_lo = owner_of(unit0, p.total, grid);
        const int contrib = int(owner_of(unit0 + units - 1, p.total, grid) - own_lo + 1);
        const int jj = int(blockIdx.x - own_lo);
        const int64_t row = rb * kRB + row_local;
#pragma unroll
        for (int tok = 0; tok < kTcMaxTokens; ++tok) {
          if (tok >= m) break;
          const int e1 = ct.e1[tok];
          float v = 0.0f;
#pragma unroll
          for (int t = kTerms - 1; t >= 0; --t)
            v = __fadd_rn(v, __fmul_rn(d[tok * kTerms + t],
                                       e1 == INT_MIN / 2 ? 0.0f : pow2f(e1 - 3 * t)));
          if (complete) {
            if (row < p.n) p.y[int64_t(tok) * p.n + row] = f32_to_bf16_rn(__fmul_rn(v, gd));
          } else {
            r.partial[((rb * p.max_contrib + jj) * kRB + row_local) * 16 + tok] = v;
          }
        }
        if (!complete) {
          // Each epilogue warp publishes its 32 rows on its own: its stores,
          // then a gpu-scope fence and a ticket.  The warp that takes the
          // last of the row block's 4 * contrib tickets adds every
          // contributor's partials in contributor order and re-arms the
          // ticket.  No barrier spans warps, so a warp that gives up on a
          // wait can never leave the others waiting.
          __syncwarp();
          unsigned last = 0;
          if (lane == 0) {
            __threadfence();
            last = atomicAdd(&r.tickets[rb], 1u) == unsigned(4 * contrib - 1);
            __threadfence();
          }
          last = __shfl_sync(0xFFFFFFFFu, last, 0);
          if (last) {
            for (int idx = lane; idx < kRB * m; idx += 32) {
              const int rl = idx / m, token = idx - rl * m;
              const int64_t rr = rb * kRB + rl;
              if (rr >= p.n) continue;
              float s = 0.0f;
              for (int c = 0; c < contrib; ++c)
                s = __fadd_rn(s, __ldcg(r.partial + ((rb * p.max_contrib + c) * kRB + rl) * 16 + token));
              p.y[int64_t(token) * p.n + rr] = f32_to_bf16_rn(__fmul_rn(s, gd));
            }
            __syncwarp();
            if (lane == 0) r.tickets[rb] = 0;
          }
        }
        u += uk1 - uk0;
      }
    }  // staging-only warps 10..13 have nothing more to do
  }
  tcx::fence_before_sync();
  __syncthreads();
  if (warp == kWarpMma) {
    tcx::fence_after_sync();
    tcx::tmem_dealloc(tmem, cols);
  }
}

bool g_attr_done[64];
std::mutex g_attr_mu;

cudaError_t set_tc_attr(int device) {
  std::lock_guard<std::mutex> lock(g_attr_mu);
  if (device >= 0 && device < 64 && g_attr_done[device]) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(tc_gemv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem);
  if (e == cudaSuccess && device >= 0 && device < 64) g_attr_done[device] = true;
  return e;
}

}  // namespace

// The stream-K plan of the tensor-core kernel: one CTA per SM.
GemvPlan plan_gemv_tc(int n, int k, const DeviceInfo &dev) {
  GemvPlan p;
  p.row_blocks = ceil_div(n, kRB);
  p.k_tiles = ceil_div(k, kTileCols);
  p.units = ceil_div(p.k_tiles, kKT);
  p.total = p.row_blocks * p.units;
  int64_t g = dev.sms;
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

// The tensor-core kernel serves a shape when the activation terms of five
// tokens (N = 32) for the longest CTA range fit next to a ring of at least
// kTcMinStages stages.  Deciding with five tokens whatever m is keeps every
// token count of 1..5 on the same kernel for a given shape.
bool tc_eligible(int n, int k, int m, const DeviceInfo &dev) {
  if (m < 1 || m > kTcMaxTokens) return false;
  const GemvPlan p = plan_gemv_tc(n, k, dev);
  const int64_t longest = ceil_div(p.total, p.grid);
  const int slots = x_slots(longest, int(p.units));
  return slots <= kTcMaxSlots && tc_stages(slots, 32) >= kTcMinStages;
}

size_t gemv_tc_workspace_bytes(int n, int k, const DeviceInfo &dev) {
  const GemvPlan p = plan_gemv_tc(n, k, dev);
  return kRestOffset + size_t(p.row_blocks) * p.max_contrib * kRB * 16 * sizeof(float);
}

cudaError_t launch_gemv_tc(const aq_nvfp4_weight &w, const uint16_t *x, int m, uint16_t *y,
                           void *ws, bool pdl, const DeviceInfo &dev, cudaStream_t st) {
  const GemvPlan plan = plan_gemv_tc(w.n, w.k, dev);
  CUtensorMap tm_w, tm_s;
  if (!encode_maps(w, &tm_w, &tm_s, 8)) return cudaErrorInvalidValue;
  const int64_t longest = ceil_div(plan.total, plan.grid);
  const int slots = x_slots(longest, int(plan.units));
  Run r{};
  uint8_t *wsb = static_cast<uint8_t *>(ws);
  r.tickets = reinterpret_cast<uint32_t *>(wsb);
  r.partial = reinterpret_cast<float *>(wsb + kRestOffset);
  r.status = dev.status;
  r.m = m;
  r.stages = tc_stages(slots, tc_n(m));
  r.x_cap = 0;
  if (r.stages < kTcMinStages) return cudaErrorInvalidConfiguration;

  Proj p{};
  p.tm_w = nullptr;  // set from the kernel's own parameters
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

  cudaError_t e = set_tc_attr(dev.ordinal);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(plan.grid);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = kTcSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, tc_gemv_kernel, tm_w, tm_s, p, r);
}

}  // namespace aq
