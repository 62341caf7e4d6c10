// gemv.cu -- one block-scaled NVFP4 GEMV launch (aq_gemv_nvfp4, and the
// per-projection launches of aq_decode_step_weights):
// y[t, i] = bf16( g_dec * sum_j sd[i, j] * sum_{k in block j} x[t, k] * e2m1(q[i, k]) )
// (Weightless docs, "GPU and cache acceleration", "Future work": a GEMV
// that dequantises the 4-bit weights in registers and streams them at full
// HBM bandwidth; AttnQuant docs, "Throughput", per-kernel MLP analysis: a
// skinny `down` projection needs split-K to fill the machine.)
//
// Design for sm_103a (device code in gemv_core.cuh):
//  * Work unit = a row block of 128 rows by 2 k-tiles of 128 columns: one
//    16 KiB TMA box of packed nibbles (128-byte swizzle) plus one 2 KiB box
//    of scale words.  Tall boxes keep HBM efficient even though each CTA
//    streams its own contiguous range of units.
//  * Units are laid out row-block-major and cut into equal contiguous
//    ranges, one per persistent CTA (stream-K), at most two CTAs per SM, so
//    every CTA streams the same number of bytes whatever the shape; the
//    grid is the smallest that keeps the longest range as short as two
//    CTAs per SM allow (plan_gemv), so the ranges are equal to within one
//    unit and a split row block has as few contributors as possible.
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
//  * One token (m = 1): the MMA's n dimension carries the tile's eight
//    16-element blocks instead of tokens (block-diagonal activation
//    operand), so D holds unscaled block sums and each block scale is one
//    fp32 multiply-add on them instead of an f16 multiply per weight pair
//    (unit_mma_bd in gemv_core.cuh).
//  * Each CTA stages only the activation columns its units touch, as f16
//    after an exact power-of-two rescale that puts each token's largest |x|
//    over those columns in [2^14, 2^15); bf16 values keep all 8 significand
//    bits in f16 there (only values 2^29 below the maximum round), and the
//    partial sums are scaled back exactly.
//  * Split-K across CTAs is deterministic: contributor 0 of a split row
//    block (the CTA whose range ends in it) adds the others' fp32 partials
//    in contributor order and writes bf16 y (finish_rows in gemv_core.cuh).
//    The partition depends only on (n, k) and the SM count, never on m, so
//    for m >= 2 each token's result is independent of the rest of the batch.
//  * The weight copies carry an evict-first L2 policy: the stream is read
//    once per step and leaves L2 to the activations, partials and the next
//    projection's prefetched units.
//  * Every mbarrier wait is bounded; a wait that gives up records
//    AQ_ERR_TIMEOUT in the device status word and the CTA winds down.
#include <cudaTypedefs.h>

#include <mutex>
#include <unordered_map>

#include "gemv_core.cuh"

namespace aq {

using namespace core;

namespace {

template <int NT, int EPI, bool BD, int RG>
__global__ void __launch_bounds__(Geo<RG>::kThreads, Geo<RG>::kCtasPerSm)
    gemv_kernel(const __grid_constant__ CUtensorMap tm_w,
                const __grid_constant__ CUtensorMap tm_s,
                const __grid_constant__ CUtensorMap tm_nw,
                const __grid_constant__ CUtensorMap tm_ns, Proj p, const Run r) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const SmemView sv = carve<RG>(smem_raw, r.stages);
  Ctrl &ct = *sv.ct;
  volatile int *aborted = &ct.aborted;
  p.tm_w = &tm_w;
  p.tm_s = &tm_s;
  p.nx_w = &tm_nw;
  p.nx_s = &tm_ns;
  if (threadIdx.x == 0) {
    init_ring<RG>(ct, r.stages);
    pdl_launch_dependents();
  }
  __syncthreads();
  RingPos pos;
  if ((threadIdx.x >> 5) == Geo<RG>::kW) {  // producer warp
    if ((threadIdx.x & 31) == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_w)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_s)) : "memory");
      if (produce<RG>(p, sv.base, ct, r.stages, pos, aborted, r.status)) prefetch_next<RG>(p);
      drain(ct, r.stages, pos.count);
    }
    return;
  }
  prefetch_x_l2<RG>(p, r.m);
  // x and the workspace may come from the previous kernel: consume() waits
  // for it once its own index work is done
  Dep dep;
  dep.kind = kDepPdl;
  consume<NT, EPI, BD, RG>(p, r, sv.base, ct, sv.xs, pos, aborted, dep);
}

// The kernels' bounded ring wait run against an mbarrier that nothing
// completes, with a short poll limit: it gives up, records AQ_ERR_TIMEOUT
// in the status word and returns, exactly as a CTA whose copies never
// arrive would.
__global__ void selftest_wait_kernel(unsigned polls, unsigned *status) {
  __shared__ uint64_t bar;
  __shared__ int aborted;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    aborted = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait_n(&bar, 0, &aborted, polls)) raise_status(status, kDevTimeout);
}

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

template <int NT, int EPI, bool BD, int RG>
cudaError_t set_smem_attr(int device) {
  static bool done[64] = {};
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (device >= 0 && device < 64 && done[device]) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(gemv_kernel<NT, EPI, BD, RG>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Geo<RG>::kSmemBudget);
  if (e == cudaSuccess && device >= 0 && device < 64) done[device] = true;
  return e;
}

template <int NT, int EPI, bool BD, int RG>
cudaError_t launch_form(const cudaLaunchConfig_t &cfg, const CUtensorMap &tm_w,
                        const CUtensorMap &tm_s, const CUtensorMap &tm_nw, const CUtensorMap &tm_ns,
                        const Proj &p, const Run &r, int device) {
  cudaError_t e = set_smem_attr<NT, EPI, BD, RG>(device);
  if (e != cudaSuccess) return e;
  return cudaLaunchKernelEx(&cfg, gemv_kernel<NT, EPI, BD, RG>, tm_w, tm_s, tm_nw, tm_ns, p, r);
}

// The instantiation for m tokens and the epilogue kind: the block-diagonal
// form for one token, one n8 block of tokens up to 8, two up to 16.
template <int EPI, int RG>
cudaError_t launch_epi(const cudaLaunchConfig_t &cfg, int m, const CUtensorMap &tm_w,
                       const CUtensorMap &tm_s, const CUtensorMap &tm_nw, const CUtensorMap &tm_ns,
                       const Proj &p, const Run &r, int device) {
  if (m == 1) return launch_form<1, EPI, true, RG>(cfg, tm_w, tm_s, tm_nw, tm_ns, p, r, device);
  if (m <= 8) return launch_form<1, EPI, false, RG>(cfg, tm_w, tm_s, tm_nw, tm_ns, p, r, device);
  return launch_form<2, EPI, false, RG>(cfg, tm_w, tm_s, tm_nw, tm_ns, p, r, device);
}
template <int RG>
cudaError_t launch_any(const cudaLaunchConfig_t &cfg, int epi, int m, const CUtensorMap &tm_w,
                       const CUtensorMap &tm_s, const CUtensorMap &tm_nw, const CUtensorMap &tm_ns,
                       const Proj &p, const Run &r, int device) {
  switch (epi) {
    case kEpiLowRank: return launch_epi<kEpiLowRank, RG>(cfg, m, tm_w, tm_s, tm_nw, tm_ns, p, r, device);
    case kEpiGlu: return launch_epi<kEpiGlu, RG>(cfg, m, tm_w, tm_s, tm_nw, tm_ns, p, r, device);
    case kEpiSegments: return launch_epi<kEpiSegments, RG>(cfg, m, tm_w, tm_s, tm_nw, tm_ns, p, r, device);
    default: return launch_epi<kEpiPlain, RG>(cfg, m, tm_w, tm_s, tm_nw, tm_ns, p, r, device);
  }
}

// Activation buffer (f16) of a single-projection launch: everything the
// longest CTA range touches when that fits in 48 KiB, else one chunk.
int x_cap_for(const GemvPlan &p, int m) {
  const int64_t longest = ceil_div(p.total, p.grid);
  const int full = m * x_stride_full(x_slots(longest, int(p.units)));
  return full * 2 <= 48 * 1024 ? full : m * x_stride_chunk(m);
}

}  // namespace

namespace core {

size_t smem_bytes(int stages, int x_cap_halves, int rg) {
  const int stage = rg == 16 ? Geo<16>::kStageBytes : Geo<8>::kStageBytes;
  return 1024 + size_t(stages) * stage + kCtrlBytes + size_t(x_cap_halves) * 2;
}

int stages_for(int x_cap_halves, int rg) {
  const int budget = rg == 16 ? Geo<16>::kSmemBudget : Geo<8>::kSmemBudget;
  const int stage = rg == 16 ? Geo<16>::kStageBytes : Geo<8>::kStageBytes;
  const int most = rg == 16 ? Geo<16>::kMaxStages : Geo<8>::kMaxStages;
  const int64_t room = int64_t(budget) - 1024 - kCtrlBytes - int64_t(x_cap_halves) * 2;
  const int64_t st = room / stage;
  return int(st > most ? most : (st < 0 ? 0 : st));
}

// Boxes of 16 rg rows of packed nibbles (128 bytes wide) and rg rows of
// scale tiles (256 bytes: the unit's two 128-column tiles).
bool encode_maps(const aq_nvfp4_weight &w, CUtensorMap *tm_w, CUtensorMap *tm_s, int rg) {
  if (!encoder()) return false;
  if (!cached_map(tm_w, w.packed, uint64_t(w.k) / 2, uint64_t(w.n), kUnitCols, 16 * rg, true))
    return false;
  const uint64_t srow = uint64_t(ceil_div(w.k, kTileCols)) * 128;
  return cached_map(tm_s, w.scales, srow, uint64_t(ceil_div(w.n, kTileRows)), kKT * 128, rg,
                    false);
}

// bf16 weight [n, k] as a byte matrix [n rows, 2k bytes]: boxes of 128 B x
// 128 rows with the 128-byte swizzle, exactly like the NVFP4 nibble boxes.
bool encode_bf16_map(const uint16_t *w, int n, int k, CUtensorMap *tm) {
  if (!encoder()) return false;
  return cached_map(tm, w, uint64_t(k) * 2, uint64_t(n), kUnitCols, kRB, true);
}

// bf16 matrix [n, k] as bytes [n rows, 2k bytes]: boxes of 128 B (64
// values) x box_rows rows with the 128-byte swizzle.
bool encode_bf16_rows_map(const uint16_t *w, int n, int k, int box_rows, CUtensorMap *tm) {
  if (!encoder()) return false;
  return cached_map(tm, w, uint64_t(k) * 2, uint64_t(n), 128, uint32_t(box_rows), true);
}

// A byte array of `bytes` bytes as a 1-D tensor, copied in boxes of `box`
// bytes; bytes past the end read as zero.
bool encode_bytes_1d(const void *base, uint64_t bytes, uint32_t box, CUtensorMap *tm) {
  if (!encoder()) return false;
  const cuuint64_t dims[1] = {bytes};
  const cuuint64_t strides[1] = {bytes};
  const cuuint32_t boxd[1] = {box};
  const cuuint32_t estr[1] = {1};
  return g_encode(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, const_cast<void *>(base), dims, strides,
                  boxd, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace core

bool encode_act_maps(const uint8_t *xq, const uint8_t *xs, int m, int k, int scale_pitch,
                     int n_box, CUtensorMap *tm_x, CUtensorMap *tm_xs) {
  if (!encoder()) return false;
  // k/16 scale columns of a row; the pitch pads the row to 16 bytes
  const cuuint64_t dims[2] = {cuuint64_t(k / 16), cuuint64_t(m)};
  const cuuint64_t strides[1] = {cuuint64_t(scale_pitch)};
  const cuuint32_t box[2] = {16, cuuint32_t(n_box)};
  const cuuint32_t estr[2] = {1, 1};
  return cached_map(tm_x, xq, uint64_t(k) / 2, uint64_t(m), kUnitCols, uint32_t(n_box), true) &&
         g_encode(tm_xs, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(xs), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

GemvPlan plan_gemv(int n, int k, const DeviceInfo &dev, int rg) {
  GemvPlan p;
  p.row_blocks = ceil_div(n, 16 * rg);
  p.k_tiles = ceil_div(k, kTileCols);
  p.units = ceil_div(p.k_tiles, kKT);
  p.total = p.row_blocks * p.units;
  // Up to two persistent CTAs per SM (the shared-memory budget of each CTA
  // is set so both are resident); tiny projections get one unit per CTA.
  // Of the grids whose longest range is as short as two CTAs per SM allow,
  // the smallest: every range then has that length (or one unit less), so
  // no CTA idles while others finish an extra unit, and fewer CTAs share
  // each split row block.  A range is never shorter than an eighth of a
  // row block's units, so at most about eight CTAs share one row block:
  // small projections with long rows would otherwise spread a row block over
  // dozens of one-unit CTAs and spend their time in the split-K reduction
  // (measured on the 1B down [1152, 6912]: 9.1 us per call with 27
  // contributors, 6.4 us with 7; the ~31B shapes' ranges are longer than
  // that already).  The grid depends only on (n, k) and the SM count, never
  // on m.
  int64_t g = int64_t(dev.sms) * (rg == 8 ? Geo<8>::kCtasPerSm : Geo<16>::kCtasPerSm);
  if (g > p.total) g = p.total;
  if (g < 1) g = 1;
  int64_t longest = (p.total + g - 1) / g;
  if (longest < (p.units + 7) / 8) longest = (p.units + 7) / 8;
  g = (p.total + longest - 1) / longest;
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

// The register-decode kernel's own need: tickets, the zero region, and
// fp32 partials [row_blocks][max_contrib][kRB][16 tokens].
size_t gemv_regdecode_workspace_bytes(int n, int k, const DeviceInfo &dev) {
  const GemvPlan p = plan_gemv(n, k, dev, kGemvRG);
  return kRestOffset + size_t(p.row_blocks) * p.max_contrib * (16 * kGemvRG) * 16 * sizeof(float);
}

// Enough for either kernel, so one workspace serves every token count.
size_t gemv_workspace_bytes(int n, int k, const DeviceInfo &dev) {
  const size_t reg = gemv_regdecode_workspace_bytes(n, k, dev);
  const size_t tc = gemv_tc_workspace_bytes(n, k, dev);
  return reg > tc ? reg : tc;
}

// The GEMV for m tokens.  Both kernels meet the same tolerance; the
// register-decode kernel is the faster one on the measured decode shapes
// today, so it serves every m unless the tcgen05 kernel is asked for.
constexpr bool kAutoPrefersTc = false;
cudaError_t launch_gemv(const aq_nvfp4_weight &w, const uint16_t *x, int m, uint16_t *y,
                        void *ws, bool pdl, const DeviceInfo &dev, cudaStream_t st,
                        const aq_nvfp4_weight *next) {
  if (kAutoPrefersTc && tc_eligible(w.n, w.k, m, dev))
    return launch_gemv_tc(w, x, m, y, ws, pdl, dev, st);
  return launch_gemv_regdecode(w, x, m, y, ws, pdl, dev, st, next);
}

cudaError_t launch_gemv_regdecode(const aq_nvfp4_weight &w, const uint16_t *x, int m,
                                  uint16_t *y, void *ws, bool pdl, const DeviceInfo &dev,
                                  cudaStream_t st, const aq_nvfp4_weight *next,
                                  const LowRank *lr, bool glu, int nseg,
                                  const int32_t *seg_end) {
  constexpr int RG = kGemvRG;
  const GemvPlan plan = plan_gemv(w.n, w.k, dev, RG);
  CUtensorMap tm_w, tm_s, tm_nw, tm_ns;
  if (!encode_maps(w, &tm_w, &tm_s, RG)) return cudaErrorInvalidValue;

  Run r{};
  uint8_t *wsb = static_cast<uint8_t *>(ws);
  r.tickets = reinterpret_cast<uint32_t *>(wsb);
  r.zero = reinterpret_cast<uint32_t *>(wsb + kTicketBytes);
  r.partial = reinterpret_cast<float *>(wsb + kRestOffset);
  r.status = dev.status;
  r.m = m;
  r.x_cap = x_cap_for(plan, m);
  r.stages = stages_for(r.x_cap, RG);
  if (r.stages < kMinStages) return cudaErrorInvalidConfiguration;

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
  p.direct = direct_partials_fit<RG>(plan.row_blocks, plan.max_contrib, m) ? 1 : 0;
  p.scale_box = 1;
  if (nseg > 0) {
    p.nseg = nseg;
    for (int i = 0; i < nseg; ++i) p.seg_end[i] = seg_end[i];
  }
  if (lr) {
    p.lr_s = lr->s;
    p.lr_u = lr->u;
    p.lr_t = lr->t;
    p.lr_r = lr->r;
  }
  p.nx_w = p.nx_s = nullptr;
  p.nx_total = 0;
  p.nx_units = p.nx_grid = p.nx_pf = 0;
  if (next) {
    if (!encode_maps(*next, &tm_nw, &tm_ns, RG)) return cudaErrorInvalidValue;
    const GemvPlan np = plan_gemv(next->n, next->k, dev, RG);
    p.nx_total = np.total;
    p.nx_units = int(np.units);
    p.nx_grid = np.grid;
    p.nx_pf = kPrefetchUnits;
  } else {
    tm_nw = tm_w;  // unused
    tm_ns = tm_s;
  }

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(plan.grid);
  cfg.blockDim = dim3(Geo<RG>::kThreads);
  cfg.dynamicSmemBytes = smem_bytes(r.stages, r.x_cap, RG);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  const int epi = glu ? kEpiGlu : lr ? kEpiLowRank : nseg > 0 ? kEpiSegments : kEpiPlain;
  return launch_any<RG>(cfg, epi, m, tm_w, tm_s, tm_nw, tm_ns, p, r, dev.ordinal);
}

cudaError_t launch_selftest_wait(unsigned polls, const DeviceInfo &dev, cudaStream_t st) {
  selftest_wait_kernel<<<1, 32, 0, st>>>(polls, dev.status);
  return cudaGetLastError();
}

// The same launch with both tensor maps encoded on the stack for this call
// only (no map cache, so nothing is allocated on the host either) and
// without programmatic dependent launch; ws is the caller's scratch.
cudaError_t launch_gemv_uncached(const aq_nvfp4_weight &w, const uint16_t *x, int m,
                                 uint16_t *y, void *ws, const DeviceInfo &dev,
                                 cudaStream_t st) {
  constexpr int RG = kGemvRG;
  const GemvPlan plan = plan_gemv(w.n, w.k, dev, RG);
  CUtensorMap tm_w, tm_s;
  if (!encoder()) return cudaErrorInvalidValue;
  if (!make_map(&tm_w, w.packed, uint64_t(w.k) / 2, uint64_t(w.n), kUnitCols, 16 * RG, true))
    return cudaErrorInvalidValue;
  const uint64_t srow = uint64_t(ceil_div(w.k, kTileCols)) * 128;
  if (!make_map(&tm_s, w.scales, srow, uint64_t(ceil_div(w.n, kTileRows)), kKT * 128, RG, false))
    return cudaErrorInvalidValue;

  Run r{};
  uint8_t *wsb = static_cast<uint8_t *>(ws);
  r.tickets = reinterpret_cast<uint32_t *>(wsb);
  r.zero = reinterpret_cast<uint32_t *>(wsb + kTicketBytes);
  r.partial = reinterpret_cast<float *>(wsb + kRestOffset);
  r.status = dev.status;
  r.m = m;
  r.x_cap = x_cap_for(plan, m);
  r.stages = stages_for(r.x_cap, RG);
  if (r.stages < kMinStages) return cudaErrorInvalidConfiguration;

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
  p.direct = direct_partials_fit<RG>(plan.row_blocks, plan.max_contrib, m) ? 1 : 0;
  p.scale_box = 1;
  p.nx_w = p.nx_s = nullptr;  // no prefetch of a next projection
  p.nx_total = 0;
  p.nx_units = p.nx_grid = p.nx_pf = 0;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(plan.grid);
  cfg.blockDim = dim3(Geo<RG>::kThreads);
  cfg.dynamicSmemBytes = smem_bytes(r.stages, r.x_cap, RG);
  cfg.stream = st;
  return launch_any<RG>(cfg, kEpiPlain, m, tm_w, tm_s, tm_w, tm_s, p, r, dev.ordinal);
}

}  // namespace aq
