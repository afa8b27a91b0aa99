// gemm.cu -- block-scaled A4W4 (tcgen05 kind::mxf4) and FP8 PTPC A8W8
// (tcgen05 kind::f8f6f4) GEMMs for sm_103a.
//
// What is computed (page "Kimi-K3 DSpark O-Proj-only MXFP4", section "Exact
// quantization coverage": "dynamic MXFP4 activations with A4W4 dispatch";
// page "Kimi-K3-DSpark-FP8-PTPC", section "Phase 1 FP8 PTPC Quantization"):
//   A4W4: y[m][n] = sum_g 2^(ea[m,g]-127) 2^(ew[n,g]-127) sum_{k in g} a[m,k] w[n,k]
//   PTPC: y[m][n] = (sum_k a[m,k] w[n,k] * sa[m]) * sw[n]
// with fp32 accumulation in TMEM and a bf16 (or fp32) epilogue.
//
// One kernel template serves both variants the dispatcher chooses from:
//   full tile  (swap = 0): MMA-A = 128 token rows, MMA-B = 256 weight rows,
//              each CTA owns whole tiles and all of K (persistent, strided;
//              in bands of token tiles when the operands exceed L2).  With
//              CTA pairs (CG = 2, clusters of two) a tile is 256 tokens x 256
//              channels: each CTA brings 128 token rows and one 128-row half
//              of the weight tile, and the even CTA issues 2-SM MMAs
//              (cta_group::2) over both -- 256 instead of 384 operand rows
//              per 128 x 256 share of output, and stages half as big.
//   split-K    (swap = 1): MMA-A = 128 weight rows, MMA-B = the (padded)
//              token rows; the (tile, K-block) units are cut evenly over the
//              CTAs (stream-K); a CTA that ends a tile part-way writes an
//              fp32 partial tile, and the reduce kernel launched right after
//              the GEMM sums the partials of each tile in slot order -- a
//              fixed order, so results are deterministic.
//
// Warp roles (192 threads): warp 0 = producer (bulk copies of operand tiles
// and weight panels, tensor-map boxes for row-major operands, scale tiles);
// warp 1 = TMEM allocator and the single MMA-issuing thread; warps 2-5 =
// epilogue (tcgen05.ld of their 32-lane quarter; for A4W4 they also move each
// stage's scale factors into TMEM, and in the full tile store y by TMA).  All
// hand-offs are mbarriers; every wait is bounded.
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <cuda_runtime.h>

#include "kernels.h"
#include "ptx.cuh"

namespace mxg {
namespace {

constexpr int kTileA = 128;      // MMA M: rows of the MMA-A operand per tile
constexpr int kRowBytes = 128;   // K bytes per row per stage (one 128-byte swizzle row)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCol = 0;    // accumulator: columns [0, BN)
// Scale factors: every pipeline stage has its own TMEM columns from kSfCol on
// (A: 2 K-tiles x 4 columns, then B: 2 K-tiles x row blocks x 4 columns), so
// the copy for the next stage never waits for the MMAs still reading the
// scales of this one.
constexpr uint32_t kSfCol = 256;
// Dynamic shared memory of a CTA: the mbarriers and a few words in the first
// 1024 bytes, then the 1024-byte-aligned pipeline stages and the epilogue's
// staging boxes, up to the 227 KB a CTA may have.
constexpr int kSmemMax = 227 * 1024;
constexpr int kSmemHead = 1024;

// KS: 128-byte K columns per pipeline stage (one column = 256 E2M1 or 128
// E4M3 values of every row).  Two columns per stage halve the number of bulk
// copies per byte, which is what bounds the weight-streaming (split-K) rate.
template <int KIND, int BN, int KS, int CG = 1>
struct Cfg {
  static constexpr int kSfBlocksB = BN >= 128 ? BN / 128 : 1;
  static constexpr int kBRows = BN / CG;  // MMA-B rows this CTA holds (the MMA's N is BN)
  static constexpr int kAColBytes = kTileA * kRowBytes;  // one column of the A operand
  static constexpr int kBColBytes = kBRows * kRowBytes;
  static constexpr int kABytes = kAColBytes * KS;
  static constexpr int kBBytes = kBColBytes * KS;
  static constexpr int kSfaBytes = KIND == 0 ? 1024 * KS : 0;  // 2 scale atoms per column
  // the scales of all BN rows of B (a CTA pair: each CTA holds both halves'
  // scales, since each CTA's MMAs cover all BN columns of its output rows)
  static constexpr int kSfbBytes = KIND == 0 ? 1024 * KS * kSfBlocksB : 0;
  static constexpr int kStageBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes;
  // one column of a 256-row weight panel: codes, then (E2M1) the 2 x 2 scale atoms
  static constexpr int kPanelBytes = 256 * kRowBytes + (KIND == 0 ? 2048 : 0);
  // Epilogue warps: one set of four (one per TMEM lane quarter) for
  // split-K, or, for the full tile, two sets that read out half of the
  // accumulator's columns each (a short-K FP8 tile's read-out outlasts its
  // MMAs) and, for A4W4, feed alternate stages' scale factors (a stage's
  // feed waits for its data and for its TMEM stores, so one set alone paces
  // the MMAs).  Full tile: per epilogue warp one (two sets) or two 32 x 32
  // bf16 staging boxes for the TMA stores of y.
  static constexpr int kEpiSets = KS == 1 ? 2 : 1;
  static constexpr int kThreads = 64 + 128 * kEpiSets;
  static constexpr int kEpiBufs = kEpiSets == 2 ? 1 : 2;
  static constexpr int kEpiBytes = KS == 1 ? 4 * kEpiSets * kEpiBufs * 2048 : 0;
  static constexpr int kStagesRaw = (kSmemMax - kSmemHead - kEpiBytes) / kStageBytes;
  static constexpr int kStages = kStagesRaw > 12 ? 12 : kStagesRaw;
  static constexpr int kBarBytes = 8 * (4 * kStages + 6) + 8;  // mbarriers, TMEM base, abort flag
  static constexpr size_t kSmem = (size_t)kSmemHead + (size_t)kStages * kStageBytes + kEpiBytes;
  // TMEM accumulators: two where the columns allow (FP8: all 512; A4W4: the
  // 256 below the scale factors), so that the epilogue of one item runs
  // beside the MMAs of the next
  static constexpr int kAccBufs = 2 * BN <= (KIND == 0 ? (int)kSfCol : (int)kTmemCols) ? 2 : 1;
  static constexpr int kChunk = BN >= 32 ? 32 : 16;  // epilogue TMEM columns per load
  static constexpr int kSteps = 4 * KS;              // MMAs (K = 64 / 32) per stage
  static constexpr uint32_t kSfColsA = 8u * KS;      // 4 TMEM columns per scale atom
  static constexpr uint32_t kSfColsPerStage = kSfColsA + 8u * KS * (uint32_t)kSfBlocksB;
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N");
  static_assert(CG == 1 || (KS == 1 && BN == 256), "CTA pairs: full tile only");
  static_assert(kStages >= 2, "pipeline depth");
  static_assert(kBarBytes <= kSmemHead && kSmem <= (size_t)kSmemMax, "shared memory");
  static_assert(KIND != 0 || kSfCol + kStages * kSfColsPerStage <= kTmemCols, "TMEM budget");
  static_assert(kSfColsPerStage % 8 == 0, "scale columns of a stage: whole 8-column stores");
};

struct Item {
  int t, ta, tb, kb0, kb1, seg, nseg;
  // grouped GEMM: the expert of token tile ta, its first token tile, its
  // first token row and its number of token rows
  int e, tile0, row0, rows;
};

// Grouped GEMM: the expert whose token tiles include global token tile ta
// (the largest e with tile_off[e] <= ta), by binary search over E + 1 offsets.
__device__ __forceinline__ int group_of_tile(const int *tile_off, int E, int ta) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(tile_off + mid) <= ta) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// CTA that owns stream-K unit u when U units are cut into G equal ranges
// [c*U/G, (c+1)*U/G): the largest c with c*U < (u+1)*G.  The host checks
// that (U+1)*G fits in 32 bits (64-bit division costs ~1 us per item on
// the single producer thread).
__device__ __forceinline__ uint32_t owner_of(uint32_t u, uint32_t U, uint32_t G) {
  return ((u + 1) * G - 1) / U;
}

// The first item cursor of this CTA (CG = 2: of its pair; both CTAs of a
// pair walk the same items).
template <int CG>
__device__ __forceinline__ uint32_t first_cursor(const GemmParams &p) {
  return p.splitk ? (blockIdx.x * (uint32_t)p.units) / gridDim.x : blockIdx.x / (uint32_t)CG;
}

// The work items of this CTA, in order; every role walks the same list.
template <int CG>
__device__ __forceinline__ bool next_item(const GemmParams &p, uint32_t &cur, Item &it) {
  const uint32_t G = gridDim.x / (uint32_t)CG;
  it.e = 0;
  if (p.groups) {
    // grouped (full tile): item i = (weight tile i / tilesA, token tile i %
    // tilesA), token tiles fastest so that the CTAs running at one time
    // share a weight tile of one expert; tilesA is the host's bound on the
    // token tiles, the items past the groups' last tile are skipped
    const int valid = __ldg(p.g_tile_off + p.groups);
    const uint32_t total = (uint32_t)(p.tilesA * p.tilesB);
    while (cur < total && (int)(cur % (uint32_t)p.tilesA) >= valid) cur += G;
    if (cur >= total) return false;
    it.t = (int)cur;
    it.ta = (int)(cur % (uint32_t)p.tilesA);
    it.tb = (int)(cur / (uint32_t)p.tilesA);
    it.kb0 = 0;
    it.kb1 = p.kblocks;
    it.seg = 0;
    it.nseg = 1;
    cur += G;
    it.e = group_of_tile(p.g_tile_off, p.groups, it.ta);
    it.tile0 = __ldg(p.g_tile_off + it.e);
    it.row0 = __ldg(p.g_row_off + it.e);
    it.rows = __ldg(p.g_row_off + it.e + 1) - it.row0;
    return true;
  }
  if (!p.splitk) {
    // full tile; a CTA pair's item is a pair of token tiles (the CTA of rank
    // r takes token tile 2 * pair + r; past the last token tile it loads no
    // activations and stores nothing)
    const uint32_t tA = CG == 2 ? ((uint32_t)p.tilesA + 1u) >> 1 : (uint32_t)p.tilesA;
    const uint32_t tB = (uint32_t)p.tilesB;
    if (cur >= tA * tB) return false;
    it.t = (int)cur;
    it.kb0 = 0;
    it.kb1 = p.kblocks;
    it.seg = 0;
    it.nseg = 1;
    const uint32_t t = cur;
    cur += G;
    if (p.raster_group > 0) {
      // bands of raster_group MMA-A (token) tiles: within a band the token
      // tile varies fastest, so the CTAs running at one time share a few
      // weight tiles and the band's activations stay in L2 -- the weights
      // are read from HBM once per band, not once per token tile
      const uint32_t g = max(1u, (uint32_t)p.raster_group / (uint32_t)CG);
      const uint32_t band = g * tB;
      const uint32_t b0 = t / band, r = t - b0 * band;
      const uint32_t ta0 = b0 * g;
      const uint32_t gsz = min(g, tA - ta0);
      it.ta = (int)(ta0 + r % gsz);
      it.tb = (int)(r / gsz);
    } else {
      it.ta = (int)(t / tB);
      it.tb = (int)(t - (uint32_t)it.ta * tB);
    }
    if (CG == 2) it.ta = 2 * it.ta + (int)(blockIdx.x & 1u);
    return true;
  }
  const uint32_t U = (uint32_t)p.units;
  const uint32_t u1 = ((blockIdx.x + 1) * U) / G;
  if (cur >= u1) return false;
  const uint32_t KB = (uint32_t)p.kblocks;
  const uint32_t t = cur / KB;
  it.t = (int)t;
  it.kb0 = (int)(cur - t * KB);
  const uint32_t room = u1 - cur;
  it.kb1 = (KB - (uint32_t)it.kb0) < room ? (int)KB : it.kb0 + (int)room;
  cur += (uint32_t)(it.kb1 - it.kb0);
  const uint32_t first = t * KB;
  const uint32_t o0 = owner_of(first, U, G);
  it.seg = (int)(blockIdx.x - o0);
  it.nseg = (int)(owner_of(first + KB - 1, U, G) - o0 + 1);
  it.ta = it.t / p.tilesB;
  it.tb = it.t - it.ta * p.tilesB;
  return true;
}

// A wait every lane of the warp takes; the outcome is made warp-uniform so
// that the .sync.aligned tcgen05 loads that follow stay convergent.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const WaitCtl &ctl) {
  const bool ok = mbar_wait(bar, parity, ctl);
  return __all_sync(0xFFFFFFFFu, ok);
}

// Wait that ignores the abort flag (used only to let in-flight async copies
// and MMAs land before the CTA exits); bounded by the same limit.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns,
                                           int *status) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > timeout_ns) {
      if (status) atomicOr(status, 0x1);
      return;
    }
  }
}

// Optional timeline: one SM-clock stamp per trace point per CTA (plus the
// global timer at entry and exit, to line CTAs up against each other).
__device__ __forceinline__ void trace_mark(const GemmParams &p, int point) {
  if (p.trace) p.trace[(size_t)blockIdx.x * kTracePoints + point] = clock64();
}
__device__ __forceinline__ void trace_set(const GemmParams &p, int point, unsigned long long v) {
  if (p.trace) p.trace[(size_t)blockIdx.x * kTracePoints + point] = v;
}

template <int N>
__device__ __forceinline__ void tmem_ld_chunk(uint32_t taddr, uint32_t (&r)[N]);
template <>
__device__ __forceinline__ void tmem_ld_chunk<32>(uint32_t taddr, uint32_t (&r)[32]) {
  tmem_ld32(taddr, r);
}
template <>
__device__ __forceinline__ void tmem_ld_chunk<16>(uint32_t taddr, uint32_t (&r)[16]) {
  tmem_ld16(taddr, r);
}

__device__ __forceinline__ void store_out(const GemmParams &p, int m, int n, float v) {
  if (p.out_f32)
    reinterpret_cast<float *>(p.y)[(size_t)m * p.ldy + n] = v;
  else
    reinterpret_cast<uint16_t *>(p.y)[(size_t)m * p.ldy + n] =
        static_cast<uint16_t>(pack_bf16x2(v, 0.0f) & 0xFFFFu);
}

// Split-K reduction: the work is cut into (tile, chunk) items, a chunk being
// kRedThreads x kRedJ float4 groups (4 consecutive rows of one column) of
// the tile's [column][128 rows] slots.  An item sums the slots in slot order
// (a fixed order: deterministic), applies the PTPC scales and writes y; all
// loads of a thread go out before its first sum (one round of L2 latency).
constexpr int kRedThreads = 128;
constexpr int kRedJ = 2;

template <int KIND>
__device__ __forceinline__ void reduce_items(const GemmParams &p, int bn, unsigned gemm_ctas) {
  const unsigned U = (unsigned)p.units, KB = (unsigned)p.kblocks;
  const int per_col = kTileA / 4;
  const int per_tile = bn * per_col;
  const int chunk = kRedThreads * kRedJ;
  const int chunks = (per_tile + chunk - 1) / chunk;
  const int items = p.tilesA * p.tilesB * chunks;
  const size_t slot4 = (size_t)bn * kTileA / 4;
  for (int item = blockIdx.x; item < items; item += gridDim.x) {
    const int t = item / chunks, c = item - t * chunks;
    const unsigned first_u = (unsigned)t * KB;
    const unsigned o0 = owner_of(first_u, U, gemm_ctas);
    const int nseg = (int)(owner_of(first_u + KB - 1, U, gemm_ctas) - o0 + 1);
    if (nseg <= 1) continue;  // one CTA owned the whole tile and wrote y itself
    const int tb = t - (t / p.tilesB) * p.tilesB;
    const int ta = t / p.tilesB;
    const int valid_cols = min(bn, p.rowsB - tb * bn);
    const float4 *base = reinterpret_cast<const float4 *>(p.ws) + (size_t)t * p.seg_max * slot4;
    int g[kRedJ];
    float4 v[kRedJ][4];
#pragma unroll
    for (int j = 0; j < kRedJ; ++j) {
      g[j] = c * chunk + j * kRedThreads + threadIdx.x;
      const bool in = g[j] < per_tile && g[j] / per_col < valid_cols;
      if (!in) g[j] = -1;
#pragma unroll
      for (int sg = 0; sg < 4; ++sg)
        v[j][sg] = (in && sg < nseg) ? __ldcg(base + sg * slot4 + g[j]) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int j = 0; j < kRedJ; ++j) {
      if (g[j] < 0) continue;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int sg = 0; sg < 4; ++sg) {
        acc.x += v[j][sg].x;
        acc.y += v[j][sg].y;
        acc.z += v[j][sg].z;
        acc.w += v[j][sg].w;
      }
      for (int sg = 4; sg < nseg; ++sg) {
        const float4 w = __ldcg(base + sg * slot4 + g[j]);
        acc.x += w.x;
        acc.y += w.y;
        acc.z += w.z;
        acc.w += w.w;
      }
      const int col = g[j] / per_col, r = (g[j] - col * per_col) * 4;
      const int m = tb * bn + col;      // token
      const int n = ta * kTileA + r;    // output channel
      float f[4] = {acc.x, acc.y, acc.z, acc.w};
      if (KIND == 1) {
        const float sa = p.tok_scale[m];
#pragma unroll
        for (int q = 0; q < 4; ++q) f[q] = (f[q] * sa) * p.chan_scale[n + q];
      }
      if (p.out_f32)
        *reinterpret_cast<float4 *>(reinterpret_cast<float *>(p.y) + (size_t)m * p.ldy + n) =
            make_float4(f[0], f[1], f[2], f[3]);
      else
        *reinterpret_cast<uint2 *>(reinterpret_cast<uint16_t *>(p.y) + (size_t)m * p.ldy + n) =
            make_uint2(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]));
    }
  }
}

template <int KIND, int BN, int KS, int CG>
__global__ void __maxnreg__(136)  // 26K registers a CTA: room for the small kernels beside it
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmY, const GemmParams p) {
  using C = Cfg<KIND, BN, KS, CG>;
  constexpr int S = C::kStages;
  constexpr int CH = C::kChunk;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  // the 128-byte swizzle needs 1024-byte aligned stages: they start at the
  // first 1024-byte boundary after the barriers
  const uint32_t base = (raw + (uint32_t)C::kBarBytes + 1023u) & ~1023u;
  if (base + (uint32_t)(C::kStages * C::kStageBytes + C::kEpiBytes) > raw + (uint32_t)C::kSmem) {
    // (the same for every CTA of the grid: none of them touches anything)
    if (threadIdx.x == 0 && p.status) atomicOr(p.status, 0x4 /* MXG_DEV_SMEM_LAYOUT */);
    return;
  }
  // Stage s is one block of kStageBytes: A codes, B codes, B scales, A scales
  // (every part 1024-byte aligned; an operand's scales follow its codes so
  // that a weight panel -- codes, then scales -- lands with one copy).
  const uint32_t sA = base;  // the whole pipeline region starts here
  auto a_smem = [&](int st) { return sA + (uint32_t)st * C::kStageBytes; };
  auto b_smem = [&](int st) { return a_smem(st) + C::kABytes; };
  auto sfb_smem = [&](int st) { return b_smem(st) + C::kBBytes; };
  auto sfa_smem = [&](int st) { return sfb_smem(st) + C::kSfbBytes; };
  const uint32_t sEpi = sA + S * C::kStageBytes;
  const uint32_t bars = raw;
  // mbarriers: per stage full / empty / ready for the MMAs (A4W4: scales in
  // TMEM) / landed in the other CTA of a pair (FP8), then per accumulator
  // full / empty, the debug stall and the MMA drain.  In a CTA pair the even
  // CTA's MMA thread waits on its own stage_ready / peer_full / acce, which
  // both CTAs arrive on; its commits land on empty / accf / mma_done of both.
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (S + s); };
  auto sf_ready = [&](int s) { return bars + 8u * (2 * S + s); };
  auto peer_full = [&](int s) { return bars + 8u * (3 * S + s); };
  const uint32_t acc_bars = bars + 8u * (4 * S);
  auto accf = [&](int b) { return acc_bars + 8u * (uint32_t)b; };
  auto acce = [&](int b) { return acc_bars + 16u + 8u * (uint32_t)b; };
  const uint32_t stall_bar = acc_bars + 32;
  const uint32_t mma_done = acc_bars + 40;
  constexpr int kAccBufs = C::kAccBufs;
  static_assert(kAccCol + kAccBufs * BN <= (KIND == 0 ? kSfCol : kTmemCols), "TMEM accumulators");
  uint8_t *misc = smem_raw + 8 * (4 * S + 6);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(misc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(misc + 4);
  // A4W4: the epilogue warps (idle during an item's main loop) move each
  // stage's scale factors into TMEM with tcgen05.st, off the tensor pipe; a
  // tcgen05.cp there would hold up the MMAs behind it in the in-order tensor
  // pipe and, through them, the release of the stage.
  constexpr bool kEpiScales = KIND == 0;
  // CTA pair: rank in the cluster; the even CTA issues the MMAs
  const uint32_t crank = CG == 2 ? cluster_rank() : 0u;
  // arrival on a barrier the (even CTA's) MMA thread waits on
  auto arrive_mma = [&](uint32_t bar) {
    if (CG == 2)
      mbar_arrive_cluster(mapa_shared(bar, 0));
    else
      mbar_arrive(bar);
  };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // The next kernel may launch now: it touches no memory this one writes or
  // reads before its own griddepcontrol.wait, which returns only when this
  // grid has completed.  Its CTAs take an SM as this kernel's leave it.
  pdl_trigger();
  if (threadIdx.x == 0) {
    trace_mark(p, kTrEntry);
    trace_set(p, kTrEntryNs, global_timer_ns());
    if (p.trace) {
      uint32_t smid;
      asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
      trace_set(p, kTrSmid, smid);
    }
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
      mbar_init(peer_full(s), 1);
    }
    for (int st = 0; st < S; ++st) mbar_init(sf_ready(st), 4 * CG);
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf(b), 1);
      mbar_init(acce(b), 4 * CG * C::kEpiSets);
    }
    mbar_init(stall_bar, 1);
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc<CG>(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish<CG>();
  }
  tc_fence_before();
  __syncthreads();
  if (CG == 2) cluster_sync();  // both CTAs' barriers are initialised before any remote arrival
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(tmem_slot);
  const WaitCtl ctl{abort_flag, p.status, p.timeout_ns};
  if (threadIdx.x == 0) trace_mark(p, kTrSetup);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    {  // all 32 lanes set up the first stages; lane 0 then runs the pipeline
      const uint64_t pol_stream = policy_evict_first();
      const uint64_t pol_keep = policy_evict_last();
      const uint64_t polA = p.swap ? pol_stream : pol_keep;  // swapped: A = weights, read once
      const uint64_t polB = pol_keep;
      // Stage kb covers the 128-byte K columns [kb*KS, kb*KS + ncol(kb)).
      auto ncol_of = [&](int kb) { return min(KS, p.kc_per_row - kb * KS); };
      // A4W4 scale atoms (512 bytes: 128 rows x 4 blocks of 32) of stage kb
      auto natoms_of = [&](int kb) { return min(2 * KS, p.G4 - 2 * KS * kb); };
      // a CTA of a pair whose token tile lies past the last one loads no
      // activations (its output rows are never stored)
      auto a_in = [&](const Item &it) { return CG == 1 || it.ta < p.tilesA; };
      // the operand and scale bytes one stage receives
      auto stage_bytes = [&](const Item &it, int kb) {
        const uint32_t na = a_in(it) ? 1u : 0u;
        uint32_t bytes = (uint32_t)ncol_of(kb) * (na * C::kAColBytes + C::kBColBytes);
        if (KIND == 0) {
          const int rb0 = (it.tb * BN) / 128;
          const int nblk = min(C::kSfBlocksB, (p.rowsB + 127) / 128 - rb0);
          // a weight panel as B brings the scales of both halves, padding included
          const int nblk_in = (p.w_panels && !p.swap) ? C::kSfBlocksB : nblk;
          bytes += (uint32_t)(natoms_of(kb) * 512) * (na + (uint32_t)nblk_in);
        }
        return bytes;
      };
      // The copies of one stage, numbered: the A operand (one bulk copy in the
      // tile layout -- the columns of a stage are adjacent, tile (row tile,
      // column) at (row tile * KC + column) * tile bytes -- else one 128-byte
      // swizzle box per column), its scales, then the B operand (token tiles:
      // one copy; 128-row weight tiles: one per column and row tile; else one
      // box per column), its scales (one per 128-row block).  Copy i of a
      // stage is issued by one lane (copy_of below), all of a stage's copies
      // in one converged instruction: they run in parallel.
      auto issue_op = [&](int i, bool want_a, bool want_b, int stage, const Item &it, int kb,
                          uint32_t fb) {
        const int nc = ncol_of(kb);
        const int rb0 = (it.tb * BN) / 128;
        const int nblk = min(C::kSfBlocksB, (p.rowsB + 127) / 128 - rb0);
        // weight panels (256 rows: the codes, then the scales of both 128-row
        // halves, per 128-byte column): split-K takes one half as its A tile
        // (codes and scales one copy each per column); the full tile takes a
        // whole panel as its B tile -- codes and scales in one copy
        const bool a_pan = p.w_panels && p.swap;
        const bool b_pan = p.w_panels && !p.swap;
        if (want_a && a_pan) {
          const uint8_t *blk0 = p.a_tiles + ((size_t)(it.ta >> 1) * p.kc_per_row + (size_t)kb * KS) * C::kPanelBytes;
          const int h = it.ta & 1;
          if (i < nc) {
            bulk_load(a_smem(stage) + i * C::kAColBytes, blk0 + (size_t)i * C::kPanelBytes + h * 16384, 16384,
                      fb, polA);
            return;
          }
          i -= nc;
          if (KIND == 0) {
            if (i < nc) {
              bulk_load(sfa_smem(stage) + i * 1024, blk0 + (size_t)i * C::kPanelBytes + 32768 + h * 1024, 1024,
                        fb, polA);
              return;
            }
            i -= nc;
          }
        } else if (want_a) {
          const int na = p.a_tiles ? 1 : nc;
          if (i < na) {
            if (!a_in(it)) return;
            if (p.a_tiles)
              bulk_load(a_smem(stage),
                        p.a_tiles + ((size_t)it.ta * p.kc_per_row + (size_t)kb * KS) * (size_t)C::kAColBytes,
                        (uint32_t)nc * C::kAColBytes, fb, polA);
            else
              tma_load_2d(a_smem(stage) + i * C::kAColBytes, &tmA, (kb * KS + i) * kRowBytes,
                          it.ta * kTileA, fb, polA);
            return;
          }
          i -= na;
          if (KIND == 0) {
            if (i == 0) {
              if (a_in(it))
                bulk_load(sfa_smem(stage), p.sfA + ((size_t)it.ta * p.G4 + 2 * KS * kb) * 512u,
                          natoms_of(kb) * 512, fb, polA);
              return;
            }
            i -= 1;
          }
        }
        if (want_b && b_pan) {  // BN == 256, one column per stage
          const uint8_t *blk = p.b_tiles + (size_t)it.e * p.w_group_bytes +
                               ((size_t)it.tb * p.kc_per_row + (size_t)kb * KS) * C::kPanelBytes;
          if (CG == 1) {
            if (i == 0) bulk_load(b_smem(stage), blk, (uint32_t)C::kPanelBytes, fb, polB);
          } else {
            // this CTA's 128-row half of the panel's codes, then (A4W4) the
            // scales of both halves
            if (i == 0)
              bulk_load(b_smem(stage), blk + crank * 16384u, 16384, fb, polB);
            else if (KIND == 0 && i == 1)
              bulk_load(sfb_smem(stage), blk + 32768, 2048, fb, polB);
          }
        } else if (want_b) {
          const bool tok = p.b_tiles && p.b_tile_rows == BN;
          constexpr int kRT = C::kBRows >= 128 ? C::kBRows / 128 : 1;  // 128-row weight tiles per column
          const int nb = tok ? 1 : p.b_tiles ? nc * kRT : nc;
          if (i < nb) {
            if (tok) {
              bulk_load(b_smem(stage),
                        p.b_tiles + ((size_t)it.tb * p.kc_per_row + (size_t)kb * KS) * (size_t)C::kBColBytes,
                        (uint32_t)nc * C::kBColBytes, fb, polB);
            } else if (p.b_tiles) {  // BN >= 128 here (the dispatcher's weight-tile case)
              const int j = i / kRT, r = i % kRT;
              // a row tile past the last weight row (N % BN != 0) re-reads the last
              // tile: its rows only feed output columns past N, which are not stored
              const int rt = min(it.tb * (BN / 128) + (int)crank * kRT + r, (p.rowsB + 127) / 128 - 1);
              bulk_load(b_smem(stage) + j * C::kBColBytes + r * 16384,
                        p.b_tiles + ((size_t)rt * p.kc_per_row + (size_t)kb * KS + j) * 16384u,
                        16384, fb, polB);
            } else {
              // (CG = 2: the map's box is the CTA's 128 rows)
              tma_load_2d(b_smem(stage) + i * C::kBColBytes, &tmB, (kb * KS + i) * kRowBytes,
                          it.tb * BN + (int)crank * C::kBRows, fb, polB);
            }
            return;
          }
          i -= nb;
          if (KIND == 0 && i < nblk)
            bulk_load(sfb_smem(stage) + i * (1024 * KS),
                      p.sfB + ((size_t)(rb0 + i) * p.G4 + 2 * KS * kb) * 512u, natoms_of(kb) * 512, fb, polB);
        }
      };
      // Stage k's copies go to lanes 8 (k % 4) .. 8 (k % 4) + 7 (a stage has at
      // most 7 copies): the copies one thread issues complete one after
      // another (~0.4 us each, whatever their size), so giving consecutive
      // stages to different lanes lets them overlap.
      auto copy_of = [&](long long k) { return (lane - 8 * (int)(k & 3)) & 31; };
      const bool w_is_a = p.swap != 0;
      // stage k of this CTA's sequence: its item and K-stage
      auto stage_of = [&](int k, Item &it, int &kb) -> bool {
        uint32_t c = first_cursor<CG>(p);
        int n = 0;
        while (next_item<CG>(p, c, it)) {
          const int len = it.kb1 - it.kb0;
          if (k < n + len) {
            kb = it.kb0 + (k - n);
            return true;
          }
          n += len;
        }
        return false;
      };
      // A grouped GEMM's tiles follow the token-tile offsets the quantizer
      // ahead of it writes: walk them only after the wait.
      if (p.groups) pdl_wait();
      // The first S stages (fewer if the CTA has fewer): weights that no
      // kernel still in flight writes stream in before griddepcontrol.wait;
      // the activation operand follows the wait.
      int pre = 0;
      {
        Item itk;
        int kbk = 0;
        while (pre < S && stage_of(pre, itk, kbk)) {
          if (p.early_w) {
            if (lane == 0) mbar_arrive_expect_tx(full_bar(pre), stage_bytes(itk, kbk));
            __syncwarp();
            issue_op(copy_of(pre), w_is_a, !w_is_a, pre, itk, kbk, full_bar(pre));
          }
          ++pre;
        }
      }
      // With the weights already in flight, what remains of the first stages
      // after the wait is the activation operand: when it is in the tile
      // layout, every one of those copies (dst, src, bytes) is worked out
      // now, and lane j issues copy j right after the wait -- one converged
      // instruction for all of them, instead of one stage after another.
      const bool act_tiles = p.swap ? (p.b_tiles && p.b_tile_rows == BN) : (p.a_tiles != nullptr);
      const int n_act = 1 + (KIND == 0 ? (p.swap ? C::kSfBlocksB : 1) : 0);  // copies per stage (at most)
      const bool fast_first = p.early_w && act_tiles && pre * n_act <= 32;
      uint32_t fc_dst = 0, fc_bytes = 0, fc_bar = 0;
      const uint8_t *fc_src = nullptr;
      if (fast_first && lane < pre * n_act) {
        const int k = lane / n_act, j = lane % n_act;
        Item itk;
        int kbk = 0;
        stage_of(k, itk, kbk);
        const int nc = ncol_of(kbk);
        fc_bar = full_bar(k);
        if (!p.swap && !a_in(itk)) {
          // nothing to load
        } else if (j == 0) {
          if (p.swap) {
            fc_dst = b_smem(k);
            fc_src = p.b_tiles + ((size_t)itk.tb * p.kc_per_row + (size_t)kbk * KS) * (size_t)C::kBColBytes;
            fc_bytes = (uint32_t)nc * C::kBColBytes;
          } else {
            fc_dst = a_smem(k);
            fc_src = p.a_tiles + ((size_t)itk.ta * p.kc_per_row + (size_t)kbk * KS) * (size_t)C::kAColBytes;
            fc_bytes = (uint32_t)nc * C::kAColBytes;
          }
        } else if (KIND == 0) {
          const int na = natoms_of(kbk);
          if (p.swap) {
            const int rb0 = (itk.tb * BN) / 128;
            const int nblk = min(C::kSfBlocksB, (p.rowsB + 127) / 128 - rb0);
            if (j - 1 < nblk) {
              fc_dst = sfb_smem(k) + (uint32_t)(j - 1) * (1024 * KS);
              fc_src = p.sfB + ((size_t)(rb0 + j - 1) * p.G4 + 2 * KS * kbk) * 512u;
              fc_bytes = (uint32_t)na * 512u;
            }
          } else {
            fc_dst = sfa_smem(k);
            fc_src = p.sfA + ((size_t)itk.ta * p.G4 + 2 * KS * kbk) * 512u;
            fc_bytes = (uint32_t)na * 512u;
          }
        }
      }
      pdl_wait();
      if (lane == 0) {
        trace_mark(p, kTrWaited);
        trace_set(p, kTrWaitedNs, global_timer_ns());
      }
      bool ok = true;
      // the rest of the first stages
      if (fast_first) {
        if (fc_bytes) bulk_load(fc_dst, fc_src, fc_bytes, fc_bar, p.swap ? polB : polA);
      }
      for (int k = 0; k < pre && !fast_first; ++k) {
        Item itk;
        int kbk = 0;
        stage_of(k, itk, kbk);
        if (p.early_w) {
          issue_op(copy_of(k), !w_is_a, w_is_a, k, itk, kbk, full_bar(k));
        } else {
          if (lane == 0) mbar_arrive_expect_tx(full_bar(k), stage_bytes(itk, kbk));
          __syncwarp();
          issue_op(copy_of(k), true, true, k, itk, kbk, full_bar(k));
        }
      }
      if (lane == 0) trace_mark(p, kTrFirstLoad);
      // steady state: the whole warp walks the stages in order; lane 0 waits
      // for a free slot and arms it, then every lane issues its copy
      uint32_t cur = first_cursor<CG>(p);
      Item it;
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      while (ok && next_item<CG>(p, cur, it)) {
        for (int kb = it.kb0; kb < it.kb1; ++kb) {
          if (issued >= pre) {
            const uint32_t fb = full_bar(stage);
            bool w_ok = true;
            if (lane == 0) {
              w_ok = mbar_wait(empty_bar(stage), phase ^ 1u, ctl);
              if (w_ok) mbar_arrive_expect_tx(fb, stage_bytes(it, kb));
            }
            if (!__shfl_sync(0xFFFFFFFFu, w_ok ? 1 : 0, 0)) {
              ok = false;
              break;
            }
            issue_op(copy_of(issued), true, true, stage, it, kb, fb);
          }
          ++issued;
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (issued < pre) issued = pre;
      if (lane == 0) {
        trace_mark(p, kTrLastLoad);
        if (!ok || *abort_flag) {
          // let every copy still in flight land before the CTA can exit
          const long long n = issued < S ? issued : S;
          for (long long k = 1; k <= n; ++k) {
            const long long pos = issued - k;
            drain_wait(full_bar((int)(pos % S)), (uint32_t)((pos / S) & 1), p.timeout_ns, p.status);
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && crank != 0) {
      // the odd CTA of a pair: tell the even CTA's MMA thread when each FP8
      // stage has landed here (A4W4: the epilogue warps' scale feed does)
      pdl_wait();
      if (KIND == 1) {
        uint32_t cur = first_cursor<CG>(p);
        Item it;
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        while (ok && next_item<CG>(p, cur, it)) {
          for (int kb = it.kb0; kb < it.kb1; ++kb) {
            if (!mbar_wait(full_bar(stage), phase, ctl)) {
              ok = false;
              break;
            }
            mbar_arrive_cluster(mapa_shared(peer_full(stage), 0));
            if (++stage == S) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      // the even CTA's last commit: every MMA that reads this CTA's shared
      // memory or writes its TMEM is done
      drain_wait(mma_done, 0, p.timeout_ns, p.status);
    } else if (lane == 0) {
      const uint32_t idesc0 = KIND == 0 ? idesc_mxf4(kTileA * CG, BN) : idesc_f8(kTileA * CG, BN);
      // the bounded waits below start counting only once the kernels this
      // one depends on have finished
      pdl_wait();
      trace_mark(p, kTrWaited);
      uint32_t cur = first_cursor<CG>(p);
      Item it;
      int stage = 0;
      uint32_t phase = 0;
      int i = 0;
      bool ok = true;
      while (ok && next_item<CG>(p, cur, it)) {
        // accumulator b of item i; its use-th use: wait until the epilogue
        // has read out its previous tile
        const int b = i % kAccBufs, use = i / kAccBufs;
        const uint32_t d_acc = tmem + kAccCol + (uint32_t)(b * BN);
        if (use > 0 && !mbar_wait(acce(b), (uint32_t)((use - 1) & 1), ctl)) break;
        tc_fence_after();
        for (int kb = it.kb0; kb < it.kb1; ++kb) {
          // A4W4: the epilogue warps (of both CTAs of a pair) signal once the
          // stage's data is in and its scales are in TMEM; FP8: the stage's
          // data is in (here, and in the other CTA of a pair)
          const bool landed = kEpiScales ? mbar_wait(sf_ready(stage), phase, ctl)
                                         : (mbar_wait(full_bar(stage), phase, ctl) &&
                                            (CG == 1 || mbar_wait(peer_full(stage), phase, ctl)));
          if (!landed) {
            ok = false;
            break;
          }
          if (i == 0 && kb == it.kb0) trace_mark(p, kTrFirstFull);
          tc_fence_after();
          const uint32_t a0 = a_smem(stage);
          const uint32_t b0 = b_smem(stage);
          // K step s of the stage: column s / 4, 32 bytes per step within it
          auto a_desc = [&](int s) {
            return sdesc_kmajor_sw128(a0 + (uint32_t)(s >> 2) * C::kAColBytes + 32u * (s & 3));
          };
          auto b_desc = [&](int s) {
            return sdesc_kmajor_sw128(b0 + (uint32_t)(s >> 2) * C::kBColBytes + 32u * (s & 3));
          };
          if constexpr (KIND == 0) {
            // this ring slot's scale factors, fed into TMEM by the epilogue warps
            const uint32_t sfa_t = tmem + kSfCol + (uint32_t)stage * C::kSfColsPerStage;
            const uint32_t sfb_t = sfa_t + C::kSfColsA;
            const int nk = min(C::kSteps, (p.K - kb * 256 * KS) / 64);
            for (int s = 0; s < nk; ++s) {
              const uint32_t sel = (uint32_t)(s & 1) * 2u;
              mma_mxf4<CG>(d_acc, a_desc(s), b_desc(s), idesc_sf_ids(idesc0, sel, sel),
                           sfa_t + 4 * (s >> 1), sfb_t + 4 * C::kSfBlocksB * (s >> 1),
                           (kb > it.kb0 || s > 0) ? 1u : 0u);
            }
          } else {
            const int nk = min(C::kSteps, (p.K - kb * 128 * KS) / 32);
            for (int s = 0; s < nk; ++s)
              mma_f8<CG>(d_acc, a_desc(s), b_desc(s), idesc0, (kb > it.kb0 || s > 0) ? 1u : 0u);
          }
          tc_commit<CG>(empty_bar(stage));
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit<CG>(accf(b));
        trace_mark(p, kTrLastCommit);
        ++i;
      }
      // every MMA issued so far must finish before TMEM is released
      tc_commit<CG>(mma_done);
      drain_wait(mma_done, 0, p.timeout_ns, p.status);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;            // TMEM lane quarter this warp may access
    const int eset = (warp - 2) >> 2;  // epilogue warp set
    constexpr int kSetCols = BN / C::kEpiSets;  // accumulator columns this set reads out
    const int c_lo = eset * kSetCols;
    const int r_in = q * 32 + lane;    // row of the MMA-A tile
    const uint32_t t_row = tmem + ((uint32_t)(q * 32) << 16) + kAccCol;
    pdl_wait();  // scales and partial tiles may come from the kernel ahead
    long long q_sf = 0;  // stage sequence number (kEpiScales)
    // A4W4: the item's stages in order; once a stage's data is in, its scale
    // atoms go smem -> registers -> this warp's TMEM lane quarter, in the
    // layout tcgen05.cp 32x128b.warpx4 makes (lane 32q+i, columns c..c+3 =
    // the atom's 16-byte row i, in every quarter q).
    // One stage's scale factors: smem -> registers -> this warp's TMEM lane
    // quarter.
    auto feed_stage = [&](const Item &it, int kb, int st) {
      const int natoms = min(2 * KS, p.G4 - 2 * KS * kb);
      const int rb0 = (it.tb * BN) / 128;
      const int nblk = min(C::kSfBlocksB, (p.rowsB + 127) / 128 - rb0);
      const uint32_t lane_base = (uint32_t)(q * 32) << 16;
      const uint32_t sfa_col = tmem + lane_base + kSfCol + (uint32_t)st * C::kSfColsPerStage;
      const uint32_t sfb_col = sfa_col + C::kSfColsA;
      if (natoms == 2 * KS && nblk == C::kSfBlocksB) {
        // a whole stage: its columns are contiguous (A atoms, then B atom a
        // of block j at 4 (blocks a + j)), gathered into registers and
        // stored with as few wide stores as there are 32 / 16 / 8 columns
        constexpr int NC = (int)C::kSfColsPerStage;
        uint32_t v[NC];
  #pragma unroll
        for (int a = 0; a < 2 * KS; ++a) {
          const uint4 w = ld_shared_v4(sfa_smem(st) + a * 512 + lane * 16);
          v[4 * a] = w.x, v[4 * a + 1] = w.y, v[4 * a + 2] = w.z, v[4 * a + 3] = w.w;
        }
  #pragma unroll
        for (int j = 0; j < C::kSfBlocksB; ++j)
  #pragma unroll
          for (int a = 0; a < 2 * KS; ++a) {
            const uint4 w = ld_shared_v4(sfb_smem(st) + j * (1024 * KS) + a * 512 + lane * 16);
            const int c = (int)C::kSfColsA + 4 * (C::kSfBlocksB * a + j);
            v[c] = w.x, v[c + 1] = w.y, v[c + 2] = w.z, v[c + 3] = w.w;
          }
        int c = 0;
  #pragma unroll
        for (; c + 32 <= NC; c += 32) tmem_st32(sfa_col + c, v + c);
        if constexpr (NC % 32 >= 16) {
          tmem_st16(sfa_col + c, v + c);
          c += 16;
        }
        if constexpr (NC % 16 >= 8) tmem_st8(sfa_col + c, v + c);
      } else {
        for (int a = 0; a < natoms; ++a)
          tmem_st4(sfa_col + 4 * a, ld_shared_v4(sfa_smem(st) + a * 512 + lane * 16));
        for (int j = 0; j < nblk; ++j)
          for (int a = 0; a < natoms; ++a)
            tmem_st4(sfb_col + 4 * C::kSfBlocksB * a + 4 * j,
                     ld_shared_v4(sfb_smem(st) + j * (1024 * KS) + a * 512 + lane * 16));
      }
    };
    auto feed = [&](const Item &it) -> bool {
      for (int kb = it.kb0; kb < it.kb1; ++kb, ++q_sf) {
        if (C::kEpiSets == 2 && (int)(q_sf & 1) != eset) continue;  // the other set's stage
        const int st = (int)(q_sf % S);
        if (!warp_wait(full_bar(st), (uint32_t)((q_sf / S) & 1), ctl)) return false;
        if (p.trace && q == 2 && lane == 0 && q_sf < 8) trace_mark(p, kTrStageLanded + (int)q_sf);
        feed_stage(it, kb, st);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) arrive_mma(sf_ready(st));
        if (p.trace && q == 2 && lane == 0 && q_sf < 8) trace_mark(p, kTrStageFed + (int)q_sf);
      }
      return true;
    };
    // Read out the accumulator of item i and store it: y (the item covers
    // all of K) or this CTA's fp32 partial tile (part of K; the reduce
    // kernel sums the partials).  Hands the accumulator back to the MMA warp.
    auto finish = [&](const Item &it, int i) -> bool {
      if (p.debug_stall && i == 0) {
        // test hook: a barrier nothing arrives at; the bounded wait gives up
        if (!warp_wait(stall_bar, 0, ctl)) return false;
      }
      const int acc_b = i % kAccBufs, acc_use = i / kAccBufs;
      if (!warp_wait(accf(acc_b), (uint32_t)(acc_use & 1), ctl)) return false;
      const uint32_t t_acc = t_row + (uint32_t)(acc_b * BN);  // this item's accumulator
      if (threadIdx.x == 64 && i < 2) trace_mark(p, i == 0 ? kTrAcc0 : kTrAcc1);
      tc_fence_after();
      const int ra = it.ta * kTileA + r_in;  // MMA-A row: token (full tile) / weight row (split)
      const int cb0 = it.tb * BN;            // first MMA-B row of the tile
      const int ncols = min(BN, p.rowsB - cb0);
      const bool whole = (it.kb0 == 0 && it.kb1 == p.kblocks);
      if (whole && !p.swap && KS == 1 && p.y_tma) {
        // rows = tokens, columns = output channels; per 32-column chunk the
        // warp's 32 x 32 bf16 box goes registers -> smem -> one TMA store
        // (rows past M and columns past N are clipped by the tensor map; a
        // box wholly past M is not stored)
        const float sa = (KIND == 1 && ra < p.M) ? p.tok_scale[ra] : 1.0f;
        const uint32_t ebuf = sEpi + (uint32_t)(warp - 2) * (C::kEpiBufs * 2048u);
        const bool box_in = it.ta * kTileA + q * 32 < p.M;
#pragma unroll 1
        for (int c = c_lo / 32; c < (box_in ? (c_lo + kSetCols) / 32 : 0); ++c) {
          uint32_t v[32];
          tmem_ld_chunk<32>(t_acc + c * 32, v);
          tmem_ld_wait();
          const int n0 = cb0 + c * 32;
          uint32_t w[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            float f0 = __uint_as_float(v[2 * j]), f1 = __uint_as_float(v[2 * j + 1]);
            if (KIND == 1) {
              f0 = (f0 * sa) * p.chan_scale[min(n0 + 2 * j, p.N - 1)];
              f1 = (f1 * sa) * p.chan_scale[min(n0 + 2 * j + 1, p.N - 1)];
            }
            w[j] = pack_bf16x2(f0, f1);
          }
          const int j = c - c_lo / 32;  // this warp's chunk count
          const uint32_t buf = ebuf + (uint32_t)(j % C::kEpiBufs) * 2048u;
          if (j >= C::kEpiBufs) {  // the box last written here must have been read out
            if (lane == 0) {
              if (C::kEpiBufs == 2)
                bulk_wait_group_read<1>();
              else
                bulk_wait_group_read<0>();
            }
            __syncwarp();
          }
#pragma unroll
          for (int k = 0; k < 4; ++k)
            st_shared_v4(buf + lane * 64u + k * 16u, w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tmY, buf, n0, it.ta * kTileA + q * 32);
            bulk_commit_group();
          }
        }
      } else if (whole && !p.swap) {
        // rows = tokens, columns = output channels: each thread writes a row
        // run (grouped: the tile's rows are the expert's rows from
        // (ta - tile0) * 128 on, stored at row0 + that, rows past the
        // expert's last token skipped)
        int yr = ra;
        bool mvalid = ra < p.M;
        if (p.groups) {
          const int lr = (it.ta - it.tile0) * kTileA + r_in;
          yr = it.row0 + lr;
          mvalid = lr < it.rows;
        }
        const float sa = (KIND == 1 && mvalid) ? p.tok_scale[yr] : 1.0f;
#pragma unroll 1
        for (int c = c_lo / CH; c < (c_lo + kSetCols) / CH; ++c) {
          uint32_t v[CH];
          tmem_ld_chunk<CH>(t_acc + c * CH, v);
          tmem_ld_wait();
          const int n0 = cb0 + c * CH;
          if (!mvalid || n0 >= p.N) continue;
          float f[CH];
#pragma unroll
          for (int j = 0; j < CH; ++j) {
            f[j] = __uint_as_float(v[j]);
            if (KIND == 1) f[j] = (f[j] * sa) * p.chan_scale[min(n0 + j, p.N - 1)];
          }
          if (n0 + CH <= p.N) {
            if (p.out_f32) {
              float4 *dst = reinterpret_cast<float4 *>(reinterpret_cast<float *>(p.y) +
                                                       (size_t)yr * p.ldy + n0);
#pragma unroll
              for (int j = 0; j < CH / 4; ++j)
                dst[j] = make_float4(f[4 * j], f[4 * j + 1], f[4 * j + 2], f[4 * j + 3]);
            } else {
              uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<uint16_t *>(p.y) +
                                                     (size_t)yr * p.ldy + n0);
#pragma unroll
              for (int j = 0; j < CH / 8; ++j)
                dst[j] = make_uint4(pack_bf16x2(f[8 * j], f[8 * j + 1]),
                                    pack_bf16x2(f[8 * j + 2], f[8 * j + 3]),
                                    pack_bf16x2(f[8 * j + 4], f[8 * j + 5]),
                                    pack_bf16x2(f[8 * j + 6], f[8 * j + 7]));
            }
          } else {
#pragma unroll
            for (int j = 0; j < CH; ++j)
              if (n0 + j < p.N) store_out(p, yr, n0 + j, f[j]);
          }
        }
      } else if (whole) {
        // swapped, one CTA covered all of K: rows = output channels, columns = tokens
        const int n = ra;
        const float sw = (KIND == 1 && n < p.N) ? p.chan_scale[n] : 1.0f;
#pragma unroll 1
        for (int c = 0; c < BN / CH; ++c) {
          uint32_t v[CH];
          tmem_ld_chunk<CH>(t_acc + c * CH, v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < CH; ++j) {
            const int m = cb0 + c * CH + j;
            if (m < p.M && n < p.N) {
              float f = __uint_as_float(v[j]);
              if (KIND == 1) f = (f * p.tok_scale[m]) * sw;
              store_out(p, m, n, f);
            }
          }
        }
      } else {
        // swapped, part of K: this CTA's fp32 partial tile ([column][128
        // rows]) into its slot of the workspace; the reduce kernel sums them
        float *mine = p.ws + ((size_t)it.t * p.seg_max + (size_t)it.seg) * ((size_t)BN * kTileA);
#pragma unroll 1
        for (int c = 0; c < BN / CH; ++c) {
          uint32_t v[CH];
          tmem_ld_chunk<CH>(t_acc + c * CH, v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < CH; ++j)
            if (c * CH + j < ncols) mine[(size_t)(c * CH + j) * kTileA + r_in] = __uint_as_float(v[j]);
        }
        if (threadIdx.x == 64 && p.trace &&
            p.trace[(size_t)blockIdx.x * kTracePoints + kTrPartStored] == 0)
          trace_mark(p, kTrPartStored);
      }
      // hand the accumulator back to the MMA warp once its TMEM reads are done
      tc_fence_before();
      __syncwarp();
      if (lane == 0) arrive_mma(acce(acc_b));
      if (threadIdx.x == 64 && i < 2) trace_mark(p, i == 0 ? kTrItem0Done : kTrItem1Done);
      return true;
    };
    // Feed ahead: with two accumulators, the scales of item i+1 go into TMEM
    // before item i is read out, so that the MMAs of item i+1 run while the
    // epilogue stores item i.
    uint32_t cur = first_cursor<CG>(p);
    Item it, held;  // held: fed, not yet finished (two accumulators only)
    bool holding = false;
    int i_fin = 0;
    bool ok = true;
    while (ok && next_item<CG>(p, cur, it)) {
      if (kEpiScales && !feed(it)) {
        ok = false;
        break;
      }
      if (kAccBufs == 1) {
        ok = finish(it, i_fin++);
      } else if (holding) {
        ok = finish(held, i_fin++);
        held = it;
      } else {
        held = it;
        holding = true;
      }
    }
    if (ok && holding) ok = finish(held, i_fin++);
    if (KS == 1 && p.y_tma && lane == 0) bulk_wait_group_all();  // y stores complete
    if (threadIdx.x == 64) {
      trace_mark(p, kTrEpiDone);
      trace_set(p, kTrItems, (unsigned long long)i_fin);
    }
  }

  tc_fence_before();
  __syncthreads();
  // a pair: neither CTA releases its TMEM or leaves (its shared memory and
  // barriers are the other's MMA operands and arrival targets) before both
  // are done
  if (CG == 2) cluster_sync();
  if (threadIdx.x == 0) {
    trace_mark(p, kTrExit);
    trace_set(p, kTrExitNs, global_timer_ns());
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<CG>(tmem, kTmemCols);
  }
}

// The split-K reduction as its own kernel, launched right after the GEMM.
template <int KIND>
__global__ void __maxnreg__(64)  // 128-thread CTAs, 3 of them beside a GEMM CTA and a quantizer CTA
    splitk_reduce_kernel(const GemmParams p, int bn, unsigned gemm_ctas) {
  pdl_trigger();  // touches nothing before the wait below
  if (p.trace && threadIdx.x == 0)
    atomicMax(p.trace + kTrRedEntryInv, ~(unsigned long long)global_timer_ns());
  pdl_wait();     // the GEMM that wrote the partial slots has completed
  reduce_items<KIND>(p, bn, gemm_ctas);
  if (p.trace) {  // (uniform over the grid)
    __syncthreads();
    if (threadIdx.x == 0) atomicMax(p.trace + kTrRedExitNs, (unsigned long long)global_timer_ns());
  }
}

template <int KIND, int BN, int KS, int CG = 1>
cudaError_t launch_t(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmY,
                     const GemmParams &p, int ctas, cudaStream_t stream) {
  using C = Cfg<KIND, BN, KS, CG>;
  auto kern = gemm_kernel<KIND, BN, KS, CG>;
  static DeviceOnce once;  // per instantiation and device (a repeat sets the same value)
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (!once.done(dev)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem);
    if (e != cudaSuccess) return e;
    once.set(dev);
  }
  if (CG == 2 && (ctas % 2) != 0) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = pdl_config(dim3(ctas), dim3(C::kThreads), C::kSmem, stream);
  cudaLaunchAttribute attr[2];
  attach_pdl(cfg, attr);
  if (CG == 2) {  // clusters of two CTAs (a portable cluster size)
    attr[cfg.numAttrs].id = cudaLaunchAttributeClusterDimension;
    attr[cfg.numAttrs].val.clusterDim.x = 2;
    attr[cfg.numAttrs].val.clusterDim.y = 1;
    attr[cfg.numAttrs].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs += 1;
  }
  return cudaLaunchKernelEx(&cfg, kern, tmA, tmB, tmY, p);
}

// Full-tile kernels (BN = 256) take one K column per stage; split-K kernels two.
template <int KIND>
cudaError_t launch_kind(int bn, const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmY,
                        const GemmParams &p, int ctas, cudaStream_t stream) {
  if (!p.splitk) {
    if (bn != 256) return cudaErrorInvalidValue;
    return p.cta_pair ? launch_t<KIND, 256, 1, 2>(tmA, tmB, tmY, p, ctas, stream)
                      : launch_t<KIND, 256, 1, 1>(tmA, tmB, tmY, p, ctas, stream);
  }
  switch (bn) {
    case 16: return launch_t<KIND, 16, 2>(tmA, tmB, tmY, p, ctas, stream);
    case 32: return launch_t<KIND, 32, 2>(tmA, tmB, tmY, p, ctas, stream);
    case 64: return launch_t<KIND, 64, 2>(tmA, tmB, tmY, p, ctas, stream);
    case 128: return launch_t<KIND, 128, 2>(tmA, tmB, tmY, p, ctas, stream);
    case 256: return launch_t<KIND, 256, 2>(tmA, tmB, tmY, p, ctas, stream);
    default: return cudaErrorInvalidValue;
  }
}

// The tensor pipe's own rate for this GEMM's instruction shapes: one CTA per
// SM, one thread issuing `iters` x 4 MMAs (M = 128, N = bn; K = 64 E2M1 with
// block scales already in TMEM, or K = 32 E4M3) on operands resident in
// shared memory (zeros: finite codes and scales), one TMEM accumulator.  The
// final commit is waited on with a bound.
template <int KIND>
__global__ void __launch_bounds__(128) mma_peak_kernel(int iters, int bn, int *status,
                                                       unsigned long long timeout_ns) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t tslot;
  __shared__ __align__(8) uint64_t bar;
  const uint32_t base = (smem_addr(smem_raw) + 1023u) & ~1023u;
  const uint32_t sA = base, sB = base + 16384, sSFA = sB + 32768, sSFB = sSFA + 1024;
  for (uint32_t o = threadIdx.x * 16u; o < 16384u + 32768u + 3072u; o += 128u * 16u)
    st_shared_v4(base + o, 0u, 0u, 0u, 0u);
  fence_proxy_async_smem();  // the zeros are read by the tensor pipe
  if (threadIdx.x < 32) {
    tmem_alloc(smem_addr(&tslot), 512);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bar), 1);
    fence_barrier_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tslot;
  if (threadIdx.x == 0) {
    const uint32_t idesc = KIND == 0 ? idesc_mxf4(128, bn) : idesc_f8(128, bn);
    const uint32_t sfa_t = tmem + 256, sfb_t = tmem + 264;
    if (KIND == 0) {
      for (int a = 0; a < 2; ++a) tc_cp_sf(sfa_t + 4 * a, sdesc_sf_block(sSFA + a * 512));
      for (int j = 0; j < 2; ++j)
        for (int a = 0; a < 2; ++a) tc_cp_sf(sfb_t + 8 * a + 4 * j, sdesc_sf_block(sSFB + j * 1024 + a * 512));
    }
    for (int it = 0; it < iters; ++it)
      for (int s = 0; s < 4; ++s) {
        if (KIND == 0) {
          const uint32_t sel = (uint32_t)(s & 1) * 2u;
          mma_mxf4(tmem, sdesc_kmajor_sw128(sA + 32 * s), sdesc_kmajor_sw128(sB + 32 * s),
                   idesc_sf_ids(idesc, sel, sel), sfa_t + 4 * (s >> 1), sfb_t + 8 * (s >> 1), 1u);
        } else {
          mma_f8(tmem, sdesc_kmajor_sw128(sA + 32 * s), sdesc_kmajor_sw128(sB + 32 * s), idesc, 1u);
        }
      }
    tc_commit(smem_addr(&bar));
    drain_wait(smem_addr(&bar), 0, timeout_ns, status);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x < 32) tmem_dealloc(tmem, 512);
}

}  // namespace

cudaError_t launch_mma_peak(int kind, int bn, int iters, int sm_count, int *status,
                            cudaStream_t stream) {
  const int smem = 200 * 1024;  // one CTA per SM
  cudaError_t e = kind == 0
                      ? cudaFuncSetAttribute(mma_peak_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)
                      : cudaFuncSetAttribute(mma_peak_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const unsigned long long tmo = 2000000000ull;
  if (kind == 0)
    mma_peak_kernel<0><<<sm_count, 128, smem, stream>>>(iters, bn, status, tmo);
  else
    mma_peak_kernel<1><<<sm_count, 128, smem, stream>>>(iters, bn, status, tmo);
  return cudaGetLastError();
}

cudaError_t launch_splitk_reduce(int kind, int bn, const GemmParams &p, int gemm_ctas,
                                 int sm_count, cudaStream_t stream) {
  const int per_tile = bn * (kTileA / 4);
  const long long chunks = (per_tile + kRedThreads * kRedJ - 1) / (kRedThreads * kRedJ);
  long long blocks = (long long)p.tilesA * p.tilesB * chunks;
  // Launched early (programmatic launch), the reduce CTAs sit beside the
  // GEMM CTAs: 3 per SM at most (64 registers a thread, 8K a CTA), so that
  // the next GEMM CTA (at most 26K registers) and a quantizer CTA (10K)
  // still fit on the SM.
  const long long cap = (long long)(sm_count > 0 ? sm_count : 152) * 3;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  cudaLaunchConfig_t cfg = pdl_config(dim3((unsigned)blocks), dim3(kRedThreads), 0, stream);
  cudaLaunchAttribute attr[1];
  attach_pdl(cfg, attr);
  cudaError_t e = kind == 0 ? prefer_shared_carveout(splitk_reduce_kernel<0>)
                            : prefer_shared_carveout(splitk_reduce_kernel<1>);
  if (e != cudaSuccess) return e;
  if (kind == 0) return cudaLaunchKernelEx(&cfg, splitk_reduce_kernel<0>, p, bn, (unsigned)gemm_ctas);
  return cudaLaunchKernelEx(&cfg, splitk_reduce_kernel<1>, p, bn, (unsigned)gemm_ctas);
}

cudaError_t launch_gemm(int kind, int bn, const CUtensorMap &tmA, const CUtensorMap &tmB,
                        const CUtensorMap &tmY, const GemmParams &p, int ctas, cudaStream_t stream) {
  return kind == 0 ? launch_kind<0>(bn, tmA, tmB, tmY, p, ctas, stream)
                   : launch_kind<1>(bn, tmA, tmB, tmY, p, ctas, stream);
}

int gemm_cols_per_stage(bool splitk) { return splitk ? 2 : 1; }

}  // namespace mxg
