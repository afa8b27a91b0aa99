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
//              in bands of token tiles when the operands exceed L2).
//   split-K    (swap = 1): MMA-A = 128 weight rows, MMA-B = the (padded)
//              token rows; the (tile, K-block) units are cut evenly over the
//              CTAs (stream-K); a CTA that ends a tile part-way writes an
//              fp32 partial tile.  The partials are summed in slot order -- a
//              fixed order, so results are deterministic -- by the reduce
//              kernel launched after the GEMM (default), by every CTA after a
//              grid barrier, by the last CTA to finish the tile, or, for CTA
//              pairs in a 2-CTA cluster, by the first CTA of the pair from its
//              partner's partial in its shared memory.
//
// Warp roles (192 threads): warp 0 = producer (bulk copies of operand tiles
// and weight panels, tensor-map boxes for row-major operands, scale tiles);
// warp 1 = TMEM allocator and the single MMA-issuing thread; warps 2-5 =
// epilogue (tcgen05.ld of their 32-lane quarter; for the full-tile A4W4 they
// also move each stage's scale factors into TMEM, and store y by TMA).  All
// hand-offs are mbarriers; every wait is bounded.
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <cuda_runtime.h>

#include "kernels.h"
#include "ptx.cuh"
#include "quant_math.cuh"

namespace mxg {
namespace {

constexpr int kThreads = 192;
constexpr int kTileA = 128;      // MMA M: rows of the MMA-A operand per tile
constexpr int kRowBytes = 128;   // K bytes per row per stage (one 128-byte swizzle row)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCol = 0;    // accumulator: columns [0, BN)
// Scale factors: every pipeline stage has its own TMEM columns from kSfCol on
// (A: 2 K-tiles x 4 columns, then B: 2 K-tiles x row blocks x 4 columns), so
// the copy for the next stage never waits for the MMAs still reading the
// scales of this one.
constexpr uint32_t kSfCol = 256;
constexpr int kSmemBudget = 220 * 1024;

// KS: 128-byte K columns per pipeline stage (one column = 256 E2M1 or 128
// E4M3 values of every row).  Two columns per stage halve the number of bulk
// copies per byte, which is what bounds the weight-streaming (split-K) rate.
template <int KIND, int BN, int KS>
struct Cfg {
  static constexpr int kSfBlocksB = BN >= 128 ? BN / 128 : 1;
  static constexpr int kAColBytes = kTileA * kRowBytes;  // one column of the A operand
  static constexpr int kBColBytes = BN * kRowBytes;
  static constexpr int kABytes = kAColBytes * KS;
  static constexpr int kBBytes = kBColBytes * KS;
  static constexpr int kSfaBytes = KIND == 0 ? 1024 * KS : 0;  // 2 scale atoms per column
  static constexpr int kSfbBytes = KIND == 0 ? 1024 * KS * kSfBlocksB : 0;
  static constexpr int kStageBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes;
  // one column of a 256-row weight panel: codes, then (E2M1) the 2 x 2 scale atoms
  static constexpr int kPanelBytes = 256 * kRowBytes + (KIND == 0 ? 2048 : 0);
  static constexpr int kStagesRaw = kSmemBudget / kStageBytes;
  static constexpr int kStages = kStagesRaw > 12 ? 12 : kStagesRaw;
  static constexpr int kBarBytes = 8 * (3 * kStages + 12) + 16;
  // full tile: per epilogue warp two 32 x 32 bf16 staging boxes for TMA stores of y
  static constexpr int kEpiBytes = KS == 1 ? 4 * 2 * 2048 : 0;
  static constexpr size_t kSmem = 1024 + (size_t)kStages * kStageBytes + kEpiBytes + kBarBytes;
  static constexpr int kChunk = BN >= 32 ? 32 : 16;  // epilogue TMEM columns per load
  static constexpr int kSteps = 4 * KS;              // MMAs (K = 64 / 32) per stage
  static constexpr uint32_t kSfColsA = 8u * KS;      // 4 TMEM columns per scale atom
  static constexpr uint32_t kSfColsPerStage = kSfColsA + 8u * KS * (uint32_t)kSfBlocksB;
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N");
  static_assert(kStages >= 2, "pipeline depth");
  static_assert(KS == 1 || 128 * BN * 4 <= kStages * kStageBytes, "CTA-pair partial tile fits the pipeline");
  static_assert(KIND != 0 || kSfCol + kStages * kSfColsPerStage <= kTmemCols, "TMEM budget");
};

struct Item {
  int t, ta, tb, kb0, kb1, seg, nseg;
};

// CTA that owns stream-K unit u when U units are cut into G equal ranges
// [c*U/G, (c+1)*U/G): the largest c with c*U < (u+1)*G.  The host checks
// that (U+1)*G fits in 32 bits (64-bit division costs ~1 us per item on
// the single producer thread).
__device__ __forceinline__ uint32_t owner_of(uint32_t u, uint32_t U, uint32_t G) {
  return ((u + 1) * G - 1) / U;
}

__device__ __forceinline__ uint32_t first_cursor(const GemmParams &p) {
  return p.splitk ? (blockIdx.x * (uint32_t)p.units) / gridDim.x : blockIdx.x;
}

// The work items of this CTA, in order; every role walks the same list.
__device__ __forceinline__ bool next_item(const GemmParams &p, uint32_t &cur, Item &it) {
  const uint32_t G = gridDim.x;
  if (!p.splitk) {
    if (cur >= (uint32_t)(p.tilesA * p.tilesB)) return false;
    it.t = (int)cur;
    it.kb0 = 0;
    it.kb1 = p.kblocks;
    it.seg = 0;
    it.nseg = 1;
    cur += G;
    if (p.raster_group > 0) {
      // bands of raster_group MMA-A (token) tiles: within a band the token
      // tile varies fastest, so the CTAs running at one time share a few
      // weight tiles and the band's activations stay in L2 -- the weights
      // are read from HBM once per band, not once per token tile
      const uint32_t g = (uint32_t)p.raster_group;
      const uint32_t band = g * (uint32_t)p.tilesB;
      const uint32_t bi = (uint32_t)it.t;
      const uint32_t b0 = bi / band, r = bi - b0 * band;
      const uint32_t ta0 = b0 * g;
      const uint32_t gsz = min(g, (uint32_t)p.tilesA - ta0);
      it.ta = (int)(ta0 + r % gsz);
      it.tb = (int)(r / gsz);
      return true;
    }
  } else {
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
  }
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

// Sum the nseg partial tiles of one output tile in slot order and write y.
// Each slot is [column][128 rows] fp32; the 128 epilogue threads take float4
// groups (4 consecutive rows of one column) so that loads and stores are
// coalesced, with the loads of up to 4 slots x kU groups in flight at once
// (one round of L2 latency per 128 * kU groups).
template <int KIND>
__device__ __forceinline__ void reduce_partials(const GemmParams &p, const float *tile_ws,
                                                size_t slot_elems, int nseg, int ncols, int row0,
                                                int col0, int tid) {
  constexpr int kU = 8;
  const int ngrp = ncols * (kTileA / 4);
  const float4 *base = reinterpret_cast<const float4 *>(tile_ws);
  const size_t slot4 = slot_elems / 4;
#pragma unroll 1
  for (int g0 = tid; g0 < ngrp; g0 += 128 * kU) {
    float4 acc[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    float4 v[4][kU];
#pragma unroll
    for (int s = 0; s < 4; ++s)
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int g = g0 + 128 * u;
        v[s][u] = (s < nseg && g < ngrp) ? __ldcg(base + s * slot4 + g) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
    for (int s = 0; s < 4; ++s)
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        acc[u].x += v[s][u].x;
        acc[u].y += v[s][u].y;
        acc[u].z += v[s][u].z;
        acc[u].w += v[s][u].w;
      }
#pragma unroll 1
    for (int s = 4; s < nseg; ++s)
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int g = g0 + 128 * u;
        if (g < ngrp) {
          const float4 t = __ldcg(base + s * slot4 + g);
          acc[u].x += t.x;
          acc[u].y += t.y;
          acc[u].z += t.z;
          acc[u].w += t.w;
        }
      }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int g = g0 + 128 * u;
      if (g >= ngrp) continue;
      const int c = g / (kTileA / 4);
      const int r = (g % (kTileA / 4)) * 4;
      const int m = col0 + c;  // token
      const int n = row0 + r;  // output channel (N % 128 == 0: always in range)
      float f[4] = {acc[u].x, acc[u].y, acc[u].z, acc[u].w};
      if (KIND == 1) {
        const float sa = p.tok_scale[m];
#pragma unroll
        for (int j = 0; j < 4; ++j) f[j] = (f[j] * sa) * p.chan_scale[n + j];
      }
      if (p.out_f32) {
        *reinterpret_cast<float4 *>(reinterpret_cast<float *>(p.y) + (size_t)m * p.ldy + n) =
            make_float4(f[0], f[1], f[2], f[3]);
      } else {
        *reinterpret_cast<uint2 *>(reinterpret_cast<uint16_t *>(p.y) + (size_t)m * p.ldy + n) =
            make_uint2(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]));
      }
    }
  }
}

// Split-K reduction: for every tile that more than one CTA touched, y = sum
// of the partial slots in slot order (fixed order: deterministic), then the
// PTPC scales, then bf16 (or fp32).  One thread per float4 group of a slot
// ([column][128 rows]), kRedJ groups per thread with all their loads issued
// before the first sum (one round of L2 latency); threads first, first +
// stride, ... so that every SM pulls a share.
constexpr int kRedThreads = 128;
constexpr int kRedJ = 2;

template <int KIND>
__device__ __forceinline__ void reduce_share(const GemmParams &p, int bn, unsigned gemm_ctas,
                                             int first, int stride) {
  const unsigned U = (unsigned)p.units, KB = (unsigned)p.kblocks;
  const int per_col = kTileA / 4;
  const int per_tile = bn * per_col;
  const int total = p.tilesA * p.tilesB * per_tile;
  const size_t slot4 = (size_t)bn * kTileA / 4;
  for (int e0 = first; e0 < total; e0 += stride * kRedJ) {
    int nseg[kRedJ];
    const float4 *src[kRedJ];
    float4 v[kRedJ][4];
#pragma unroll
    for (int j = 0; j < kRedJ; ++j) {
      const int e = e0 + j * stride;
      nseg[j] = 0;
      src[j] = nullptr;
      if (e < total) {
        const int t = e / per_tile;
        const int g = e - t * per_tile;
        const unsigned first_u = (unsigned)t * KB;
        const unsigned o0 = owner_of(first_u, U, gemm_ctas);
        const int ns = (int)(owner_of(first_u + KB - 1, U, gemm_ctas) - o0 + 1);
        const int tb = t - (t / p.tilesB) * p.tilesB;
        const int c = g / per_col;
        // one CTA owned the whole tile and wrote y itself; padding columns
        if (ns > 1 && c < min(bn, p.rowsB - tb * bn)) {
          nseg[j] = ns;
          src[j] = reinterpret_cast<const float4 *>(p.ws) + (size_t)t * p.seg_max * slot4 + g;
        }
      }
#pragma unroll
      for (int s = 0; s < 4; ++s)
        v[j][s] = s < nseg[j] ? __ldcg(src[j] + s * slot4) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int j = 0; j < kRedJ; ++j) {
      if (nseg[j] == 0) continue;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        acc.x += v[j][s].x;
        acc.y += v[j][s].y;
        acc.z += v[j][s].z;
        acc.w += v[j][s].w;
      }
      for (int s = 4; s < nseg[j]; ++s) {
        const float4 w = __ldcg(src[j] + s * slot4);
        acc.x += w.x;
        acc.y += w.y;
        acc.z += w.z;
        acc.w += w.w;
      }
      const int e = e0 + j * stride;
      const int t = e / per_tile;
      const int g = e - t * per_tile;
      const int ta = t / p.tilesB, tb = t - ta * p.tilesB;
      const int c = g / per_col, r = (g - c * per_col) * 4;
      const int m = tb * bn + c;      // token
      const int n = ta * kTileA + r;  // output channel
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

// Fused activation phase (A4W4 split-K): the M x K/128 units (one row, 128
// values = 16 chunks of 8) are cut evenly over the CTAs; 128 threads = 8
// half-warps take one unit each per round, two rounds' loads in flight.
// Codes go to the token tiles (T = BN rows, 128-byte columns), scales to the
// 128x4-tile layout; padding rows stay unwritten (their columns of the
// accumulator are never stored).  Every lane of a warp runs every round:
// the block amax is a 4-lane shuffle.
__device__ __forceinline__ void quant_share(const GemmParams &p, int T, int tid) {
  const int upr = p.K >> 7;
  const long long W = (long long)p.M * upr;
  const long long u0 = (long long)blockIdx.x * W / gridDim.x;
  const long long u1 = (long long)(blockIdx.x + 1) * W / gridDim.x;
  const int hw = tid >> 4, hl = tid & 15;
  const int kc = p.K >> 8;  // 128-byte code columns per row
  const int G = p.K >> 5;   // MX blocks per row
  uint8_t *codes = const_cast<uint8_t *>(p.b_tiles);
  uint8_t *sf = const_cast<uint8_t *>(p.sfB);
  for (long long base = u0; base < u1; base += 16) {
    uint4 v[2];
    int r[2], ch[2];
    bool ok[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const long long u = base + hw + 8 * j;
      ok[j] = u < u1;
      r[j] = ok[j] ? (int)(u / upr) : 0;
      ch[j] = ok[j] ? (int)(u - (long long)r[j] * upr) * 16 + hl : 0;
      v[j] = ok[j] ? ld_stream_v4(p.x + (size_t)r[j] * p.ldx + (size_t)ch[j] * 8)
                   : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      uint32_t scode;
      const uint32_t packed = mx_encode_chunk(v[j], scode);
      if (ok[j]) *reinterpret_cast<uint32_t *>(codes + tiled_offset(r[j], ch[j] * 4, kc, T)) = packed;
      const uint32_t word = mx_scale_word(scode);
      if (ok[j] && hl == 0)
        *reinterpret_cast<uint32_t *>(sf + sf_swizzled_offset(r[j], ch[j] >> 2, G)) = word;
    }
  }
}

// L2 prefetch of this CTA's share of x (contiguous runs within a row).
__device__ __forceinline__ void prefetch_x_share(const GemmParams &p) {
  const int upr = p.K >> 7;
  const long long W = (long long)p.M * upr;
  long long u = (long long)blockIdx.x * W / gridDim.x;
  const long long u1 = (long long)(blockIdx.x + 1) * W / gridDim.x;
  while (u < u1) {
    const long long r = u / upr;
    const long long hi = min(u1, (r + 1) * upr);
    prefetch_l2_bulk(p.x + (size_t)r * p.ldx + (size_t)(u - r * upr) * 128, (uint32_t)(hi - u) * 256u);
    u = hi;
  }
}

template <int KIND, int BN, int KS>
__global__ void __maxnreg__(136)  // 26K registers a CTA: room for the small kernels beside it
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmY, const GemmParams p) {
  using C = Cfg<KIND, BN, KS>;
  constexpr int S = C::kStages;
  constexpr int CH = C::kChunk;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  // Stage s is one block of kStageBytes: A codes, B codes, B scales, A scales
  // (every part 1024-byte aligned; an operand's scales follow its codes so
  // that a weight panel -- codes, then scales -- lands with one copy).
  const uint32_t sA = base;  // the whole pipeline region starts here
  auto a_smem = [&](int st) { return sA + (uint32_t)st * C::kStageBytes; };
  auto b_smem = [&](int st) { return a_smem(st) + C::kABytes; };
  auto sfb_smem = [&](int st) { return b_smem(st) + C::kBBytes; };
  auto sfa_smem = [&](int st) { return sfb_smem(st) + C::kSfbBytes; };
  const uint32_t sEpi = sA + S * C::kStageBytes;
  const uint32_t bars = sEpi + C::kEpiBytes;
  const uint32_t acc_full = bars + 8 * (2 * S);
  const uint32_t acc_empty = acc_full + 8;
  const uint32_t part_bar = acc_full + 16;
  const uint32_t dec_bar = acc_full + 24;
  const uint32_t stall_bar = acc_full + 32;
  const uint32_t mma_done = acc_full + 40;
  const uint32_t acts_ready = acc_full + 48;  // fused path: token tiles of every CTA written
  const uint32_t sf_bars = acc_full + 56;     // full tile: a stage's scales are in TMEM
  const uint32_t pull_bar = sf_bars + 8 * S;  // last-CTA split-K: the partial tiles are in smem
  // CTA-pair split-K: rank 0's pair_bar completes once rank 1's partial tile
  // is in rank 0's shared memory; rank 1's ready_bar once rank 0's pipeline
  // shared memory is free to receive it
  const uint32_t pair_bar = pull_bar + 8;
  const uint32_t ready_bar = pull_bar + 16;
  // FP8 full tile: two accumulators (TMEM columns [0, 256) and [256, 512)),
  // so that the epilogue of one tile overlaps the MMAs of the next; A4W4
  // needs TMEM columns for its scale factors and keeps one
  constexpr int kAccBufs = (KIND == 1 && KS == 1) ? 2 : 1;
  static_assert(kAccCol + kAccBufs * BN <= (KIND == 0 ? kSfCol : kTmemCols), "TMEM accumulators");
  const uint32_t acc_full1 = pull_bar + 24;
  const uint32_t acc_empty1 = pull_bar + 32;
  auto accf = [&](int b) { return b ? acc_full1 : acc_full; };
  auto acce = [&](int b) { return b ? acc_empty1 : acc_empty; };
  uint8_t *misc = smem_raw + (bars - raw) + 8 * (3 * S + 12);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(misc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(misc + 4);
  volatile int *decision = reinterpret_cast<volatile int *>(misc + 8);
  volatile int *reduce_go = reinterpret_cast<volatile int *>(misc + 12);
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (S + s); };
  auto sf_ready = [&](int s) { return sf_bars + 8u * s; };
  // Full-tile A4W4: the epilogue warps (idle during a tile's main loop) move
  // each stage's scale factors into TMEM with tcgen05.st, off the tensor
  // pipe; a tcgen05.cp there would hold up the MMAs behind it and, through
  // them, the release of the stage.
  constexpr bool kEpiScales = KIND == 0;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    trace_mark(p, kTrEntry);
    trace_set(p, kTrEntryNs, global_timer_ns());
    if (p.trace) {
      uint32_t smid;
      asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
      trace_set(p, kTrSmid, smid);
    }
  }
  // The next kernel may launch now: it touches no memory this one writes or
  // reads before its own griddepcontrol.wait, which returns only when this
  // grid has completed.  Its CTAs take an SM as this kernel's leave it.
  pdl_trigger();

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 4);
    mbar_init(part_bar, 128);
    mbar_init(dec_bar, 1);
    mbar_init(stall_bar, 1);
    mbar_init(mma_done, 1);
    mbar_init(acts_ready, 1);
    for (int st = 0; st < S; ++st) mbar_init(sf_ready(st), 4);
    mbar_init(pull_bar, 1);
    mbar_init(pair_bar, 128);
    mbar_init(ready_bar, 1);
    mbar_init(acc_full1, 1);
    mbar_init(acc_empty1, 4);
    *abort_flag = 0;
    *decision = 0;
    *reduce_go = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  // the peer CTA arrives on this CTA's barriers later: their init must be
  // visible across the cluster first
  if (p.pair_reduce) cluster_sync_all();
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
      // the operand and scale bytes one stage receives
      auto stage_bytes = [&](const Item &it, int kb) {
        uint32_t bytes = (uint32_t)ncol_of(kb) * (C::kAColBytes + C::kBColBytes);
        if (KIND == 0) {
          const int rb0 = (it.tb * BN) / 128;
          const int nblk = min(C::kSfBlocksB, (p.rowsB + 127) / 128 - rb0);
          // a weight panel as B brings the scales of both halves, padding included
          const int nblk_in = (p.w_panels && !p.swap) ? C::kSfBlocksB : nblk;
          bytes += (uint32_t)(natoms_of(kb) * 512 * (1 + nblk_in));
        }
        return bytes;
      };
      // The copies of one stage, numbered: the A operand (one bulk copy in the
      // tile layout -- the columns of a stage are adjacent, tile (row tile,
      // column) at (row tile * KC + column) * tile bytes -- else one 128-byte
      // swizzle box per column), its scales, then the B operand (token tiles:
      // one copy; 128-row weight tiles: one per column and row tile; else one
      // box per column), its scales (one per 128-row block).  Lane i issues
      // copy i: copies from one converged instruction run in parallel, while
      // copies that one thread issues one after another complete one after
      // another (~0.2-0.4 us each).
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
              bulk_load(sfa_smem(stage), p.sfA + ((size_t)it.ta * p.G4 + 2 * KS * kb) * 512u,
                        natoms_of(kb) * 512, fb, polA);
              return;
            }
            i -= 1;
          }
        }
        if (want_b && b_pan) {  // BN == 256, one column per stage
          if (i == 0)
            bulk_load(b_smem(stage),
                      p.b_tiles + ((size_t)it.tb * p.kc_per_row + (size_t)kb * KS) * C::kPanelBytes,
                      (uint32_t)C::kPanelBytes, fb, polB);
        } else if (want_b) {
          const bool tok = p.b_tiles && p.b_tile_rows == BN;
          const int nb = tok ? 1 : p.b_tiles ? nc * (BN >= 128 ? BN / 128 : 1) : nc;
          if (i < nb) {
            if (tok) {
              bulk_load(b_smem(stage),
                        p.b_tiles + ((size_t)it.tb * p.kc_per_row + (size_t)kb * KS) * (size_t)C::kBColBytes,
                        (uint32_t)nc * C::kBColBytes, fb, polB);
            } else if (p.b_tiles) {  // BN >= 128 here (the dispatcher's weight-tile case)
              constexpr int kRT = BN >= 128 ? BN / 128 : 1;
              const int j = i / kRT, r = i % kRT;
              // a row tile past the last weight row (N % BN != 0) re-reads the last
              // tile: its rows only feed output columns past N, which are not stored
              const int rt = min(it.tb * kRT + r, (p.rowsB + 127) / 128 - 1);
              bulk_load(b_smem(stage) + j * C::kBColBytes + r * 16384,
                        p.b_tiles + ((size_t)rt * p.kc_per_row + (size_t)kb * KS + j) * 16384u,
                        16384, fb, polB);
            } else {
              tma_load_2d(b_smem(stage) + i * C::kBColBytes, &tmB, (kb * KS + i) * kRowBytes,
                          it.tb * BN, fb, polB);
            }
            return;
          }
          i -= nb;
          if (KIND == 0 && i < nblk)
            bulk_load(sfb_smem(stage) + i * (1024 * KS),
                      p.sfB + ((size_t)(rb0 + i) * p.G4 + 2 * KS * kb) * 512u, natoms_of(kb) * 512, fb, polB);
        }
      };
      const bool w_is_a = p.swap != 0;
      // stage k of this CTA's sequence: its item and K-stage
      auto stage_of = [&](int k, Item &it, int &kb) -> bool {
        uint32_t c = first_cursor(p);
        int n = 0;
        while (next_item(p, c, it)) {
          const int len = it.kb1 - it.kb0;
          if (k < n + len) {
            kb = it.kb0 + (k - n);
            return true;
          }
          n += len;
        }
        return false;
      };
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
            issue_op(lane, w_is_a, !w_is_a, pre, itk, kbk, full_bar(pre));
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
        if (j == 0) {
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
      if (p.fuse_quant) {
        // the token tiles are written by every CTA of this grid; the epilogue
        // warps signal once the grid barrier after that phase has passed
        ok = mbar_wait(acts_ready, 0, ctl) && !*abort_flag;
        ok = __all_sync(0xFFFFFFFFu, ok);
        fence_proxy_async_global();
      }
      // the rest of the first stages -- also when the fused phase failed:
      // every armed stage must land before the CTA exits (contents are then
      // irrelevant; every address stays in bounds)
      if (fast_first) {
        if (fc_bytes) bulk_load(fc_dst, fc_src, fc_bytes, fc_bar, p.swap ? polB : polA);
      }
      for (int k = 0; k < pre && !fast_first; ++k) {
        Item itk;
        int kbk = 0;
        stage_of(k, itk, kbk);
        if (p.early_w) {
          issue_op(lane, !w_is_a, w_is_a, k, itk, kbk, full_bar(k));
        } else {
          if (lane == 0) mbar_arrive_expect_tx(full_bar(k), stage_bytes(itk, kbk));
          __syncwarp();
          issue_op(lane, true, true, k, itk, kbk, full_bar(k));
        }
      }
      if (lane == 0) trace_mark(p, kTrFirstLoad);
      // steady state: the whole warp walks the stages in order; lane 0 waits
      // for a free slot and arms it, then every lane issues its copy
      uint32_t cur = first_cursor(p);
      Item it;
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      while (ok && next_item(p, cur, it)) {
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
            issue_op(lane, true, true, stage, it, kb, fb);
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
    if (lane == 0) {
      const uint32_t idesc0 = KIND == 0 ? idesc_mxf4(kTileA, BN) : idesc_f8(kTileA, BN);
      // the bounded waits below start counting only once the kernels this
      // one depends on have finished
      pdl_wait();
      trace_mark(p, kTrWaited);
      uint32_t cur = first_cursor(p);
      Item it;
      int stage = 0;
      uint32_t phase = 0;
      int i = 0;
      bool ok = true;
      while (ok && next_item(p, cur, it)) {
        // accumulator b of item i; its use-th use: wait until the epilogue
        // has read out its previous tile
        const int b = i % kAccBufs, use = i / kAccBufs;
        const uint32_t d_acc = tmem + kAccCol + (uint32_t)(b * BN);
        if (use > 0 && !mbar_wait(acce(b), (uint32_t)((use - 1) & 1), ctl)) break;
        tc_fence_after();
        for (int kb = it.kb0; kb < it.kb1; ++kb) {
          // full tile A4W4: the epilogue warps signal once the stage's data is
          // in and its scales are in TMEM
          if (!mbar_wait(kEpiScales ? sf_ready(stage) : full_bar(stage), phase, ctl)) {
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
          if (KIND == 0) {
            // scale factors: smem -> the TMEM columns of this ring slot
            const int natoms = min(2 * KS, p.G4 - 2 * KS * kb);
            const int rb0 = (it.tb * BN) / 128;
            const int nblk = min(C::kSfBlocksB, (p.rowsB + 127) / 128 - rb0);
            const uint32_t sfa_t = tmem + kSfCol + (uint32_t)stage * C::kSfColsPerStage;
            const uint32_t sfb_t = sfa_t + C::kSfColsA;
            if (!kEpiScales) {
              for (int a = 0; a < natoms; ++a)
                tc_cp_sf(sfa_t + 4 * a, sdesc_sf_block(sfa_smem(stage) + a * 512));
              for (int j = 0; j < nblk; ++j)
                for (int a = 0; a < natoms; ++a)
                  tc_cp_sf(sfb_t + 4 * C::kSfBlocksB * a + 4 * j,
                           sdesc_sf_block(sfb_smem(stage) + j * (1024 * KS) + a * 512));
            }
            const int nk = min(C::kSteps, (p.K - kb * 256 * KS) / 64);
            for (int s = 0; s < nk; ++s) {
              const uint32_t sel = (uint32_t)(s & 1) * 2u;
              mma_mxf4(d_acc, a_desc(s), b_desc(s), idesc_sf_ids(idesc0, sel, sel),
                       sfa_t + 4 * (s >> 1), sfb_t + 4 * C::kSfBlocksB * (s >> 1),
                       (kb > it.kb0 || s > 0) ? 1u : 0u);
            }
          } else {
            const int nk = min(C::kSteps, (p.K - kb * 128 * KS) / 32);
            for (int s = 0; s < nk; ++s)
              mma_f8(d_acc, a_desc(s), b_desc(s), idesc0, (kb > it.kb0 || s > 0) ? 1u : 0u);
          }
          tc_commit(empty_bar(stage));
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(accf(b));
        trace_mark(p, kTrLastCommit);
        ++i;
      }
      // every MMA issued so far must finish before TMEM is released
      tc_commit(mma_done);
      drain_wait(mma_done, 0, p.timeout_ns, p.status);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;            // TMEM lane quarter this warp may access
    const int r_in = q * 32 + lane;    // row of the MMA-A tile
    const uint32_t t_row = tmem + ((uint32_t)(q * 32) << 16) + kAccCol;
    if (p.fuse_quant && threadIdx.x == 64) prefetch_x_share(p);  // L2 only: safe before the wait
    pdl_wait();  // x, scales, counters and partial tiles may come from the previous kernel
    if (p.fuse_quant) {
      quant_share(p, BN, threadIdx.x - 64);
      fence_proxy_async_global();  // these generic stores are read by other CTAs' bulk copies
      named_barrier(1, 128);
      if (threadIdx.x == 64) {
        trace_mark(p, kTrQuantDone);
        grid_barrier(p.gbar, p.gbar + 32, gridDim.x, ctl);  // raises the abort flag on failure
        trace_mark(p, kTrPartStored);  // (fused path: the first grid barrier passed)
        fence_proxy_async_global();
        mbar_arrive(acts_ready);
      }
      __syncwarp();
    }
    uint32_t cur = first_cursor(p);
    Item it;
    int i = 0;
    uint32_t part_phase = 0;
    long long q_sf = 0;  // stage sequence number (kEpiScales)
    while (next_item(p, cur, it)) {
      if (kEpiScales) {
        // The item's stages in order: once the stage's data is in, its scale
        // atoms go smem -> registers -> this warp's TMEM lane quarter, in the
        // layout tcgen05.cp 32x128b.warpx4 makes (lane 32q+i, columns c..c+3
        // = the atom's 16-byte row i, in every quarter q).
        bool fed = true;
        for (int kb = it.kb0; kb < it.kb1; ++kb, ++q_sf) {
          const int st = (int)(q_sf % S);
          if (!warp_wait(full_bar(st), (uint32_t)((q_sf / S) & 1), ctl)) {
            fed = false;
            break;
          }
          if (p.trace && threadIdx.x == 64 && q_sf < 8) trace_mark(p, kTrStageLanded + (int)q_sf);
          const int natoms = min(2 * KS, p.G4 - 2 * KS * kb);
          const int rb0 = (it.tb * BN) / 128;
          const int nblk = min(C::kSfBlocksB, (p.rowsB + 127) / 128 - rb0);
          const uint32_t lane_base = (uint32_t)(q * 32) << 16;
          const uint32_t sfa_col = tmem + lane_base + kSfCol + (uint32_t)st * C::kSfColsPerStage;
          const uint32_t sfb_col = sfa_col + C::kSfColsA;
          for (int a = 0; a < natoms; ++a)
            tmem_st4(sfa_col + 4 * a, ld_shared_v4(sfa_smem(st) + a * 512 + lane * 16));
          for (int j = 0; j < nblk; ++j)
            for (int a = 0; a < natoms; ++a)
              tmem_st4(sfb_col + 4 * C::kSfBlocksB * a + 4 * j,
                       ld_shared_v4(sfb_smem(st) + j * (1024 * KS) + a * 512 + lane * 16));
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(sf_ready(st));
          if (p.trace && threadIdx.x == 64 && q_sf < 8) trace_mark(p, kTrStageFed + (int)q_sf);
        }
        if (!fed) break;
      }
      if (p.debug_stall && i == 0) {
        // test hook: a barrier nothing arrives at; the bounded wait gives up
        if (!warp_wait(stall_bar, 0, ctl)) break;
      }
      const int acc_b = i % kAccBufs, acc_use = i / kAccBufs;
      if (!warp_wait(accf(acc_b), (uint32_t)(acc_use & 1), ctl)) break;
      const uint32_t t_acc = t_row + (uint32_t)(acc_b * BN);  // this item's accumulator
      if (threadIdx.x == 64 && i < 2) trace_mark(p, i == 0 ? kTrAcc0 : kTrAcc1);
      tc_fence_after();
      const int ra = it.ta * kTileA + r_in;  // MMA-A row: token (full tile) / weight row (split)
      const int cb0 = it.tb * BN;            // first MMA-B row of the tile
      const int ncols = min(BN, p.rowsB - cb0);
      const bool whole = (it.kb0 == 0 && it.kb1 == p.kblocks);
      bool ok = true;
      bool released = false;
      // write this CTA's fp32 partial of the tile ([column][128 rows]) into
      // its slot of the workspace; returns the tile's first slot
      auto publish_partial = [&]() -> float * {
        const size_t slot_elems = (size_t)BN * kTileA;
        float *tile_ws = p.ws + (size_t)it.t * p.seg_max * slot_elems;
        float *mine = tile_ws + (size_t)it.seg * slot_elems;
#pragma unroll 1
        for (int c = 0; c < BN / CH; ++c) {
          uint32_t v[CH];
          tmem_ld_chunk<CH>(t_acc + c * CH, v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < CH; ++j)
            if (c * CH + j < ncols) mine[(size_t)(c * CH + j) * kTileA + r_in] = __uint_as_float(v[j]);
        }
        return tile_ws;
      };
      // hand the accumulator back to the MMA warp once its TMEM reads are done
      auto release_acc = [&]() {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acce(acc_b));
        released = true;
      };
      if (whole && !p.swap && KS == 1 && p.y_tma) {
        // rows = tokens, columns = output channels; per 32-column chunk the
        // warp's 32 x 32 bf16 box goes registers -> smem -> one TMA store
        // (rows past M and columns past N are clipped by the tensor map)
        const float sa = (KIND == 1 && ra < p.M) ? p.tok_scale[ra] : 1.0f;
        const uint32_t ebuf = sEpi + (uint32_t)(warp - 2) * 4096u;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
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
          const uint32_t buf = ebuf + (uint32_t)(c & 1) * 2048u;
          if (c >= 2) {  // the box written two chunks ago must have been read out
            if (lane == 0) bulk_wait_group_read<1>();
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
        // rows = tokens, columns = output channels: each thread writes a row run
        const bool mvalid = ra < p.M;
        const float sa = (KIND == 1 && mvalid) ? p.tok_scale[ra] : 1.0f;
#pragma unroll 1
        for (int c = 0; c < BN / CH; ++c) {
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
                                                       (size_t)ra * p.ldy + n0);
#pragma unroll
              for (int j = 0; j < CH / 4; ++j)
                dst[j] = make_float4(f[4 * j], f[4 * j + 1], f[4 * j + 2], f[4 * j + 3]);
            } else {
              uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<uint16_t *>(p.y) +
                                                     (size_t)ra * p.ldy + n0);
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
              if (n0 + j < p.N) store_out(p, ra, n0 + j, f[j]);
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
      } else if (p.pair_reduce) {
        // A CTA pair (one cluster) shares the tile: rank 0 holds the first
        // part of K, rank 1 the rest.  Rank 1 pushes its fp32 partial into
        // rank 0's pipeline shared memory (idle once rank 0's MMAs are done:
        // each CTA of a pair has this one item); rank 0 adds it to its own,
        // (partial 0 + partial 1, as the reduce kernel sums the slots) and
        // writes y.  Row r's 16-byte chunk k sits at r * BN * 4 +
        // ((k ^ (r % 8)) * 16), so that 8 consecutive rows cover all banks.
        constexpr int kChunks = BN / 4;
        constexpr int kSw = kChunks >= 8 ? 7 : kChunks - 1;
        auto pofs = [&](int r, int k) -> uint32_t {
          return (uint32_t)r * (uint32_t)(BN * 4) + (uint32_t)((k ^ (r & kSw)) << 4);
        };
        if (it.seg == 1) {
          ok = __all_sync(0xFFFFFFFFu, mbar_wait_cluster(ready_bar, 0, ctl));
          if (ok) {
            const uint32_t dst = mapa_shared(sA, 0);
#pragma unroll 1
            for (int c = 0; c < BN / CH; ++c) {
              uint32_t v[CH];
              tmem_ld_chunk<CH>(t_acc + c * CH, v);
              tmem_ld_wait();
#pragma unroll
              for (int j = 0; j < CH / 4; ++j)
                st_cluster_v4(dst + pofs(r_in, c * (CH / 4) + j), v[4 * j], v[4 * j + 1], v[4 * j + 2],
                              v[4 * j + 3]);
            }
          }
          release_acc();
          if (ok) mbar_arrive_remote(mapa_shared(pair_bar, 0));
        } else {
          if (threadIdx.x == 64) mbar_arrive_remote(mapa_shared(ready_bar, 1));
          ok = __all_sync(0xFFFFFFFFu, mbar_wait_cluster(pair_bar, 0, ctl));
          if (ok) {
            const int n = ra;
            const float sw = (KIND == 1 && n < p.N) ? p.chan_scale[n] : 1.0f;
#pragma unroll 1
            for (int c = 0; c < BN / CH; ++c) {
              uint32_t v[CH];
              tmem_ld_chunk<CH>(t_acc + c * CH, v);
              tmem_ld_wait();
#pragma unroll
              for (int j = 0; j < CH / 4; ++j) {
                const uint4 u = ld_shared_v4(sA + pofs(r_in, c * (CH / 4) + j));
                const uint32_t o[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const int m = cb0 + c * CH + 4 * j + e;
                  if (m < p.M && n < p.N) {
                    float f = 0.0f;
                    f += __uint_as_float(v[4 * j + e]);
                    f += __uint_as_float(o[e]);
                    if (KIND == 1) f = (f * p.tok_scale[m]) * sw;
                    store_out(p, m, n, f);
                  }
                }
              }
            }
          }
        }
      } else if (p.defer_reduce || p.grid_reduce) {
        // swapped, part of K: publish this CTA's fp32 partial tile into its
        // slot; the split-K reduce kernel that follows (or every CTA of this
        // grid, after a grid barrier) sums the slots
        publish_partial();
        release_acc();  // the MMA may start the next item during the hand-off
        if (threadIdx.x == 64 && !p.fuse_quant && p.trace &&
            p.trace[(size_t)blockIdx.x * kTracePoints + kTrPartStored] == 0)
          trace_mark(p, kTrPartStored);
      } else if (!whole) {
        // (in-kernel variant) the last CTA of the tile reduces the partials
        const size_t slot_elems = (size_t)BN * kTileA;
        float *tile_ws = publish_partial();
        fence_proxy_async_global();  // the last CTA may read them with bulk copies
        release_acc();
        // the arrive (release, CTA scope) orders this thread's partial stores
        // before the leader's acquire-release counter increment (GPU scope)
        mbar_arrive(part_bar);
        if (warp == 2 && lane == 0) {
          const bool okp = mbar_wait(part_bar, part_phase, ctl);
          int last = 0;
          if (okp) {
            // one acquire-release increment both publishes this CTA's partial
            // (the part_bar arrivals order the other threads' stores before
            // it) and, for the last arriver, makes the other partials visible
            const unsigned old =
                atom_add_acq_rel_gpu(reinterpret_cast<unsigned *>(p.counters) + it.t, 1u);
            last = (old == (unsigned)(it.nseg - 1)) ? 1 : 0;
            if (last) p.counters[it.t] = 0;  // every segment arrived: left zero for the next call
          }
          *decision = okp ? last : -1;
          if (p.trace && p.trace[(size_t)blockIdx.x * kTracePoints + kTrDecision] == 0)
            trace_mark(p, kTrDecision);
          mbar_arrive(dec_bar);
        }
        ok = warp_wait(dec_bar, part_phase, ctl);
        part_phase ^= 1u;
        const int dec = ok ? *decision : -1;
        if (dec < 0) {
          ok = false;
        } else if (dec == 1) {
          // The tile's last item in this CTA's range and nothing after it: the
          // pipeline's shared memory is idle (the MMAs behind acc_full have
          // consumed every stage), so the partial slots come in by bulk copies,
          // one lane per slot, and are summed from smem.
          uint32_t cur2 = cur;
          Item nxt;
          const bool more = next_item(p, cur2, nxt);
          const uint32_t slot_bytes = (uint32_t)(slot_elems * sizeof(float));
          if (!more && (size_t)it.nseg * slot_bytes <= (size_t)S * C::kStageBytes) {
            if (warp == 2) {
              fence_proxy_async_global();  // the slots were stored by other CTAs' generic stores
              if (lane == 0) mbar_arrive_expect_tx(pull_bar, (uint32_t)it.nseg * slot_bytes);
              __syncwarp();
              if (lane < it.nseg)
                bulk_load(sA + (uint32_t)lane * slot_bytes,
                          reinterpret_cast<const uint8_t *>(tile_ws + (size_t)lane * slot_elems), slot_bytes,
                          pull_bar, policy_evict_first());
            }
            ok = warp_wait(pull_bar, 0, ctl);
            if (ok) {
              const int tid = threadIdx.x - 64;
              const int ngrp = ncols * (kTileA / 4);
              const int row0 = it.ta * kTileA;
              for (int g = tid; g < ngrp; g += 128) {
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int sgi = 0; sgi < it.nseg; ++sgi) {
                  const uint32_t a = sA + (uint32_t)sgi * slot_bytes + (uint32_t)g * 16u;
                  const uint4 u = ld_shared_v4(a);
                  acc.x += __uint_as_float(u.x);
                  acc.y += __uint_as_float(u.y);
                  acc.z += __uint_as_float(u.z);
                  acc.w += __uint_as_float(u.w);
                }
                const int c = g / (kTileA / 4);
                const int r = (g % (kTileA / 4)) * 4;
                const int m = cb0 + c;    // token
                const int n = row0 + r;   // output channel
                float f[4] = {acc.x, acc.y, acc.z, acc.w};
                if (KIND == 1) {
                  const float sa = p.tok_scale[m];
#pragma unroll
                  for (int j = 0; j < 4; ++j) f[j] = (f[j] * sa) * p.chan_scale[n + j];
                }
                if (p.out_f32)
                  *reinterpret_cast<float4 *>(reinterpret_cast<float *>(p.y) + (size_t)m * p.ldy + n) =
                      make_float4(f[0], f[1], f[2], f[3]);
                else
                  *reinterpret_cast<uint2 *>(reinterpret_cast<uint16_t *>(p.y) + (size_t)m * p.ldy + n) =
                      make_uint2(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]));
              }
            }
          } else {
            reduce_partials<KIND>(p, tile_ws, slot_elems, it.nseg, ncols, it.ta * kTileA, cb0,
                                  threadIdx.x - 64);
          }
          if (threadIdx.x == 64) trace_mark(p, kTrReduced);
        }
      }
      if (!released) release_acc();
      if (threadIdx.x == 64 && i < 2) trace_mark(p, i == 0 ? kTrItem0Done : kTrItem1Done);
      if (!ok) break;
      ++i;
    }
    if (KS == 1 && p.y_tma && lane == 0) bulk_wait_group_all();  // y stores complete
    if (threadIdx.x == 64) {
      trace_mark(p, kTrEpiDone);
      trace_set(p, kTrItems, (unsigned long long)i);
    }
    if (p.grid_reduce) {
      // every CTA's partial slots are stored: sum a share of all of them
      named_barrier(1, 128);
      if (threadIdx.x == 64) {
        *reduce_go = (!*abort_flag && grid_barrier(p.gbar + 64, p.gbar + 96, gridDim.x, ctl)) ? 1 : 0;
        trace_mark(p, kTrDecision);
      }
      named_barrier(1, 128);
      if (*reduce_go) {
        reduce_share<KIND>(p, BN, gridDim.x, blockIdx.x * 128 + (threadIdx.x - 64), gridDim.x * 128);
        if (threadIdx.x == 64) trace_mark(p, kTrReduced);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) {
    trace_mark(p, kTrExit);
    trace_set(p, kTrExitNs, global_timer_ns());
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// The split-K reduction as its own kernel, launched right after the GEMM.
template <int KIND>
__global__ void __maxnreg__(48)  // 128-thread CTAs, 3 of them beside a GEMM CTA and a quantizer CTA
    splitk_reduce_kernel(const GemmParams p, int bn, unsigned gemm_ctas) {
  pdl_trigger();  // touches nothing before the wait below
  if (p.trace && threadIdx.x == 0)
    atomicMax(p.trace + kTrRedEntryInv, ~(unsigned long long)global_timer_ns());
  pdl_wait();     // the GEMM that wrote the partial slots has completed
  reduce_share<KIND>(p, bn, gemm_ctas, blockIdx.x * blockDim.x + threadIdx.x, gridDim.x * blockDim.x);
  if (p.trace) {  // (uniform over the grid)
    __syncthreads();
    if (threadIdx.x == 0) atomicMax(p.trace + kTrRedExitNs, (unsigned long long)global_timer_ns());
  }
}

template <int KIND, int BN, int KS>
cudaError_t launch_t(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmY,
                     const GemmParams &p, int ctas, cudaStream_t stream) {
  using C = Cfg<KIND, BN, KS>;
  auto kern = gemm_kernel<KIND, BN, KS>;
  static DeviceOnce once;  // per instantiation and device (a repeat sets the same value)
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (!once.done(dev)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem);
    if (e != cudaSuccess) return e;
    once.set(dev);
  }
  cudaLaunchConfig_t cfg = pdl_config(dim3(ctas), dim3(kThreads), C::kSmem, stream);
  cudaLaunchAttribute attr[3];
  attach_pdl(cfg, attr);
  if (p.pair_reduce) {
    // CTA pairs (2j, 2j + 1) share a tile and exchange partials through
    // distributed shared memory
    if (ctas % 2 != 0) return cudaErrorInvalidValue;
    attr[cfg.numAttrs].id = cudaLaunchAttributeClusterDimension;
    attr[cfg.numAttrs].val.clusterDim.x = 2;
    attr[cfg.numAttrs].val.clusterDim.y = 1;
    attr[cfg.numAttrs].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs += 1;
  }
  if (p.fuse_quant || p.grid_reduce) {
    // grid barriers: every CTA must be resident at once, also when other
    // streams run kernels of their own (a cooperative launch guarantees it)
    if (cooperative_enabled()) {
      attr[cfg.numAttrs].id = cudaLaunchAttributeCooperative;
      attr[cfg.numAttrs].val.cooperative = 1;
      cfg.attrs = attr;
      cfg.numAttrs += 1;
    }
  }
  return cudaLaunchKernelEx(&cfg, kern, tmA, tmB, tmY, p);
}

// Full-tile kernels (BN = 256) take one K column per stage; split-K kernels two.
template <int KIND>
cudaError_t launch_kind(int bn, const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmY,
                        const GemmParams &p, int ctas, cudaStream_t stream) {
  if (!p.splitk)
    return bn == 256 ? launch_t<KIND, 256, 1>(tmA, tmB, tmY, p, ctas, stream) : cudaErrorInvalidValue;
  switch (bn) {
    case 16: return launch_t<KIND, 16, 2>(tmA, tmB, tmY, p, ctas, stream);
    case 32: return launch_t<KIND, 32, 2>(tmA, tmB, tmY, p, ctas, stream);
    case 64: return launch_t<KIND, 64, 2>(tmA, tmB, tmY, p, ctas, stream);
    case 128: return launch_t<KIND, 128, 2>(tmA, tmB, tmY, p, ctas, stream);
    case 256: return launch_t<KIND, 256, 2>(tmA, tmB, tmY, p, ctas, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <int KIND>
int stages_kind(int bn, bool splitk) {
  if (!splitk) return bn == 256 ? Cfg<KIND, 256, 1>::kStages : 0;
  switch (bn) {
    case 16: return Cfg<KIND, 16, 2>::kStages;
    case 32: return Cfg<KIND, 32, 2>::kStages;
    case 64: return Cfg<KIND, 64, 2>::kStages;
    case 128: return Cfg<KIND, 128, 2>::kStages;
    case 256: return Cfg<KIND, 256, 2>::kStages;
    default: return 0;
  }
}

template <int KIND>
size_t smem_kind(int bn, bool splitk) {
  if (!splitk) return bn == 256 ? Cfg<KIND, 256, 1>::kSmem : 0;
  switch (bn) {
    case 16: return Cfg<KIND, 16, 2>::kSmem;
    case 32: return Cfg<KIND, 32, 2>::kSmem;
    case 64: return Cfg<KIND, 64, 2>::kSmem;
    case 128: return Cfg<KIND, 128, 2>::kSmem;
    case 256: return Cfg<KIND, 256, 2>::kSmem;
    default: return 0;
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
  const long long total = (long long)p.tilesA * p.tilesB * bn * (kTileA / 4);
  long long blocks = (total + kRedThreads * kRedJ - 1) / (kRedThreads * kRedJ);
  // Launched early (programmatic launch), the reduce CTAs sit beside the
  // GEMM CTAs of a layer chain: 3 per SM at most (48 registers a thread),
  // so that a GEMM CTA (26K registers) and a quantizer CTA still fit.
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

int gemm_stages(int kind, int bn, bool splitk) {
  return kind == 0 ? stages_kind<0>(bn, splitk) : stages_kind<1>(bn, splitk);
}

size_t gemm_smem_bytes(int kind, int bn, bool splitk) {
  return kind == 0 ? smem_kind<0>(bn, splitk) : smem_kind<1>(bn, splitk);
}

int gemm_cols_per_stage(bool splitk) { return splitk ? 2 : 1; }

}  // namespace mxg
