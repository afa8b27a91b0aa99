// api.cu -- the C ABI declared in include/mxgemm.h: argument checks, device
// checks, the dispatcher, TMA tensor-map encoding and kernel launches.
// Every host-detectable error is returned before anything is launched.
#include <algorithm>
#include <cudaTypedefs.h>
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "kernels.h"
#include "mxgemm.h"

namespace {

constexpr int kMaxDevices = 64;
// Workspace layout: the quantized activations of the fused A4W4 path (when
// the call quantizes x itself), then the split-K partial tiles.  Nothing in
// it needs to start at any particular value.

struct DevInfo {
  bool init = false;
  int major = 0, minor = 0, sm_count = 0;
};
std::mutex g_mu;
DevInfo g_dev[kMaxDevices];

// Current device must be compute capability 10.3; returns its SM count.
mxg_status check_device(int *sm_count) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MXG_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MXG_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lk(g_mu);
  DevInfo &d = g_dev[dev];
  if (!d.init) {
    if (cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return MXG_ERR_CUDA;
    d.init = true;
  }
  if (d.major != 10 || d.minor != 3) return MXG_ERR_UNSUPPORTED_DEVICE;
  if (sm_count) *sm_count = d.sm_count;
  return MXG_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D byte matrix (rows x row_bytes, contiguous) read in boxes of 128 bytes x
// box_rows rows with the 128-byte swizzle; rows past the end read as zero.
mxg_status make_operand_map(CUtensorMap *m, const void *ptr, uint64_t row_bytes, uint64_t rows,
                            uint32_t box_rows) {
  auto enc = tensor_map_encoder();
  if (!enc) return MXG_ERR_CUDA;
  cuuint64_t dims[2] = {row_bytes, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {128u, box_rows};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(ptr), dims, strides, box,
                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MXG_OK : MXG_ERR_CUDA;
}

// y (M rows of N bf16, leading dimension ldy) for the full-tile epilogue's
// TMA stores: 32 x 32 boxes, no swizzle; out-of-bounds elements are skipped.
mxg_status make_output_map(CUtensorMap *m, void *y, int M, int N, int ldy) {
  auto enc = tensor_map_encoder();
  if (!enc) return MXG_ERR_CUDA;
  cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)M};
  cuuint64_t strides[1] = {(cuuint64_t)ldy * 2u};
  cuuint32_t box[2] = {32u, 32u};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, y, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MXG_OK : MXG_ERR_CUDA;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t align256(size_t x) { return (x + 255u) & ~static_cast<size_t>(255u); }

// Full-tile rasterization: operands above kL2KeepBytes (together) do not stay
// in the 129 MB L2 across a wave of tiles, so the tiles go in bands of token
// tiles.  Each die's half of the L2 caches what that die's SMs read, and the
// SMs of both dies read every token tile of a band: a band's activations are
// held twice, so one copy of them takes at most kL2ActBudget.
constexpr uint64_t kL2KeepBytes = 96ull << 20;
constexpr uint64_t kL2ActBudget = 32ull << 20;

// The split-K reduce kernel chained behind a GEMM, in K-stages of one CTA's
// time (see plan_impl).
constexpr long long kReduceStages = 7;

// CTA that owns stream-K unit u (must equal the device-side owner_of).
long long owner_of(long long u, long long U, long long G) { return ((u + 1) * G - 1) / U; }

mxg_status plan_impl(int kind, int M, int N, int K, int sm_count, const mxg_gemm_opts *opts,
                     mxg_plan *pl) {
  if (!pl || (kind != 0 && kind != 1) || M < 1 || N < 1 || K < 1 || sm_count < 1)
    return MXG_ERR_INVALID_ARG;
  if (K % 128 != 0 || N % 128 != 0) return MXG_ERR_UNSUPPORTED_SHAPE;
  int variant = opts ? opts->variant : MXG_VARIANT_AUTO;
  if (variant < MXG_VARIANT_AUTO || variant > MXG_VARIANT_SPLITK) return MXG_ERR_INVALID_ARG;
  // pipeline stages along K: 128-byte K columns (256 E2M1 / 128 E4M3
  // values), one per stage in the full-tile kernel, two in the split-K one
  const int kcol = kind == 0 ? 256 : 128;
  const int KC = (K + kcol - 1) / kcol;
  if (variant == MXG_VARIANT_AUTO) {
    // Measured on GB300 (quantizer + GEMM, o_proj / FP8 gate_up / FP8 down):
    // a full wave of 128 x 256 tiles streams the weights as fast as split-K
    // and needs no reduction; below a wave, split-K wins for M <= 128, and
    // up to M = 256 when K is long (a few long tiles leave SMs idle), while
    // split-K with 256-token tiles (two pipeline stages) loses beyond that.
    const long long full_tiles = (long long)((M + 127) / 128) * ((N + 255) / 256);
    if (10 * full_tiles >= 9LL * sm_count)
      variant = MXG_VARIANT_FULL;
    else if (M <= 128 || (M <= 256 && KC > 64))
      variant = MXG_VARIANT_SPLITK;
    else
      variant = MXG_VARIANT_FULL;
  }
  const int per = mxg::gemm_cols_per_stage(variant == MXG_VARIANT_SPLITK);
  const int KB = (KC + per - 1) / per;
  std::memset(pl, 0, sizeof(*pl));
  pl->variant = variant;
  pl->kblocks = KB;
  pl->bm = 128;
  if (variant == MXG_VARIANT_FULL) {
    pl->bn = 256;
    const long long tA = (M + 127) / 128, tB = (N + 255) / 256;
    if (tA * tB + sm_count >= (1LL << 31)) return MXG_ERR_UNSUPPORTED_SHAPE;
    if (opts && opts->cta_pair && tA >= 2 && sm_count >= 2) {
      // on request, with two token tiles or more: CTA pairs with 2-SM MMAs
      // over 256 x 256 tiles, one pair per two SMs
      const long long tiles = ((tA + 1) / 2) * tB;
      const long long pairs = sm_count / 2;
      pl->bm = 256;
      pl->cta_pair = 1;
      pl->tiles = (int)tiles;
      pl->ctas = (int)(2 * (tiles < pairs ? tiles : pairs));
    } else {
      const long long tiles = tA * tB;
      pl->tiles = (int)tiles;
      pl->ctas = (int)(tiles < sm_count ? tiles : sm_count);
    }
    pl->seg_max = 1;
    pl->ws_bytes = 0;
  } else {
    pl->bn = M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : M <= 128 ? 128 : 256;
    const long long tilesA = N / 128, tilesB = (M + pl->bn - 1) / pl->bn;
    const long long tiles = tilesA * tilesB;
    const long long U = tiles * KB;
    if (U > (1LL << 40) / 4) return MXG_ERR_UNSUPPORTED_SHAPE;
    // persistent: at most one CTA per SM
    const bool fixed = opts && opts->ctas > 0;
    long long G = (fixed && opts->ctas < sm_count) ? opts->ctas : sm_count;
    if (G > U) G = U;
    auto segments = [&](long long g) {  // most CTAs that share one tile
      int sm_ = 1;
      for (long long t = 0; t < tiles; ++t) {
        const long long n = owner_of(t * KB + KB - 1, U, g) - owner_of(t * KB, U, g) + 1;
        if (n > sm_) sm_ = (int)n;
      }
      return sm_;
    };
    int seg_max = segments(G);
    // Without a CTA count from the caller: whole tiles (one CTA a tile, no
    // partial sums, no reduce kernel) when they fit in one wave and cost no
    // more than stream-K does.  Measured on GB300, a CTA's time grows by about
    // one unit per K-stage it takes (~0.5 us) and the reduce kernel chained
    // behind the GEMM costs about kReduceStages of them (~3.5 us).
    if (!fixed && tiles <= sm_count && seg_max > 1 && KB <= (U + G - 1) / G + kReduceStages) {
      G = tiles;
      seg_max = 1;
    }
    // the kernel walks its stream-K range in 32-bit arithmetic
    if ((U + 1) * G >= (1LL << 32)) return MXG_ERR_UNSUPPORTED_SHAPE;
    pl->tiles = (int)tiles;
    pl->ctas = (int)G;
    pl->seg_max = seg_max;
    pl->ws_bytes = seg_max > 1 ? (size_t)tiles * seg_max * pl->bn * 128 * sizeof(float) : 0;
  }
  return MXG_OK;
}

mxg_status check_rows_arg(const void *x, int rows, int K, int ld) {
  if (!x || rows < 1 || K < 1 || ld < K) return MXG_ERR_INVALID_ARG;
  if (K % 128 != 0) return MXG_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(x) || (ld % 8) != 0) return MXG_ERR_MISALIGNED;
  return MXG_OK;
}

// Bytes of activation codes (row bytes `row_bytes`) for M rows, row-major
// (tile_rows == 0) or in tiles of tile_rows rows (the last tile padded).
size_t act_code_bytes(int M, size_t row_bytes, int tile_rows) {
  const size_t rows = tile_rows ? (size_t)((M + tile_rows - 1) / tile_rows) * tile_rows : (size_t)M;
  return rows * row_bytes;
}

// Token-tile height of the activation codes a plan reads as tiles: the MMA-N
// tile in the split-K variant (tokens are the MMA-B operand), 128 otherwise.
int plan_act_tile_rows(const mxg_plan &pl) {
  return pl.variant == MXG_VARIANT_SPLITK ? pl.bn : 128;
}

// Workspace bytes of the fused path's quantized activations (codes in tiles
// of tile_rows rows, then the 128x4-tile scales).
size_t fused_act_bytes(int M, int K, int tile_rows) {
  return align256(act_code_bytes(M, (size_t)K / 2, tile_rows)) +
         align256(mxg_sf_bytes(M, K, MXG_SF_SWIZZLED));
}

bool valid_tile_rows(int t) { return t == 16 || t == 32 || t == 64 || t == 128 || t == 256; }

struct GemmOperands {
  const uint8_t *a, *a_sf, *w, *w_sf;  // codes (A4W4) or E4M3 bytes (PTPC)
  const float *sa, *sw;                // PTPC scales
};

// ws: the caller's workspace base; part_off: where the partial tiles start
// (after the quantized activations on the fused path).
// act_tile_rows: 0 = activations row-major, else in the tile layout with
// tiles of that many rows (must match the plan: plan_act_tile_rows).
mxg_status run_gemm(int kind, const GemmOperands &op, int M, int N, int K, void *y, int ldy,
                    mxg_out_dtype out_dtype, const mxg_gemm_opts *opts, void *ws, size_t ws_bytes,
                    size_t part_off, int act_tile_rows, int sm_count,
                    cudaStream_t stream) {
  mxg_plan pl;
  mxg_status st = plan_impl(kind, M, N, K, sm_count, opts, &pl);
  if (st != MXG_OK) return st;
  if (pl.ws_bytes > 0) {
    if (!ws || ws_bytes < part_off + pl.ws_bytes) return MXG_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MXG_ERR_MISALIGNED;
  }

  const bool swap = pl.variant == MXG_VARIANT_SPLITK;
  const uint64_t row_bytes = kind == 0 ? (uint64_t)K / 2 : (uint64_t)K;
  const bool w_tiled = opts && opts->weights_tiled;
  const bool w_panels = opts && opts->weights_tiled == 2;
  if (opts && (opts->weights_tiled < 0 || opts->weights_tiled > 2)) return MXG_ERR_INVALID_ARG;
  if (w_tiled && (row_bytes % 128 != 0 || N % 128 != 0)) return MXG_ERR_UNSUPPORTED_SHAPE;
  // a full-tile GEMM takes a whole 256-row panel as its B tile
  if (w_panels && !swap && pl.bn != mxg::kPanelRows) return MXG_ERR_UNSUPPORTED_SHAPE;
  if (act_tile_rows && act_tile_rows != plan_act_tile_rows(pl)) return MXG_ERR_INVALID_ARG;
  if (act_tile_rows && row_bytes % 128 != 0) return MXG_ERR_UNSUPPORTED_SHAPE;
  CUtensorMap tmA, tmB, tmY;
  std::memset(&tmY, 0, sizeof(tmY));
  const uint8_t *A = swap ? op.w : op.a;
  const uint8_t *B = swap ? op.a : op.w;
  const int rowsA = swap ? N : M, rowsB = swap ? M : N;
  if ((st = make_operand_map(&tmA, A, row_bytes, rowsA, 128)) != MXG_OK) return st;
  // (a CTA pair's CTA holds 128 rows of the BN-row weight tile)
  if ((st = make_operand_map(&tmB, B, row_bytes, rowsB, (uint32_t)(pl.cta_pair ? 128 : pl.bn))) != MXG_OK)
    return st;

  mxg::GemmParams p;
  std::memset(&p, 0, sizeof(p));
  p.sfA = swap ? op.w_sf : op.a_sf;
  p.sfB = swap ? op.a_sf : op.w_sf;
  p.tok_scale = op.sa;
  p.chan_scale = op.sw;
  p.y = y;
  p.ldy = ldy;
  p.out_f32 = out_dtype == MXG_OUT_F32 ? 1 : 0;
  if (!swap && !p.out_f32 && (reinterpret_cast<uintptr_t>(y) & 15u) == 0 && (ldy % 8) == 0) {
    if ((st = make_output_map(&tmY, y, M, N, ldy)) != MXG_OK) return st;
    p.y_tma = 1;
  }
  p.M = M;
  p.N = N;
  p.K = K;
  p.swap = swap ? 1 : 0;
  p.rowsA = rowsA;
  p.rowsB = rowsB;
  p.tilesA = (rowsA + 127) / 128;
  p.tilesB = (rowsB + pl.bn - 1) / pl.bn;
  p.kblocks = pl.kblocks;
  p.G4 = K / 128;
  p.splitk = swap ? 1 : 0;
  p.cta_pair = pl.cta_pair;
  p.units = (long long)p.tilesA * p.tilesB * p.kblocks;
  if (pl.ws_bytes > 0) p.ws = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + part_off);
  p.seg_max = pl.seg_max;
  p.status = opts ? opts->dev_status : nullptr;
  const uint32_t tmo = (opts && opts->timeout_ms) ? opts->timeout_ms : 1000u;
  p.timeout_ns = (unsigned long long)tmo * 1000000ull;
  p.debug_stall = (opts && opts->debug_stall == 1) ? 1 : 0;
  p.early_w = (opts && opts->weights_static) ? 1 : 0;

  p.trace = opts ? static_cast<unsigned long long *>(opts->trace) : nullptr;
  p.kc_per_row = (int)((row_bytes + 127) / 128);  // the last column may be half (TMA pads it)
  if (!swap) {
    // Full tile: when the two operands together exceed what L2 keeps
    // (129 MB), walk the tiles in bands of token tiles (as few bands as keep
    // each band's activations within kL2ActBudget, of equal size), so that
    // every weight tile is read from HBM once per band (in row order every
    // wave of CTAs would sweep all the weights).
    const uint64_t a_tile = 128ull * (row_bytes + (kind == 0 ? row_bytes / 16 : 0));
    const uint64_t total = (uint64_t)(rowsA + rowsB) * row_bytes;
    if (total > kL2KeepBytes) {
      const uint64_t tiles = (uint64_t)p.tilesA;
      const uint64_t bands = std::max<uint64_t>(1, (tiles * a_tile + kL2ActBudget - 1) / kL2ActBudget);
      p.raster_group = (int)((tiles + bands - 1) / bands);
    }
  }
  // operands in the tile layout are fetched by bulk copy (their tensor map
  // above is then unused)
  if (w_tiled) {
    if (swap) {
      p.a_tiles = op.w;
    } else {
      p.b_tiles = op.w;
      p.b_tile_rows = w_panels ? mxg::kPanelRows : 128;
    }
    p.w_panels = w_panels ? 1 : 0;
  }
  if (act_tile_rows) {
    if (swap) {
      p.b_tiles = op.a;
      p.b_tile_rows = act_tile_rows;
    } else {
      p.a_tiles = op.a;
    }
  }
  cudaError_t e = mxg::launch_gemm(kind, pl.bn, tmA, tmB, tmY, p, pl.ctas, stream);
  if (e == cudaSuccess && swap && pl.seg_max > 1)
    e = mxg::launch_splitk_reduce(kind, pl.bn, p, pl.ctas, sm_count, stream);
  return e == cudaSuccess ? MXG_OK : MXG_ERR_CUDA;
}

mxg_status check_gemm_common(int M, int N, int K, const void *y, int ldy, mxg_out_dtype od,
                             const mxg_gemm_opts *opts) {
  if (M < 1 || N < 1 || K < 1 || !y || ldy < N) return MXG_ERR_INVALID_ARG;
  if (od != MXG_OUT_BF16 && od != MXG_OUT_F32) return MXG_ERR_INVALID_ARG;
  if (K % 128 != 0 || N % 128 != 0) return MXG_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(y) || ((size_t)ldy * (od == MXG_OUT_F32 ? 4 : 2)) % 16 != 0)
    return MXG_ERR_MISALIGNED;
  if (opts && (opts->variant < 0 || opts->variant > 2 || opts->ctas < 0))
    return MXG_ERR_INVALID_ARG;
  if (opts && opts->splitk_reduce != MXG_REDUCE_DEFAULT && opts->splitk_reduce != MXG_REDUCE_KERNEL)
    return MXG_ERR_INVALID_ARG;
  if (opts && (opts->weights_tiled < 0 || opts->weights_tiled > 2)) return MXG_ERR_INVALID_ARG;
  if (opts && (opts->cta_pair < 0 || opts->cta_pair > 1)) return MXG_ERR_INVALID_ARG;
  if (opts && opts->act_tile_rows && !valid_tile_rows(opts->act_tile_rows))
    return MXG_ERR_INVALID_ARG;
  return MXG_OK;
}

}  // namespace

extern "C" {

size_t mxg_sf_bytes(int rows, int K, mxg_sf_layout layout) {
  if (rows < 1 || K < 32) return 0;
  const size_t G = (size_t)K / 32;
  if (layout == MXG_PANEL) return 0;  // the scales live inside the panels
  if (layout == MXG_SF_SWIZZLED || layout == MXG_TILED) return (size_t)((rows + 127) / 128) * 128u * G;
  return (size_t)rows * G;
}

size_t mxg_weight_bytes(int kind, int N, int K, mxg_sf_layout layout) {
  if ((kind != 0 && kind != 1) || N < 1 || K < 1) return 0;
  const size_t row_bytes = kind == 0 ? (size_t)K / 2 : (size_t)K;
  if (layout == MXG_PANEL) {
    if (row_bytes % 128 != 0) return 0;
    return (size_t)((N + mxg::kPanelRows - 1) / mxg::kPanelRows) * (row_bytes / 128) *
           (size_t)(kind == 0 ? mxg::kMxPanelBytes : mxg::kF8PanelBytes);
  }
  if (layout == MXG_SF_ROWMAJOR || layout == MXG_SF_SWIZZLED || layout == MXG_TILED)
    return (size_t)N * row_bytes;
  return 0;
}

mxg_status mxg_plan_gemm(int kind, int M, int N, int K, int sm_count, const mxg_gemm_opts *opts,
                         mxg_plan *plan) {
  return plan_impl(kind, M, N, K, sm_count, opts, plan);
}

size_t mxg_gemm_workspace_bytes(int kind, int fused, int M, int N, int K,
                                const mxg_gemm_opts *opts) {
  int sm = 0;
  if (check_device(&sm) != MXG_OK) return 0;
  mxg_plan pl;
  if (plan_impl(kind, M, N, K, sm, opts, &pl) != MXG_OK) return 0;
  const size_t act = (kind == 0 && fused) ? fused_act_bytes(M, K, plan_act_tile_rows(pl)) : 0;
  return act + pl.ws_bytes;
}

namespace {
mxg_status mx_quantize_rows(const void *w_bf16, int N, int K, int ldw, uint8_t *codes, uint8_t *sf,
                            mxg_sf_layout layout, bool act, mxg_stream_t stream) {
  mxg_status st = check_rows_arg(w_bf16, N, K, ldw);
  if (st != MXG_OK) return st;
  const bool panel = layout == MXG_PANEL;
  if (!codes || (!sf && !panel) ||
      (layout != MXG_SF_ROWMAJOR && layout != MXG_SF_SWIZZLED && layout != MXG_TILED && !panel))
    return MXG_ERR_INVALID_ARG;
  if (layout == MXG_TILED && (N % 128 != 0 || K % 256 != 0)) return MXG_ERR_UNSUPPORTED_SHAPE;
  if (panel && K % 256 != 0) return MXG_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(codes) || (!panel && !aligned16(sf))) return MXG_ERR_MISALIGNED;
  int sm = 0;
  if ((st = check_device(&sm)) != MXG_OK) return st;
  cudaError_t e = mxg::launch_mx_quant(w_bf16, ldw, N, K, codes, sf, layout != MXG_SF_ROWMAJOR,
                                       panel                 ? mxg::kPanelLayout
                                       : layout == MXG_TILED ? 128
                                                             : 0,
                                       act, sm, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MXG_OK : MXG_ERR_CUDA;
}
}  // namespace

mxg_status mx_quantize_weight(const void *w_bf16, int N, int K, int ldw, uint8_t *codes,
                              uint8_t *sf, mxg_sf_layout layout, mxg_stream_t stream) {
  return mx_quantize_rows(w_bf16, N, K, ldw, codes, sf, layout, false, stream);
}

mxg_status mx_quantize_act(const void *x_bf16, int M, int K, int ldx, uint8_t *codes, uint8_t *sf,
                           mxg_stream_t stream) {
  return mx_quantize_rows(x_bf16, M, K, ldx, codes, sf, MXG_SF_SWIZZLED, true, stream);
}

mxg_status fp8_quantize_act(const void *x_bf16, int M, int K, int ldx, uint8_t *q, float *scale,
                            mxg_stream_t stream) {
  mxg_status st = check_rows_arg(x_bf16, M, K, ldx);
  if (st != MXG_OK) return st;
  if (!q || !scale) return MXG_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(scale)) return MXG_ERR_MISALIGNED;
  int sm = 0;
  if ((st = check_device(&sm)) != MXG_OK) return st;
  cudaError_t e = mxg::launch_fp8_quant(x_bf16, ldx, M, K, q, scale, 0, true, sm,
                                        reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MXG_OK : MXG_ERR_CUDA;
}

size_t mxg_act_tiled_bytes(int kind, int M, int K, int tile_rows) {
  if ((kind != 0 && kind != 1) || M < 1 || K < 1 || !valid_tile_rows(tile_rows)) return 0;
  return act_code_bytes(M, kind == 0 ? (size_t)K / 2 : (size_t)K, tile_rows);
}

mxg_status mx_quantize_act_tiled(const void *x_bf16, int M, int K, int ldx, int tile_rows,
                                 uint8_t *codes, uint8_t *sf, mxg_stream_t stream) {
  mxg_status st = check_rows_arg(x_bf16, M, K, ldx);
  if (st != MXG_OK) return st;
  if (!codes || !sf || !valid_tile_rows(tile_rows)) return MXG_ERR_INVALID_ARG;
  if (K % 256 != 0) return MXG_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(codes) || !aligned16(sf)) return MXG_ERR_MISALIGNED;
  int sm = 0;
  if ((st = check_device(&sm)) != MXG_OK) return st;
  cudaError_t e = mxg::launch_mx_quant(x_bf16, ldx, M, K, codes, sf, true, tile_rows, true, sm,
                                       reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MXG_OK : MXG_ERR_CUDA;
}

mxg_status fp8_quantize_act_tiled(const void *x_bf16, int M, int K, int ldx, int tile_rows,
                                  uint8_t *q, float *scale, mxg_stream_t stream) {
  mxg_status st = check_rows_arg(x_bf16, M, K, ldx);
  if (st != MXG_OK) return st;
  if (!q || !scale || !valid_tile_rows(tile_rows)) return MXG_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(scale)) return MXG_ERR_MISALIGNED;
  int sm = 0;
  if ((st = check_device(&sm)) != MXG_OK) return st;
  cudaError_t e = mxg::launch_fp8_quant(x_bf16, ldx, M, K, q, scale, tile_rows, true, sm,
                                        reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MXG_OK : MXG_ERR_CUDA;
}

mxg_status swiglu_fp8_quantize(const void *gu_bf16, int M, int I, int ldgu, int tile_rows, uint8_t *q,
                               float *scale, void *h_bf16, int ldh, mxg_stream_t stream) {
  if (!gu_bf16 || M < 1 || I < 1 || ldgu < 2 * I || !q || !scale) return MXG_ERR_INVALID_ARG;
  if (tile_rows != 0 && !valid_tile_rows(tile_rows)) return MXG_ERR_INVALID_ARG;
  if (h_bf16 && ldh < I) return MXG_ERR_INVALID_ARG;
  if (I % 128 != 0 || I > mxg::kSwigluMaxI) return MXG_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(gu_bf16) || (ldgu % 8) != 0 || !aligned16(q) || !aligned16(scale) ||
      (h_bf16 && (!aligned16(h_bf16) || (ldh % 8) != 0)))
    return MXG_ERR_MISALIGNED;
  int sm = 0;
  mxg_status st = check_device(&sm);
  if (st != MXG_OK) return st;
  cudaError_t e = mxg::launch_swiglu_fp8(gu_bf16, ldgu, M, I, tile_rows, h_bf16, ldh, q, scale, sm,
                                         reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MXG_OK : MXG_ERR_CUDA;
}

mxg_status fp8_quantize_weight(const void *w_bf16, int N, int K, int ldw, uint8_t *q, float *scale,
                               mxg_sf_layout layout, mxg_stream_t stream) {
  mxg_status st = check_rows_arg(w_bf16, N, K, ldw);
  if (st != MXG_OK) return st;
  if (!q || !scale || (layout != MXG_SF_ROWMAJOR && layout != MXG_TILED && layout != MXG_PANEL))
    return MXG_ERR_INVALID_ARG;
  if (layout == MXG_TILED && N % 128 != 0) return MXG_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(q) || !aligned16(scale)) return MXG_ERR_MISALIGNED;
  int sm = 0;
  if ((st = check_device(&sm)) != MXG_OK) return st;
  const int tile_rows = layout == MXG_PANEL ? mxg::kPanelLayout : layout == MXG_TILED ? 128 : 0;
  cudaError_t e = mxg::launch_fp8_quant(w_bf16, ldw, N, K, q, scale, tile_rows, false, sm,
                                        reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MXG_OK : MXG_ERR_CUDA;
}

namespace {
// The operand checks of mx_gemm_a4w4 (everything it can reject on the host
// before touching the device).
mxg_status check_a4w4_args(const uint8_t *a_codes, const uint8_t *a_sf, const void *x_bf16, int ldx,
                           const uint8_t *w_codes, const uint8_t *w_sf, int M, int N, int K,
                           const void *y, int ldy, mxg_out_dtype out_dtype, const mxg_gemm_opts *opts) {
  mxg_status st = check_gemm_common(M, N, K, y, ldy, out_dtype, opts);
  if (st != MXG_OK) return st;
  // weight panels carry their scales; w_sf is then unused (may be NULL)
  const bool w_panels = opts && opts->weights_tiled == 2;
  if (!w_codes || (!w_sf && !w_panels)) return MXG_ERR_INVALID_ARG;
  if (a_codes == nullptr) {
    if (!x_bf16 || a_sf) return MXG_ERR_INVALID_ARG;
    if ((st = check_rows_arg(x_bf16, M, K, ldx)) != MXG_OK) return st;
  } else if (!a_sf) {
    return MXG_ERR_INVALID_ARG;
  }
  if (!aligned16(w_codes) || (w_sf && !aligned16(w_sf)) || (a_codes && (!aligned16(a_codes) || !aligned16(a_sf))))
    return MXG_ERR_MISALIGNED;
  return MXG_OK;
}
}  // namespace

mxg_status mx_gemm_a4w4(const uint8_t *a_codes, const uint8_t *a_sf, const void *x_bf16, int ldx,
                        const uint8_t *w_codes, const uint8_t *w_sf, int M, int N, int K, void *y,
                        int ldy, mxg_out_dtype out_dtype, const mxg_gemm_opts *opts,
                        mxg_stream_t stream) {
  mxg_status st = check_a4w4_args(a_codes, a_sf, x_bf16, ldx, w_codes, w_sf, M, N, K, y, ldy, out_dtype, opts);
  if (st != MXG_OK) return st;
  const bool fused = a_codes == nullptr;
  int sm = 0;
  if ((st = check_device(&sm)) != MXG_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t *ws = opts ? static_cast<uint8_t *>(opts->workspace) : nullptr;
  size_t ws_bytes = opts ? opts->ws_bytes : 0;
  size_t part_off = 0;
  int act_tile_rows = opts ? opts->act_tile_rows : 0;
  if (fused) {
    // plan first: the activations are quantized straight into the tile
    // layout the plan reads, and a too-small workspace is reported before
    // any launch
    mxg_plan pl;
    if ((st = plan_impl(0, M, N, K, sm, opts, &pl)) != MXG_OK) return st;
    act_tile_rows = K % 256 == 0 ? plan_act_tile_rows(pl) : 0;
    const size_t need = fused_act_bytes(M, K, act_tile_rows);
    if (!ws || ws_bytes < need + pl.ws_bytes) return MXG_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MXG_ERR_MISALIGNED;
    uint8_t *codes = ws;
    uint8_t *sf = codes + align256(act_code_bytes(M, (size_t)K / 2, act_tile_rows));
    a_codes = codes;
    a_sf = sf;
    part_off += need;
    mxg::QuantWatch watch;
    if (opts) {
      watch.status = opts->dev_status;
      watch.timeout_ns = (unsigned long long)(opts->timeout_ms ? opts->timeout_ms : 1000u) * 1000000ull;
      watch.debug_stall = opts->debug_stall == 2 ? 1 : 0;
    }
    cudaError_t e = mxg::launch_mx_quant(x_bf16, ldx, M, K, codes, sf, true, act_tile_rows, true, sm, s, watch);
    if (e != cudaSuccess) return MXG_ERR_CUDA;
  }
  GemmOperands op{a_codes, a_sf, w_codes, w_sf, nullptr, nullptr};
  return run_gemm(0, op, M, N, K, y, ldy, out_dtype, opts, ws, ws_bytes, part_off, act_tile_rows,
                  sm, s);
}

namespace {
// Grouped A4W4: a bound on the 128-row token tiles when each of E groups
// starts a new tile, and the workspace layout [tile offsets][codes][scales].
long long grouped_tiles(int M_total, int E) { return (long long)(M_total + 127) / 128 + E; }
struct GroupedWs {
  size_t tile_off, codes, sf, total;
};
GroupedWs grouped_ws(int M_total, int K, int E) {
  GroupedWs w;
  const size_t rows = (size_t)grouped_tiles(M_total, E) * 128;
  w.tile_off = 0;
  w.codes = align256((size_t)(E + 1) * sizeof(int));
  w.sf = w.codes + align256(rows * (size_t)K / 2);
  w.total = w.sf + align256(rows * (size_t)K / 32);
  return w;
}
}  // namespace

size_t mxg_grouped_workspace_bytes(int M_total, int K, int E) {
  if (M_total < 0 || K < 256 || E < 1 || E > mxg::kMaxGroups) return 0;
  return grouped_ws(M_total, K, E).total;
}

mxg_status mx_gemm_a4w4_grouped(const void *x_bf16, int ldx, const int *row_off, int E,
                                const uint8_t *w_panels, int M_total, int N, int K, void *y, int ldy,
                                mxg_out_dtype out_dtype, const mxg_gemm_opts *opts, mxg_stream_t stream) {
  // with no token routed, x and y may be empty (null) tensors
  if ((M_total > 0 && (!x_bf16 || !y)) || !row_off || !w_panels || E < 1 || E > mxg::kMaxGroups ||
      M_total < 0 || N < 1 || K < 1 || ldx < K || ldy < N)
    return MXG_ERR_INVALID_ARG;
  if (out_dtype != MXG_OUT_BF16 && out_dtype != MXG_OUT_F32) return MXG_ERR_INVALID_ARG;
  if (opts && ((opts->variant != MXG_VARIANT_AUTO && opts->variant != MXG_VARIANT_FULL) ||
               (opts->weights_tiled != 0 && opts->weights_tiled != 2) || opts->act_tile_rows != 0 ||
               (opts->splitk_reduce != MXG_REDUCE_DEFAULT && opts->splitk_reduce != MXG_REDUCE_KERNEL) ||
               opts->cta_pair != 0))
    return MXG_ERR_INVALID_ARG;
  if (K % 256 != 0 || N % 128 != 0) return MXG_ERR_UNSUPPORTED_SHAPE;
  if ((x_bf16 && !aligned16(x_bf16)) || (ldx % 8) != 0 || !aligned16(w_panels) || (y && !aligned16(y)) ||
      ((size_t)ldy * (out_dtype == MXG_OUT_F32 ? 4 : 2)) % 16 != 0 || (reinterpret_cast<uintptr_t>(row_off) & 3u))
    return MXG_ERR_MISALIGNED;
  const GroupedWs wl = grouped_ws(M_total, K, E);
  uint8_t *ws = opts ? static_cast<uint8_t *>(opts->workspace) : nullptr;
  if (!ws || opts->ws_bytes < wl.total) return MXG_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MXG_ERR_MISALIGNED;
  const long long TA = grouped_tiles(M_total, E);
  const long long tilesB = (N + 255) / 256;
  if (TA * tilesB >= (1LL << 31)) return MXG_ERR_UNSUPPORTED_SHAPE;
  int sm = 0;
  mxg_status st = check_device(&sm);
  if (st != MXG_OK) return st;
  if (M_total == 0) return MXG_OK;  // no token was routed: nothing to compute
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int *tile_off = reinterpret_cast<int *>(ws + wl.tile_off);
  uint8_t *codes = ws + wl.codes, *sf = ws + wl.sf;
  cudaError_t e = mxg::launch_mx_quant_grouped(x_bf16, ldx, M_total, K, row_off, E, tile_off, codes, sf, sm, s);
  if (e != cudaSuccess) return MXG_ERR_CUDA;

  const uint64_t row_bytes = (uint64_t)K / 2;
  CUtensorMap tmA, tmB, tmY;
  std::memset(&tmY, 0, sizeof(tmY));
  if ((st = make_operand_map(&tmA, codes, row_bytes, (uint64_t)TA * 128, 128)) != MXG_OK) return st;
  if ((st = make_operand_map(&tmB, w_panels, row_bytes, (uint64_t)N, 256)) != MXG_OK) return st;
  mxg::GemmParams p;
  std::memset(&p, 0, sizeof(p));
  p.sfA = sf;
  p.y = y;
  p.ldy = ldy;
  p.out_f32 = out_dtype == MXG_OUT_F32 ? 1 : 0;
  p.M = M_total;
  p.N = N;
  p.K = K;
  p.swap = 0;
  p.rowsA = (int)(TA * 128);
  p.rowsB = N;
  p.tilesA = (int)TA;
  p.tilesB = (int)tilesB;
  p.kblocks = K / 256;  // one 128-byte code column (256 values) per stage
  p.G4 = K / 128;
  p.splitk = 0;
  p.units = TA * tilesB * p.kblocks;
  p.seg_max = 1;
  p.status = opts->dev_status;
  const uint32_t tmo = opts->timeout_ms ? opts->timeout_ms : 1000u;
  p.timeout_ns = (unsigned long long)tmo * 1000000ull;
  p.debug_stall = opts->debug_stall == 1 ? 1 : 0;
  p.early_w = opts->weights_static ? 1 : 0;
  p.trace = static_cast<unsigned long long *>(opts->trace);
  p.a_tiles = codes;
  p.b_tiles = w_panels;
  p.b_tile_rows = mxg::kPanelRows;
  p.w_panels = 1;
  p.kc_per_row = (int)(row_bytes / 128);
  p.groups = E;
  p.g_tile_off = tile_off;
  p.g_row_off = row_off;
  p.w_group_bytes = mxg_weight_bytes(0, N, K, MXG_PANEL);
  const long long ctas = std::min<long long>(TA * tilesB, sm);
  e = mxg::launch_gemm(0, mxg::kPanelRows, tmA, tmB, tmY, p, (int)ctas, s);
  return e == cudaSuccess ? MXG_OK : MXG_ERR_CUDA;
}

mxg_status fp8_gemm_ptpc(const uint8_t *qa, const float *sa, const uint8_t *qw, const float *sw,
                         int M, int N, int K, void *y, int ldy, mxg_out_dtype out_dtype,
                         const mxg_gemm_opts *opts, mxg_stream_t stream) {
  mxg_status st = check_gemm_common(M, N, K, y, ldy, out_dtype, opts);
  if (st != MXG_OK) return st;
  if (!qa || !sa || !qw || !sw) return MXG_ERR_INVALID_ARG;
  if (!aligned16(qa) || !aligned16(qw) || (reinterpret_cast<uintptr_t>(sa) & 3u) ||
      (reinterpret_cast<uintptr_t>(sw) & 3u))
    return MXG_ERR_MISALIGNED;
  int sm = 0;
  if ((st = check_device(&sm)) != MXG_OK) return st;
  GemmOperands op{qa, nullptr, qw, nullptr, sa, sw};
  return run_gemm(1, op, M, N, K, y, ldy, out_dtype, opts, opts ? opts->workspace : nullptr,
                  opts ? opts->ws_bytes : 0, 0, opts ? opts->act_tile_rows : 0, sm,
                  reinterpret_cast<cudaStream_t>(stream));
}

mxg_status mxg_mma_peak(int kind, int n, int iters, double *tflops, mxg_stream_t stream) {
  if ((kind != 0 && kind != 1) || (n != 128 && n != 256) || iters < 1 || iters > (1 << 22) || !tflops)
    return MXG_ERR_INVALID_ARG;
  int sm = 0;
  mxg_status st = check_device(&sm);
  if (st != MXG_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int *status = nullptr;
  if (cudaMalloc(&status, sizeof(int)) != cudaSuccess) return MXG_ERR_CUDA;
  cudaEvent_t a = nullptr, b = nullptr;
  float ms = 0.0f;
  bool ok = cudaMemsetAsync(status, 0, sizeof(int), s) == cudaSuccess &&
            cudaEventCreate(&a) == cudaSuccess && cudaEventCreate(&b) == cudaSuccess &&
            mxg::launch_mma_peak(kind, n, iters / 8 + 1, sm, status, s) == cudaSuccess &&  // warm-up
            cudaEventRecord(a, s) == cudaSuccess &&
            mxg::launch_mma_peak(kind, n, iters, sm, status, s) == cudaSuccess &&
            cudaEventRecord(b, s) == cudaSuccess && cudaEventSynchronize(b) == cudaSuccess &&
            cudaEventElapsedTime(&ms, a, b) == cudaSuccess;
  int h = 0;
  ok = ok && cudaMemcpy(&h, status, sizeof(int), cudaMemcpyDeviceToHost) == cudaSuccess;
  if (a) cudaEventDestroy(a);
  if (b) cudaEventDestroy(b);
  cudaFree(status);
  if (!ok) return MXG_ERR_CUDA;
  if (h) return MXG_ERR_TIMEOUT;
  const double k = kind == 0 ? 64.0 : 32.0;
  *tflops = (double)sm * iters * 4.0 * 2.0 * 128.0 * n * k / (ms * 1e-3) / 1e12;
  return MXG_OK;
}

mxg_status mxg_query_status(int *dev_status, mxg_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return MXG_ERR_CUDA;
  if (!dev_status) return MXG_OK;
  int h = 0;
  if (cudaMemcpy(&h, dev_status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MXG_ERR_CUDA;
  if (h != 0 && cudaMemset(dev_status, 0, sizeof(int)) != cudaSuccess) return MXG_ERR_CUDA;
  if (h & MXG_DEV_TIMEOUT) return MXG_ERR_TIMEOUT;
  if (h != 0) return MXG_ERR_CUDA;
  return MXG_OK;
}

const char *mxg_status_string(mxg_status s) {
  switch (s) {
    case MXG_OK: return "MXG_OK";
    case MXG_ERR_INVALID_ARG: return "MXG_ERR_INVALID_ARG";
    case MXG_ERR_UNSUPPORTED_SHAPE: return "MXG_ERR_UNSUPPORTED_SHAPE";
    case MXG_ERR_MISALIGNED: return "MXG_ERR_MISALIGNED";
    case MXG_ERR_UNSUPPORTED_DEVICE: return "MXG_ERR_UNSUPPORTED_DEVICE";
    case MXG_ERR_CUDA: return "MXG_ERR_CUDA";
    case MXG_ERR_TIMEOUT: return "MXG_ERR_TIMEOUT";
    case MXG_ERR_WORKSPACE: return "MXG_ERR_WORKSPACE";
  }
  return "MXG_UNKNOWN";
}

// ---------------------------------------------------------------------------
// mx_gemm_a4w4_noalloc: the A4W4 GEMM for callers that cannot allocate device
// memory.  Its scratch (fused activations, partial tiles -- the same layout
// as the caller workspace of mx_gemm_a4w4) lives in
// this file-scope device array, which every GPU that loads the library holds
// until the process exits.  Host code must not use the array's name as a
// device address: the address comes from cudaGetSymbolAddress, once per
// device, with that device current.
static __device__ __align__(256) uint8_t g_noalloc_scratch[MXG_NOALLOC_SCRATCH_BYTES];

namespace {
std::mutex g_noalloc_mu;
void *g_noalloc_ptr[kMaxDevices];

// Device address of the scratch array on the current device (looked up on
// the first call for that device).
mxg_status noalloc_scratch(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MXG_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MXG_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return MXG_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return MXG_OK;
}
}  // namespace

mxg_status mx_gemm_a4w4_noalloc(const uint8_t *a_codes, const uint8_t *a_sf, const void *x_bf16,
                                int ldx, const uint8_t *w_codes, const uint8_t *w_sf, int M, int N,
                                int K, void *y, int ldy, mxg_out_dtype out_dtype, int weights_tiled,
                                mxg_stream_t stream) {
  mxg_gemm_opts opts;
  std::memset(&opts, 0, sizeof(opts));
  opts.variant = MXG_VARIANT_AUTO;
  opts.weights_tiled = weights_tiled;
  // every operand check first: a rejected call touches no device memory
  // (in particular not the shared scratch another stream may be using)
  mxg_status st = check_a4w4_args(a_codes, a_sf, x_bf16, ldx, w_codes, w_sf, M, N, K, y, ldy, out_dtype,
                                  &opts);
  if (st != MXG_OK) return st;
  int sm = 0;
  if ((st = check_device(&sm)) != MXG_OK) return st;
  // the scratch this call needs, exactly as mx_gemm_a4w4 would ask for it
  mxg_plan pl;
  if ((st = plan_impl(0, M, N, K, sm, &opts, &pl)) != MXG_OK) return st;
  const bool fused = a_codes == nullptr;
  const size_t act =
      fused ? fused_act_bytes(M, K, K % 256 == 0 ? plan_act_tile_rows(pl) : 0) : 0;
  const size_t need = act + pl.ws_bytes;
  if (need > (size_t)MXG_NOALLOC_SCRATCH_BYTES) return MXG_ERR_WORKSPACE;
  void *scratch = nullptr;
  if ((st = noalloc_scratch(&scratch)) != MXG_OK) return st;
  // every byte of scratch a call reads, that call has written first, so
  // whatever the previous call left in the array is never used
  opts.workspace = scratch;
  opts.ws_bytes = MXG_NOALLOC_SCRATCH_BYTES;
  return mx_gemm_a4w4(a_codes, a_sf, x_bf16, ldx, w_codes, w_sf, M, N, K, y, ldy, out_dtype, &opts,
                      stream);
}

}  // extern "C"
