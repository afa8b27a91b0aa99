// kernels.h -- internal launchers (not part of the public C ABI).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cstdlib>
#include <deque>
#include <mutex>
#include <utility>
#include <cuda.h>
#include <cuda_runtime.h>

namespace mxg {

// Launch configuration with programmatic stream serialization: the kernel
// may begin while the previous kernel in the stream is still running; every
// kernel of this library calls griddepcontrol.wait before it touches memory
// the previous kernel may write or read.
inline cudaLaunchConfig_t pdl_config(dim3 grid, dim3 block, size_t smem, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  return cfg;
}
// MXG_DISABLE_PDL=1 in the environment turns the overlap off (for A/B timing).
inline bool pdl_enabled() {
  static const bool on = [] {
    const char *e = std::getenv("MXG_DISABLE_PDL");
    return !(e && e[0] == '1');
  }();
  return on;
}
template <int N>
inline void attach_pdl(cudaLaunchConfig_t &cfg, cudaLaunchAttribute (&attr)[N]) {
  if (!pdl_enabled()) return;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
}
// Small kernels (quantizers, split-K reduce) run beside, and just before,
// GEMM CTAs that need ~210 KB of shared memory.  An SM whose L1/shared split
// was set for an L1-preferring kernel cannot take a GEMM CTA until it drains,
// so these kernels ask for the maximum shared-memory carveout (set once per
// kernel; a repeated or concurrent call sets the same value).
// A per-device "already done" bit set (devices 0..63; beyond that, always redo).
struct DeviceOnce {
  unsigned long long bits = 0;
  bool done(int dev) const { return dev >= 0 && dev < 64 && ((bits >> dev) & 1ull); }
  void set(int dev) {
    if (dev >= 0 && dev < 64) __atomic_fetch_or(&bits, 1ull << dev, __ATOMIC_RELAXED);
  }
};

// The "done" bits of one kernel, found by its address (kernels of one
// signature share the template instance, so a static per instance would not
// tell them apart).
inline DeviceOnce &carveout_once(const void *kern) {
  static std::mutex mu;
  static std::deque<std::pair<const void *, DeviceOnce>> done;  // appends keep references valid
  std::lock_guard<std::mutex> lock(mu);
  for (auto &d : done)
    if (d.first == kern) return d.second;
  done.emplace_back(kern, DeviceOnce{});
  return done.back().second;
}

template <class Kernel>
inline cudaError_t prefer_shared_carveout(Kernel *kern) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  {
    DeviceOnce &once = carveout_once(reinterpret_cast<const void *>(kern));
    if (once.done(dev)) return cudaSuccess;
  }
  e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                           (int)cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess) carveout_once(reinterpret_cast<const void *>(kern)).set(dev);
  return e;
}

// CTAs of `kern` (`threads` per CTA, `smem` bytes of dynamic shared memory)
// that one SM holds at once; a grid-stride kernel launched with this many
// per SM starts every CTA in one wave.
template <class Kernel>
inline cudaError_t resident_ctas_per_sm(Kernel *kern, int threads, size_t smem, int *n) {
  *n = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(n, kern, threads, smem);
  if (e == cudaSuccess && *n < 1) *n = 1;
  return e;
}

// tile_rows: 0 = row-major codes / bytes, kPanelLayout = the weight panel
// layout (256-row panels, MXFP4 scales inside them; rows padded to a multiple
// of 256 with zero codes), else the tile layout with tiles of that many rows
// (128 for weights, the GEMM's token tile for activations).
constexpr int kPanelLayout = -1;
constexpr int kPanelRows = 256;
constexpr int kMxPanelBytes = 256 * 128 + 2048;  // per 128-byte column
constexpr int kF8PanelBytes = 256 * 128;
// Bounded-wait controls of a quantizer that streams rows through shared
// memory (more than 512 rows): the caller's status word (may be null), the
// wait limit, and the test hook that makes its first wait one that nothing
// satisfies.
struct QuantWatch {
  int *status = nullptr;
  unsigned long long timeout_ns = 1000000000ull;
  int debug_stall = 0;
};

// act: the input is an activation; the next kernel may launch at once.  For
// weights (act = false) no later kernel starts before this one has finished.
cudaError_t launch_mx_quant(const void *x, long long ldx, int rows, int K, uint8_t *codes,
                            uint8_t *sf, bool swizzled, int tile_rows, bool act, int sm_count,
                            cudaStream_t stream, const QuantWatch &watch = QuantWatch{});

cudaError_t launch_fp8_quant(const void *x, long long ldx, int rows, int K, uint8_t *q,
                             float *scale, int tile_rows, bool act, int sm_count,
                             cudaStream_t stream);

// SwiGLU of a [gate | up] row (I values each) fused with the per-token FP8
// quantization of h = bf16(silu(gate) * up); q in the layout tile_rows names
// (0 = row-major, else token tiles), h_out (nullable) receives h.
cudaError_t launch_swiglu_fp8(const void *gu, long long ldgu, int rows, int I, int tile_rows, void *h_out,
                              long long ldh, uint8_t *q, float *scale, int sm_count, cudaStream_t stream);
constexpr int kSwigluMaxI = 102400;  // h of one row lives in shared memory (2 bytes a value)

// Everything one GEMM launch needs besides the two tensor maps.
struct GemmParams {
  const uint8_t *sfA;  // A4W4: scale factors of the MMA-A / MMA-B operands,
  const uint8_t *sfB;  //       128x4-tile layout
  const float *tok_scale;   // PTPC: per-token activation scale sa (M)
  const float *chan_scale;  // PTPC: per-output-channel weight scale sw (N)
  void *y;
  long long ldy;
  int out_f32;
  int M, N, K;
  int swap;            // 1: MMA-A = weight rows (N), MMA-B = token rows (M)
  int rowsA, rowsB;    // rows of the MMA-A / MMA-B operand
  int tilesA, tilesB;  // ceil(rowsA / 128), ceil(rowsB / BN)
  int kblocks;         // pipeline stages along K per tile (gemm_cols_per_stage columns each)
  int G4;              // K / 128: 512-byte scale tiles per 128-row block
  int splitk;          // 1: stream-K over (tile, K-block) units
  long long units;     // tilesA * tilesB * kblocks
  float *ws;           // split-K partial tiles: [tile][slot][BN columns][128 rows] fp32
  int seg_max;         // partial slots per tile
  int *status;         // optional device status word
  unsigned long long timeout_ns;
  int debug_stall;
  unsigned long long *trace;  // optional: kTracePoints SM-clock stamps per CTA
  const uint8_t *a_tiles;  // non-null: the MMA-A operand in the weight tile layout (bulk copies)
  const uint8_t *b_tiles;  // non-null: the MMA-B operand in the tile layout, b_tile_rows rows
  int b_tile_rows;         //   per tile: 128 (weights, full-tile mode) or BN (activations)
  int w_panels;            // the weight operand (a_tiles when swapped, else b_tiles) is in
                           //   256-row panels with their scales appended (MXG_PANEL)
  int kc_per_row;          // 128-byte chunks per operand row (tile layout)
  int raster_group;        // full tile: 0 = tiles in row order (token tile slowest), else
                           //   bands of this many token tiles, the token tile fastest
  int cta_pair;            // full tile: 1 = clusters of two CTAs issuing 2-SM MMAs over
                           //   256-token x 256-channel tiles (each CTA holds 128 token rows
                           //   and one 128-row half of the weight tile)
  int early_w;         // 1: no kernel still in flight writes the weights, so their first
                       //    stages may load before griddepcontrol.wait
  int y_tma;           // full tile, bf16 out: the epilogue stores y through tensor map tmY
  // Grouped (MoE) full tile, A4W4: groups = number of experts E (0 = a plain
  // GEMM).  The MMA-A operand is token tiles (a_tiles) in which each
  // expert's rows start a new 128-row tile; g_tile_off / g_row_off (device,
  // E + 1 each) give each expert's first token tile and first token row
  // (y row); the MMA-B operand is E weight panel sets, w_group_bytes apart.
  int groups;
  const int *g_tile_off;
  const int *g_row_off;
  size_t w_group_bytes;
};

// Timeline trace points (index into a CTA's kTracePoints slots): SM clock64
// values, except the *Ns slots (global timer, ns).  Row 0 also holds the span
// of the split-K reduce kernel that follows the GEMM: kTrRedEntryInv = the
// bitwise NOT of its first CTA's entry time (so that an atomic max finds the
// earliest), kTrRedExitNs = its last CTA's exit time.
enum TracePoint {
  kTrEntry = 0, kTrSetup = 1, kTrFirstLoad = 2, kTrLastLoad = 3, kTrFirstFull = 4,
  kTrLastCommit = 5, kTrAcc0 = 6, kTrItem0Done = 7, kTrAcc1 = 8, kTrItem1Done = 9,
  kTrEpiDone = 10, kTrExit = 11, kTrPartStored = 12,  // 13, 14: unused
  kTrItems = 15, kTrEntryNs = 16, kTrExitNs = 17, kTrWaited = 18,  // 19: unused
  kTrWaitedNs = 20, kTrSmid = 21, kTrRedEntryInv = 22, kTrRedExitNs = 23,
  // A4W4, per pipeline stage k < 8 of the CTA's sequence, seen by the first
  // epilogue warp: the stage's data landed / its scales are in TMEM
  kTrStageLanded = 24, kTrStageFed = 32,
  kTracePoints = 40
};

// kind 0 = A4W4 (kind::mxf4), 1 = PTPC (kind::f8f6f4); bn = MMA-B tile rows.
cudaError_t launch_gemm(int kind, int bn, const CUtensorMap &tmA, const CUtensorMap &tmB,
                        const CUtensorMap &tmY, const GemmParams &p, int ctas, cudaStream_t stream);

// Split-K reduction of a GEMM whose tiles have several partials (the same
// params, its grid size gemm_ctas); launched right after it on the stream.
cudaError_t launch_splitk_reduce(int kind, int bn, const GemmParams &p, int gemm_ctas,
                                 int sm_count, cudaStream_t stream);

// Grouped MXFP4 activation quantizer: x (M_total rows sorted by expert,
// row_off: E + 1 device offsets) -> codes in 128-row token tiles where each
// expert's rows start a new tile, scales in the 128x4 layout over those
// padded rows; every CTA forms the tile offsets from row_off, and the first
// one also writes them to tile_off (E + 1 ints) for the GEMM.
cudaError_t launch_mx_quant_grouped(const void *x, long long ldx, int M_total, int K, const int *row_off,
                                    int E, int *tile_off, uint8_t *codes, uint8_t *sf, int sm_count,
                                    cudaStream_t stream);
constexpr int kMaxGroups = 1024;

// The tensor-pipe rate probe behind mxg_mma_peak: sm_count CTAs, one per SM.
cudaError_t launch_mma_peak(int kind, int bn, int iters, int sm_count, int *status,
                            cudaStream_t stream);

// Pipeline stages a (kind, bn, variant) kernel uses, its dynamic shared
// memory, and the 128-byte K columns one stage covers (p.kblocks counts
// stages of that many columns).
int gemm_cols_per_stage(bool splitk);

}  // namespace mxg
