// kernels.h -- internal launchers (not part of the public C ABI).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cstdlib>
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
inline void attach_pdl(cudaLaunchConfig_t &cfg, cudaLaunchAttribute (&attr)[1]) {
  if (!pdl_enabled()) return;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
}

// tile_rows: 0 = row-major codes / bytes, else the tile layout with tiles of
// that many rows (128 for weights, the GEMM's token tile for activations).
// act: the input is an activation; the next kernel may launch at once.  For
// weights (act = false) no later kernel starts before this one has finished.
cudaError_t launch_mx_quant(const void *x, long long ldx, int rows, int K, uint8_t *codes,
                            uint8_t *sf, bool swizzled, int tile_rows, bool act, int sm_count,
                            cudaStream_t stream);

cudaError_t launch_fp8_quant(const void *x, long long ldx, int rows, int K, uint8_t *q,
                             float *scale, int tile_rows, bool act, int sm_count,
                             cudaStream_t stream);

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
  int kblocks;         // K-blocks per tile (one pipeline stage each)
  int G4;              // K / 128: 512-byte scale tiles per 128-row block
  int splitk;          // 1: stream-K over (tile, K-block) units
  long long units;     // tilesA * tilesB * kblocks
  float *ws;           // split-K partial tiles
  int *counters;       // split-K arrival counters, one per tile
  int seg_max;         // partial slots per tile
  int *status;         // optional device status word
  unsigned long long timeout_ns;
  int debug_stall;
  unsigned long long *trace;  // optional: kTracePoints SM-clock stamps per CTA
  const uint8_t *a_tiles;  // non-null: the MMA-A operand in the weight tile layout (bulk copies)
  const uint8_t *b_tiles;  // non-null: the MMA-B operand in the tile layout, b_tile_rows rows
  int b_tile_rows;         //   per tile: 128 (weights, full-tile mode) or BN (activations)
  int kc_per_row;          // 128-byte chunks per operand row (tile layout)
  int defer_reduce;        // split-K: partial tiles are summed by launch_splitk_reduce, not by
                           //          the last CTA of each tile
  int early_w;         // 1: no kernel still in flight writes the weights, so their first
                       //    stages may load before griddepcontrol.wait
};

// Timeline trace points (index into a CTA's 16 slots): SM clock64 values.
enum TracePoint {
  kTrEntry = 0, kTrSetup = 1, kTrFirstLoad = 2, kTrLastLoad = 3, kTrFirstFull = 4,
  kTrLastCommit = 5, kTrAcc0 = 6, kTrItem0Done = 7, kTrAcc1 = 8, kTrItem1Done = 9,
  kTrEpiDone = 10, kTrExit = 11, kTrPartStored = 12, kTrDecision = 13, kTrReduced = 14,
  kTrItems = 15, kTrEntryNs = 16, kTrExitNs = 17, kTrWaited = 18, kTracePoints = 20
};

// kind 0 = A4W4 (kind::mxf4), 1 = PTPC (kind::f8f6f4); bn = MMA-B tile rows.
cudaError_t launch_gemm(int kind, int bn, const CUtensorMap &tmA, const CUtensorMap &tmB,
                        const GemmParams &p, int ctas, cudaStream_t stream);

// Split-K reduction of a GEMM launched with p.defer_reduce = 1 (the same
// params, its grid size gemm_ctas); launched right after it on the stream.
cudaError_t launch_splitk_reduce(int kind, int bn, const GemmParams &p, int gemm_ctas,
                                 int sm_count, cudaStream_t stream);

// Pipeline stages a (kind, bn) kernel uses, and its dynamic shared memory.
int gemm_stages(int kind, int bn);
size_t gemm_smem_bytes(int kind, int bn);

}  // namespace mxg
