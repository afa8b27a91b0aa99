// kernels.h -- internal launchers (not part of the public C ABI).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace mxg {

cudaError_t launch_mx_quant(const void *x, long long ldx, int rows, int K, uint8_t *codes,
                            uint8_t *sf, bool swizzled, int sm_count, cudaStream_t stream);

cudaError_t launch_fp8_quant(const void *x, long long ldx, int rows, int K, uint8_t *q,
                             float *scale, int sm_count, cudaStream_t stream);

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
};

// kind 0 = A4W4 (kind::mxf4), 1 = PTPC (kind::f8f6f4); bn = MMA-B tile rows.
cudaError_t launch_gemm(int kind, int bn, const CUtensorMap &tmA, const CUtensorMap &tmB,
                        const GemmParams &p, int ctas, cudaStream_t stream);

// Pipeline stages a (kind, bn) kernel uses, and its dynamic shared memory.
int gemm_stages(int kind, int bn);
size_t gemm_smem_bytes(int kind, int bn);

}  // namespace mxg
