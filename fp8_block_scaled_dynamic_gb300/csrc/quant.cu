// quant.cu -- HBM-bound quantizer kernels.
//
//  * mx_quant_kernel: OCP-MX MXFP4 quantization of bf16 rows ("Kimi-K3 DSpark
//    O-Proj-only MXFP4", "Exact quantization coverage": E2M1 codes, one E8M0
//    scale per 32 consecutive input channels).  One thread owns one 16-byte
//    chunk (8 values = a quarter block); the block amax is a max over 4
//    lanes by warp shuffles; codes leave as packed nibbles and scales go
//    straight into the row-major, 128x4-tile or panel layout.  Large inputs
//    stream through shared memory by bulk copies.
//  * mx_quant_grouped_kernel: the same for token rows grouped by expert.
//  * fp8_quant_kernel / fp8_quant_staged_kernel: per-row E4M3 quantization
//    with an FP32 scale ("Kimi-K3-DSpark-FP8-PTPC", "Phase 1 FP8 PTPC
//    Quantization": dynamic per-token activations; per-output-channel
//    weights are per-row of W), two passes over a row or (large inputs) one
//    read of rows streamed through shared memory.
//  * swiglu_fp8_kernel: SwiGLU of the packed gate_up output fused with the
//    per-token FP8 quantization of its result.
//
// Numerics (shared readings, see the public header): MX scale e =
// clamp(floor(log2 amax) - 2, -127, 127), code = E2M1_RNE_sat(x * 2^-e) with
// the sign of x; FP8 s = amax / 448 (1 for an all-zero row), q =
// E4M3_RNE_sat(x / s).  Built without fast-math: x * 2^-e is an exact fp32
// product (subnormal inputs included), and x / s is the IEEE division or,
// where it decides the same code (RowDivisor), Markstein's correction step.
#include <algorithm>
#include <cstdint>
#include <cuda_runtime.h>
#include <type_traits>

#include "kernels.h"
#include "ptx.cuh"
#include "quant_math.cuh"

namespace mxg {

namespace {

constexpr int kMxThreads = 256;

// grid: x = chunk groups along the row, y = rows (grid-stride).
// rows_iter >= rows: rows in [rows, rows_iter) are padding (swizzled layout
// only) -- their scales are written as 0 and no codes are stored.
// tile_rows: 0 = row-major codes, kPanelLayout = weight panels (codes and
// scales; padding rows get zero codes), else the tile layout with that tile
// height.
// CPT: 16-byte chunks per thread per row (4 for large inputs: a CTA covers a
// whole 8192-value row and its per-row address work is shared by more
// chunks; 2 for decode-sized inputs, whose latency wants more, smaller CTAs).
// kStaged (large inputs): the CTA's parts of its rows stream into a ring of
// kMxSlots buffers in shared memory by bulk copies that one thread issues,
// so that the bytes in flight are not bounded by registers; otherwise two
// row buffers in registers are used in turn.
constexpr uint64_t kQuantWaitNs = 1000000000ull;  // a copy that has not landed in 1 s never will

// Bounded wait for a copy still in flight before the CTA exits (its shared
// memory must not be reused while the copy can still write it).
__device__ __forceinline__ void drain_copy(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > kQuantWaitNs) return;
}

constexpr int kMxSlots = 2;
constexpr uint32_t kMxSlotBytes = 4 * kMxThreads * 16;  // a CTA's part of a row at CPT = 4
constexpr size_t kMxStagedSmem = (size_t)kMxSlots * kMxSlotBytes + 8u * (kMxSlots + 1);

template <bool kSwizzled, int CPT, bool kStaged>
__global__ void __launch_bounds__(kMxThreads) mx_quant_kernel(const uint16_t *__restrict__ x,
                                                              long long ldx, int rows,
                                                              int rows_iter, int K, int tile_rows,
                                                              int early_trigger,
                                                              uint8_t *__restrict__ codes,
                                                              uint8_t *__restrict__ sf, int *status,
                                                              unsigned long long timeout_ns, int debug_stall) {
  const int cpr = K >> 3;  // 16-byte chunks per row; K % 128 == 0 => cpr % 16 == 0
  const int G = K >> 5;    // MX blocks per row
  const int lane = threadIdx.x & 31;
  // An activation quantizer lets the next kernel launch at once: every kernel
  // of this library waits for its predecessor before it touches memory that
  // one may write.  A weight quantizer never triggers, so no later kernel
  // starts (and streams weights before its own wait) until it has finished.
  if (early_trigger) pdl_trigger();
  // Warm L2 with this CTA's part of its first row while the kernel ahead
  // finishes; the loads below come after the wait.
  if (threadIdx.x == 0 && (int)blockIdx.y < rows) {
    const int c0 = blockIdx.x * CPT * kMxThreads;
    const int nc = min(CPT * kMxThreads, cpr - c0);
    if (nc > 0) prefetch_l2_bulk(x + (size_t)blockIdx.y * ldx + (size_t)c0 * 8, (uint32_t)nc * 16u);
  }
  // x may be the previous kernel's output and codes/sf may still be read by it
  pdl_wait();
  const bool panel = tile_rows == kPanelLayout;
  const int KC = K >> 8;  // 128-byte code columns per row
  const int t_shift = (tile_rows > 0) ? __ffs(tile_rows) - 1 : 0;  // tile_rows is a power of 2
  // where a row's codes go: 128-byte column c at row_base + c * col_stride,
  // its 16-byte unit j at ((j ^ rsw) * 16) (row-major: rsw = 0)
  const size_t col_stride = panel ? (size_t)kMxPanelBytes : tile_rows > 0 ? (size_t)tile_rows * 128u : 128u;
  // this thread's chunks c0 + 256 i, i < CPT: in the row or past it (cpr %
  // 16 == 0: a half-warp is wholly inside the row or wholly past it; past
  // it, it reads the row's first chunk so that the shuffles have data, and
  // stores nothing).  Within a row, chunk i's codes go at code_col0 + i *
  // code_step (the same 16-byte unit of a column 8 columns on) and its scale
  // word at sf_col0 + i * sf_step (4 blocks = 16 chunks further on).
  const int c0 = blockIdx.x * CPT * kMxThreads + threadIdx.x;
  const size_t code_col0 = (size_t)(c0 >> 5) * col_stride + (size_t)((c0 * 4) & 15);
  const size_t code_step = 8 * col_stride;
  const uint32_t unit = (uint32_t)(c0 >> 2) & 7u;  // 16-byte unit of the column (byte 4 c0 / 16)
  const int g0 = c0 >> 2;                          // first of the 4 blocks of a scale word
  const size_t sf_col0 = panel       ? (size_t)(g0 >> 3) * 34816u + (size_t)((g0 >> 2) & 1) * 512u
                         : kSwizzled ? (size_t)(g0 >> 2) * 512u
                                     : (size_t)g0;
  const size_t sf_step = panel ? 8u * 34816u : kSwizzled ? 16u * 512u : 64u;
  const bool sf_lane = (lane & 15) == 0;
  auto in_row = [&](int i) { return c0 + i * kMxThreads < cpr; };
  uint8_t *const sf_dst = panel ? codes : sf;
  // this CTA's part of a row: chunks cta_c0 .. cta_c0 + cta_nc - 1
  const int cta_c0 = blockIdx.x * CPT * kMxThreads;
  const int cta_nc = min(CPT * kMxThreads, cpr - cta_c0);
  auto load_row = [&](int r, uint4 (&v)[CPT]) {
    if (r >= rows) return;  // padding: not read
    const uint16_t *xr = x + (size_t)r * ldx;
#pragma unroll
    for (int i = 0; i < CPT; ++i) v[i] = ld_stream_v4(xr + (in_row(i) ? (size_t)(c0 + i * kMxThreads) * 8 : 0));
    // the row two steps on heads for L2 now, so that its register loads
    // (issued one row later) wait for L2, not for HBM
    const int rp = r + 2 * (int)gridDim.y;
    if (threadIdx.x == 0 && rp < rows && cta_nc > 0) {
      const uint16_t *xp = x + (size_t)rp * ldx + (size_t)cta_c0 * 8;
      for (int c = 0; c < cta_nc; c += 1024)
        prefetch_l2_bulk(xp + (size_t)c * 8, (uint32_t)min(1024, cta_nc - c) * 16u);
    }
  };
  // where row r's codes and scale words go
  auto row_dest = [&](int r, size_t &row_base, size_t &sf_row, uint32_t &rsw) {
    if (panel) {
      row_base = (size_t)(r >> 8) * KC * kMxPanelBytes + (size_t)((r >> 7) & 1) * 16384u + (size_t)(r & 127) * 128u;
      rsw = r & 7;
      sf_row = (size_t)(r >> 8) * KC * 34816u + 32768u + (size_t)((r >> 7) & 1) * 1024u + (size_t)(r & 31) * 16u +
               (size_t)((r >> 5) & 3) * 4u;
    } else {
      if (tile_rows > 0) {
        const int rr = r & (tile_rows - 1);
        row_base = ((size_t)(r >> t_shift) * KC << (t_shift + 7)) + (size_t)rr * 128u;
        rsw = rr & 7;
      } else {
        row_base = (size_t)r * (K >> 1);
        rsw = 0;
      }
      sf_row = kSwizzled ? (size_t)(r >> 7) * (size_t)(G >> 2) * 512u + (size_t)(r & 31) * 16u + (size_t)((r >> 5) & 3) * 4u
                         : (size_t)r * G;
    }
  };
  auto do_row = [&](int r, const uint4 (&v)[CPT]) {
    size_t row_base, sf_row;
    uint32_t rsw;
    row_dest(r, row_base, sf_row, rsw);
    uint8_t *const code_at = codes + row_base + code_col0 + ((unit ^ rsw) << 4);
    uint8_t *const sf_at = sf_dst + sf_row + sf_col0;
    if (r >= rows) {  // padding (uniform over the CTA): zero scales, and zero codes in a panel
#pragma unroll
      for (int i = 0; i < CPT; ++i) {
        if (panel) st_global_b32_if(code_at + i * code_step, 0u, in_row(i));
        st_global_b32_if(sf_at + i * sf_step, 0u, in_row(i) && sf_lane);
      }
      return;
    }
#pragma unroll
    for (int i = 0; i < CPT; ++i) {
      uint32_t scode;
      const uint32_t packed = mx_encode_chunk(v[i], scode);
      st_global_b32_if(code_at + i * code_step, packed, in_row(i));
      const uint32_t word = mx_scale_word(scode);
      st_global_b32_if(sf_at + i * sf_step, word, in_row(i) && sf_lane);
    }
  };
  uint4 va[CPT], vb[CPT];
  if constexpr (kStaged) {
    // kMxSlots row parts, then one mbarrier a slot and one that nothing
    // arrives at (the debug_stall test hook waits on it)
    extern __shared__ __align__(128) uint8_t ring[];
    __shared__ int abort_flag;
    const uint32_t slots = smem_addr(ring);
    const uint32_t bars = slots + kMxSlots * kMxSlotBytes;
    const uint32_t never = bars + 8u * kMxSlots;
    if (threadIdx.x == 0) {
      for (int i = 0; i <= kMxSlots; ++i) mbar_init(bars + 8u * i, 1);
      abort_flag = 0;
      fence_barrier_init();
    }
    __syncthreads();
    const WaitCtl ctl{&abort_flag, status, timeout_ns};
    const uint32_t part_bytes = (uint32_t)cta_nc * 16u;  // cta_nc % 16 == 0
    // row k of this CTA is blockIdx.y + k * gridDim.y; thread 0 copies its
    // part into slot k % kMxSlots (padding rows are not read)
    auto row_of = [&](int k) { return (int)blockIdx.y + k * (int)gridDim.y; };
    auto issue = [&](int k) {
      const int r = row_of(k);
      if (r >= rows || cta_nc <= 0) return;
      const uint32_t bar = bars + 8u * (uint32_t)(k % kMxSlots);
      mbar_arrive_expect_tx(bar, part_bytes);
      bulk_load(slots + (uint32_t)(k % kMxSlots) * kMxSlotBytes, x + (size_t)r * ldx + (size_t)cta_c0 * 8, part_bytes,
                bar, policy_evict_first());
    };
    if (threadIdx.x == 0)
      for (int k = 0; k < kMxSlots; ++k) issue(k);
    for (int k = 0; row_of(k) < rows_iter; ++k) {
      const int r = row_of(k);
      if (r >= rows) {  // padding (uniform over the CTA; after every real row)
        do_row(r, va);
        continue;
      }
      const bool landed = (debug_stall && k == 0)
                              ? mbar_wait(never, 0u, ctl)
                              : mbar_wait(bars + 8u * (uint32_t)(k % kMxSlots), (uint32_t)(k / kMxSlots) & 1u, ctl);
      if (__syncthreads_or(!landed)) {
        // a copy did not land: let every copy still in flight finish
        // (bounded), give this CTA's remaining rows NaN scales (E8M0 0xFF),
        // and leave
        if (threadIdx.x == 0)
          for (int j = k; j < k + kMxSlots; ++j)
            if (row_of(j) < rows) drain_copy(bars + 8u * (uint32_t)(j % kMxSlots), (uint32_t)(j / kMxSlots) & 1u);
        for (int j = k; row_of(j) < rows; ++j) {
          size_t row_base, sf_row;
          uint32_t rsw;
          row_dest(row_of(j), row_base, sf_row, rsw);
#pragma unroll
          for (int i = 0; i < CPT; ++i) st_global_b32_if(sf_dst + sf_row + sf_col0 + i * sf_step, 0xFFFFFFFFu, in_row(i) && sf_lane);
        }
        return;
      }
      const uint32_t slot = slots + (uint32_t)(k % kMxSlots) * kMxSlotBytes;
#pragma unroll
      for (int i = 0; i < CPT; ++i)
        va[i] = ld_shared_v4(slot + (in_row(i) ? (uint32_t)(threadIdx.x + i * kMxThreads) * 16u : 0u));
      __syncthreads();  // every thread has read its chunks of the slot
      if (threadIdx.x == 0) {
        fence_proxy_async_smem();
        issue(k + kMxSlots);  // the slot's next row
      }
      do_row(r, va);
    }
  } else {
    // two row buffers in turn: the next row's loads go out before this row's
    // arithmetic, with no copy between the buffers
    const int step = gridDim.y;
    int r = blockIdx.y;
    load_row(r, va);
    while (r < rows_iter) {
      const int r1 = r + step;
      if (r1 < rows_iter) load_row(r1, vb);
      do_row(r, va);
      if (r1 >= rows_iter) break;
      const int r2 = r1 + step;
      if (r2 < rows_iter) load_row(r2, va);
      do_row(r1, vb);
      r = r2;
    }
  }
}

// Grouped activations (MoE experts): the rows of x arrive sorted by expert,
// expert e owning rows row_off[e] .. row_off[e+1]-1.  Each expert's rows
// start a new 128-row token tile: compact row r of expert e goes to padded
// row 128 tile_off[e] + (r - row_off[e]), tile_off the running sum of
// ceil(rows_e / 128).  Every CTA forms tile_off in shared memory; the first
// also writes it out for the GEMM.  Codes go to 128-row token tiles, scales
// to the 128x4 layout over the padded rows; the padding rows of an expert's
// last tile are left unwritten (they only feed output rows that are never
// stored).  A half-warp covers 16 chunks (4 blocks) of one row, as in
// mx_quant_kernel.
__global__ void __launch_bounds__(kMxThreads) mx_quant_grouped_kernel(const uint16_t *__restrict__ x,
                                                                      long long ldx, int M_total, int K,
                                                                      const int *__restrict__ row_off,
                                                                      int E, int *__restrict__ tile_off_out,
                                                                      uint8_t *__restrict__ codes,
                                                                      uint8_t *__restrict__ sf) {
  __shared__ int s_row[kMaxGroups + 1];
  __shared__ int s_tile[kMaxGroups + 1];
  const int lane = threadIdx.x & 31;
  pdl_trigger();  // an activation step: the next kernel may launch now
  pdl_wait();     // x and row_off may come from the kernel ahead
  for (int e = threadIdx.x; e <= E; e += blockDim.x) s_row[e] = row_off[e];
  __syncthreads();
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int e = 0; e < E; ++e) {
      s_tile[e] = acc;
      acc += (s_row[e + 1] - s_row[e] + 127) >> 7;
    }
    s_tile[E] = acc;
  }
  __syncthreads();
  if (blockIdx.x == 0)
    for (int e = threadIdx.x; e <= E; e += blockDim.x) tile_off_out[e] = s_tile[e];
  const int cpr = K >> 3;  // 16-byte chunks per row, a multiple of 16
  const int G = K >> 5;
  const int KC = K >> 8;   // 128-byte code columns per row
  for (int r = blockIdx.x; r < M_total; r += gridDim.x) {
    int lo = 0, hi = E - 1;  // the expert of row r: the largest e with row_off[e] <= r
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_row[mid] <= r) lo = mid;
      else hi = mid - 1;
    }
    const int pr = (s_tile[lo] << 7) + (r - s_row[lo]);  // padded row
    for (int c0 = 0; c0 < cpr; c0 += kMxThreads) {
      const int c = c0 + (int)threadIdx.x;
      const bool in_row = c < cpr;  // uniform over a half-warp (cpr % 16 == 0)
      const uint4 v = in_row ? ld_stream_v4(x + (size_t)r * ldx + (size_t)c * 8) : make_uint4(0u, 0u, 0u, 0u);
      uint32_t scode;
      const uint32_t packed = mx_encode_chunk(v, scode);
      const uint32_t word = mx_scale_word(scode);
      if (in_row) {
        *reinterpret_cast<uint32_t *>(codes + tiled_offset(pr, c * 4, KC, 128)) = packed;
        if ((lane & 15) == 0)
          *reinterpret_cast<uint32_t *>(sf + sf_swizzled_offset(pr, c >> 2, G)) = word;
      }
    }
  }
}

constexpr int kF8Threads = 256;

// Read-only 16-byte load that stays in L1: the second pass over a row finds it there.
__device__ __forceinline__ uint4 ld_keep_v4(const uint16_t *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::evict_last.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t amax_bf16x8(const uint4 &w) {
  const uint32_t m2 = __vmaxu2(__vmaxu2(w.x & 0x7FFF7FFFu, w.y & 0x7FFF7FFFu),
                               __vmaxu2(w.z & 0x7FFF7FFFu, w.w & 0x7FFF7FFFu));
  return max(m2 & 0xFFFFu, m2 >> 16);
}

// x / s for the values x of one row and its scale s, rounded as the IEEE
// division is where it decides a code.  Markstein's correction step (P.
// Markstein, "IA-64 and Elementary Functions: Speed and Precision", 2000):
// with r = RN(1/s), q = RN(x r) and the exact residual e = x - q s (one
// FMA), RN(q + e r) is the correctly rounded quotient -- three operations a
// value instead of a division.  Checked exhaustively on GB300 over the
// quantizers' whole domain (every bf16 x with |x| <= amax, every finite bf16
// amax with s = RN(amax / 448) >= 2^-100): the quotient equals the IEEE one
// bit for bit wherever |x / s| >= 2^-10 (below, every quotient encodes to
// +-0), and the E4M3 codes are the same everywhere once the sign of x is
// set on the code, as fp8_quant8 does.  Rows with a smaller s (the residual
// would underflow) divide.
struct RowDivisor {
  float s, r;
  bool fast;
  __device__ __forceinline__ explicit RowDivisor(float s_) {
    s = s_;
    r = __fdiv_rn(1.0f, s_);
    fast = s_ >= 7.8886090522101181e-31f;  // 2^-100
  }
  // x / s on a fast row: one multiply, two fused multiply-adds
  __device__ __forceinline__ float correct(float x) const {
    const float q = __fmul_rn(x, r);
    return __fmaf_rn(__fmaf_rn(-q, s, x), r, q);
  }
};

// 8 bf16 values -> 8 E4M3 bytes: q = E4M3_RNE_sat(x / s), the sign of x kept
// on codes that round to zero (the correction step turns x = -0 into +0, so
// the sign bits are set from x).  kFast: the row's divisor is fast (the
// choice is made once per row, outside the loops over its chunks, so that
// the division's instructions stay out of the fast loop).
template <bool kFast>
__device__ __forceinline__ uint2 fp8_quant8(const uint4 &w, const RowDivisor &d) {
  auto q = [&](float x) { return kFast ? d.correct(x) : __fdiv_rn(x, d.s); };
  const uint32_t lo = e4m3x2(q(bf16_lo(w.x)), q(bf16_hi(w.x))) | (e4m3x2(q(bf16_lo(w.y)), q(bf16_hi(w.y))) << 16);
  const uint32_t hi = e4m3x2(q(bf16_lo(w.z)), q(bf16_hi(w.z))) | (e4m3x2(q(bf16_lo(w.w)), q(bf16_hi(w.w))) << 16);
  return make_uint2(lo | e4m3_signs4(w.x, w.y), hi | e4m3_signs4(w.z, w.w));
}

// Runs f(std::true_type) on a fast row, f(std::false_type) otherwise.
template <class F>
__device__ __forceinline__ void by_divisor(const RowDivisor &d, F &&f) {
  if (d.fast)
    f(std::true_type{});
  else
    f(std::false_type{});
}

// Where row r of a per-row FP8 output of K bytes goes: 128-byte column c of
// the row at base + c * col_stride, its 16-byte unit j at ((j ^ rsw) * 16).
// tile_rows: 0 = row-major, kPanelLayout = weight panels, else token tiles.
struct Fp8RowDest {
  size_t base, col_stride;
  int rsw;
  __device__ __forceinline__ Fp8RowDest(int r, int K, int tile_rows) {
    const int KC = K >> 7;  // 128-byte columns per row
    if (tile_rows == kPanelLayout) {
      base = (size_t)(r >> 8) * KC * kF8PanelBytes + (size_t)((r >> 7) & 1) * 16384u + (size_t)(r & 127) * 128u;
      col_stride = kF8PanelBytes;
      rsw = r & 7;
    } else if (tile_rows > 0) {
      const int t_shift = __ffs(tile_rows) - 1;  // tile_rows is a power of 2
      const int rr = r & (tile_rows - 1);
      base = ((size_t)(r >> t_shift) * KC << (t_shift + 7)) + (size_t)rr * 128u;
      col_stride = (size_t)tile_rows * 128u;
      rsw = rr & 7;
    } else {
      base = (size_t)r * K;
      col_stride = 128;
      rsw = 0;
    }
  }
  // the 8 bytes of 8-value chunk c
  __device__ __forceinline__ uint2 *chunk(uint8_t *q, int c) const {
    const int b = c * 8;
    return reinterpret_cast<uint2 *>(q + base + (size_t)(b >> 7) * col_stride +
                                     (size_t)((((b >> 4) & 7) ^ rsw) << 4) + (b & 15));
  }
};

// One CTA per row (grid-stride over rows), two passes over the row: the
// amax, then the codes (the row is re-read from L1).  Few registers, so the
// CTAs fit beside a resident GEMM CTA.  tile_rows: 0 = row-major q,
// kPanelLayout = weight panels (rows_iter = rows rounded up to the panel;
// the padding rows get zero bytes and no scale), else the tile layout with
// that tile height.
__global__ void __maxnreg__(40) fp8_quant_kernel(const uint16_t *__restrict__ x,
                                                               long long ldx, int rows,
                                                               int rows_iter, int K,
                                                               int tile_rows, int early_trigger,
                                                               uint8_t *__restrict__ q,
                                                               float *__restrict__ scale) {
  __shared__ uint32_t red[kF8Threads / 32];
  const int cpr = K >> 3;
  const int tid = threadIdx.x;
  if (early_trigger) pdl_trigger();  // activations only, as in mx_quant_kernel
  if (threadIdx.x == 0 && (int)blockIdx.x < rows) {  // warm L2 with the first row
    const uint16_t *xr = x + (size_t)blockIdx.x * ldx;
    for (int c = 0; c < cpr; c += 1024)  // 16 KiB pieces
      prefetch_l2_bulk(xr + (size_t)c * 8, (uint32_t)min(1024, cpr - c) * 16u);
  }
  pdl_wait();
  for (int r = blockIdx.x; r < rows_iter; r += gridDim.x) {
    const Fp8RowDest dst(r, K, tile_rows);
    if (r >= rows) {  // panel padding (uniform over the CTA)
      for (int c = tid; c < cpr; c += kF8Threads) *dst.chunk(q, c) = make_uint2(0u, 0u);
      continue;
    }
    const uint16_t *xr = x + (size_t)r * ldx;
    uint32_t amax = 0;
    int c = tid;
    for (; c + 3 * kF8Threads < cpr; c += 4 * kF8Threads) {  // 4 loads in flight
      const uint4 a = ld_keep_v4(xr + (size_t)c * 8);
      const uint4 b = ld_keep_v4(xr + (size_t)(c + kF8Threads) * 8);
      const uint4 d = ld_keep_v4(xr + (size_t)(c + 2 * kF8Threads) * 8);
      const uint4 e = ld_keep_v4(xr + (size_t)(c + 3 * kF8Threads) * 8);
      amax = max(max(amax, amax_bf16x8(a)), max(amax_bf16x8(b), max(amax_bf16x8(d), amax_bf16x8(e))));
    }
    for (; c < cpr; c += kF8Threads) amax = max(amax, amax_bf16x8(ld_keep_v4(xr + (size_t)c * 8)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = max(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    if ((tid & 31) == 0) red[tid >> 5] = amax;
    __syncthreads();
    amax = red[0];
#pragma unroll
    for (int i = 1; i < kF8Threads / 32; ++i) amax = max(amax, red[i]);
    __syncthreads();  // red[] is reused by the next row

    if (amax >= 0x7F80u) {  // Inf or NaN in the row
      if (tid == 0) scale[r] = __uint_as_float(0x7FC00000u);
      for (int c = tid; c < cpr; c += kF8Threads) *dst.chunk(q, c) = make_uint2(0u, 0u);
      continue;
    }
    const float s = (amax == 0u) ? 1.0f : __fdiv_rn(__uint_as_float(amax << 16), 448.0f);
    if (tid == 0) scale[r] = s;
    const RowDivisor dv(s);
    by_divisor(dv, [&](auto fast) {
      for (int c = tid; c < cpr; c += kF8Threads)
        *dst.chunk(q, c) = fp8_quant8<decltype(fast)::value>(ld_keep_v4(xr + (size_t)c * 8), dv);
    });
  }
}

// The same per-row FP8 quantization for large inputs with K <= 8192: the
// CTA's rows stream into a ring of kF8Slots row buffers in shared memory by
// bulk copies (one thread issues them; the bytes in flight are not bounded
// by registers), each row read from shared memory once into registers
// (kF8Hold chunks of 8 values per thread), reduced, and quantized.  (The
// two-pass kernel above, at 40 registers and no shared memory, is kept for
// decode-sized inputs, whose CTAs sit beside GEMM CTAs of a layer chain.)
constexpr int kF8Hold = 4;
constexpr int kF8Slots = 3;
size_t fp8_staged_smem(int K) { return (size_t)kF8Slots * ((size_t)K * 2u) + 8u * kF8Slots; }

__global__ void __launch_bounds__(kF8Threads) fp8_quant_staged_kernel(const uint16_t *__restrict__ x,
                                                                      long long ldx, int rows, int rows_iter,
                                                                      int K, int tile_rows, int early_trigger,
                                                                      uint8_t *__restrict__ q,
                                                                      float *__restrict__ scale) {
  extern __shared__ __align__(128) uint8_t ring[];  // kF8Slots rows of K bf16, then one mbarrier a slot
  __shared__ uint32_t red[2][kF8Threads / 32];
  __shared__ int abort_flag;
  const int cpr = K >> 3;  // <= kF8Hold * kF8Threads
  const int tid = threadIdx.x;
  const uint32_t row_bytes = (uint32_t)K * 2u;  // a multiple of 256
  const uint32_t slots = smem_addr(ring);
  const uint32_t bars = slots + kF8Slots * row_bytes;
  if (early_trigger) pdl_trigger();
  if (tid == 0) {
    for (int i = 0; i < kF8Slots; ++i) mbar_init(bars + 8u * i, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  pdl_wait();  // x may be the previous kernel's output
  const WaitCtl ctl{&abort_flag, nullptr, kQuantWaitNs};
  // row k of this CTA is blockIdx.x + k * gridDim.x; thread 0 copies it into
  // slot k % kF8Slots (rows past the input -- panel padding -- are not read)
  auto row_of = [&](int k) { return (int)blockIdx.x + k * (int)gridDim.x; };
  auto issue = [&](int k) {
    const int r = row_of(k);
    if (r >= rows) return;
    const uint32_t bar = bars + 8u * (uint32_t)(k % kF8Slots);
    mbar_arrive_expect_tx(bar, row_bytes);
    bulk_load(slots + (uint32_t)(k % kF8Slots) * row_bytes, x + (size_t)r * ldx, row_bytes, bar,
              policy_evict_first());
  };
  if (tid == 0)
    for (int k = 0; k < kF8Slots; ++k) issue(k);
  // this thread's chunks tid + 256 i, i < kF8Hold: in the row or past it
  // (past it, a thread reads the row's first chunk -- a repeat does not
  // change the row's amax -- and stores nothing).  Within a row, chunk i's
  // codes go at col0 + i * step (the same 16-byte unit of a column 16
  // columns on).
  const size_t col_stride = tile_rows == kPanelLayout ? (size_t)kF8PanelBytes
                            : tile_rows > 0           ? (size_t)tile_rows * 128u
                                                      : 128u;
  const size_t col0 = (size_t)(tid >> 4) * col_stride + (size_t)((tid & 1) * 8);
  const size_t step = 16 * col_stride;
  const uint32_t unit = (uint32_t)(tid >> 1) & 7u;
  auto in_row = [&](int i) { return tid + i * kF8Threads < cpr; };
  int parity = 0;
  for (int k = 0; row_of(k) < rows_iter; ++k) {
    const int r = row_of(k);
    const Fp8RowDest dst(r, K, tile_rows);
    uint8_t *const at = q + dst.base + col0 + ((unit ^ (uint32_t)dst.rsw) << 4);
    if (r >= rows) {  // panel padding (uniform over the CTA; after every real row): zero bytes, no scale
#pragma unroll
      for (int i = 0; i < kF8Hold; ++i) st_global_v2_if(at + i * step, make_uint2(0u, 0u), in_row(i));
      continue;
    }
    const uint32_t slot = slots + (uint32_t)(k % kF8Slots) * row_bytes;
    const bool landed = mbar_wait(bars + 8u * (uint32_t)(k % kF8Slots), (uint32_t)(k / kF8Slots) & 1u, ctl);
    if (__syncthreads_or(!landed)) {
      // a copy did not land: let every copy still in flight finish (bounded),
      // mark this CTA's rows from here on with NaN scales, and leave
      if (tid == 0)
        for (int j = k; j < k + kF8Slots; ++j)
          if (row_of(j) < rows) drain_copy(bars + 8u * (uint32_t)(j % kF8Slots), (uint32_t)(j / kF8Slots) & 1u);
      for (int j = k; tid == 0 && row_of(j) < rows; ++j) scale[row_of(j)] = __uint_as_float(0x7FC00000u);
      return;
    }
    uint4 v[kF8Hold];
#pragma unroll
    for (int i = 0; i < kF8Hold; ++i) v[i] = ld_shared_v4(slot + (in_row(i) ? (uint32_t)(tid + i * kF8Threads) * 16u : 0u));
    uint32_t amax = 0;
#pragma unroll
    for (int i = 0; i < kF8Hold; ++i) amax = max(amax, amax_bf16x8(v[i]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = max(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    // two reduction buffers, alternating over the rows that reduce: one
    // barrier a row suffices (a buffer is rewritten only after the barrier
    // of the row between, which every reader of it has passed)
    if ((tid & 31) == 0) red[parity][tid >> 5] = amax;
    __syncthreads();  // also: every thread has read its chunks of the slot
    if (tid == 0) {
      fence_proxy_async_smem();
      issue(k + kF8Slots);  // the slot's next row
    }
    amax = red[parity][0];
#pragma unroll
    for (int i = 1; i < kF8Threads / 32; ++i) amax = max(amax, red[parity][i]);
    parity ^= 1;
    if (amax >= 0x7F80u) {  // Inf or NaN in the row
      if (tid == 0) scale[r] = __uint_as_float(0x7FC00000u);
#pragma unroll
      for (int i = 0; i < kF8Hold; ++i) st_global_v2_if(at + i * step, make_uint2(0u, 0u), in_row(i));
      continue;
    }
    const float s = (amax == 0u) ? 1.0f : __fdiv_rn(__uint_as_float(amax << 16), 448.0f);
    if (tid == 0) scale[r] = s;
    const RowDivisor dv(s);
    by_divisor(dv, [&](auto fast) {
#pragma unroll
      for (int i = 0; i < kF8Hold; ++i)
        st_global_v2_if(at + i * step, fp8_quant8<decltype(fast)::value>(v[i], dv), in_row(i));
    });
  }
}

// ---------------------------------------------------------------------------
// SwiGLU between the packed gate_up projection and the down projection, fused
// with the per-token FP8 quantization of its output ("Kimi-K3-DSpark-FP8-PTPC",
// "Phase 1 FP8 PTPC Quantization": gate_proj and up_proj packed into one
// gate_up_proj; the activation is the SwiGLU reading).  A gate_up output row
// is [gate (I) | up (I)]; h = bf16(silu(gate) * up) with
//   silu(g) * u = (g / (1 + e^-g)) * u
// formed in binary32 one IEEE operation at a time (no contraction), and e^t
// by the method of Cody and Waite (Software Manual for the Elementary
// Functions, 1980): n = rint(t / ln2), r = (t - n L1) - n L2 with ln2 split
// so that n L1 is exact, e^r by its Taylor series through r^7/7! (Horner,
// each step one fused multiply-add), times 2^n.  h is then quantized per row exactly as fp8_quant_kernel does.
__device__ __forceinline__ float cw_exp(float t) {
  if (t != t) return t;
  if (t > 88.72283f) return __int_as_float(0x7F800000);
  if (t < -87.3f) return 0.0f;
  const float log2e = 0x1.715476p+0f;   // 1/ln2 rounded to binary32
  const float L1 = 0x1.62e4p-1f;        // 15 significant bits: n * L1 exact for |n| <= 128
  const float L2 = 0x1.7f7d1cp-20f;     // ln2 - L1 rounded to binary32
  // n = rint(t log2e), round half to even: for |t log2e| < 2^22, adding
  // 1.5 2^23 rounds to an integer in the low mantissa bits and subtracting
  // it back is exact -- the same n as rintf, and n's bits come for free
  const float big = __fadd_rn(__fmul_rn(t, log2e), 0x1.8p+23f);
  const float nf = __fsub_rn(big, 0x1.8p+23f);
  const int n = (int)(__float_as_uint(big) & 0x7FFFFFu) - 0x400000;
  float r = __fsub_rn(t, __fmul_rn(nf, L1));
  r = __fsub_rn(r, __fmul_rn(nf, L2));
  float p = 0x1.a01a02p-13f;                   // 1/7!
  p = __fmaf_rn(p, r, 0x1.6c16c2p-10f);         // 1/6!
  p = __fmaf_rn(p, r, 0x1.111112p-7f);          // 1/5!
  p = __fmaf_rn(p, r, 0x1.555556p-5f);          // 1/4!
  p = __fmaf_rn(p, r, 0x1.555556p-3f);          // 1/3!
  p = __fmaf_rn(p, r, 0.5f);
  p = __fmaf_rn(p, r, 1.0f);
  p = __fmaf_rn(p, r, 1.0f);
  if (n > 127) return __fmul_rn(__fmul_rn(p, __uint_as_float(254u << 23)), 2.0f);
  return __fmul_rn(p, __uint_as_float((uint32_t)(n + 127) << 23));
}

// silu(g) = g / (1 + e^-g) in binary32
__device__ __forceinline__ float silu_f32(float g) { return __fdiv_rn(g, __fadd_rn(1.0f, cw_exp(-g))); }

// silu depends on the bf16 gate alone: a table of it over the gates with
// 2^-25 <= |g| < 2^7 (biased exponents kSiluE0 .. kSiluE0 + 31, both signs;
// what a bf16 gate_up output holds nearly always), index sign * 4096 +
// (exponent - kSiluE0) * 128 + mantissa, each entry formed by silu_f32
// itself.  Gates outside it (zeros, tiny, huge, non-finite) take silu_f32
// directly, so the result is the same bit for bit either way.
constexpr uint32_t kSiluE0 = 102;
constexpr int kSiluEntries = 2 * 32 * 128;
constexpr int kSiluTableBytes = kSiluEntries * 4;

__device__ __forceinline__ float silu_of_bits(uint32_t gb, const float *tab) {
  if (tab) {
    const uint32_t rel = (gb & 0x7FFFu) - (kSiluE0 << 7);  // wraps above 4095 below the range
    if (rel < (32u << 7)) return tab[((gb >> 15) << 12) | rel];
  }
  return silu_f32(__uint_as_float(gb << 16));
}

// two bf16 gate values and the matching up values -> two bf16 h values,
// h = bf16(silu(g) * u)
__device__ __forceinline__ uint32_t swiglu2(uint32_t g, uint32_t u, const float *tab) {
  return pack_bf16x2(__fmul_rn(silu_of_bits(g & 0xFFFFu, tab), bf16_lo(u)),
                     __fmul_rn(silu_of_bits(g >> 16, tab), bf16_hi(u)));
}

// A chunk of 8 gates with any of them outside the table: each value on its
// own (not inlined, so that none of silu_f32 lands in the table path).
__device__ __noinline__ uint4 swiglu8_any(uint4 g, uint4 u, const float *tab) {
  return make_uint4(swiglu2(g.x, u.x, tab), swiglu2(g.y, u.y, tab), swiglu2(g.z, u.z, tab),
                    swiglu2(g.w, u.w, tab));
}

// For the two bf16 gates of g: (|g| | 0x8000) - (kSiluE0 << 7) per half (no
// borrow crosses the halves), which lies in [0x8000, 0x9000) -- its low 12
// bits the table index without the sign -- exactly when the gate is inside
// the table.
__device__ __forceinline__ uint32_t table_rel2(uint32_t g) {
  return ((g & 0x7FFF7FFFu) | 0x80008000u) - (kSiluE0 << 7) * 0x10001u;
}

// two gates known to be inside the table
__device__ __forceinline__ uint32_t swiglu2_table(uint32_t g, uint32_t t, uint32_t u, const float *tab) {
  const uint32_t i_lo = (t & 0xFFFu) | ((g >> 3) & 0x1000u);
  const uint32_t i_hi = ((t >> 16) & 0xFFFu) | ((g >> 19) & 0x1000u);
  return pack_bf16x2(__fmul_rn(tab[i_lo], bf16_lo(u)), __fmul_rn(tab[i_hi], bf16_hi(u)));
}

__device__ __forceinline__ uint4 swiglu8(const uint4 &g, const uint4 &u, const float *tab) {
  if (tab) {
    // each half of a t word lies in [0x4D00, 0xCCFF]: its top four bits are
    // 8 inside the table and another nonzero value outside, so OR-ed over
    // the chunk they are 8 only if every gate is inside
    const uint4 t = make_uint4(table_rel2(g.x), table_rel2(g.y), table_rel2(g.z), table_rel2(g.w));
    if (((t.x | t.y | t.z | t.w) & 0xF000F000u) == 0x80008000u)
      return make_uint4(swiglu2_table(g.x, t.x, u.x, tab), swiglu2_table(g.y, t.y, u.y, tab),
                        swiglu2_table(g.z, t.z, u.z, tab), swiglu2_table(g.w, t.w, u.w, tab));
  }
  return swiglu8_any(g, u, tab);
}

constexpr int kSwThreads = 256;
constexpr int kSwUnroll = 3;  // chunk pairs (gate, up) whose loads are in flight together

// One CTA per row (grid-stride over rows): pass 1 forms h for the row into
// shared memory (I bf16) and takes its amax; pass 2 quantizes h from shared
// memory into q (row-major or the down GEMM's token tiles) and writes the
// row's scale.  h_out (optional) receives h itself.  kTable: the silu table
// sits in shared memory after the row (filled before the dependency wait,
// while the kernel ahead finishes).
template <bool kTable>
__global__ void __launch_bounds__(kSwThreads) swiglu_fp8_kernel(const uint16_t *__restrict__ gu,
                                                                long long ldgu, int rows, int I,
                                                                int tile_rows, uint16_t *__restrict__ h_out,
                                                                long long ldh, uint8_t *__restrict__ q,
                                                                float *__restrict__ scale) {
  extern __shared__ uint4 hrow[];  // I / 8 chunks of 8 bf16, then (kTable) the silu table
  __shared__ uint32_t red[kSwThreads / 32];
  const int tid = threadIdx.x;
  const int cpr = I >> 3;
  pdl_trigger();  // an activation step: the next kernel may launch now
  if (tid == 0 && (int)blockIdx.x < rows) {  // warm L2 with the first row
    const uint16_t *g = gu + (size_t)blockIdx.x * ldgu;
    for (int c = 0; c < 2 * cpr; c += 1024)
      prefetch_l2_bulk(g + (size_t)c * 8, (uint32_t)min(1024, 2 * cpr - c) * 16u);
  }
  float *tab = nullptr;
  if (kTable) {
    tab = reinterpret_cast<float *>(hrow + cpr);
    for (int i = tid; i < kSiluEntries; i += kSwThreads) {
      const uint32_t gb = ((uint32_t)(i >> 12) << 15) | ((kSiluE0 << 7) + (uint32_t)(i & 0xFFF));
      tab[i] = silu_f32(__uint_as_float(gb << 16));
    }
    __syncthreads();
  }
  pdl_wait();  // gu comes from the kernel ahead (the gate_up GEMM)
  for (int r = blockIdx.x; r < rows; r += gridDim.x) {
    const uint16_t *gr = gu + (size_t)r * ldgu;
    const uint16_t *ur = gr + I;
    if (tid == 0 && r + (int)gridDim.x < rows) {  // warm L2 with this CTA's next row
      const uint16_t *g = gu + (size_t)(r + gridDim.x) * ldgu;
      for (int c = 0; c < 2 * cpr; c += 1024)
        prefetch_l2_bulk(g + (size_t)c * 8, (uint32_t)min(1024, 2 * cpr - c) * 16u);
    }
    uint32_t amax = 0;
    for (int c0 = tid; c0 < cpr; c0 += kSwUnroll * kSwThreads) {
      uint4 g[kSwUnroll], u[kSwUnroll];
#pragma unroll
      for (int j = 0; j < kSwUnroll; ++j) {
        const int c = c0 + j * kSwThreads;
        if (c < cpr) {
          g[j] = ld_stream_v4(gr + (size_t)c * 8);
          u[j] = ld_stream_v4(ur + (size_t)c * 8);
        }
      }
#pragma unroll
      for (int j = 0; j < kSwUnroll; ++j) {
        const int c = c0 + j * kSwThreads;
        if (c < cpr) {
          const uint4 h = swiglu8(g[j], u[j], tab);
          hrow[c] = h;
          if (h_out) *reinterpret_cast<uint4 *>(h_out + (size_t)r * ldh + (size_t)c * 8) = h;
          amax = max(amax, amax_bf16x8(h));
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = max(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    if ((tid & 31) == 0) red[tid >> 5] = amax;
    __syncthreads();  // also: hrow complete
    amax = red[0];
#pragma unroll
    for (int i = 1; i < kSwThreads / 32; ++i) amax = max(amax, red[i]);
    const Fp8RowDest dst(r, I, tile_rows);
    if (amax >= 0x7F80u) {  // Inf or NaN in h
      if (tid == 0) scale[r] = __uint_as_float(0x7FC00000u);
      for (int c = tid; c < cpr; c += kSwThreads) *dst.chunk(q, c) = make_uint2(0u, 0u);
    } else {
      const float s = (amax == 0u) ? 1.0f : __fdiv_rn(__uint_as_float(amax << 16), 448.0f);
      if (tid == 0) scale[r] = s;
      const RowDivisor dv(s);
      by_divisor(dv, [&](auto fast) {
        for (int c = tid; c < cpr; c += kSwThreads)
          *dst.chunk(q, c) = fp8_quant8<decltype(fast)::value>(hrow[c], dv);
      });
    }
    __syncthreads();  // red[] and hrow are reused by the next row
  }
}

}  // namespace

cudaError_t launch_mx_quant(const void *x, long long ldx, int rows, int K, uint8_t *codes,
                            uint8_t *sf, bool swizzled, int tile_rows, bool act, int sm_count,
                            cudaStream_t stream, const QuantWatch &watch) {
  const int cpr = K / 8;
  const bool big = rows > 512;
  const int per_block = kMxThreads * (big ? 4 : 2);
  const int gx = (cpr + per_block - 1) / per_block;
  const int rows_iter = tile_rows == kPanelLayout ? ((rows + kPanelRows - 1) / kPanelRows) * kPanelRows
                        : swizzled                   ? ((rows + 127) / 128) * 128
                                                     : rows;
  auto kern = swizzled ? (big ? mx_quant_kernel<true, 4, true> : mx_quant_kernel<true, 2, false>)
                       : (big ? mx_quant_kernel<false, 4, true> : mx_quant_kernel<false, 2, false>);
  const size_t smem = big ? kMxStagedSmem : 0;
  cudaError_t e = prefer_shared_carveout(kern);
  if (e != cudaSuccess) return e;
  if (big) {
    static DeviceOnce once[2];
    int dev = -1;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if (!once[swizzled].done(dev)) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMxStagedSmem);
      if (e != cudaSuccess) return e;
      once[swizzled].set(dev);
    }
  }
  // as many CTAs as are resident at once (one wave), rows beyond that
  // grid-strided; for a decode-sized activation (a few hundred rows at most)
  // one CTA per SM: launched early beside the GEMMs of a layer chain, a
  // second quantizer CTA on an SM would leave no registers for the next GEMM
  // CTA
  int per_sm = 1;
  if (!(act && rows <= 512) && (e = resident_ctas_per_sm(kern, kMxThreads, smem, &per_sm)) != cudaSuccess) return e;
  int gy = rows_iter;
  const int sms = sm_count > 0 ? sm_count : 152;
  const int cap = sms * per_sm;
  if (gy * gx > cap) gy = (cap + gx - 1) / gx;
  if (gy > 65535) gy = 65535;
  if (gy < 1) gy = 1;
  cudaLaunchConfig_t cfg = pdl_config(dim3(gx, gy), dim3(kMxThreads), smem, stream);
  cudaLaunchAttribute attr[1];
  attach_pdl(cfg, attr);
  const uint16_t *xp = static_cast<const uint16_t *>(x);
  return cudaLaunchKernelEx(&cfg, kern, xp, ldx, rows, rows_iter, K, tile_rows, act ? 1 : 0, codes, sf,
                            watch.status, watch.timeout_ns, watch.debug_stall);
}

cudaError_t launch_fp8_quant(const void *x, long long ldx, int rows, int K, uint8_t *q,
                             float *scale, int tile_rows, bool act, int sm_count,
                             cudaStream_t stream) {
  const int rows_iter =
      tile_rows == kPanelLayout ? ((rows + kPanelRows - 1) / kPanelRows) * kPanelRows : rows;
  // large inputs whose rows fit in the CTA's registers: rows staged in
  // shared memory by bulk copies, one read of each
  const bool staged = rows > 512 && K / 8 <= kF8Hold * kF8Threads;
  auto kern = staged ? fp8_quant_staged_kernel : fp8_quant_kernel;
  const size_t smem = staged ? fp8_staged_smem(K) : 0;
  cudaError_t e = prefer_shared_carveout(kern);
  if (e != cudaSuccess) return e;
  if (staged) {
    static DeviceOnce once;
    int dev = -1;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if (!once.done(dev)) {
      e = cudaFuncSetAttribute(fp8_quant_staged_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)fp8_staged_smem(8192));
      if (e != cudaSuccess) return e;
      once.set(dev);
    }
  }
  // one CTA per row, at most as many as are resident at once (one wave)
  int per_sm = 1;
  if ((e = resident_ctas_per_sm(kern, kF8Threads, smem, &per_sm)) != cudaSuccess) return e;
  int g = rows_iter;
  const int cap = (sm_count > 0 ? sm_count : 152) * per_sm;
  if (g > cap) g = cap;
  cudaLaunchConfig_t cfg = pdl_config(dim3(g), dim3(kF8Threads), smem, stream);
  cudaLaunchAttribute attr[1];
  attach_pdl(cfg, attr);
  return cudaLaunchKernelEx(&cfg, kern, static_cast<const uint16_t *>(x), ldx, rows, rows_iter, K, tile_rows,
                            act ? 1 : 0, q, scale);
}

cudaError_t launch_mx_quant_grouped(const void *x, long long ldx, int M_total, int K, const int *row_off,
                                    int E, int *tile_off, uint8_t *codes, uint8_t *sf, int sm_count,
                                    cudaStream_t stream) {
  cudaError_t e = prefer_shared_carveout(mx_quant_grouped_kernel);
  if (e != cudaSuccess) return e;
  int per_sm = 1;  // one wave of CTAs, rows grid-strided
  if ((e = resident_ctas_per_sm(mx_quant_grouped_kernel, kMxThreads, 0, &per_sm)) != cudaSuccess) return e;
  int g = M_total < 1 ? 1 : M_total;
  const int cap = (sm_count > 0 ? sm_count : 152) * per_sm;
  if (g > cap) g = cap;
  cudaLaunchConfig_t cfg = pdl_config(dim3(g), dim3(kMxThreads), 0, stream);
  cudaLaunchAttribute attr[1];
  attach_pdl(cfg, attr);
  return cudaLaunchKernelEx(&cfg, mx_quant_grouped_kernel, static_cast<const uint16_t *>(x), ldx, M_total, K,
                            row_off, E, tile_off, codes, sf);
}

cudaError_t launch_swiglu_fp8(const void *gu, long long ldgu, int rows, int I, int tile_rows, void *h_out,
                              long long ldh, uint8_t *q, float *scale, int sm_count, cudaStream_t stream) {
  constexpr size_t kMaxSmem = 200u * 1024u;
  const bool table = (size_t)I * 2u + kSiluTableBytes <= kMaxSmem;
  const size_t smem = (size_t)I * 2u + (table ? kSiluTableBytes : 0);
  auto kern = table ? swiglu_fp8_kernel<true> : swiglu_fp8_kernel<false>;
  static DeviceOnce once[2];
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (!once[table].done(dev)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMaxSmem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    once[table].set(dev);
  }
  int per_sm = 1;  // one wave of CTAs, rows grid-strided
  if ((e = resident_ctas_per_sm(kern, kSwThreads, smem, &per_sm)) != cudaSuccess) return e;
  int g = rows;
  const int cap = (sm_count > 0 ? sm_count : 152) * per_sm;
  if (g > cap) g = cap;
  cudaLaunchConfig_t cfg = pdl_config(dim3(g), dim3(kSwThreads), smem, stream);
  cudaLaunchAttribute attr[1];
  attach_pdl(cfg, attr);
  return cudaLaunchKernelEx(&cfg, kern, static_cast<const uint16_t *>(gu), ldgu, rows, I, tile_rows,
                            static_cast<uint16_t *>(h_out), ldh, q, scale);
}

}  // namespace mxg
