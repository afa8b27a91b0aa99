// quant_math.cuh -- the per-value arithmetic and the output layouts of the
// quantizer kernels.
//
// OCP-MX MXFP4 ("Kimi-K3 DSpark O-Proj-only MXFP4", "Exact quantization
// coverage"): a 32-value block gets the E8M0 scale e = clamp(floor(log2 amax)
// - 2, -127, 127) and codes E2M1_RNE_sat(x * 2^-e) with the sign of x.
// FP8 PTPC ("Kimi-K3-DSpark-FP8-PTPC", "Phase 1 FP8 PTPC Quantization"): s =
// amax / 448, q = E4M3_RNE_sat(x / s).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace mxg {

// Two fp32 values -> one byte of two E2M1 codes (lo in the low nibble),
// round to nearest even, saturating to +-6.
__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi) {
  uint16_t r;
  asm("{\n\t.reg .b8 t;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
      "cvt.u16.u8 %0, t;\n\t}"
      : "=h"(r)
      : "f"(hi), "f"(lo));
  return r;
}

// Two fp32 values -> two E4M3 bytes (lo in the low byte), RNE, saturating.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// The sign bits of the four bf16 values in (a, b) (a's low, a's high, b's
// low, b's high) at bits 7, 15, 23 and 31: the sign bits of their four E4M3
// bytes.  One byte permute whose selectors (source bytes 1, 3, 5, 7, the
// high bytes of the four values) have the sign-replicate bit set, then the
// byte sign bits kept.
__device__ __forceinline__ uint32_t e4m3_signs4(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, 0xFDB9;" : "=r"(r) : "r"(a), "r"(b));
  return r & 0x80808080u;
}


__device__ __forceinline__ uint4 ld_stream_v4(const uint16_t *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Byte offset of (row r, byte b of the row) in the tile layout with T-row
// tiles (T = 128 for weights; the GEMM's token tile for activations): tile
// (r / T, b / 128) of T rows x 128 bytes at ((r/T)*KC + b/128) * T * 128, and
// the 16-byte unit j of row r at (r % T) * 128 + ((j ^ (r % 8)) * 16).
__device__ __forceinline__ size_t tiled_offset(int r, int b, int kc_per_row, int T) {
  const int j = (b >> 4) & 7;
  const int rt = r / T;
  return ((size_t)rt * kc_per_row + (b >> 7)) * (size_t)T * 128u + (size_t)(r - rt * T) * 128u +
         (size_t)((j ^ (r & 7)) << 4) + (b & 15);
}

// Weight panel layout: rows in panels of 256; per panel and 128-byte column
// kc one block of panel_bytes holding the codes of the panel's two 128-row
// halves (16 KiB each, laid out as a tile above: byte b of row r at
// ((r / 256) * KC + b / 128) * panel_bytes + ((r / 128) % 2) * 16384 +
// (r % 128) * 128 + (((b / 16) % 8) ^ (r % 8)) * 16 + b % 16), then -- MXFP4
// -- the scale atoms of the two halves (1 KiB each: the column's two 512-byte
// atoms of the 128x4-tile scale layout).  The 4-byte scale word of groups
// g..g+3 (g % 4 == 0) of row r (MXFP4: 8 groups per column, panel_bytes =
// 34816) sits at:
__device__ __forceinline__ size_t panel_sf_offset(int r, int g, int kc_per_row) {
  return ((size_t)(r >> 8) * kc_per_row + (g >> 3)) * 34816u + 32768u + (size_t)((r >> 7) & 1) * 1024u +
         (size_t)((g >> 2) & 1) * 512u + (size_t)(r & 31) * 16u + (size_t)((r >> 5) & 3) * 4u;
}

// One 16-byte chunk (8 bf16 = a quarter of an MX block) per lane; four
// consecutive lanes hold one block.  Returns the 8 packed E2M1 codes (value
// 2i in the low nibble of byte i) and the block's E8M0 code in `scode`.
// Every lane of the warp must call it (the block amax is a 4-lane shuffle).
__device__ __forceinline__ uint32_t mx_encode_chunk(const uint4 &w, uint32_t &scode) {
  const unsigned kFull = 0xFFFFFFFFu;
  // |x| as bf16 bits; unsigned max orders finite < inf < nan.
  const uint32_t m2 = __vmaxu2(__vmaxu2(w.x & 0x7FFF7FFFu, w.y & 0x7FFF7FFFu),
                               __vmaxu2(w.z & 0x7FFF7FFFu, w.w & 0x7FFF7FFFu));
  uint32_t amax = max(m2 & 0xFFFFu, m2 >> 16);
  amax = max(amax, __shfl_xor_sync(kFull, amax, 1));
  amax = max(amax, __shfl_xor_sync(kFull, amax, 2));
  // floor(log2 amax) = ef - 127 for a normal amax; a zero or subnormal amax
  // clamps to e = -127 like ef in {1, 2}: e = max(ef, 2) - 129.  A block
  // holding Inf or NaN (amax >= 0x7F80) gets scale code 0xFF and zero codes;
  // its conversions below run on a finite 2^-e (ef <= 255) and are dropped.
  const bool bad = amax >= 0x7F80u;
  const int ef = max(static_cast<int>(amax >> 7), 2);
  scode = bad ? 0xFFu : static_cast<uint32_t>(ef - 2);
  const float inv = __uint_as_float(static_cast<uint32_t>(256 - ef) << 23);  // 2^-e
  // four conversions of two values each, the four code bytes packed by one
  // vector move (value 2i in the low nibble of byte i); the conversion keeps
  // the sign of a value that rounds to zero (-0 -> code 0x8)
  uint32_t packed;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(packed)
      : "f"(bf16_lo(w.x) * inv), "f"(bf16_hi(w.x) * inv), "f"(bf16_lo(w.y) * inv), "f"(bf16_hi(w.y) * inv),
        "f"(bf16_lo(w.z) * inv), "f"(bf16_hi(w.z) * inv), "f"(bf16_lo(w.w) * inv), "f"(bf16_hi(w.w) * inv));
  return bad ? 0u : packed;
}

// The scales of 4 consecutive blocks (lanes 0, 4, 8, 12 of a half-warp) as
// one 32-bit word, valid in lanes 0 and 16: two blocks per word in lanes 0,
// 8, 16, 24 first, then the pairs joined.  Every lane must call it.
__device__ __forceinline__ uint32_t mx_scale_word(uint32_t scode) {
  const unsigned kFull = 0xFFFFFFFFu;
  const uint32_t two = scode | (__shfl_down_sync(kFull, scode, 4) << 8);
  return two | (__shfl_down_sync(kFull, two, 8) << 16);
}

// A 64-bit global store that only the lanes with `pred` make.
__device__ __forceinline__ void st_global_v2_if(void *p, uint2 v, bool pred) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %3, 0;\n\t"
      "@p st.global.v2.b32 [%0], {%1, %2};\n\t}" ::"l"(p),
      "r"(v.x), "r"(v.y), "r"((uint32_t)pred)
      : "memory");
}

// A 32-bit global store that only the lanes with `pred` make (a predicated
// store, no branch around it).
__device__ __forceinline__ void st_global_b32_if(void *p, uint32_t v, bool pred) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %2, 0;\n\t"
      "@p st.global.b32 [%0], %1;\n\t}" ::"l"(p),
      "r"(v), "r"((uint32_t)pred)
      : "memory");
}

// Byte offset of the scale of (row r, block g) -- g % 4 == 0 for a word -- in
// the 128x4-tile layout: 512-byte tiles of 128 rows x 4 blocks, row-block
// major, then (r % 32) * 16 + ((r % 128) / 32) * 4 + g % 4.  G = blocks/row.
__device__ __forceinline__ size_t sf_swizzled_offset(int r, int g, int G) {
  return ((size_t)(r >> 7) * (size_t)(G >> 2) + (size_t)(g >> 2)) * 512u + (size_t)(r & 31) * 16u +
         (size_t)((r >> 5) & 3) * 4u;
}

}  // namespace mxg
