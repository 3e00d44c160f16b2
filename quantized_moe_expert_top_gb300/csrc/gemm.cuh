// Definitions shared by the grouped GEMM kernels and the activation
// quantiser: the activation scale-factor layout, E4M3 decoding, the tcgen05
// instruction descriptors and the token-tile tensor maps.
#pragma once

#include <cuda.h>

#include "common.cuh"
#include "internal.h"

namespace ds4moe {

// Activation scales use the K-block-major chunk layout [K/128][rows/128][512]
// so the chunks of consecutive 128-row blocks are adjacent; inside a chunk,
// row r and 32-element block kb sit at (r % 32) * 16 + (r % 128 / 32) * 4 + kb % 4
// (the layout one tcgen05.cp 32x128b.warpx4 moves into tensor memory).
__device__ __forceinline__ size_t act_sf_index(size_t row, int kblk, int r128) {
  return ((size_t)(kblk / 4) * r128 + row / 128) * kSfChunk + (row % 32) * 16 + ((row % 128) / 32) * 4 + (kblk % 4);
}

// Two E4M3 codes (low byte first) -> their values as f32.
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint32_t two) {
  uint32_t h;
  asm("{ .reg .b16 t; cvt.u16.u32 t, %1; cvt.rn.f16x2.e4m3x2 %0, t; }" : "=r"(h) : "r"(two));
  return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

// E8M0 exponent of an MXFP8 block with largest magnitude `amax`:
// floor(log2 amax) - 8 clamped to [-127, 127], 0 for an all-zero block.
__device__ __forceinline__ int mxfp8_exponent(float amax) {
  return amax > 0.f ? max(-127, min(127, floor_log2_f32(amax) - 8)) : 0;
}

// MXFP8 of one 32-value block: E8M0 exponent s (floor(log2 amax) - 8, clamped;
// 0 for an all-zero block) and the 32 codes packed little-endian in 8 words.
__device__ __forceinline__ int mxfp8_block(const float (&v)[32], uint32_t (&packed)[8]) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const int s = mxfp8_exponent(amax);
  const float inv = exp2i(-s);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t lo = f32x2_to_e4m3x2(v[4 * i] * inv, v[4 * i + 1] * inv);
    const uint32_t hi = f32x2_to_e4m3x2(v[4 * i + 2] * inv, v[4 * i + 3] * inv);
    packed[i] = lo | (hi << 16);
  }
  return s;
}

// MXFP8 of a block and of its residual: hi = MXFP8(v) (returned exponent,
// codes in hi), lo = MXFP8(v - hi) (exponent in s_lo, codes in lo), so that
// hi + lo carries about twice the E4M3 mantissa.  v is overwritten by the
// residual.
__device__ __forceinline__ int mxfp8_split_block(float (&v)[32], uint32_t (&hi)[8], uint32_t (&lo)[8], int& s_lo) {
  const int s = mxfp8_block(v, hi);
  const float sc = exp2i_e8m0(s);  // s = -127 for a block of subnormals
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float2 a = e4m3x2_to_f32x2(hi[i] & 0xFFFFu), b = e4m3x2_to_f32x2(hi[i] >> 16);
    v[4 * i] -= a.x * sc;
    v[4 * i + 1] -= a.y * sc;
    v[4 * i + 2] -= b.x * sc;
    v[4 * i + 3] -= b.y * sc;
  }
  s_lo = mxfp8_block(v, lo);
  return s;
}

// Instruction descriptor, kind::mxf8f6f4 with block scaling: A/B formats
// (E4M3 = 0, E2M1 = 5), K-major A and B, N >> 3, E8M0 scales, M >> 4, and the
// byte of the 32-bit scale word (one per 32-K step) used for A and B.
__device__ __forceinline__ uint32_t idesc_mx(int M, int N, uint32_t sf_id) {
  constexpr uint32_t kE2M1 = 5, kE4M3 = 0;
  return (sf_id << 4) | (kE2M1 << 7) | (kE4M3 << 10) | ((uint32_t)(N >> 3) << 17) | (1u << 23) |
         ((uint32_t)(M >> 4) << 24) | (sf_id << 29);
}

// Instruction descriptor, kind::f16: f16 A and B, f32 D, K-major, N >> 3, M >> 4.
__device__ __forceinline__ uint32_t idesc_f16(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Token-tile tensor maps, one per box height 16, 32, ..., 192 rows.
struct alignas(128) BoxMaps {
  CUtensorMap m[kNumBoxMaps];
};

__device__ __forceinline__ int round16(int n) { return (n + 15) & ~15; }
__device__ __forceinline__ int round32(int n) { return (n + 31) & ~31; }

}  // namespace ds4moe
