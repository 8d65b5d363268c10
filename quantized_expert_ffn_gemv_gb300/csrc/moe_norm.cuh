// Residual add + RMSNorm pieces shared by residual_rmsnorm_kernel and the
// fused decode kernel's prologue, so that both give the same bits.
//
// Per token, 256 threads; thread v takes the 8-element chunks v, v + 256, ...
// (elements 8i .. 8i + 7 of chunk i), adds the residual, rounds to bf16 and
// accumulates the squares in element order; the 32 lane sums are added by an
// xor butterfly and the 8 warp sums in warp order.
#pragma once
#include <cuda_bf16.h>
#include <cstdint>

namespace moe {

constexpr int kNormThreads = 256;  // threads per token

// x + y (y optional) of one chunk rounded to bf16; the squares of the
// rounded values are added to ss in element order.
__device__ __forceinline__ uint4 resid_chunk(const uint4& xv, const uint4& yv, bool has_y, float& ss) {
  const uint32_t w[4] = {xv.x, xv.y, xv.z, xv.w}, u[4] = {yv.x, yv.y, yv.z, yv.w};
  uint32_t o[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float a0 = __uint_as_float(w[j] << 16), a1 = __uint_as_float(w[j] & 0xFFFF0000u);
    if (has_y) {
      a0 += __uint_as_float(u[j] << 16);
      a1 += __uint_as_float(u[j] & 0xFFFF0000u);
    }
    const uint32_t b0 = __bfloat16_as_ushort(__float2bfloat16_rn(a0));
    const uint32_t b1 = __bfloat16_as_ushort(__float2bfloat16_rn(a1));
    const float r0 = __uint_as_float(b0 << 16), r1 = __uint_as_float(b1 << 16);
    ss = fmaf(r0, r0, ss);
    ss = fmaf(r1, r1, ss);
    o[j] = b0 | (b1 << 16);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// bf16(v * inv) of one bf16 chunk.
__device__ __forceinline__ uint4 scale_chunk(const uint4& v, float inv) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t o[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(w[j] << 16) * inv));
    const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(w[j] & 0xFFFF0000u) * inv));
    o[j] = lo | (hi << 16);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

}  // namespace moe
