// 4-bit block-32 weights on the legacy tensor path (mma.sync m16n8k16): the
// A-fragment dequantization of one GPU-layout word and the 16 x 64 super-tile
// product with exact fp32 block scaling, shared by the fused decode kernel,
// the batched kernels and the prefill kernel's small-chunk path.
#pragma once

#include <cuda_fp16.h>
#include <cstdint>

namespace moe {

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// 8 packed nibbles (GPU layout word) -> the 4 f16x2 registers of an A fragment,
// holding q = u - 8 exactly.  A low nibble of a half becomes 1024 + u through
// the 0x6400 exponent (minus 1032 -> q); a high nibble becomes 1024 + 16u
// (times 1/16 minus 72 -> q).
__device__ __forceinline__ void dequant_frag(uint32_t w, uint32_t (&a)[4]) {
  const uint32_t lo0 = (w & 0x000F000Fu) | 0x64006400u;
  const uint32_t hi0 = (w & 0x00F000F0u) | 0x64006400u;
  const uint32_t w8 = w >> 8;
  const uint32_t lo1 = (w8 & 0x000F000Fu) | 0x64006400u;
  const uint32_t hi1 = (w8 & 0x00F000F0u) | 0x64006400u;
  const __half2 k1032 = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));
  const __half2 k16th = __halves2half2(__ushort_as_half(0x2C00), __ushort_as_half(0x2C00));
  const __half2 km72 = __halves2half2(__ushort_as_half(0xD480), __ushort_as_half(0xD480));
  __half2 r0 = __hsub2(*reinterpret_cast<const __half2*>(&lo0), k1032);
  __half2 r1 = __hsub2(*reinterpret_cast<const __half2*>(&lo1), k1032);
  __half2 r2 = __hfma2(*reinterpret_cast<const __half2*>(&hi0), k16th, km72);
  __half2 r3 = __hfma2(*reinterpret_cast<const __half2*>(&hi1), k16th, km72);
  a[0] = *reinterpret_cast<uint32_t*>(&r0);  // row g,   k 2t..2t+1
  a[1] = *reinterpret_cast<uint32_t*>(&r1);  // row g+8, k 2t..2t+1
  a[2] = *reinterpret_cast<uint32_t*>(&r2);  // row g,   k 2t+8..2t+9
  a[3] = *reinterpret_cast<uint32_t*>(&r3);  // row g+8, k 2t+8..2t+9
}

// Codebook format: weight = scale * C[u] with C a fixed table of 16 integer
// levels.  `lut` is this lane's register holding level (lane % 16) as fp16
// in its low half (codebook_lut); the word's eight indices are looked up by
// shuffles across the warp (all 32 lanes call this together) and paired into
// the same A-fragment registers dequant_frag produces.
__device__ __forceinline__ void dequant_frag_cb(uint32_t w, uint32_t (&a)[4], uint32_t lut) {
  uint32_t v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __shfl_sync(0xffffffffu, lut, (int)((w >> (4 * i)) & 15u));
  a[0] = __byte_perm(v[0], v[4], 0x5410);  // row g,   k 2t..2t+1   (bits 0-3, 16-19)
  a[1] = __byte_perm(v[2], v[6], 0x5410);  // row g+8, k 2t..2t+1   (bits 8-11, 24-27)
  a[2] = __byte_perm(v[1], v[5], 0x5410);  // row g,   k 2t+8..2t+9 (bits 4-7, 20-23)
  a[3] = __byte_perm(v[3], v[7], 0x5410);  // row g+8, k 2t+8..2t+9 (bits 12-15, 28-31)
}

// The codebook levels as fp16 bit patterns: the standard normal's quantiles
// at (u + 1/2) / 16 scaled to +-127 and rounded (see include/moe.h).
__device__ __forceinline__ uint32_t codebook_lut(int lane) {
  const int lv[16] = {-127, -90, -69, -53, -39, -27, -16, -5, 5, 16, 27, 39, 53, 69, 90, 127};
  int v = 0;
#pragma unroll
  for (int i = 0; i < 16; ++i) v = (lane % 16 == i) ? lv[i] : v;
  return (uint32_t)__half_as_ushort(__int2half_rn(v));
}

__device__ __forceinline__ float half_lo(uint32_t v) { return __half2float(__ushort_as_half((uint16_t)(v & 0xFFFF))); }
__device__ __forceinline__ float half_hi(uint32_t v) { return __half2float(__ushort_as_half((uint16_t)(v >> 16))); }

// One 16 x 64 super-tile against one n8 group of activations: 2 scale blocks,
// each the exact fp32 scaling of a 32-long integer-weight dot product.  b01
// and b23 hold the lane's B-fragment halves of the four k16 blocks: block j's
// k 2t, 2t+1 and 2t+8, 2t+9 (t = lane % 4) of column n = lane / 4.
// fmt 0: linear 4-bit (d * (u - 8)); fmt 1: codebook (d * C[u], lut from
// codebook_lut).  fmt is uniform across the warp.
__device__ __forceinline__ void supertile_mma(float (&acc)[4], const uint4& nib, const uint2& sc, const uint4& b01,
                                              const uint4& b23, int fmt = 0, uint32_t lut = 0u) {
  const uint32_t words[4] = {nib.x, nib.y, nib.z, nib.w};
  const uint32_t bb[4][2] = {{b01.x, b01.y}, {b01.z, b01.w}, {b23.x, b23.y}, {b23.z, b23.w}};
  const float d[4] = {half_lo(sc.x), half_hi(sc.x), half_lo(sc.y), half_hi(sc.y)};
#pragma unroll
  for (int blk = 0; blk < 2; ++blk) {
    float tmp[4] = {0.f, 0.f, 0.f, 0.f};
    uint32_t a[4];
    if (fmt == 1)
      dequant_frag_cb(words[2 * blk], a, lut);
    else
      dequant_frag(words[2 * blk], a);
    mma16816(tmp, a, bb[2 * blk][0], bb[2 * blk][1]);
    if (fmt == 1)
      dequant_frag_cb(words[2 * blk + 1], a, lut);
    else
      dequant_frag(words[2 * blk + 1], a);
    mma16816(tmp, a, bb[2 * blk + 1][0], bb[2 * blk + 1][1]);
    const float dg = d[2 * blk], dg8 = d[2 * blk + 1];
    acc[0] = fmaf(dg, tmp[0], acc[0]);
    acc[1] = fmaf(dg, tmp[1], acc[1]);
    acc[2] = fmaf(dg8, tmp[2], acc[2]);
    acc[3] = fmaf(dg8, tmp[3], acc[3]);
  }
}

// A 16 x 64 super-tile dequantized once (its four words' A fragments), for
// kernels that multiply the same weights against several n8 token groups.
struct SupertileA {
  uint32_t a[4][4];
  float d[4];
};

__device__ __forceinline__ SupertileA dequant_supertile(const uint4& nib, const uint2& sc) {
  SupertileA t;
  dequant_frag(nib.x, t.a[0]);
  dequant_frag(nib.y, t.a[1]);
  dequant_frag(nib.z, t.a[2]);
  dequant_frag(nib.w, t.a[3]);
  t.d[0] = half_lo(sc.x);
  t.d[1] = half_hi(sc.x);
  t.d[2] = half_lo(sc.y);
  t.d[3] = half_hi(sc.y);
  return t;
}

// The same product as supertile_mma, from pre-dequantized fragments.
__device__ __forceinline__ void supertile_mma_pre(float (&acc)[4], const SupertileA& A, const uint4& b01,
                                                  const uint4& b23) {
  const uint32_t bb[4][2] = {{b01.x, b01.y}, {b01.z, b01.w}, {b23.x, b23.y}, {b23.z, b23.w}};
#pragma unroll
  for (int blk = 0; blk < 2; ++blk) {
    float tmp[4] = {0.f, 0.f, 0.f, 0.f};
    mma16816(tmp, A.a[2 * blk], bb[2 * blk][0], bb[2 * blk][1]);
    mma16816(tmp, A.a[2 * blk + 1], bb[2 * blk + 1][0], bb[2 * blk + 1][1]);
    const float dg = A.d[2 * blk], dg8 = A.d[2 * blk + 1];
    acc[0] = fmaf(dg, tmp[0], acc[0]);
    acc[1] = fmaf(dg, tmp[1], acc[1]);
    acc[2] = fmaf(dg8, tmp[2], acc[2]);
    acc[3] = fmaf(dg8, tmp[3], acc[3]);
  }
}

}  // namespace moe
