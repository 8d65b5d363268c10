// Router logits in compensated (double-float) fp32 arithmetic, and the
// 64-bit order keys every top-k selection of the library compares.
//
// Routing must pick the same experts as a binary64 evaluation of the
// router (Betelgeuse news page, section "bit-exact 的确切含义": the top-10
// routing is never changed).  A plain fp32 dot product of 2048 terms can be
// off by about 1e-4 and so swap two experts whose logits are that close.
// Here every product is split exactly (TwoProduct through fma) and every
// running sum carries its rounding error (TwoSum), the compensated dot
// product of Ogita, Rump and Oishi ("Accurate sum and dot product", SIAM J.
// Sci. Comput. 26, 2005, algorithm Dot2).  Its error is bounded by
// gamma_n^2 * sum |w x| (n = 64 terms per lane at H = 2048 plus five tree
// levels): below 5e-10 there, and typically far smaller.
//
// Canonical summation order (every kernel follows it, so a logit has the
// same bits on every path):  the H inputs split into four quarters; in
// quarter q, lane l of a warp accumulates the float4 groups l, l + 32,
// l + 64, ... of the quarter in that order (components x, y, z, w); the 32
// lane partials are combined by an xor butterfly (offsets 16, 8, 4, 2, 1);
// the quarters are then added in the order ((q0 + q1) + q2) + q3, then the
// bias.  The pair (s, c) is finally normalised to hi + lo.
//
// Key: the pair mapped to an unsigned integer that orders like its value
// (NaN lowest, -0 = +0), keeping 52 high bits (2^-36 relative resolution
// below hi's own 2^-24).  The low 12 bits of the 64-bit
// words built from a key hold either the expert's complement 4095 - e (so
// one unsigned compare ranks by logit, then lower index), or a call tag.
#pragma once

#include <cstdint>

namespace moe {

struct DF {
  float s, c;  // running sum and its accumulated rounding error
};

// s + e == a + b exactly (Knuth's TwoSum; no fused or reordered operations).
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// One term w * x of a compensated dot product: p + pe == w * x exactly.
__device__ __forceinline__ void dot2_acc(DF& d, float w, float x) {
  const float p = __fmul_rn(w, x);
  const float pe = __fmaf_rn(w, x, -p);
  float s, se;
  two_sum(d.s, p, s, se);
  d.s = s;
  d.c = __fadd_rn(d.c, __fadd_rn(se, pe));
}

__device__ __forceinline__ void dot2_acc4(DF& d, const float4& w, const float4& x) {
  dot2_acc(d, w.x, x.x);
  dot2_acc(d, w.y, x.y);
  dot2_acc(d, w.z, x.z);
  dot2_acc(d, w.w, x.w);
}

// a + b; commutative bit for bit (the error term of TwoSum is exact).
__device__ __forceinline__ DF df_add(DF a, DF b) {
  float s, e;
  two_sum(a.s, b.s, s, e);
  return DF{s, __fadd_rn(__fadd_rn(a.c, b.c), e)};
}

// The xor butterfly over the warp; every lane ends with the same sum.
__device__ __forceinline__ DF warp_sum_df(DF d) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    DF other;
    other.s = __shfl_xor_sync(0xffffffffu, d.s, o);
    other.c = __shfl_xor_sync(0xffffffffu, d.c, o);
    d = df_add(d, other);
  }
  return d;
}

// bf16 pair (one 32-bit word) -> two floats, exactly.
__device__ __forceinline__ float bf_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// Lane partial of one quarter: W quarter row (fp32, 16-byte aligned) against
// the matching quarter of x given as bf16 (n4 float4 groups in the quarter).
__device__ __forceinline__ DF quarter_partial_bf16(const float* wq, const uint16_t* xq, int n4, int lane) {
  DF d{0.f, 0.f};
  for (int j = lane; j < n4; j += 32) {
    const float4 w = *reinterpret_cast<const float4*>(wq + 4 * j);
    const uint2 xv = *reinterpret_cast<const uint2*>(xq + 4 * j);
    dot2_acc4(d, w, make_float4(bf_lo(xv.x), bf_hi(xv.x), bf_lo(xv.y), bf_hi(xv.y)));
  }
  return d;
}

// Order-preserving 32-bit image of a float (-0 as +0).
__device__ __forceinline__ uint32_t fkey(float f) {
  const uint32_t u = __float_as_uint(__fadd_rn(f, 0.f));
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// ((q0 + q1) + q2) + q3 + bias as a 52-bit key.  The sum is normalised to
// hi + lo with hi = fl(hi + lo) (TwoSum, exact); hi then orders the values
// and lo breaks ties of hi, so the 64-bit word fkey(hi) : fkey(lo) orders
// exactly like hi + lo.  The key keeps its top 52 bits (lo to 12 of its
// bits: 2^-36 relative).  Float arithmetic only: this GPU's FP64 units are
// few and a handful of double operations stalled CTAs for microseconds.
__device__ __forceinline__ uint64_t logit_key(DF q0, DF q1, DF q2, DF q3, float bias) {
  DF d = df_add(df_add(df_add(q0, q1), q2), q3);
  float s, e;
  two_sum(d.s, bias, s, e);
  float hi, lo;
  if (isfinite(s)) {
    two_sum(s, __fadd_rn(d.c, e), hi, lo);
  } else {  // an infinite sum (a -inf bias masks an expert) keeps its value
    hi = s;
    lo = 0.f;
  }
  if (hi != hi || lo != lo) return 1ull;  // NaN ranks below every number, -inf included
  const uint64_t k = (((uint64_t)fkey(hi) << 32) | fkey(lo)) >> 12;
  return k ? k : 1ull;  // 0 is reserved for "no entry"
}

// The logit a key stands for, as fp32 (its hi part; for the softmax weights).
__device__ __forceinline__ float key_value(uint64_t key52) {
  const uint32_t k = (uint32_t)(key52 >> 20);
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// One unsigned compare ranks (larger logit, then lower expert index); 0 = none.
__device__ __forceinline__ uint64_t rank_word(uint64_t key52, int e) {
  return key52 ? ((key52 << 12) | (uint64_t)(4095 - e)) : 0ull;
}
__device__ __forceinline__ uint64_t word_key(uint64_t w) { return w >> 12; }
__device__ __forceinline__ int word_expert(uint64_t w) { return 4095 - (int)(w & 4095u); }

// Warp-wide maximum of a 64-bit word.
__device__ __forceinline__ uint64_t warp_max_u64(uint64_t v) {
  const uint32_t hi = (uint32_t)(v >> 32);
  const uint32_t mh = __reduce_max_sync(0xffffffffu, hi);
  const uint32_t ml = __reduce_max_sync(0xffffffffu, hi == mh ? (uint32_t)v : 0u);
  return ((uint64_t)mh << 32) | ml;
}

// n bf16 activations (n a multiple of 8, 16-byte aligned) -> fp32 in shared
// memory by NT threads: every thread's loads are issued before any of its
// stores, so the staging costs one global round trip, not one per element.
template <int NT>
__device__ __forceinline__ void stage_x_f32(const uint16_t* src, int n, float* dst, int tid) {
  constexpr int kPer = 8;  // 16-byte loads per thread in flight together
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
  const int n8 = n / 8;
  for (int i0 = 0; i0 < n8; i0 += NT * kPer) {
    uint4 v[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int i = i0 + j * NT + tid;
      v[j] = i < n8 ? __ldcg(s4 + i) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int i = i0 + j * NT + tid;
      if (i < n8) {
        float4* d = reinterpret_cast<float4*>(dst + 8 * i);
        d[0] = make_float4(bf_lo(v[j].x), bf_hi(v[j].x), bf_lo(v[j].y), bf_hi(v[j].y));
        d[1] = make_float4(bf_lo(v[j].z), bf_hi(v[j].z), bf_lo(v[j].w), bf_hi(v[j].w));
      }
    }
  }
}

// One warp: the k best of one token's rank words staged in shared memory
// (lr[0..E), every word nonzero), in rank order, by k rounds of a warp
// maximum; a selected word is cleared in lr.  Every lane returns the same
// experts sel[r] and logits selv[r].
__device__ inline void warp_select_k(unsigned long long* lr, int E, int k, int* sel, float* selv) {
  const int lane = threadIdx.x & 31;
  for (int r = 0; r < k; ++r) {
    uint64_t best = 0ull;
    for (int e = lane; e < E; e += 32) {
      const uint64_t v = lr[e];
      best = v > best ? v : best;
    }
    const uint64_t m = warp_max_u64(best);
    const int e = word_expert(m);
    if (lane == (e & 31)) lr[e] = 0ull;
    sel[r] = e;
    selv[r] = key_value(word_key(m));
    __syncwarp();
  }
}

// Lane 0: the selection (rank order in sel/selv, sel[0] the largest logit)
// reordered to ascending expert index, with softmax weights renormalised over
// the k: w_j = exp(v_j - v_max) / z, z summed in ascending expert order.
__device__ inline void softmax_ascending(int* sel, float* selv, int k, int* idx_out, float* w_out) {
  const float m = selv[0];
  for (int i = 1; i < k; ++i) {
    const int ki = sel[i];
    const float kv = selv[i];
    int j = i - 1;
    while (j >= 0 && sel[j] > ki) {
      sel[j + 1] = sel[j];
      selv[j + 1] = selv[j];
      --j;
    }
    sel[j + 1] = ki;
    selv[j + 1] = kv;
  }
  float z = 0.f;
  for (int j = 0; j < k; ++j) z += expf(selv[j] - m);
  for (int j = 0; j < k; ++j) {
    idx_out[j] = sel[j];
    w_out[j] = expf(selv[j] - m) / z;
  }
}

}  // namespace moe
