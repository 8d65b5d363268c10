// Prefill path (T > 64 tokens per call): the layer as three GEMMs on the
// 5th-generation tensor cores.  Prefill is compute-bound where decode is
// bandwidth-bound (halogen-flash-server README, section "Measured"), and a
// chunk's cost per token keeps falling up to a few thousand tokens (Basalt
// README, section "Prompt chunks").
//
//   prep       W_r (fp32) -> three bf16 pieces W0 + W1 + W2 (24 + bits, so
//              the router keeps fp32 accuracy on bf16 tensor cores: x is
//              bf16 already, each product is exact, sums are fp32);
//              x -> fp16 rows for the expert GEMMs
//   router     tcgen05 GEMM: logits [T][E] = sum of the three pieces' products
//   top-k      warp per token: the k largest logits (ties to the lower
//              index), made exact by recomputing, with the compensated
//              router, the experts whose tensor-core logits lie within the
//              GEMM's error bound of the k-th/(k+1)-th boundary; ascending
//              expert order, softmax over the selection; bit t of the
//              expert's token bitmap
//   prefix     warp per expert: set bits before each bitmap word
//   scan       per-expert counts -> pair offsets, chunk records of up to 256
//              tokens for the tensor cores, and an expert's last chunk of at
//              most 16 tokens for the mma.sync path
//   pairs      thread per (token, rank): its place in the expert's token
//              list (ascending token: a stable counting sort)
//   small      the chunks of at most 16 tokens: the chunk's x (or h) rows
//              staged in shared memory, each 16-row strip's packed weights
//              read once and applied with mma.sync (gate/up + SiLU, or down)
//   gate/up    grouped GEMM, M = 128 (64 gate rows and the 64 matching up
//              rows), N = the chunk's tokens (<= 256, rounded up to 16),
//              K = H in steps of 64.  One warp streams the packed 4-bit
//              tiles into shared memory (batched bulk copies); eight warps
//              dequantize them to fp16 d*q, written with stmatrix in the
//              128-byte-swizzled K-major layout; eight warps gather the
//              chunk's activation rows with cp.async; one thread issues the
//              MMAs into a double-buffered TMEM accumulator; eight epilogue
//              warps compute h = silu(g) * u.
//   down       the same engine, M = 128 output rows, K = I, B = the pairs'
//              h rows; the epilogue writes each pair's expert output z as
//              fp16.
//   combine    y[t] = sum_j w_j z_j (ascending expert) + z_shared in fp32,
//              rounded once to bf16.
#include <cfloat>
#include <climits>

#include "moe.h"
#include "moe_internal.h"
#include "moe_mma.cuh"
#include "moe_prefill.h"
#include "moe_route.cuh"

namespace moe {
namespace {

constexpr uint64_t kPipeTimeoutNs = 4000000000ull;  // a pipeline wait that exceeds this is an error

// ------------------------------------------------------------------ PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
// Potentially blocking test: the thread sleeps (up to the hint, 20 us)
// until the phase completes instead of spinning on issue slots that the
// MMA thread and the epilogue need.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(20000u)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ int ld_cg_i32(const int* p) {
  int r;
  asm volatile("ld.global.cg.s32 %0, [%1];" : "=r"(r) : "l"(p));
  return r;
}
__device__ __forceinline__ uint4 ld_cg4(const void* p) {
  uint4 r;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}
// Four 8x8 b16 matrices from mma-fragment registers; lane l gives the shared
// address of row (l & 7) of matrix (l >> 3).
__device__ __forceinline__ void stmatrix_x4(uint32_t addr, uint32_t r0, uint32_t r1, uint32_t r2, uint32_t r3) {
  asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(r0), "r"(r1),
               "r"(r2), "r"(r3)
               : "memory");
}
// 1-D bulk copy global -> shared, completion counted on `bar` in bytes.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"((uint64_t)map), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(dst),
      "l"((uint64_t)map), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(
          d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
// 16 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tc_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor, K-major, 128-byte swizzle: rows of 128 B
// (64 fp16), 8-row atoms 1024 B apart, bit 46 = descriptor version, layout
// type 2 = 128-byte swizzle.  A K-slice of 16 starts 32 B further.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | (1ull << 16) | ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) |
         (2ull << 61);
}
// Instruction descriptor of kind::f16: D f32, M = 128, N; A and B both f16
// (bf16 = false) or both bf16, K-major.
__device__ __forceinline__ uint32_t instr_desc(int n, bool bf16) {
  return (1u << 4) | (bf16 ? ((1u << 7) | (1u << 10)) : 0u) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(128 >> 4) << 24);
}
// Byte offset of 16-byte chunk c (k 8c .. 8c+7) of row r in a swizzled tile.
__device__ __forceinline__ uint32_t sw128_off(int r, int c) { return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)); }

__device__ void set_error(const LayerArgs& a, int code) {
  atomicCAS(&a.st->error, 0, code);
  volatile int32_t* m = &a.hm->error;
  if (*m == 0) *m = code;
  __threadfence_system();
}

// Bounded wait on an mbarrier phase.  backoff_ns > 0 puts the warp to sleep
// between tests so that waiting warps leave the issue slots to the ones
// doing work (the MMA thread waits without it).
#ifndef PF_BACKOFF_NS
#define PF_BACKOFF_NS 64
#endif
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const LayerArgs& a, uint64_t deadline,
                                         bool& ok, unsigned backoff_ns = PF_BACKOFF_NS) {
  if (!ok) return false;
  int spins = 0;
  while (!mbar_try_wait(bar, parity)) {
    if (backoff_ns) __nanosleep(backoff_ns);
    if (((++spins) & 15) == 0 && global_ns() > deadline) {
      set_error(a, MOE_ERR_TIMEOUT);
      ok = false;
      return false;
    }
  }
  return true;
}

// One GPU-layout nibble word (lane 4g + t, one 16-wide k-tile) -> q = u - 8
// as four f16x2: [0] row g, k 2t..2t+1; [1] row g+8, k 2t..2t+1;
// [2] row g, k 2t+8..2t+9; [3] row g+8, k 2t+8..2t+9.  Exponent-bias trick:
// 0x6400 | u is 1024 + u; 0x6400 | 16u is 1024 + 16u.
__device__ __forceinline__ void dequant_word(uint32_t w, __half2 (&q)[4]) {
  const uint32_t lo0 = (w & 0x000F000Fu) | 0x64006400u;
  const uint32_t hi0 = (w & 0x00F000F0u) | 0x64006400u;
  const uint32_t w8 = w >> 8;
  const uint32_t lo1 = (w8 & 0x000F000Fu) | 0x64006400u;
  const uint32_t hi1 = (w8 & 0x00F000F0u) | 0x64006400u;
  const __half2 k1032 = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));
  const __half2 k16th = __halves2half2(__ushort_as_half(0x2C00), __ushort_as_half(0x2C00));
  const __half2 km72 = __halves2half2(__ushort_as_half(0xD480), __ushort_as_half(0xD480));
  q[0] = __hsub2(*reinterpret_cast<const __half2*>(&lo0), k1032);
  q[1] = __hsub2(*reinterpret_cast<const __half2*>(&lo1), k1032);
  q[2] = __hfma2(*reinterpret_cast<const __half2*>(&hi0), k16th, km72);
  q[3] = __hfma2(*reinterpret_cast<const __half2*>(&hi1), k16th, km72);
}
__device__ __forceinline__ uint32_t h2u(__half2 v) { return *reinterpret_cast<uint32_t*>(&v); }

// ------------------------------------------------------------------ prep, top-k, grouping

// W_r -> bf16 pieces (W = W0 + W1 + W2 up to 2^-27 relative) and x -> fp16.
__global__ void __launch_bounds__(256) prefill_prep_kernel(LayerArgs a, PrefillArgs p) {
  const size_t nw = (size_t)a.E * a.H, nx = (size_t)a.T * a.H;
  const size_t stride = (size_t)gridDim.x * 256;
  for (size_t i = (size_t)blockIdx.x * 256 + threadIdx.x; i < nw; i += stride) {
    const float w = a.W_r[i];
    const __nv_bfloat16 w0 = __float2bfloat16_rn(w);
    const float r0 = w - __bfloat162float(w0);
    const __nv_bfloat16 w1 = __float2bfloat16_rn(r0);
    const __nv_bfloat16 w2 = __float2bfloat16_rn(r0 - __bfloat162float(w1));
    p.w_split[i] = __bfloat16_as_ushort(w0);
    p.w_split[nw + i] = __bfloat16_as_ushort(w1);
    p.w_split[2 * nw + i] = __bfloat16_as_ushort(w2);
  }
  // router row norms, for the recheck bound of the top-k kernel (fp32 sum of
  // squares rounded up by 0.1 %, far more than its own rounding error)
  {
    const int lane = threadIdx.x & 31;
    const int gw = (int)((blockIdx.x * 256 + threadIdx.x) >> 5), nwarps = (int)(gridDim.x * 8);
    for (int e = gw; e < a.E; e += nwarps) {
      const float* wr = a.W_r + (size_t)e * a.H;
      float ss = 0.f;
      for (int h = lane; h < a.H; h += 32) ss = fmaf(wr[h], wr[h], ss);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      if (lane == 0) p.wnorm[e] = sqrtf(ss) * 1.001f;
    }
  }
  // x -> fp16 rows, and each token's norm (warp per token), for the same bound
  int bad = 0;
  {
    const int lane = threadIdx.x & 31;
    const int gw = (int)((blockIdx.x * 256 + threadIdx.x) >> 5), nwarps = (int)(gridDim.x * 8);
    for (int t = gw; t < a.T; t += nwarps) {
      float ss = 0.f;
      for (int h8 = lane * 8; h8 < a.H; h8 += 256) {
        const size_t i = (size_t)t * a.H + h8;
        const uint4 v = *reinterpret_cast<const uint4*>(a.x + i);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float f0 = __uint_as_float(w[q] << 16), f1 = __uint_as_float(w[q] & 0xFFFF0000u);
          bad |= !(fabsf(f0) < 65504.f) || !(fabsf(f1) < 65504.f);
          ss = fmaf(f0, f0, fmaf(f1, f1, ss));
          o[q] = h2u(__floats2half2_rn(f0, f1));
        }
        *reinterpret_cast<uint4*>(p.x16p + i) = make_uint4(o[0], o[1], o[2], o[3]);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      if (lane == 0) p.xnorm[t] = sqrtf(ss) * 1.001f;
    }
  }
  (void)nx;
  if (bad) set_error(a, MOE_ERR_DEVICE);
}

// Bound on |tensor-core logit - exact logit| per unit of |W_r[e]| |x_t|:
// the router GEMM adds 3 * H / 16 MMA steps of exact bf16 x bf16 products
// into an fp32 accumulator (at most 2^-23 relative per step even without
// round-to-nearest: 4.6e-5 at H = 2048), and the three bf16 pieces miss W_r
// by at most 2^-27 relative; 1.25e-4 leaves a factor 2.5 over their sum.
constexpr float kTcBound = 1.25e-4f;

__device__ __forceinline__ uint64_t shfl_u64(uint64_t v, int src) {
  const uint32_t lo = __shfl_sync(0xffffffffu, (uint32_t)v, src);
  const uint32_t hi = __shfl_sync(0xffffffffu, (uint32_t)(v >> 32), src);
  return ((uint64_t)hi << 32) | lo;
}
__device__ __forceinline__ uint64_t shfl_up_u64(uint64_t v, int d) {
  const uint32_t lo = __shfl_up_sync(0xffffffffu, (uint32_t)v, d);
  const uint32_t hi = __shfl_up_sync(0xffffffffu, (uint32_t)(v >> 32), d);
  return ((uint64_t)hi << 32) | lo;
}

// Warp per token: k + 1 rounds of a warp argmax (value desc, index asc) over
// the token's tensor-core logits, held in registers (CPL per lane; CPL = 0:
// read from memory each round, for very large E).  The selection is exact:
// when the k-th and (k+1)-th tensor-core logits are closer than twice the
// error bound delta_t (kTcBound * max_e |W_r[e]| * |x_t|), every expert
// whose logit lies within 2 delta_t of that boundary is recomputed with the
// compensated router in the library's canonical order (moe_route.cuh), and
// the places the experts above the band do not fill go to the best of those
// by exact key.  Sets bit t of each selected expert's bitmap row; the
// per-expert counts come from the bitmap.
template <int CPL>
__global__ void __launch_bounds__(256) prefill_topk_kernel(LayerArgs a, PrefillArgs p) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int E = a.E, k = a.k, H = a.H;
  __shared__ unsigned int s_wmax;  // max row norm (positive floats order as their bits)
  if (threadIdx.x == 0) s_wmax = 0u;
  __syncthreads();
  {
    unsigned int m = 0u;
    for (int e = threadIdx.x; e < E; e += 256) m = max(m, __float_as_uint(p.wnorm[e]));
    atomicMax(&s_wmax, m);
  }
  __syncthreads();
  if (t >= a.T) return;
  const float* lt = a.logits + (size_t)t * E;
  constexpr int kRegs = CPL > 0 ? CPL : 1;
  float lv[kRegs];
#pragma unroll
  for (int i = 0; i < kRegs; ++i) lv[i] = (CPL > 0 && lane + 32 * i < E) ? lt[lane + 32 * i] : -FLT_MAX;
  int my_e = INT_MAX;   // lane r <= k: the expert of rank r
  float my_v = 0.f;     // and its logit
  uint32_t taken[kMaxExperts / 1024] = {};  // bit i: logit lane + 32 i already selected
  const int rounds = k < E ? k + 1 : k;
  bool boundary = k < E;  // a (k+1)-th comparable logit exists
  for (int r = 0; r < rounds; ++r) {
    float bv = -FLT_MAX;
    int bi = INT_MAX;
    if (CPL > 0) {
#pragma unroll
      for (int i = 0; i < kRegs; ++i) {
        const int e = lane + 32 * i;
        const bool free = e < E && !((taken[0] >> i) & 1u);
        if (free && (lv[i] > bv || (lv[i] == bv && e < bi))) {
          bv = lv[i];
          bi = e;
        }
      }
    } else {
      for (int e = lane, i = 0; e < E; e += 32, ++i) {
        if ((taken[i >> 5] >> (i & 31)) & 1u) continue;
        const float v = lt[e];
        if (v > bv || (v == bv && e < bi)) {
          bv = v;
          bi = e;
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ov > bv || (ov == bv && oi < bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if (bi == INT_MAX) {
      if (r == k) {  // only k comparable logits: no boundary to check
        boundary = false;
        break;
      }
      if (lane == 0) set_error(a, MOE_ERR_DEVICE);  // fewer than k comparable logits (NaN): flagged
      bi = r;                                       // keep the indices distinct
    }
    if (lane == (bi & 31)) {
      if (CPL > 0)
        taken[0] |= 1u << ((bi >> 5) & 31);  // CPL <= 32: one word
      else
        taken[(bi >> 5) >> 5] |= 1u << ((bi >> 5) & 31);
    }
    if (lane == r) {
      my_e = bi;
      my_v = bv;
    }
  }
  if (boundary) {
    const float lk = __shfl_sync(0xffffffffu, my_v, k - 1), lk1 = __shfl_sync(0xffffffffu, my_v, k);
    const float delta = kTcBound * __uint_as_float(s_wmax) * __ldg(p.xnorm + t) + 1e-6f * (fabsf(lk) + 1.f);
    if (lk - lk1 <= 2.f * delta) {
      // above hi: surely selected; below lo: surely not; in between: exact
      const float hi = lk + 2.f * delta, lo = lk1 - 2.f * delta;
      const int n_in = __popc(__ballot_sync(0xffffffffu, lane < k && my_v > hi));
      const int pick = k - n_in;
      uint64_t best = 0ull;  // lanes 0 .. pick-1: the best exact words so far, in rank order
      int nchk = 0;
      auto consider = [&](int e) {
        DF q4[4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
          q4[q] = warp_sum_df(quarter_partial_bf16(a.W_r + (size_t)e * H + q * (H / 4),
                                                   a.x + (size_t)t * H + q * (H / 4), H / 16, lane));
        const uint64_t w = rank_word(logit_key(q4[0], q4[1], q4[2], q4[3], a.bias ? a.bias[e] : 0.f), e);
        const unsigned below = __ballot_sync(0xffffffffu, lane < pick && best < w);
        if (below) {
          const int pos = __ffs(below) - 1;
          const uint64_t up = shfl_up_u64(best, 1);
          if (lane > pos && lane < pick) best = up;
          if (lane == pos) best = w;
        }
        ++nchk;
      };
      if (CPL > 0) {
#pragma unroll
        for (int i = 0; i < kRegs; ++i) {
          const int e = lane + 32 * i;
          unsigned b = __ballot_sync(0xffffffffu, e < E && lv[i] >= lo && lv[i] <= hi);
          while (b) {
            const int src = __ffs(b) - 1;
            b &= b - 1;
            consider(src + 32 * i);
          }
        }
      } else {
        for (int i = 0; i < (E + 31) / 32; ++i) {
          const int e = lane + 32 * i;
          const float v = e < E ? lt[e] : -FLT_MAX;
          unsigned b = __ballot_sync(0xffffffffu, e < E && v >= lo && v <= hi);
          while (b) {
            const int src = __ffs(b) - 1;
            b &= b - 1;
            consider(src + 32 * i);
          }
        }
      }
      const uint64_t got = shfl_u64(best, lane >= n_in ? lane - n_in : 0);
      if (lane >= n_in && lane < k) {
        my_e = word_expert(got);
        my_v = key_value(word_key(got));
      }
      if (lane == 0) atomicAdd(&a.st->rechecks, (unsigned long long)nchk);
    }
  }
  // in parallel, lane r for rank r: its place in ascending expert order, the
  // weight exp(v - m) / z with z summed in ascending expert order (m = lane
  // 0's logit, the largest up to the recheck band)
  const float m = __shfl_sync(0xffffffffu, my_v, 0);
  int pos = 0;
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {
    const int ej = __shfl_sync(0xffffffffu, my_e, j);
    pos += (int)((j < k) & (ej < my_e));
  }
  const float ex = lane < k ? expf(my_v - m) : 0.f;
  float z = 0.f;
  for (int q = 0; q < k; ++q) {
    const unsigned src = __ballot_sync(0xffffffffu, lane < k && pos == q);
    z += __shfl_sync(0xffffffffu, ex, __ffs(src) - 1);
  }
  if (lane < k) {
    a.topk_idx[t * k + pos] = my_e;
    a.topk_w[t * k + pos] = ex / z;
    atomicOr(&p.bitmap[(size_t)my_e * p.words + (t >> 5)], 1u << (t & 31));
  }
}

// Warp per routed expert: prefix[e][w] = set bits of bitmap row e before
// word w; counts[e] = all of them.
__global__ void __launch_bounds__(256) prefill_prefix_kernel(LayerArgs a, PrefillArgs p) {
  const int lane = threadIdx.x & 31;
  const int e = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (e >= a.E) return;
  const int words = (a.T + 31) >> 5;
  const uint32_t* row = p.bitmap + (size_t)e * p.words;
  int32_t* pre = p.prefix + (size_t)e * p.words;
  int run = 0;
  for (int w0 = 0; w0 < words; w0 += 32) {
    const int w = w0 + lane;
    const int c = (w < words) ? __popc(row[w]) : 0;
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (w < words) pre[w] = run + incl - c;
    run += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) p.counts[e] = run;
}

// One CTA: offsets and chunk records of the E routed experts and the shared
// expert (entry E, all T tokens): tensor-core chunks and small chunks; layer
// statistics.
__global__ void __launch_bounds__(1024) prefill_scan_kernel(LayerArgs a, PrefillArgs p) {
  __shared__ int wsum[3][32];
  __shared__ int s_used;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = a.E, NE = E + a.n_shared;
  const int per = (NE + 1023) / 1024;
  if (tid == 0) s_used = 0;
  __syncthreads();
  // an entry's tokens make full kPfN chunks plus a remainder: a remainder of
  // more than kSmallN tokens is one more tensor-core chunk, a smaller one a
  // small chunk
  int c_cnt = 0, c_chk = 0, c_sml = 0, used = 0;
  for (int i = 0; i < per; ++i) {
    const int e = tid * per + i;
    if (e < NE) {
      const int cnt = (e < E) ? p.counts[e] : a.T;
      const int rem = cnt % kPfN;
      c_cnt += cnt;
      c_chk += cnt / kPfN + (rem > kSmallN);
      c_sml += (rem > 0 && rem <= kSmallN);
      used += (e < E && cnt > 0);
    }
  }
  if (used) atomicAdd(&s_used, used);
  int ia = c_cnt, ib = c_chk, ic = c_sml;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int va = __shfl_up_sync(0xffffffffu, ia, o), vb = __shfl_up_sync(0xffffffffu, ib, o),
              vc = __shfl_up_sync(0xffffffffu, ic, o);
    if (lane >= o) {
      ia += va;
      ib += vb;
      ic += vc;
    }
  }
  if (lane == 31) {
    wsum[0][warp] = ia;
    wsum[1][warp] = ib;
    wsum[2][warp] = ic;
  }
  __syncthreads();
  int ba = 0, bb = 0, bc = 0, ta = 0, tb = 0, tc = 0;
  for (int w = 0; w < 32; ++w) {
    if (w < warp) {
      ba += wsum[0][w];
      bb += wsum[1][w];
      bc += wsum[2][w];
    }
    ta += wsum[0][w];
    tb += wsum[1][w];
    tc += wsum[2][w];
  }
  int oa = ba + ia - c_cnt, ob = bb + ib - c_chk, oc = bc + ic - c_sml;
  for (int i = 0; i < per; ++i) {
    const int e = tid * per + i;
    if (e < NE) {
      const int cnt = (e < E) ? p.counts[e] : a.T;
      const int full = cnt / kPfN, rem = cnt - full * kPfN;
      p.offsets[e] = oa;
      p.chunk_off[e] = ob;
      for (int c = 0; c < full; ++c) p.chunk_rec[ob + c] = make_int4(e, oa + c * kPfN, kPfN, 0);
      if (rem > kSmallN)
        p.chunk_rec[ob + full] = make_int4(e, oa + full * kPfN, rem, 0);
      else if (rem > 0)
        p.small_rec[oc++] = make_int4(e, oa + full * kPfN, rem, 0);
      oa += cnt;
      ob += full + (rem > kSmallN);
    }
  }
  if (tid == 0) {
    p.offsets[NE] = ta;
    p.chunk_off[NE] = tb;
    p.n_chunks[0] = tb;
    p.n_chunks[1] = tc;
    a.st->forwards += 1ull;
    a.st->hits += (unsigned long long)s_used;
  }
}

// Thread per (t, rank j): place t in expert e's ascending token list.  The
// shared expert's pairs are token t at offsets[E] + t, rank k.
__global__ void __launch_bounds__(256) prefill_pairs_kernel(LayerArgs a, PrefillArgs p) {
  const int i = blockIdx.x * 256 + threadIdx.x;
  const int T = a.T, k = a.k;
  if (i < T * k) {
    const int t = i / k, j = i - t * k;
    const int e = a.topk_idx[i];
    const size_t w = (size_t)e * p.words + (t >> 5);
    const int pos = p.offsets[e] + p.prefix[w] + __popc(p.bitmap[w] & ((1u << (t & 31)) - 1u));
    p.pair_token[pos] = t;
    p.pair_z[pos] = t * (k + 1) + j;
  } else if (a.n_shared && i < T * k + T) {
    const int t = i - T * k;
    const int pos = p.offsets[a.E] + t;
    p.pair_token[pos] = t;
    p.pair_z[pos] = t * (k + 1) + k;
  }
}

// ------------------------------------------------------------------ GEMMs on tcgen05

constexpr int kTile = 128 * 128;  // one operand tile: 128 rows x 64 fp16/bf16 (128-byte rows)
constexpr int kMmaWarp = 9;       // allocates TMEM; lane 0 issues the MMAs
constexpr int kEpi0 = 10;         // warps 10-13: epilogue; TMEM lane quadrant = warp % 4
constexpr int kGemmThreads = (kEpi0 + 4) * 32;

__device__ __forceinline__ int4 ld_cg_int4(const int4* p) {
  int4 r;
  asm volatile("ld.global.cg.v4.s32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
// Arrive on `bar` once every cp.async this thread issued so far has landed
// (the barrier's expected count includes these arrivals).
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// ---- router GEMM: M-block = 128 experts, N = 128 tokens, K = H; A = the
//      three bf16 pieces of W_r, B = x, both by TMA; logits = acc + bias.
//      Warp 0 loads, warp 9 issues, warps 10-13 drain.
constexpr int kRtStages = 3;
constexpr int kRtOffB = kRtStages * 3 * kTile;
constexpr int kRtOffBar = kRtOffB + kRtStages * kTile;
constexpr int kRtOffTmem = kRtOffBar + 8 * (2 * kRtStages + 5);
constexpr int kRtSmem = kRtOffTmem + 16 + 1024;

__global__ void __launch_bounds__(kGemmThreads, 1)
    prefill_router_kernel(LayerArgs a, const __grid_constant__ CUtensorMap mapW, const __grid_constant__ CUtensorMap mapX) {
  constexpr int S = kRtStages;
  extern __shared__ __align__(1024) unsigned char smraw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(sm);
  const uint32_t bar0 = sbase + kRtOffBar;
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (S + s); };
  auto acc_full = [&](int b) { return bar0 + 8u * (2 * S + b); };
  auto acc_empty = [&](int b) { return bar0 + 8u * (2 * S + 2 + b); };
  const uint32_t drain = bar0 + 8u * (2 * S + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kRtOffTmem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = a.E, T = a.T;
  const int MB = (E + 127) / 128, KS = a.H / 64;
  const int n_tasks = MB * ((T + 127) / 128);
  const uint64_t deadline = global_ns() + kPipeTimeoutNs;
  bool ok = true;
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(acc_full(b), 1);
      mbar_init(acc_empty(b), 4);
    }
    mbar_init(drain, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 256;" ::"r"(smem_u32(tmem_slot)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      int g = 0;
      for (int t = blockIdx.x; t < n_tasks && ok; t += gridDim.x) {
        const int mb = t % MB, n0 = (t / MB) * 128;
        for (int ks = 0; ks < KS; ++ks, ++g) {
          const int s = g % S, use = g / S;
          if (use > 0 && !wait_bar(empty(s), (use - 1) & 1, a, deadline, ok)) break;
          const uint32_t sA = sbase + s * 3 * kTile, sB = sbase + kRtOffB + s * kTile;
          mbar_expect_tx(full(s), 4 * kTile);
#pragma unroll
          for (int pc = 0; pc < 3; ++pc) tma_3d(sA + pc * kTile, &mapW, ks * 64, mb * 128, pc, full(s));
          tma_2d(sB, &mapX, ks * 64, n0, full(s));
        }
      }
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      int g = 0, i = 0;
      for (int t = blockIdx.x; t < n_tasks && ok; t += gridDim.x, ++i) {
        const int nt = min(128, T - (t / MB) * 128);
        const uint32_t idesc = instr_desc((nt + 15) & ~15, true);
        const int b = i & 1, ub = i >> 1;
        if (ub > 0 && !wait_bar(acc_empty(b), (ub - 1) & 1, a, deadline, ok)) break;
        tc_fence_after();
        const uint32_t dt = tmem + (uint32_t)(b * 128);
        for (int ks = 0; ks < KS; ++ks, ++g) {
          const int s = g % S, use = g / S;
          if (!wait_bar(full(s), use & 1, a, deadline, ok, 0)) break;
          tc_fence_after();
          const uint32_t sA = sbase + s * 3 * kTile, sB = sbase + kRtOffB + s * kTile;
#pragma unroll
          for (int pc = 0; pc < 3; ++pc)
#pragma unroll
            for (int j = 0; j < 4; ++j)
              tc_mma(dt, desc_sw128(sA + pc * kTile + j * 32), desc_sw128(sB + j * 32), idesc,
                     (ks > 0 || j > 0 || pc > 0) ? 1u : 0u);
          tc_commit(empty(s));
        }
        if (!ok) break;
        tc_commit(acc_full(b));
      }
      tc_commit(drain);
      bool dok = true;
      wait_bar(drain, 0, a, deadline + kPipeTimeoutNs, dok);
    }
    __syncwarp();
  } else if (warp >= kEpi0) {
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    int i = 0;
    for (int t = blockIdx.x; t < n_tasks && ok; t += gridDim.x, ++i) {
      const int mb = t % MB, n0 = (t / MB) * 128, nt = min(128, T - n0);
      const int b = i & 1, ub = i >> 1;
      if (!wait_bar(acc_full(b), ub & 1, a, deadline, ok)) break;
      tc_fence_after();
      const uint32_t taddr = tmem + (uint32_t)(b * 128) + ((uint32_t)(quad * 32) << 16);
      const int e = mb * 128 + row;
      const float bias = (a.bias && e < E) ? a.bias[e] : 0.f;
      for (int c0 = 0; c0 < nt; c0 += 16) {
        float v[16];
        tc_ld16(taddr + (uint32_t)c0, v);
        if (e < E) {
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (c0 + j < nt) a.logits[(size_t)(n0 + c0 + j) * E + e] = v[j] + bias;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty(b));
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 256;" ::"r"(tmem));
}

// ---- grouped expert GEMMs.
// A tcgen05.mma costs the issuing thread about as long as the tensor core
// needs for 128 x 256 x 16, so chunks are up to 256 tokens (N = 256) and a
// k-step issues its four MMAs and one commit.
// Warp 0 (lanes 0-15): bulk copies of the packed 4-bit tiles, kRawR k-steps
//   per copy and strip, into a ring of kRawStages raw stages.
// Warps 1-8 (dequant): warp w dequantizes strip w of each k-step's packed
//   tile into the swizzled fp16 A tile (stmatrix) and signals a_full.
// Warps 9-16 (gather): their 256 threads copy the chunk's B rows with
//   cp.async as far ahead as the B ring allows, each signalling b_full when
//   its copies land.  A k-step's commit arrives on its B stage's empty barrier; the A
//   ring (kAStages <= kBStages) is reused once the MMA of k-step g - kAStages
//   has completed, i.e. when that k-step's B stage is released.  With more A
//   than B stages that barrier could run two phases past the awaited one.  The MMA
//   thread orders both halves (generic-proxy writes) before its tensor-core
//   reads with one proxy fence after its waits.
// Warp 17: TMEM allocation (2 x 256 columns); lane 0 issues the MMAs.
// Warps 18-25: epilogue, two per TMEM lane quadrant (warp % 4), each taking
//   half of the chunk's columns.
constexpr int kAStages = 3;
constexpr int kBStages = 4;
static_assert(kAStages <= kBStages, "A stages are released through the B stages' empty barriers");
constexpr int kRawR = 2;
constexpr int kRawStages = 2;
constexpr int kProd = 8;    // dequant warps
constexpr int kGather = 8;  // gather warps
constexpr int kXMmaWarp = 1 + kProd + kGather;
constexpr int kXEpi0 = kXMmaWarp + 1;
constexpr int kXEpiWarps = 8;
constexpr int kExpThreads = (kXEpi0 + kXEpiWarps) * 32;
constexpr int kBTile = kPfN * 128;  // B tile: kPfN rows x 64 fp16
constexpr int kRawBytes = 8 * kRawR * (512 + 64);
constexpr int kOffB = kAStages * kTile;
constexpr int kOffRaw = kOffB + kBStages * kBTile;
constexpr int kNumBars = 2 * kRawStages + kAStages + 2 * kBStages + 5;
constexpr int kOffBar = kOffRaw + kRawStages * kRawBytes;
constexpr int kOffTmem = kOffBar + 8 * kNumBars;
constexpr int kGemmSmem = kOffTmem + 16 + 1024;
static_assert(kGemmSmem <= 232448, "shared memory");

struct Task {
  int e, poff, nt, mb;
};
// Task t: chunk t / MB (its record: expert list entry, first pair, tokens)
// and M-block t % MB.  The M-blocks of one chunk are consecutive tasks, so
// CTAs running them at once share the chunk's B rows in L2.
__device__ __forceinline__ Task load_task(const PrefillArgs& p, int MB, int t) {
  const int4 r = ld_cg_int4(&p.chunk_rec[t / MB]);
  return Task{r.x, r.y, r.z, t % MB};
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tc_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
      "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// MODE 0: gate/up; M-block mb = intermediate rows 64 mb .. 64 mb + 63 of gate
//   and of up, K = H.  Tile row of local gate row i: 16 (i / 8) + i % 8; the
//   matching up row is 8 further, so an epilogue lane pairs with lane ^ 8.
// MODE 1: down; M-block mb = output rows 128 mb .. 128 mb + 127, K = I.
// ---- small chunks: an entry's last chunk of at most kSmallN tokens
//
// A tensor-core tile costs a full pass of MMA issues whatever its N, so a
// chunk of a few tokens is cheaper on the legacy path.  A block takes a group
// of strips of one chunk: it stages the chunk's B rows (x for gate/up, h for
// down; at most 16) in shared memory with cp.async, then reads each strip's
// packed weights once from global memory and applies them to the two n8 token
// groups with mma.sync.  MODE 0: gate/up + SiLU -> h rows, four strips per
// block, each strip's K split over eight warps (one batch of weight loads
// each); MODE 1: down -> z rows, sixteen strips per block, a warp per strip
// over the whole K.  Same outputs, in the same places, as the tensor-core
// epilogues.
__host__ __device__ constexpr int sm_warps(int mode) { return mode == 0 ? 8 : 4; }
constexpr int kSmBatch = 4;  // super-tiles of a warp with their weight loads in flight together
__host__ __device__ constexpr int sm_strips(int mode) { return mode == 0 ? 4 : 16; }
// B rows staged with a 16-byte pad: the eight token columns of a fragment
// load fall in different banks
__host__ __device__ inline int sm_row(int K) { return K + 8; }
__host__ __device__ inline size_t sm_smem(int mode, int K) {
  return (size_t)kSmallN * sm_row(K) * 2 + (mode == 0 ? sizeof(float) * sm_warps(0) * 2 * 32 * 8 : 0);
}

// Weights of kSmBatch super-tiles st0, st0 + step, ... (gate and, for MODE 0, up).
template <int MODE>
__device__ __forceinline__ void sm_load_w(const uint8_t* strip, int K, int st0, int step, int nst, int lane, int g,
                                          uint4 (&w0)[kSmBatch], uint2 (&s0)[kSmBatch], uint4 (&w1)[kSmBatch],
                                          uint2 (&s1)[kSmBatch]) {
#pragma unroll
  for (int b = 0; b < kSmBatch; ++b) {
    const int st = st0 + step * b;
    if (st < nst) {
      w0[b] = ld_cg4(strip + st * 512 + lane * 16);
      s0[b] = __ldg(reinterpret_cast<const uint2*>(strip + 8 * K + st * 64 + g * 8));
      if (MODE == 0) {
        w1[b] = ld_cg4(strip + 9 * K + st * 512 + lane * 16);
        s1[b] = __ldg(reinterpret_cast<const uint2*>(strip + 17 * K + st * 64 + g * 8));
      }
    }
  }
}

// B fragments of super-tile st for n8 group q from the staged rows (natural K
// order: k16 block j holds k 16j + 2t, +1 and 16j + 8 + 2t, +1).
__device__ __forceinline__ void sm_load_b(const __half* bs, int K, int q, int st, int g, int t4, uint4& b01,
                                          uint4& b23) {
  const uint32_t* r = reinterpret_cast<const uint32_t*>(bs + (size_t)(q * 8 + g) * sm_row(K) + st * 64 + 2 * t4);
  b01 = make_uint4(r[0], r[4], r[8], r[12]);
  b23 = make_uint4(r[16], r[20], r[24], r[28]);
}

template <int MODE>
__global__ void __launch_bounds__(sm_warps(MODE) * 32) prefill_small_kernel(LayerArgs a, PrefillArgs p) {
  extern __shared__ __align__(16) unsigned char sms[];
  constexpr int NW = sm_warps(MODE), NT = NW * 32;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t4 = lane & 3;
  const int H = a.H, I = a.I, E = a.E;
  const int K = MODE == 0 ? H : I;
  const int nst = K / 64;
  constexpr int SG = sm_strips(MODE);
  const int groups = (MODE == 0 ? I / 16 : H / 16) / SG;
  __half* bs = reinterpret_cast<__half*>(sms);                                          // [16][K + 8]
  float* red = reinterpret_cast<float*>(sms + (size_t)kSmallN * sm_row(K) * 2);  // MODE 0: [NW][2][32][8]
  const int n_tasks = ld_cg_i32(&p.n_chunks[1]) * groups;
  for (int task = blockIdx.x; task < n_tasks; task += gridDim.x) {
    const int c = task / groups, sg = task - c * groups;
    const int4 rec = ld_cg_int4(&p.small_rec[c]);
    const int e = rec.x, poff = rec.y, nt = rec.z;
    const int ng = (nt + 7) >> 3;
    const uint8_t* base = (e < E) ? (p.base ? p.base[e] : a.arena + (int64_t)e * a.blob) : a.shared;
    // the chunk's B rows; rows past nt are zero (row addresses looked up once)
    __shared__ const __half* s_row[kSmallN];
    if (tid < kSmallN)
      s_row[tid] = tid >= nt ? nullptr
                 : MODE == 0 ? p.x16p + (size_t)ld_cg_i32(&p.pair_token[poff + tid]) * H
                             : p.h16p + (size_t)(poff + tid) * I;
    __syncthreads();
    const int per_row = K / 8;
    for (int o = tid; o < kSmallN * per_row; o += NT) {
      const int n = o / per_row, cc = o - n * per_row;
      __half* dst = bs + (size_t)n * sm_row(K) + cc * 8;
      const __half* src = s_row[n];
      if (src)
        cp_async16(smem_u32(dst), src + cc * 8);
      else
        *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();
    uint4 w0[kSmBatch], w1[kSmBatch];
    uint2 s0[kSmBatch], s1[kSmBatch];
    if (MODE == 0) {
      for (int si = 0; si < SG; ++si) {
        const int s = sg * SG + si;
        const uint8_t* strip = base + (int64_t)s * gu_strip_bytes(H);
        float ag[2][4] = {}, au[2][4] = {};
        for (int st0 = warp; st0 < nst; st0 += NW * kSmBatch) {
          sm_load_w<0>(strip, K, st0, NW, nst, lane, g, w0, s0, w1, s1);
#pragma unroll
          for (int b = 0; b < kSmBatch; ++b) {
            const int st = st0 + NW * b;
            if (st < nst) {
#pragma unroll
              for (int q = 0; q < 2; ++q) {
                if (q < ng) {
                  uint4 b01, b23;
                  sm_load_b(bs, K, q, st, g, t4, b01, b23);
                  supertile_mma(ag[q], w0[b], s0[b], b01, b23);
                  supertile_mma(au[q], w1[b], s1[b], b01, b23);
                }
              }
            }
          }
        }
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          float4* dst = reinterpret_cast<float4*>(red + ((warp * 2 + q) * 32 + lane) * 8);
          dst[0] = make_float4(ag[q][0], ag[q][1], ag[q][2], ag[q][3]);
          dst[1] = make_float4(au[q][0], au[q][1], au[q][2], au[q][3]);
        }
        __syncthreads();
        if (warp < ng) {  // warp q sums the K slices of n8 group q, in warp order
          const int q = warp;
          float gv[4] = {0.f, 0.f, 0.f, 0.f}, uv[4] = {0.f, 0.f, 0.f, 0.f};
          for (int w = 0; w < NW; ++w) {
            const float4* src = reinterpret_cast<const float4*>(red + ((w * 2 + q) * 32 + lane) * 8);
            const float4 x0 = src[0], x1 = src[1];
            gv[0] += x0.x; gv[1] += x0.y; gv[2] += x0.z; gv[3] += x0.w;
            uv[0] += x1.x; uv[1] += x1.y; uv[2] += x1.z; uv[3] += x1.w;
          }
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            const int row = s * 16 + ((cc < 2) ? g : g + 8), n = q * 8 + 2 * t4 + (cc & 1);
            if (n < nt)
              p.h16p[(size_t)(poff + n) * I + row] =
                  __float2half_rn(__fdividef(gv[cc], 1.0f + __expf(-gv[cc])) * uv[cc]);
          }
        }
        __syncthreads();  // red is reused by the next strip
      }
    } else {
      int zr[2][2];  // z rows of this lane's output columns
#pragma unroll
      for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int n = q * 8 + 2 * t4 + h;
          zr[q][h] = n < nt ? ld_cg_i32(&p.pair_z[poff + n]) : 0;
        }
      for (int si = warp; si < SG; si += NW) {
        const int s = sg * SG + si;
        const uint8_t* strip = base + down_base(H, I) + (int64_t)s * down_strip_bytes(I);
        float acc[2][4] = {};
        for (int st0 = 0; st0 < nst; st0 += kSmBatch) {
          sm_load_w<1>(strip, K, st0, 1, nst, lane, g, w0, s0, w1, s1);
#pragma unroll
          for (int b = 0; b < kSmBatch; ++b) {
            const int st = st0 + b;
            if (st < nst) {
#pragma unroll
              for (int q = 0; q < 2; ++q) {
                if (q < ng) {
                  uint4 b01, b23;
                  sm_load_b(bs, K, q, st, g, t4, b01, b23);
                  supertile_mma(acc[q], w0[b], s0[b], b01, b23);
                }
              }
            }
          }
        }
#pragma unroll
        for (int q = 0; q < 2; ++q)
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            const int row = s * 16 + ((cc < 2) ? g : g + 8), n = q * 8 + 2 * t4 + (cc & 1);
            if (n < nt) p.z16[(size_t)zr[q][cc & 1] * H + row] = __float2half_rn(acc[q][cc]);
          }
      }
    }
    __syncthreads();  // the staged rows are replaced by the next task's
  }
}

template <int MODE>
__global__ void __launch_bounds__(kExpThreads, 1) prefill_expert_kernel(LayerArgs a, PrefillArgs p) {
  extern __shared__ __align__(1024) unsigned char smraw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(sm);
  const uint32_t bar0 = sbase + kOffBar;
  auto raw_full = [&](int r) { return bar0 + 8u * r; };
  auto raw_empty = [&](int r) { return bar0 + 8u * (kRawStages + r); };
  auto a_full = [&](int s) { return bar0 + 8u * (2 * kRawStages + s); };
  auto b_empty = [&](int s) { return bar0 + 8u * (2 * kRawStages + kAStages + s); };
  auto b_full = [&](int s) { return bar0 + 8u * (2 * kRawStages + kAStages + kBStages + s); };
  const int acc0 = 2 * kRawStages + kAStages + 2 * kBStages;
  auto acc_full = [&](int b) { return bar0 + 8u * (acc0 + b); };
  auto acc_empty = [&](int b) { return bar0 + 8u * (acc0 + 2 + b); };
  const uint32_t drain = bar0 + 8u * (acc0 + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kOffTmem);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = a.H, I = a.I, E = a.E;
  const int MB = MODE == 0 ? I / 64 : H / 128;
  const int KS = MODE == 0 ? H / 64 : I / 64;
  const int Kdim = MODE == 0 ? H : I;
  const int n_tasks = ld_cg_i32(&p.n_chunks[0]) * MB;
  const uint64_t deadline = global_ns() + kPipeTimeoutNs;
  bool ok = true;

  if (tid == 0) {
    for (int r = 0; r < kRawStages; ++r) {
      mbar_init(raw_full(r), 1);
      mbar_init(raw_empty(r), kProd);
    }
    for (int s = 0; s < kAStages; ++s) mbar_init(a_full(s), kProd);
    for (int s = 0; s < kBStages; ++s) {
      mbar_init(b_empty(s), 1);
      mbar_init(b_full(s), kGather * 32);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(acc_full(b), 1);
      mbar_init(acc_empty(b), kXEpiWarps);
    }
    mbar_init(drain, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kXMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(tmem_slot)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---- packed tiles: lanes 0-7 the nibbles of strip lane, 8-15 its scales
    int rb = 0;
    for (int t = blockIdx.x; t < n_tasks && ok; t += gridDim.x) {
      const Task tk = load_task(p, MB, t);
      const uint8_t* base = (tk.e < E) ? (p.base ? p.base[tk.e] : a.arena + (int64_t)tk.e * a.blob) : a.shared;
      const int strip = lane & 7;
      const uint8_t* sp;
      if (MODE == 0)
        sp = base + (int64_t)(tk.mb * 4 + (strip & 3)) * gu_strip_bytes(H) + ((strip >> 2) ? 9ll * H : 0);
      else
        sp = base + down_base(H, I) + (int64_t)(tk.mb * 8 + strip) * down_strip_bytes(I);
      for (int ks0 = 0; ks0 < KS; ks0 += kRawR, ++rb) {
        const int len = min(kRawR, KS - ks0);
        const int r = rb % kRawStages, use = rb / kRawStages;
        if (lane == 0 && use > 0) wait_bar(raw_empty(r), (use - 1) & 1, a, deadline, ok);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        if (lane == 0) mbar_expect_tx(raw_full(r), (uint32_t)(8 * len * (512 + 64)));
        __syncwarp();
        const uint32_t sRaw = sbase + kOffRaw + r * kRawBytes;
        if (lane < 8)
          bulk_g2s(sRaw + lane * (kRawR * 512), sp + ks0 * 512, len * 512, raw_full(r));
        else if (lane < 16)
          bulk_g2s(sRaw + 8 * kRawR * 512 + strip * (kRawR * 64), sp + 8 * Kdim + ks0 * 64, len * 64, raw_full(r));
      }
    }
  } else if (warp <= kProd) {
    // ---- dequant: warp w, strip w, all four k-tiles of each k-step
    const int w = warp - 1;
    const int gg = lane >> 2;
    const int R0 = (MODE == 0) ? 32 * (w & 3) + 8 * (w >> 2) : 16 * w;  // tile row of strip row 0
    const int rstep = (MODE == 0) ? 16 : 8;                              // tile rows from g to g + 8
    const int mi = lane >> 3;  // stmatrix matrix: (row g | g + 8) x (low | high 8 k of the k-tile)
    const int st_row = R0 + (lane & 7) + ((mi & 1) ? rstep : 0);
    int rb = 0, g = 0;
    for (int t = blockIdx.x; t < n_tasks && ok; t += gridDim.x) {
      for (int ks = 0; ks < KS && ok; ++ks, ++g) {
        const int j = ks % kRawR;
        const int r = rb % kRawStages;
        if (j == 0 && !wait_bar(raw_full(r), (rb / kRawStages) & 1, a, deadline, ok)) break;
        const unsigned char* raw = sm + kOffRaw + r * kRawBytes;
        const uint4 nib = *reinterpret_cast<const uint4*>(raw + (w * kRawR + j) * 512 + lane * 16);
        const uint2 sc = *reinterpret_cast<const uint2*>(raw + 8 * kRawR * 512 + (w * kRawR + j) * 64 + gg * 8);
        const int len = min(kRawR, KS - (ks - j));
        if (j == len - 1) {  // the raw stage is consumed (this warp's part is in registers)
          __syncwarp();
          if (lane == 0) mbar_arrive(raw_empty(r));
          ++rb;
        }
        // A stage g % kAStages is free once the MMA of k-step g - kAStages completed
        const int s = g % kAStages;
        if (g >= kAStages) {
          const int gp = g - kAStages;
          if (!wait_bar(b_empty(gp % kBStages), (gp / kBStages) & 1, a, deadline, ok)) break;
        }
        const uint32_t sA = sbase + s * kTile;
        const uint32_t words[4] = {nib.x, nib.y, nib.z, nib.w};
#pragma unroll
        for (int kt = 0; kt < 4; ++kt) {
          const uint32_t scw = (kt < 2) ? sc.x : sc.y;  // k-tiles 0, 1: first block of 32; 2, 3: second
          const __half2 dg = __half2half2(__ushort_as_half((uint16_t)(scw & 0xFFFFu)));
          const __half2 dg8 = __half2half2(__ushort_as_half((uint16_t)(scw >> 16)));
          __half2 q[4];
          dequant_word(words[kt], q);
          stmatrix_x4(sA + sw128_off(st_row, 2 * kt + (mi >> 1)), h2u(__hmul2(q[0], dg)), h2u(__hmul2(q[1], dg8)),
                      h2u(__hmul2(q[2], dg)), h2u(__hmul2(q[3], dg8)));
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(a_full(s));
      }
    }
  } else if (warp <= kProd + kGather) {
    // ---- gather: B rows of k-step gb into B stage gb % kBStages, running up
    //      to kBStages - kAStages k-steps ahead of the MMA
    const int gt = tid - 32 * (1 + kProd);  // 0 .. 255
    const int bc = gt & 7;                  // 16-byte chunk of rows (gt >> 3) + 32 q
    constexpr int kRows = kPfN / 32;
    int gb = 0;
    for (int t = blockIdx.x; t < n_tasks && ok; t += gridDim.x) {
      const Task tk = load_task(p, MB, t);
      const __half* brow[kRows];
#pragma unroll
      for (int q = 0; q < kRows; ++q) {
        const int n = (gt >> 3) + 32 * q;
        brow[q] = (n >= tk.nt) ? nullptr
                               : (MODE == 0 ? p.x16p + (size_t)ld_cg_i32(&p.pair_token[tk.poff + n]) * H
                                            : p.h16p + (size_t)(tk.poff + n) * I);
      }
      for (int ks = 0; ks < KS && ok; ++ks, ++gb) {
        const int s = gb % kBStages;
        if (gb >= kBStages && !wait_bar(b_empty(s), (gb / kBStages - 1) & 1, a, deadline, ok)) break;
        const uint32_t sB = sbase + kOffB + s * kBTile;
#pragma unroll
        for (int q = 0; q < kRows; ++q)
          if (brow[q]) cp_async16(sB + sw128_off((gt >> 3) + 32 * q, bc), brow[q] + ks * 64 + bc * 8);
        cp_async_arrive_noinc(b_full(s));
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else if (warp == kXMmaWarp) {
    // ---- MMA issue: one thread, double-buffered accumulator (2 x 256 columns)
    if (lane == 0) {
      int g = 0, i = 0;
      Task nxt = blockIdx.x < n_tasks ? load_task(p, MB, blockIdx.x) : Task{};
      for (int t = blockIdx.x; t < n_tasks && ok; t += gridDim.x, ++i) {
        const Task tk = nxt;
        if (t + (int)gridDim.x < n_tasks) nxt = load_task(p, MB, t + gridDim.x);
        const uint32_t idesc = instr_desc((tk.nt + 15) & ~15, false);
        const int b = i & 1, ub = i >> 1;
        if (ub > 0 && !wait_bar(acc_empty(b), (ub - 1) & 1, a, deadline, ok, 0)) break;
        tc_fence_after();
        const uint32_t dt = tmem + (uint32_t)(b * kPfN);
        for (int ks = 0; ks < KS; ++ks, ++g) {
          const int sa = g % kAStages, sb = g % kBStages;
          if (!wait_bar(a_full(sa), (g / kAStages) & 1, a, deadline, ok, 0)) break;
          if (!wait_bar(b_full(sb), (g / kBStages) & 1, a, deadline, ok, 0)) break;
          // the stage was written through the generic proxy (stmatrix, cp.async)
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          tc_fence_after();
          const uint32_t sA = sbase + sa * kTile, sB = sbase + kOffB + sb * kBTile;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            tc_mma(dt, desc_sw128(sA + j * 32), desc_sw128(sB + j * 32), idesc, (ks > 0 || j > 0) ? 1u : 0u);
          tc_commit(b_empty(sb));
        }
        if (!ok) break;
        tc_commit(acc_full(b));
      }
      // every MMA this thread issued completes before TMEM is released
      tc_commit(drain);
      bool dok = true;
      wait_bar(drain, 0, a, deadline + kPipeTimeoutNs, dok);
    }
    __syncwarp();
  } else {
    // ---- epilogue: TMEM lanes 32 (warp % 4) .. + 31 are tile rows; two warps
    //      per quadrant, each half of the columns
    const int quad = warp & 3, ehalf = (warp - kXEpi0) >> 2;
    const int row = quad * 32 + lane;
    int i = 0;
    Task nxt = blockIdx.x < n_tasks ? load_task(p, MB, blockIdx.x) : Task{};
    for (int t = blockIdx.x; t < n_tasks && ok; t += gridDim.x, ++i) {
      const Task tk = nxt;
      if (t + (int)gridDim.x < n_tasks) nxt = load_task(p, MB, t + gridDim.x);
      const int cbeg = ehalf * (kPfN / 2), cend = min(tk.nt, cbeg + kPfN / 2);
      int zq[kPfN / 64];  // MODE 1: z rows of the pairs cbeg + lane + 32 q
      if (MODE == 1) {
#pragma unroll
        for (int q = 0; q < kPfN / 64; ++q) {
          const int n = cbeg + lane + 32 * q;
          zq[q] = n < cend ? ld_cg_i32(&p.pair_z[tk.poff + n]) : 0;
        }
      }
      const int b = i & 1, ub = i >> 1;
      if (!wait_bar(acc_full(b), ub & 1, a, deadline, ok)) break;
      tc_fence_after();
      const uint32_t taddr = tmem + (uint32_t)(b * kPfN) + ((uint32_t)(quad * 32) << 16);
      for (int c0 = cbeg; c0 < cend; c0 += 32) {
        float v[32];
        tc_ld32(taddr + (uint32_t)c0, v);
        if (MODE == 0) {
          // lanes l (gate row) and l ^ 8 (its up row): the gate lane finishes the
          // even columns, the up lane the odd ones, without divergence
          const bool up = (row & 8) != 0;
          const int fi = tk.mb * 64 + 8 * (row >> 4) + (row & 7);
          __half* hbase = p.h16p + (size_t)(tk.poff + c0 + (up ? 1 : 0)) * I + fi;
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            const float send = up ? v[2 * q] : v[2 * q + 1];
            const float recv = __shfl_xor_sync(0xffffffffu, send, 8);
            const float gv = up ? recv : v[2 * q], uv = up ? v[2 * q + 1] : recv;
            const float h = __fdividef(gv, 1.0f + __expf(-gv)) * uv;
            if (c0 + 2 * q + (up ? 1 : 0) < cend) hbase[(size_t)(2 * q) * I] = __float2half_rn(h);
          }
        } else {
          const int orow = tk.mb * 128 + row;
          const int zb = (c0 - cbeg) >> 5;
          const int zsel = zb == 0 ? zq[0] : zb == 1 ? zq[1] : zb == 2 ? zq[2] : zq[3];
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int zr = __shfl_sync(0xffffffffu, zsel, j);
            if (c0 + j < cend) p.z16[(size_t)zr * H + orow] = __float2half_rn(v[j]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty(b));
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kXMmaWarp) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem));
}

// y[t][r] = sum_j w_tj z[t][j][r] in ascending expert order, + z[t][k][r]; 8 outputs per thread.
__global__ void __launch_bounds__(256) prefill_combine_kernel(LayerArgs a, PrefillArgs p) {
  const int H = a.H, k = a.k;
  const long long i = (long long)blockIdx.x * 256 + threadIdx.x;
  const int t = (int)(i / (H / 8)), c8 = (int)(i % (H / 8)) * 8;
  if (t >= a.T) return;
  float acc[8] = {};
  for (int j = 0; j < k; ++j) {
    const float w = a.topk_w[t * k + j];
    const uint4 zv = ld_cg4(p.z16 + ((size_t)t * (k + 1) + j) * H + c8);
    const __half2* z2 = reinterpret_cast<const __half2*>(&zv);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 f = __half22float2(z2[q]);
      acc[2 * q] = fmaf(w, f.x, acc[2 * q]);
      acc[2 * q + 1] = fmaf(w, f.y, acc[2 * q + 1]);
    }
  }
  if (a.n_shared) {
    const uint4 zv = ld_cg4(p.z16 + ((size_t)t * (k + 1) + k) * H + c8);
    const __half2* z2 = reinterpret_cast<const __half2*>(&zv);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 f = __half22float2(z2[q]);
      acc[2 * q] += f.x;
      acc[2 * q + 1] += f.y;
    }
  }
  uint32_t out[4];
#pragma unroll
  for (int q = 0; q < 4; ++q)
    out[q] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * q])) |
             ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * q + 1])) << 16);
  *reinterpret_cast<uint4*>(a.y + (size_t)t * H + c8) = make_uint4(out[0], out[1], out[2], out[3]);
}

size_t pf_align(size_t b) { return (b + 255) & ~size_t(255); }

bool encode(TensorMapEncodeFn enc, CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base,
            const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box) {
  const cuuint32_t es[3] = {1, 1, 1};
  return enc(m, dt, (cuuint32_t)rank, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

size_t prefill_scratch_bytes(int H, int I, int E, int k, int Tm) {
  if (Tm <= kMaxTokens) return 0;
  const size_t P = (size_t)Tm * (k + 1), words = (size_t)(Tm + 31) / 32;
  const size_t chunks = (size_t)E + 2 + P / kPfN;
  return pf_align(4ull * (E + 1)) + 2 * pf_align(4ull * (E + 2)) + pf_align(8) + pf_align(16 * chunks) +
         pf_align(16ull * (E + 1)) +
         2 * pf_align(4 * P) +
         2 * pf_align(4ull * E * words) + pf_align(6ull * E * H) + pf_align(4ull * E) + pf_align(4ull * Tm) +
         pf_align(2ull * Tm * H) +
         pf_align(2 * P * I) +
         pf_align(2 * P * H) +
         pf_align(8ull * E) + pf_align(16 * chunks) + pf_align(16ull * (E + 1)) + pf_align(8);
}

PrefillArgs prefill_carve(void* block, int H, int I, int E, int k, int Tm) {
  const size_t P = (size_t)Tm * (k + 1), words = (size_t)(Tm + 31) / 32;
  uint8_t* b = (uint8_t*)block;
  size_t off = 0;
  auto carve = [&](size_t bytes) {
    uint8_t* r = b + off;
    off += pf_align(bytes);
    return r;
  };
  PrefillArgs p;
  p.counts = (int32_t*)carve(4ull * (E + 1));
  p.offsets = (int32_t*)carve(4ull * (E + 2));
  p.chunk_off = (int32_t*)carve(4ull * (E + 2));
  p.n_chunks = (int32_t*)carve(8);
  p.chunk_rec = (int4*)carve(16 * ((size_t)E + 2 + P / kPfN));
  p.small_rec = (int4*)carve(16 * ((size_t)E + 1));
  p.pair_token = (int32_t*)carve(4 * P);
  p.pair_z = (int32_t*)carve(4 * P);
  p.bitmap = (uint32_t*)carve(4ull * E * words);
  p.prefix = (int32_t*)carve(4ull * E * words);
  p.w_split = (uint16_t*)carve(6ull * E * H);
  p.wnorm = (float*)carve(4ull * E);
  p.xnorm = (float*)carve(4ull * Tm);
  p.x16p = (__half*)carve(2ull * Tm * H);
  p.h16p = (__half*)carve(2 * P * I);
  p.z16 = (__half*)carve(2 * P * H);
  p.words = (int)words;
  p.base = nullptr;  // resident layer; a pooled call points it at its wave table
  p.wave_chunk_rec = (int4*)carve(16 * ((size_t)E + 2 + P / kPfN));
  p.wave_small_rec = (int4*)carve(16 * ((size_t)E + 1));
  p.wave_n = (int32_t*)carve(8);
  p.base_table = (const uint8_t**)carve(8ull * E);
  return p;
}

bool prefill_encode_maps(TensorMapEncodeFn enc, const PrefillArgs& p, int H, int I, int E, int k, int Tm,
                         PrefillMaps* m) {
  (void)I;
  (void)k;
  (void)Tm;
  const cuuint64_t dims[3] = {(cuuint64_t)H, (cuuint64_t)E, 3};
  const cuuint64_t strides[2] = {(cuuint64_t)H * 2, (cuuint64_t)E * H * 2};
  const cuuint32_t box[3] = {64, 128, 1};
  return encode(enc, &m->w_split, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, p.w_split, dims, strides, box);
}

bool prefill_encode_x(TensorMapEncodeFn enc, const void* x, int H, int T, PrefillMaps* m) {
  const cuuint64_t dims[2] = {(cuuint64_t)H, (cuuint64_t)T};
  const cuuint64_t strides[1] = {(cuuint64_t)H * 2};
  const cuuint32_t box[2] = {64, 128};
  return encode(enc, &m->x_bf16, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, x, dims, strides, box);
}

cudaError_t prefill_configure() {
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(prefill_expert_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem)))
    return e;
  if ((e = cudaFuncSetAttribute(prefill_expert_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem)))
    return e;
  if ((e = cudaFuncSetAttribute(prefill_small_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)sm_smem(0, kMaxHidden))))
    return e;
  if ((e = cudaFuncSetAttribute(prefill_small_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)sm_smem(1, kMaxInter))))
    return e;
  return cudaFuncSetAttribute(prefill_router_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kRtSmem);
}

cudaError_t launch_prefill_route(const LayerArgs& a, const PrefillArgs& p, const PrefillMaps& m, int sm_count,
                                 cudaStream_t s) {
  cudaError_t e;
  if ((e = cudaMemsetAsync(p.counts, 0, sizeof(int32_t) * (size_t)(a.E + 1), s)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(p.bitmap, 0, sizeof(uint32_t) * (size_t)a.E * p.words, s)) != cudaSuccess) return e;
  prefill_prep_kernel<<<sm_count * 4, 256, 0, s>>>(a, p);
  const int router_tasks = ((a.E + 127) / 128) * ((a.T + 127) / 128);
  prefill_router_kernel<<<router_tasks < sm_count ? router_tasks : sm_count, kGemmThreads, kRtSmem, s>>>(
      a, m.w_split, m.x_bf16);
  const int tk_grid = (a.T + 7) / 8;
  if (a.E <= 32)
    prefill_topk_kernel<1><<<tk_grid, 256, 0, s>>>(a, p);
  else if (a.E <= 64)
    prefill_topk_kernel<2><<<tk_grid, 256, 0, s>>>(a, p);
  else if (a.E <= 128)
    prefill_topk_kernel<4><<<tk_grid, 256, 0, s>>>(a, p);
  else if (a.E <= 256)
    prefill_topk_kernel<8><<<tk_grid, 256, 0, s>>>(a, p);
  else if (a.E <= 512)
    prefill_topk_kernel<16><<<tk_grid, 256, 0, s>>>(a, p);
  else if (a.E <= 1024)
    prefill_topk_kernel<32><<<tk_grid, 256, 0, s>>>(a, p);
  else
    prefill_topk_kernel<0><<<tk_grid, 256, 0, s>>>(a, p);
  prefill_prefix_kernel<<<(a.E + 7) / 8, 256, 0, s>>>(a, p);
  prefill_scan_kernel<<<1, 1024, 0, s>>>(a, p);
  prefill_pairs_kernel<<<(a.T * (a.k + 1) + 255) / 256, 256, 0, s>>>(a, p);
  return cudaGetLastError();
}

namespace {

void launch_experts(const LayerArgs& a, const PrefillArgs& p, int sm_count, cudaStream_t s) {
  prefill_small_kernel<0><<<sm_count * 2, sm_warps(0) * 32, sm_smem(0, a.H), s>>>(a, p);
  prefill_expert_kernel<0><<<sm_count, kExpThreads, kGemmSmem, s>>>(a, p);
  prefill_small_kernel<1><<<sm_count * 8, sm_warps(1) * 32, sm_smem(1, a.I), s>>>(a, p);
  prefill_expert_kernel<1><<<sm_count, kExpThreads, kGemmSmem, s>>>(a, p);
}

// This wave's chunk records: those whose expert has a base in p.base (the
// shared expert's in wave 0), in any order (each chunk writes its own rows).
__global__ void __launch_bounds__(1024) prefill_wave_kernel(LayerArgs a, PrefillArgs p, int wave0) {
  __shared__ int c0, c1;
  const int tid = threadIdx.x, E = a.E;
  if (tid == 0) c0 = c1 = 0;
  __syncthreads();
  const int n0 = ld_cg_i32(&p.n_chunks[0]), n1 = ld_cg_i32(&p.n_chunks[1]);
  for (int i = tid; i < n0; i += blockDim.x) {
    const int4 r = ld_cg_int4(&p.chunk_rec[i]);
    if (r.x >= E ? wave0 != 0 : p.base[r.x] != nullptr) p.wave_chunk_rec[atomicAdd(&c0, 1)] = r;
  }
  for (int i = tid; i < n1; i += blockDim.x) {
    const int4 r = ld_cg_int4(&p.small_rec[i]);
    if (r.x >= E ? wave0 != 0 : p.base[r.x] != nullptr) p.wave_small_rec[atomicAdd(&c1, 1)] = r;
  }
  __syncthreads();
  if (tid == 0) {
    p.wave_n[0] = c0;
    p.wave_n[1] = c1;
  }
}

}  // namespace

cudaError_t launch_prefill_wave(const LayerArgs& a, const PrefillArgs& p, int sm_count, bool wave0, cudaStream_t s) {
  PrefillArgs q = p;
  q.base = p.base_table;
  prefill_wave_kernel<<<1, 1024, 0, s>>>(a, q, wave0 ? 1 : 0);
  q.n_chunks = p.wave_n;
  q.chunk_rec = p.wave_chunk_rec;
  q.small_rec = p.wave_small_rec;
  launch_experts(a, q, sm_count, s);
  return cudaGetLastError();
}

cudaError_t launch_prefill_combine(const LayerArgs& a, const PrefillArgs& p, cudaStream_t s) {
  const long long n = (long long)a.T * (a.H / 8);
  prefill_combine_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(a, p);
  return cudaGetLastError();
}

cudaError_t launch_prefill(const LayerArgs& a, const PrefillArgs& p, const PrefillMaps& m, int sm_count,
                           cudaStream_t s) {
  cudaError_t e = launch_prefill_route(a, p, m, sm_count, s);
  if (e != cudaSuccess) return e;
  launch_experts(a, p, sm_count, s);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  return launch_prefill_combine(a, p, s);
}

}  // namespace moe
