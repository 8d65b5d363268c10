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
//              index), ascending expert order, softmax over the selection;
//              bit t of the expert's token bitmap
//   prefix     warp per expert: set bits before each bitmap word
//   scan       per-expert counts -> pair offsets and 128-token chunks
//   pairs      thread per (token, rank): its place in the expert's token
//              list (ascending token: a stable counting sort)
//   gate/up    grouped GEMM, M = 128 (64 gate rows and the 64 matching up
//              rows), N = the chunk's tokens (<= 128, rounded up to 16),
//              K = H in steps of 64.  One TMA warp streams the packed 4-bit
//              tiles into shared memory (bulk copies) and gathers the
//              chunk's activation rows (tile::gather4); eight warps
//              dequantize the tiles to fp16 d*q and write them with stmatrix
//              in the 128-byte-swizzled K-major layout; one thread issues the
//              MMAs into a double-buffered TMEM accumulator; four epilogue
//              warps compute h = silu(g) * u.
//   down       the same engine, M = 128 output rows, K = I, B = the pairs'
//              h rows (contiguous, tiled TMA); the epilogue writes each
//              pair's expert output z as fp16.
//   combine    y[t] = sum_j w_j z_j (ascending expert) + z_shared in fp32,
//              rounded once to bf16.
#include <cfloat>
#include <climits>

#include "moe.h"
#include "moe_internal.h"
#include "moe_prefill.h"

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
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
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
// Four rows (r0..r3) x 64 elements at column c0 -> 512 consecutive shared bytes.
__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* map, int c0, int r0, int r1, int r2,
                                            int r3, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, "
      "%4, %5, %6}], [%7];" ::"r"(dst),
      "l"((uint64_t)map), "r"(c0), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(bar)
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

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const LayerArgs& a, uint64_t deadline,
                                         bool& ok) {
  if (!ok) return false;
  int spins = 0;
  while (!mbar_try_wait(bar, parity)) {
    if (((++spins) & 255) == 0 && global_ns() > deadline) {
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
  int bad = 0;
  for (size_t i = ((size_t)blockIdx.x * 256 + threadIdx.x) * 8; i < nx; i += stride * 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(a.x + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float f0 = __uint_as_float(w[q] << 16), f1 = __uint_as_float(w[q] & 0xFFFF0000u);
      bad |= !(fabsf(f0) < 65504.f) || !(fabsf(f1) < 65504.f);
      o[q] = h2u(__floats2half2_rn(f0, f1));
    }
    *reinterpret_cast<uint4*>(p.x16p + i) = make_uint4(o[0], o[1], o[2], o[3]);
  }
  if (bad) set_error(a, MOE_ERR_DEVICE);
}

// Warp per token: k rounds of a warp argmax (value desc, index asc).
__global__ void __launch_bounds__(256) prefill_topk_kernel(LayerArgs a, PrefillArgs p) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int E = a.E, k = a.k;
  if (t >= a.T) return;
  const float* lt = a.logits + (size_t)t * E;
  int sel[kMaxTopK];
  float selv[kMaxTopK];
  uint32_t taken[kMaxExperts / 1024] = {};  // bit i: logit lane + 32 i already selected
  for (int r = 0; r < k; ++r) {
    float bv = -FLT_MAX;
    int bi = INT_MAX;
    for (int e = lane, i = 0; e < E; e += 32, ++i) {
      if ((taken[i >> 5] >> (i & 31)) & 1u) continue;
      const float v = lt[e];
      if (v > bv || (v == bv && e < bi)) {
        bv = v;
        bi = e;
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
    if (bi == INT_MAX) {  // fewer than k comparable logits (NaN): flagged; keep the indices distinct
      if (lane == 0) set_error(a, MOE_ERR_DEVICE);
      bi = r;
    }
    if (lane == (bi & 31)) taken[(bi >> 5) >> 5] |= 1u << ((bi >> 5) & 31);
    sel[r] = bi;
    selv[r] = bv;
  }
  if (lane == 0) {
    const float m = selv[0];
    for (int i = 1; i < k; ++i) {  // ascending expert index
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
      a.topk_idx[t * k + j] = sel[j];
      a.topk_w[t * k + j] = expf(selv[j] - m) / z;
      atomicAdd(&p.counts[sel[j]], 1);
      atomicOr(&p.bitmap[(size_t)sel[j] * p.words + (t >> 5)], 1u << (t & 31));
    }
  }
}

// Warp per routed expert: prefix[e][w] = set bits of bitmap row e before word w.
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
}

// One CTA: offsets and chunk offsets of the E routed experts and the shared
// expert (entry E, all T tokens); layer statistics.
__global__ void __launch_bounds__(1024) prefill_scan_kernel(LayerArgs a, PrefillArgs p) {
  __shared__ int wsum[2][32];
  __shared__ int s_used;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = a.E, NE = E + a.n_shared;
  const int per = (NE + 1023) / 1024;
  if (tid == 0) s_used = 0;
  __syncthreads();
  int c_cnt = 0, c_chk = 0, used = 0;
  for (int i = 0; i < per; ++i) {
    const int e = tid * per + i;
    if (e < NE) {
      const int cnt = (e < E) ? p.counts[e] : a.T;
      c_cnt += cnt;
      c_chk += (cnt + kPfN - 1) / kPfN;
      used += (e < E && cnt > 0);
    }
  }
  if (used) atomicAdd(&s_used, used);
  int ia = c_cnt, ib = c_chk;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int va = __shfl_up_sync(0xffffffffu, ia, o), vb = __shfl_up_sync(0xffffffffu, ib, o);
    if (lane >= o) {
      ia += va;
      ib += vb;
    }
  }
  if (lane == 31) {
    wsum[0][warp] = ia;
    wsum[1][warp] = ib;
  }
  __syncthreads();
  int ba = 0, bb = 0, ta = 0, tb = 0;
  for (int w = 0; w < 32; ++w) {
    if (w < warp) {
      ba += wsum[0][w];
      bb += wsum[1][w];
    }
    ta += wsum[0][w];
    tb += wsum[1][w];
  }
  int oa = ba + ia - c_cnt, ob = bb + ib - c_chk;
  for (int i = 0; i < per; ++i) {
    const int e = tid * per + i;
    if (e < NE) {
      const int cnt = (e < E) ? p.counts[e] : a.T;
      p.offsets[e] = oa;
      p.chunk_off[e] = ob;
      oa += cnt;
      ob += (cnt + kPfN - 1) / kPfN;
    }
  }
  if (tid == 0) {
    p.offsets[NE] = ta;
    p.chunk_off[NE] = tb;
    p.n_chunks[0] = tb;
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
constexpr int kRaw = 8 * 512 + 8 * 64;  // packed 4-bit tile of 128 rows x 64 k: 8 strips of nibbles + scales
constexpr int kTmaWarp = 0;
constexpr int kDeq0 = 1;     // warps 1-8: dequantize one 16-row strip each
constexpr int kMmaWarp = 9;  // allocates TMEM; lane 0 issues the MMAs
constexpr int kEpi0 = 10;    // warps 10-13: epilogue; TMEM lane quadrant = warp % 4
constexpr int kGemmThreads = (kEpi0 + 4) * 32;

// MODE 0 gate/up, 1 down: stages of [A tile][B tile][raw packed tile]
// MODE 2 router: stages of [3 A tiles (weight pieces)][B tile]
template <int MODE>
struct Cfg {
  static constexpr int kStages = MODE == 2 ? 3 : 5;
  static constexpr int kA = MODE == 2 ? 3 * kTile : kTile;
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kStages * kA;
  static constexpr int kOffRaw = kOffB + kStages * kTile;
  static constexpr int kOffBar = kOffRaw + (MODE == 2 ? 0 : kStages * kRaw);
  // barriers: raw_full[S], b_full[S], a_full[S], empty[S], acc_full[2], acc_empty[2], drain
  static constexpr int kOffTmem = kOffBar + 8 * (4 * kStages + 5);
  static constexpr int kBytes = kOffTmem + 16 + 1024;  // + alignment slack
};

struct Task {
  int e, n0, nt, mb;
};

// Tasks of the grouped GEMMs: t -> expert list entry e, first pair n0 of the
// chunk within e, its tokens nt and the M-block.  M-blocks of one chunk are
// consecutive tasks, so CTAs running them at once share the chunk's rows in L2.
__device__ __forceinline__ Task task_decode(const PrefillArgs& p, int NE, int MB, int t) {
  Task r;
  r.mb = t % MB;
  const int ch = t / MB;
  int lo = 0, hi = NE;  // the largest e with chunk_off[e] <= ch
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (ld_cg_i32(&p.chunk_off[mid]) <= ch)
      lo = mid;
    else
      hi = mid;
  }
  r.e = lo;
  r.n0 = (ch - ld_cg_i32(&p.chunk_off[lo])) * kPfN;
  const int cnt = ld_cg_i32(&p.offsets[lo + 1]) - ld_cg_i32(&p.offsets[lo]);
  r.nt = min(kPfN, cnt - r.n0);
  return r;
}
// Router tasks: t -> (M-block of 128 experts, 128-token block).
__device__ __forceinline__ Task router_task(int E, int T, int t) {
  const int MB = (E + 127) / 128;
  Task r;
  r.e = 0;
  r.mb = t % MB;
  r.n0 = (t / MB) * 128;
  r.nt = min(128, T - r.n0);
  return r;
}

// MODE 0: gate/up; M-block mb = intermediate rows 64 mb .. 64 mb + 63 of gate
//   and of up, K = H.  Tile row of local gate row i: 16 (i / 8) + i % 8; the
//   matching up row is 8 further, so an epilogue lane pairs with lane + 8.
// MODE 1: down; M-block mb = output rows 128 mb .. 128 mb + 127, K = I.
// MODE 2: router; M-block = 128 experts, N = 128 tokens, K = H, bf16 pieces.
template <int MODE>
__global__ void __launch_bounds__(kGemmThreads, 1)
    prefill_gemm_kernel(LayerArgs a, PrefillArgs p, const __grid_constant__ CUtensorMap mapA,
                        const __grid_constant__ CUtensorMap mapB) {
  using C = Cfg<MODE>;
  constexpr int S = C::kStages;
  extern __shared__ __align__(1024) unsigned char smraw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(sm);
  const uint32_t bar0 = sbase + C::kOffBar;
  auto raw_full = [&](int s) { return bar0 + 8u * s; };
  auto b_full = [&](int s) { return bar0 + 8u * (S + s); };
  auto a_full = [&](int s) { return bar0 + 8u * (2 * S + s); };
  auto empty = [&](int s) { return bar0 + 8u * (3 * S + s); };
  auto acc_full = [&](int b) { return bar0 + 8u * (4 * S + b); };
  auto acc_empty = [&](int b) { return bar0 + 8u * (4 * S + 2 + b); };
  const uint32_t drain = bar0 + 8u * (4 * S + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::kOffTmem);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = a.H, I = a.I, E = a.E;
  const int NE = E + a.n_shared;
  const int MB = MODE == 0 ? I / 64 : MODE == 1 ? H / 128 : (E + 127) / 128;
  const int KS = MODE == 1 ? I / 64 : H / 64;
  const int n_tasks = MODE == 2 ? MB * ((a.T + 127) / 128) : ld_cg_i32(&p.n_chunks[0]) * MB;
  const uint64_t deadline = global_ns() + kPipeTimeoutNs;
  bool ok = true;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(raw_full(s), 1);
      mbar_init(b_full(s), 1);
      mbar_init(a_full(s), 8);
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

  if (warp == kTmaWarp) {
    // ---- loads: packed weight tiles (bulk copies) and B rows (tensor maps)
    int g = 0;
    for (int t = blockIdx.x; t < n_tasks && ok; t += gridDim.x) {
      const Task tk = MODE == 2 ? router_task(E, a.T, t) : task_decode(p, NE, MB, t);
      const int nn = (tk.nt + 15) & ~15;
      const uint8_t* src = nullptr;  // this lane's packed source (lanes 0-7 nibbles, 8-15 scales of strip lane % 8)
      int tok[4] = {0, 0, 0, 0};
      int poff = 0;
      if (MODE != 2) {
        const uint8_t* base = (tk.e < E) ? a.arena + (int64_t)tk.e * a.blob : a.shared;
        const int strip = lane & 7;
        const uint8_t* sp;
        if (MODE == 0)
          sp = base + (int64_t)(tk.mb * 4 + (strip & 3)) * gu_strip_bytes(H) + ((strip >> 2) ? 9ll * H : 0);
        else
          sp = base + down_base(H, I) + (int64_t)(tk.mb * 8 + strip) * down_strip_bytes(I);
        src = (lane < 8) ? sp : sp + 8 * (MODE == 0 ? H : I);
        poff = ld_cg_i32(&p.offsets[tk.e]) + tk.n0;
        if (MODE == 0 && 4 * lane < nn) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int n = min(4 * lane + q, tk.nt - 1);
            tok[q] = ld_cg_i32(&p.pair_token[poff + n]);
          }
        }
      }
      for (int ks = 0; ks < KS; ++ks, ++g) {
        const int s = g % S, use = g / S;
        if (lane == 0 && use > 0) wait_bar(empty(s), (use - 1) & 1, a, deadline, ok);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        const uint32_t sA = sbase + C::kOffA + s * C::kA, sB = sbase + C::kOffB + s * kTile;
        if (MODE == 2) {
          if (lane == 0) {
            mbar_expect_tx(b_full(s), 4 * kTile);
#pragma unroll
            for (int pc = 0; pc < 3; ++pc) tma_3d(sA + pc * kTile, &mapA, ks * 64, tk.mb * 128, pc, b_full(s));
            tma_2d(sB, &mapB, ks * 64, tk.n0, b_full(s));
          }
        } else {
          if (lane == 0) {
            mbar_expect_tx(raw_full(s), kRaw);
            mbar_expect_tx(b_full(s), (uint32_t)nn * 128);
          }
          __syncwarp();
          const uint32_t sRaw = sbase + C::kOffRaw + s * kRaw;
          if (lane < 8)
            bulk_g2s(sRaw + lane * 512, src + ks * 512, 512, raw_full(s));
          else if (lane < 16)
            bulk_g2s(sRaw + 4096 + (lane - 8) * 64, src + ks * 64, 64, raw_full(s));
          if (MODE == 0) {
            if (4 * lane < nn) tma_gather4(sB + lane * 512, &mapB, ks * 64, tok[0], tok[1], tok[2], tok[3], b_full(s));
          } else {
            if (16 * lane < nn) tma_2d(sB + lane * 2048, &mapB, ks * 64, poff + 16 * lane, b_full(s));
          }
        }
      }
    }
  } else if (MODE != 2 && warp >= kDeq0 && warp < kDeq0 + 8) {
    // ---- dequantize strip w of the packed tile into the swizzled fp16 A tile
    const int w = warp - kDeq0;
    const int gg = lane >> 2;
    const int R0 = (MODE == 0) ? 32 * (w & 3) + 8 * (w >> 2) : 16 * w;  // tile row of strip row 0
    const int rstep = (MODE == 0) ? 16 : 8;                              // tile rows from g to g + 8
    // stmatrix: matrix mi = lane >> 3 is (row g | g + 8) x (low | high 8 k of the k-tile)
    const int mi = lane >> 3;
    const int st_row = R0 + (lane & 7) + ((mi & 1) ? rstep : 0);
    int my_tasks = 0;
    for (int t = blockIdx.x; t < n_tasks; t += gridDim.x) ++my_tasks;
    const int steps = my_tasks * KS;
    for (int g = 0; g < steps && ok; ++g) {
      const int s = g % S, use = g / S;
      if (!wait_bar(raw_full(s), use & 1, a, deadline, ok)) break;
      const unsigned char* raw = sm + C::kOffRaw + s * kRaw;
      const uint4 nib = *reinterpret_cast<const uint4*>(raw + w * 512 + lane * 16);
      const uint2 sc = *reinterpret_cast<const uint2*>(raw + 4096 + w * 64 + gg * 8);
      const uint32_t sA = sbase + C::kOffA + s * C::kA;
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
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(a_full(s));
    }
  } else if (warp == kMmaWarp) {
    // ---- MMA issue: one thread, double-buffered accumulator (2 x 128 columns)
    if (lane == 0) {
      int g = 0, i = 0;
      for (int t = blockIdx.x; t < n_tasks && ok; t += gridDim.x, ++i) {
        const Task tk = MODE == 2 ? router_task(E, a.T, t) : task_decode(p, NE, MB, t);
        const uint32_t idesc = instr_desc((tk.nt + 15) & ~15, MODE == 2);
        const int b = i & 1, ub = i >> 1;
        if (ub > 0 && !wait_bar(acc_empty(b), (ub - 1) & 1, a, deadline, ok)) break;
        tc_fence_after();
        const uint32_t dt = tmem + (uint32_t)(b * 128);
        for (int ks = 0; ks < KS; ++ks, ++g) {
          const int s = g % S, use = g / S;
          if (!wait_bar(b_full(s), use & 1, a, deadline, ok)) break;
          if (MODE != 2 && !wait_bar(a_full(s), use & 1, a, deadline, ok)) break;
          tc_fence_after();
          const uint32_t sA = sbase + C::kOffA + s * C::kA, sB = sbase + C::kOffB + s * kTile;
#pragma unroll
          for (int pc = 0; pc < (MODE == 2 ? 3 : 1); ++pc)
#pragma unroll
            for (int j = 0; j < 4; ++j)
              tc_mma(dt, desc_sw128(sA + pc * kTile + j * 32), desc_sw128(sB + j * 32), idesc,
                     (ks > 0 || j > 0 || pc > 0) ? 1u : 0u);
          tc_commit(empty(s));
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
  } else if (warp >= kEpi0) {
    // ---- epilogue: TMEM lanes 32 (warp % 4) .. + 31 are tile rows
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    int i = 0;
    for (int t = blockIdx.x; t < n_tasks && ok; t += gridDim.x, ++i) {
      const Task tk = MODE == 2 ? router_task(E, a.T, t) : task_decode(p, NE, MB, t);
      const int b = i & 1, ub = i >> 1;
      if (!wait_bar(acc_full(b), ub & 1, a, deadline, ok)) break;
      tc_fence_after();
      const int poff = MODE == 2 ? 0 : ld_cg_i32(&p.offsets[tk.e]) + tk.n0;
      const uint32_t taddr = tmem + (uint32_t)(b * 128) + ((uint32_t)(quad * 32) << 16);
      const int e = tk.mb * 128 + row;
      const float bias = (MODE == 2 && a.bias && e < E) ? a.bias[e] : 0.f;
      for (int c0 = 0; c0 < tk.nt; c0 += 16) {
        float v[16];
        tc_ld16(taddr + (uint32_t)c0, v);
        if (MODE == 0) {
          const bool gate = (row & 8) == 0;
          const int fi = tk.mb * 64 + 8 * (row >> 4) + (row & 7);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float u = __shfl_xor_sync(0xffffffffu, v[j], 8);
            if (gate && c0 + j < tk.nt) {
              const float gv = v[j];
              p.h16p[(size_t)(poff + c0 + j) * I + fi] = __float2half_rn(gv / (1.0f + expf(-gv)) * u);
            }
          }
        } else if (MODE == 1) {
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (c0 + j < tk.nt) {
              const int zr = ld_cg_i32(&p.pair_z[poff + c0 + j]);
              p.z16[(size_t)zr * H + e] = __float2half_rn(v[j]);
            }
        } else {
          if (e < E) {
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (c0 + j < tk.nt) a.logits[(size_t)(tk.n0 + c0 + j) * E + e] = v[j] + bias;
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
  if (warp == kMmaWarp) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 256;" ::"r"(tmem));
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
  return pf_align(4ull * (E + 1)) + 2 * pf_align(4ull * (E + 2)) + pf_align(4) + 2 * pf_align(4 * P) +
         2 * pf_align(4ull * E * words) + pf_align(6ull * E * H) + pf_align(2ull * Tm * H) + pf_align(2 * P * I) +
         pf_align(2 * P * H);
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
  p.n_chunks = (int32_t*)carve(4);
  p.pair_token = (int32_t*)carve(4 * P);
  p.pair_z = (int32_t*)carve(4 * P);
  p.bitmap = (uint32_t*)carve(4ull * E * words);
  p.prefix = (int32_t*)carve(4ull * E * words);
  p.w_split = (uint16_t*)carve(6ull * E * H);
  p.x16p = (__half*)carve(2ull * Tm * H);
  p.h16p = (__half*)carve(2 * P * I);
  p.z16 = (__half*)carve(2 * P * H);
  p.words = (int)words;
  return p;
}

bool prefill_encode_maps(TensorMapEncodeFn enc, const PrefillArgs& p, int H, int I, int E, int k, int Tm,
                         PrefillMaps* m) {
  const cuuint64_t P = (cuuint64_t)Tm * (k + 1);
  {
    const cuuint64_t dims[3] = {(cuuint64_t)H, (cuuint64_t)E, 3};
    const cuuint64_t strides[2] = {(cuuint64_t)H * 2, (cuuint64_t)E * H * 2};
    const cuuint32_t box[3] = {64, 128, 1};
    if (!encode(enc, &m->w_split, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, p.w_split, dims, strides, box)) return false;
  }
  {
    const cuuint64_t dims[2] = {(cuuint64_t)H, (cuuint64_t)Tm};
    const cuuint64_t strides[1] = {(cuuint64_t)H * 2};
    const cuuint32_t box[2] = {64, 1};
    if (!encode(enc, &m->x16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, p.x16p, dims, strides, box)) return false;
  }
  {
    const cuuint64_t dims[2] = {(cuuint64_t)I, P};
    const cuuint64_t strides[1] = {(cuuint64_t)I * 2};
    const cuuint32_t box[2] = {64, 16};
    if (!encode(enc, &m->h16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, p.h16p, dims, strides, box)) return false;
  }
  return true;
}

bool prefill_encode_x(TensorMapEncodeFn enc, const void* x, int H, int T, PrefillMaps* m) {
  const cuuint64_t dims[2] = {(cuuint64_t)H, (cuuint64_t)T};
  const cuuint64_t strides[1] = {(cuuint64_t)H * 2};
  const cuuint32_t box[2] = {64, 128};
  return encode(enc, &m->x_bf16, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, x, dims, strides, box);
}

cudaError_t prefill_configure() {
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(prefill_gemm_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<0>::kBytes)))
    return e;
  if ((e = cudaFuncSetAttribute(prefill_gemm_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<1>::kBytes)))
    return e;
  return cudaFuncSetAttribute(prefill_gemm_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<2>::kBytes);
}

cudaError_t launch_prefill(const LayerArgs& a, const PrefillArgs& p, const PrefillMaps& m, int sm_count,
                           cudaStream_t s) {
  cudaError_t e;
  if ((e = cudaMemsetAsync(p.counts, 0, sizeof(int32_t) * (size_t)(a.E + 1), s)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(p.bitmap, 0, sizeof(uint32_t) * (size_t)a.E * p.words, s)) != cudaSuccess) return e;
  prefill_prep_kernel<<<sm_count * 4, 256, 0, s>>>(a, p);
  const int router_tasks = ((a.E + 127) / 128) * ((a.T + 127) / 128);
  prefill_gemm_kernel<2><<<router_tasks < sm_count ? router_tasks : sm_count, kGemmThreads, Cfg<2>::kBytes, s>>>(
      a, p, m.w_split, m.x_bf16);
  prefill_topk_kernel<<<(a.T + 7) / 8, 256, 0, s>>>(a, p);
  prefill_prefix_kernel<<<(a.E + 7) / 8, 256, 0, s>>>(a, p);
  prefill_scan_kernel<<<1, 1024, 0, s>>>(a, p);
  prefill_pairs_kernel<<<(a.T * (a.k + 1) + 255) / 256, 256, 0, s>>>(a, p);
  prefill_gemm_kernel<0><<<sm_count, kGemmThreads, Cfg<0>::kBytes, s>>>(a, p, m.x16, m.x16);
  prefill_gemm_kernel<1><<<sm_count, kGemmThreads, Cfg<1>::kBytes, s>>>(a, p, m.h16, m.h16);
  const long long n = (long long)a.T * (a.H / 8);
  prefill_combine_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(a, p);
  return cudaGetLastError();
}

}  // namespace moe
