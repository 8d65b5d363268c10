// Prefill path (T > 64 tokens per call): the same layer as two grouped GEMMs
// on the 5th-generation tensor cores.  Prefill is compute-bound where decode
// is bandwidth-bound (halogen-flash-server README, section "Measured"), and a
// chunk's cost per token keeps falling up to a few thousand tokens (Basalt
// README, section "Prompt chunks").
//
//   router     fp32 SIMT tiled GEMM: logits [T][E]; x -> fp16 rows
//   top-k      warp per token: the k largest logits (ties to the lower
//              index), ascending expert order, softmax over the selection;
//              sets bit t of the expert's token bitmap
//   scan       per-expert counts -> pair offsets and 128-token chunks
//   group      warp per expert: the expert's tokens in ascending order
//              (a stable counting sort) -> (token, z row) pairs
//   gate/up    tcgen05.mma kind::f16, cta_group::1, M = 128 (64 gate rows
//              and the 64 matching up rows), N = the chunk's tokens (<= 128,
//              rounded up to 16), K = H in steps of 64.  Eight producer warps
//              dequantize 4-bit tiles to fp16 d*q and write them with
//              stmatrix in the no-swizzle K-major core-matrix layout; one
//              thread issues the MMAs into a double-buffered TMEM
//              accumulator; four epilogue warps compute h = silu(g) * u.
//   down       the same engine with M = 128 output rows and K = I; the
//              epilogue writes each pair's expert output z as fp16.
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
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
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
__device__ __forceinline__ uint4 ld_nc4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}
__device__ __forceinline__ uint2 ld_nc_u64(const void* p) {
  uint2 r;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
  return r;
}
// Four 8x8 b16 matrices from mma-fragment registers; lane l gives the shared
// address of row (l & 7) of matrix (l >> 3).
__device__ __forceinline__ void stmatrix_x4(uint32_t addr, uint32_t r0, uint32_t r1, uint32_t r2, uint32_t r3) {
  asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(r0), "r"(r1),
               "r"(r2), "r"(r3)
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
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
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

// Shared-memory matrix descriptor, no swizzle, K-major: core matrices of
// 8 rows x 16 bytes, `lbo` bytes apart along K and `sbo` bytes apart along
// M (or N); bit 46 is the descriptor version.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}
// Instruction descriptor of kind::f16: D f32, A and B f16, both K-major, M = 128.
__device__ __forceinline__ uint32_t instr_desc(int n) {
  return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

__device__ void set_error(const LayerArgs& a, int code) {
  atomicCAS(&a.st->error, 0, code);
  volatile int32_t* m = &a.hm->error;
  if (*m == 0) *m = code;
  __threadfence_system();
}

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, const LayerArgs& a, uint64_t deadline,
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

// Byte offset of core-matrix row (r, k-core c) in a [rows][64] fp16 operand tile:
// 8-row groups 1024 B apart, k-cores (8 elements) 128 B apart, rows 16 B apart.
__device__ __forceinline__ uint32_t core_off(int r, int c) {
  return (uint32_t)((r >> 3) * 1024 + c * 128 + (r & 7) * 16);
}

// ------------------------------------------------------------------ router, top-k, grouping

constexpr int kRtTile = 64, kRtK = 32;

// logits[t][e] = sum_h W_r[e][h] x[t][h] + bias[e]; 64 x 64 tile per CTA.
__global__ void __launch_bounds__(256) prefill_router_kernel(LayerArgs a, PrefillArgs p) {
  __shared__ __align__(16) float xs[kRtK][kRtTile + 4];
  __shared__ __align__(16) float ws[kRtK][kRtTile + 4];
  const int tid = threadIdx.x;
  const int t0 = blockIdx.x * kRtTile, e0 = blockIdx.y * kRtTile;
  const int H = a.H, E = a.E, T = a.T;
  const int tr = (tid / 16) * 4, ec = (tid % 16) * 4;
  float acc[4][4] = {};
  int bad = 0;
  for (int k0 = 0; k0 < H; k0 += kRtK) {
    for (int i = tid; i < kRtTile * kRtK; i += 256) {
      const int r = i / kRtK, kk = i % kRtK;
      const int t = t0 + r, e = e0 + r;
      float xv = 0.f;
      if (t < T) {
        const uint16_t bits = a.x[(size_t)t * H + k0 + kk];
        xv = __uint_as_float((uint32_t)bits << 16);
        if (blockIdx.y == 0) {
          bad |= !(fabsf(xv) < 65504.f);
          p.x16p[(size_t)t * H + k0 + kk] = __float2half_rn(xv);
        }
      }
      xs[kk][r] = xv;
      ws[kk][r] = (e < E) ? a.W_r[(size_t)e * H + k0 + kk] : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < kRtK; ++kk) {
      const float4 xv = *reinterpret_cast<const float4*>(&xs[kk][tr]);
      const float4 wv = *reinterpret_cast<const float4*>(&ws[kk][ec]);
      const float xa[4] = {xv.x, xv.y, xv.z, xv.w}, wa[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(xa[i], wa[j], acc[i][j]);
    }
    __syncthreads();
  }
  if (bad) set_error(a, MOE_ERR_DEVICE);
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int t = t0 + tr + i, e = e0 + ec + j;
      if (t < T && e < E) a.logits[(size_t)t * E + e] = acc[i][j] + (a.bias ? a.bias[e] : 0.f);
    }
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
      if (v > bv || (v == bv && e < bi)) { bv = v; bi = e; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
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
    const int words = (a.T + 31) >> 5;
    for (int j = 0; j < k; ++j) {
      a.topk_idx[t * k + j] = sel[j];
      a.topk_w[t * k + j] = expf(selv[j] - m) / z;
      atomicAdd(&p.counts[sel[j]], 1);
      atomicOr(&p.bitmap[(size_t)sel[j] * words + (t >> 5)], 1u << (t & 31));
    }
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

// Warp per expert list entry: its tokens in ascending order (a stable
// counting sort of the (token, rank) pairs by expert).  Pair -> token and z
// row t*(k+1) + rank; the shared expert's rank is k.  Clears the bitmap row.
__global__ void __launch_bounds__(256) prefill_group_kernel(LayerArgs a, PrefillArgs p) {
  const int lane = threadIdx.x & 31;
  const int e = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int E = a.E, k = a.k, T = a.T;
  if (e >= E + a.n_shared) return;
  const int base = p.offsets[e];
  if (e == E) {
    for (int t = lane; t < T; t += 32) {
      p.pair_token[base + t] = t;
      p.pair_z[base + t] = t * (k + 1) + k;
    }
    return;
  }
  const int words = (T + 31) >> 5;
  uint32_t* row = p.bitmap + (size_t)e * words;
  int run = 0;
  for (int w0 = 0; w0 < words; w0 += 32) {
    const int w = w0 + lane;
    const uint32_t bits = (w < words) ? row[w] : 0u;
    if (bits) row[w] = 0u;
    const int c = __popc(bits);
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int pos = base + run + incl - c;
    for (uint32_t b = bits; b; b &= b - 1) {
      const int t = (w << 5) + __ffs(b) - 1;
      int j = 0;
      while (j < k - 1 && a.topk_idx[t * k + j] != e) ++j;
      p.pair_token[pos] = t;
      p.pair_z[pos] = t * (k + 1) + j;
      ++pos;
    }
    run += __shfl_sync(0xffffffffu, incl, 31);
  }
}

// ------------------------------------------------------------------ grouped GEMM on tcgen05

constexpr int kPfStages = 4;
constexpr int kProducers = 8;  // warps 0-7: one 16-row weight strip each
constexpr int kMmaWarp = 8;    // warp 8: allocates TMEM; lane 0 issues the MMAs
constexpr int kEpi0 = 9;       // warps 9-12: epilogue, TMEM lane quadrant warp % 4
constexpr int kPfThreads = (kEpi0 + 4) * 32;
constexpr int kTileBytes = 128 * 64 * 2;  // one fp16 operand tile: 128 rows x 64 k

struct PfSmem {
  unsigned char a[kPfStages][kTileBytes];
  unsigned char b[kPfStages][kTileBytes];
  uint64_t full[kPfStages], empty[kPfStages], acc_full[2], acc_empty[2], drain;
  uint32_t tmem;
};

struct Task {
  int e, n0, nt, mb;
};

// Task t -> expert list entry e, first pair n0 of the chunk within e, its
// tokens nt and the M-block.  M-blocks of one chunk are consecutive tasks,
// so CTAs running them at once share the chunk's activation rows in L2.
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

// MODE 0: gate/up; M-block mb = intermediate rows 64 mb .. 64 mb + 63 of gate
//   and of up, K = H.  Tile row of local gate row i: 16 (i / 8) + i % 8; the
//   matching up row is 8 further, so an epilogue lane pairs with lane + 8.
// MODE 1: down; M-block mb = output rows 128 mb .. 128 mb + 127, K = I.
template <int MODE>
__global__ void __launch_bounds__(kPfThreads, 1) prefill_gemm_kernel(LayerArgs a, PrefillArgs p) {
  extern __shared__ __align__(1024) unsigned char smraw[];
  PfSmem& S = *reinterpret_cast<PfSmem*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = a.H, I = a.I, E = a.E;
  const int NE = E + a.n_shared;
  const int MB = (MODE == 0) ? I / 64 : H / 128;
  const int KS = (MODE == 0) ? H / 64 : I / 64;
  const int n_tasks = ld_cg_i32(&p.n_chunks[0]) * MB;
  const uint64_t deadline = global_ns() + kPipeTimeoutNs;
  bool ok = true;

  if (tid == 0) {
    for (int s = 0; s < kPfStages; ++s) {
      mbar_init(&S.full[s], kProducers);
      mbar_init(&S.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&S.acc_full[b], 1);
      mbar_init(&S.acc_empty[b], 4);
    }
    mbar_init(&S.drain, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 256;" ::"r"(smem_u32(&S.tmem)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem;

  if (warp < kProducers) {
    // ---- producers: warp w dequantizes weight strip w of the A tile; all
    //      eight gather the B tile
    const int gg = lane >> 2;
    const int Kdim = (MODE == 0) ? H : I;
    const int R0 = (MODE == 0) ? 32 * (warp & 3) + 8 * (warp >> 2) : 16 * warp;  // tile row of strip row 0
    const int rstep = (MODE == 0) ? 16 : 8;                                       // tile rows from g to g + 8
    // stmatrix: matrix mi = lane >> 3 is (row g | g + 8) x (k-core 2 kt | 2 kt + 1)
    const int mi = lane >> 3;
    const uint32_t st_off = core_off(R0 + (lane & 7) + ((mi & 1) ? rstep : 0), mi >> 1);
    int g = 0;  // k-steps produced so far
    for (int t = blockIdx.x; t < n_tasks && ok; t += gridDim.x) {
      const Task tk = task_decode(p, NE, MB, t);
      const uint8_t* base = (tk.e < E) ? a.arena + (int64_t)tk.e * a.blob : a.shared;
      const uint8_t* sp;
      if (MODE == 0)
        sp = base + (int64_t)(tk.mb * 4 + (warp & 3)) * gu_strip_bytes(H) + ((warp >> 2) ? 9ll * H : 0);
      else
        sp = base + down_base(H, I) + (int64_t)(tk.mb * 8 + warp) * down_strip_bytes(I);
      const int poff = ld_cg_i32(&p.offsets[tk.e]) + tk.n0;
      const int nt = tk.nt;
      for (int ks = 0; ks < KS; ++ks, ++g) {
        const int s = g % kPfStages, use = g / kPfStages;
        const uint4 nib = ld_nc4(sp + ks * 512 + lane * 16);
        const uint2 sc = ld_nc_u64(sp + 8 * Kdim + ks * 64 + gg * 8);
        if (use > 0 && !wait_bar(&S.empty[s], (use - 1) & 1, a, deadline, ok)) break;
        const uint32_t sa = smem_u32(S.a[s]);
        unsigned char* sb = S.b[s];
        const uint32_t words[4] = {nib.x, nib.y, nib.z, nib.w};
#pragma unroll
        for (int kt = 0; kt < 4; ++kt) {
          const uint32_t scw = (kt < 2) ? sc.x : sc.y;  // k-tiles 0, 1: block 2 ks; 2, 3: block 2 ks + 1
          const __half2 dg = __half2half2(__ushort_as_half((uint16_t)(scw & 0xFFFFu)));
          const __half2 dg8 = __half2half2(__ushort_as_half((uint16_t)(scw >> 16)));
          __half2 q[4];
          dequant_word(words[kt], q);
          stmatrix_x4(sa + st_off + (uint32_t)(kt * 256), h2u(__hmul2(q[0], dg)), h2u(__hmul2(q[1], dg8)),
                      h2u(__hmul2(q[2], dg)), h2u(__hmul2(q[3], dg8)));
        }
        // B: rows n < nt in 16-byte k-cores; lanes 0-7 of a phase take 8 rows of one k-core
        const int nrow8 = (nt + 7) >> 3;
        for (int i = tid; i < nrow8 * 64; i += kProducers * 32) {
          const int n = (i & 7) + 8 * (i >> 6), c = (i >> 3) & 7;
          if (n < nt) {
            const __half* src;
            if (MODE == 0) {
              const int tok = ld_cg_i32(&p.pair_token[poff + n]);
              src = p.x16p + (size_t)tok * H + ks * 64 + c * 8;
            } else {
              src = p.h16p + (size_t)(poff + n) * I + ks * 64 + c * 8;
            }
            *reinterpret_cast<uint4*>(sb + core_off(n, c)) = ld_cg4(src);
          }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.full[s]);
      }
    }
  } else if (warp == kMmaWarp) {
    // ---- MMA issue: one thread, double-buffered accumulator (2 x 128 columns)
    if (lane == 0) {
      int g = 0, i = 0;
      for (int t = blockIdx.x; t < n_tasks && ok; t += gridDim.x, ++i) {
        const Task tk = task_decode(p, NE, MB, t);
        const uint32_t idesc = instr_desc((tk.nt + 15) & ~15);
        const int b = i & 1, ub = i >> 1;
        if (ub > 0 && !wait_bar(&S.acc_empty[b], (ub - 1) & 1, a, deadline, ok)) break;
        tc_fence_after();
        const uint32_t dt = tmem + (uint32_t)(b * 128);
        for (int ks = 0; ks < KS; ++ks, ++g) {
          const int s = g % kPfStages, use = g / kPfStages;
          if (!wait_bar(&S.full[s], use & 1, a, deadline, ok)) break;
          tc_fence_after();
          const uint32_t sa = smem_u32(S.a[s]), sb = smem_u32(S.b[s]);
#pragma unroll
          for (int j = 0; j < 4; ++j)
            tc_mma(dt, smem_desc(sa + j * 256, 128, 1024), smem_desc(sb + j * 256, 128, 1024), idesc,
                   (ks > 0 || j > 0) ? 1u : 0u);
          tc_commit(&S.empty[s]);
        }
        if (!ok) break;
        tc_commit(&S.acc_full[b]);
      }
      // every MMA this thread issued completes before TMEM is released
      tc_commit(&S.drain);
      bool dok = true;
      wait_bar(&S.drain, 0, a, deadline + kPipeTimeoutNs, dok);
    }
    __syncwarp();
  } else {
    // ---- epilogue: TMEM lanes 32 (warp % 4) .. + 31 are tile rows
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    int i = 0;
    for (int t = blockIdx.x; t < n_tasks && ok; t += gridDim.x, ++i) {
      const Task tk = task_decode(p, NE, MB, t);
      const int b = i & 1, ub = i >> 1;
      if (!wait_bar(&S.acc_full[b], ub & 1, a, deadline, ok)) break;
      tc_fence_after();
      const int poff = ld_cg_i32(&p.offsets[tk.e]) + tk.n0;
      const uint32_t taddr = tmem + (uint32_t)(b * 128) + ((uint32_t)(quad * 32) << 16);
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
        } else {
          const int orow = tk.mb * 128 + row;
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (c0 + j < tk.nt) {
              const int zr = ld_cg_i32(&p.pair_z[poff + c0 + j]);
              p.z16[(size_t)zr * H + orow] = __float2half_rn(v[j]);
            }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.acc_empty[b]);
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

constexpr size_t kGemmSmem = sizeof(PfSmem) + 1024;

size_t pf_align(size_t b) { return (b + 255) & ~size_t(255); }

}  // namespace

size_t prefill_scratch_bytes(int H, int I, int E, int k, int Tm) {
  if (Tm <= kMaxTokens) return 0;
  const size_t P = (size_t)Tm * (k + 1), words = (size_t)(Tm + 31) / 32;
  return pf_align(4ull * (E + 1)) + 2 * pf_align(4ull * (E + 2)) + pf_align(4) + 2 * pf_align(4 * P) +
         pf_align(2ull * Tm * H) + pf_align(2 * P * I) + pf_align(2 * P * H) + pf_align(4ull * E * words);
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
  p.x16p = (__half*)carve(2ull * Tm * H);
  p.h16p = (__half*)carve(2 * P * I);
  p.z16 = (__half*)carve(2 * P * H);
  p.bitmap = (uint32_t*)carve(4ull * E * words);
  return p;
}

cudaError_t prefill_configure() {
  cudaError_t e =
      cudaFuncSetAttribute(prefill_gemm_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGemmSmem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(prefill_gemm_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGemmSmem);
}

cudaError_t launch_prefill(const LayerArgs& a, const PrefillArgs& p, int sm_count, cudaStream_t s) {
  cudaError_t e;
  if ((e = cudaMemsetAsync(p.counts, 0, sizeof(int32_t) * (size_t)(a.E + 1), s)) != cudaSuccess) return e;
  prefill_router_kernel<<<dim3((a.T + kRtTile - 1) / kRtTile, (a.E + kRtTile - 1) / kRtTile), 256, 0, s>>>(a, p);
  prefill_topk_kernel<<<(a.T + 7) / 8, 256, 0, s>>>(a, p);
  prefill_scan_kernel<<<1, 1024, 0, s>>>(a, p);
  prefill_group_kernel<<<(a.E + a.n_shared + 7) / 8, 256, 0, s>>>(a, p);
  prefill_gemm_kernel<0><<<sm_count, kPfThreads, kGemmSmem, s>>>(a, p);
  prefill_gemm_kernel<1><<<sm_count, kPfThreads, kGemmSmem, s>>>(a, p);
  const long long n = (long long)a.T * (a.H / 8);
  prefill_combine_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(a, p);
  return cudaGetLastError();
}

}  // namespace moe
