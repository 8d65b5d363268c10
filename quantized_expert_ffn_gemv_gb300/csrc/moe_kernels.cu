// Batched decode kernels of the quantized MoE FFN layer (sm_103a), for
// calls the fused decode kernel does not take (9..64 tokens, or shapes it
// declines), plus the separate residual + RMSNorm kernel.
//
// One moe_forward = four stream-ordered kernels chained with programmatic
// dependent launch (griddepcontrol), so each grid is already resident when
// its predecessor finishes:
//   route_kernel   router GEMV in plain fp32 (four warps per expert row,
//                  blocks of 16 tokens) and the router rows' norms;
//   route_select_kernel  CTA per token: the k best experts, exact (the
//                  experts the fp32 error bound leaves in doubt are
//                  recomputed with the canonical compensated router of
//                  moe_route.cuh), softmax weights from the exact keys; the
//                  last-arriving CTA groups the (token, expert) pairs.
//   gateup_kernel  per (expert, 16-row strip): 4-bit gate and up rows
//                  dequantized in registers into mma.m16n8k16 fragments,
//                  fp32 accumulation with exact per-block scaling, then
//                  h = silu(g) * u stored as fp16.
//   down_kernel    CTA per 16-row output strip: every selected expert's down
//                  rows (warps over (expert, 8-token group) items), then the
//                  routing-weighted combine in ascending expert order (shared
//                  expert last) and one bf16 rounding.
// These kernels serve layers whose experts are all resident (slot = expert);
// a layer with a slot pool runs the fused decode kernel, which holds the
// hit check (Betelgeuse news page, section 机制: 调度 and 显存 rows).
#include <cfloat>
#include <climits>

#include "moe.h"
#include "moe_internal.h"
#include "moe_mma.cuh"
#include "moe_norm.cuh"
#include "moe_route.cuh"

namespace moe {
namespace {

// ------------------------------------------------------------------ PTX helpers

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ int ld_cg_i32(const int* p) {
  int r;
  asm volatile("ld.global.cg.s32 %0, [%1];" : "=r"(r) : "l"(p));
  return r;
}

__device__ void set_error(const LayerArgs& a, int code) {
  atomicCAS(&a.st->error, 0, code);
  volatile int32_t* m = &a.hm->error;
  if (*m == 0) *m = code;
  __threadfence_system();
}

__device__ __forceinline__ int dev_error(const LayerArgs& a) { return ld_cg_i32(&a.st->error); }

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

// ------------------------------------------------------------------ route

constexpr int kRouteRows = 2;        // expert rows per CTA (four warps per row, one per quarter of H)
constexpr int kRouteThreads = 256;
constexpr int kSelThreads = 512;     // route_select_kernel: 16 warps, about one candidate each
constexpr int kRouteTok = 4;         // tokens whose x loads are in flight together
constexpr int kRouteTokBlock = 16;   // tokens per route_kernel block
constexpr int kRouteVec = kMaxHidden / 512;  // float4 per lane per quarter row

struct FinishSmem {
  size_t lrow, tokmask, uidx, poff, sidx, sw, misc, total;
};

__host__ __device__ inline size_t align16(size_t v) { return (v + 15) & ~size_t(15); }

// route_select_kernel's own layout (its last CTA reuses the memory for route_finish)
struct SelectSmem {
  size_t cand, words, sel, total;
};

__host__ __device__ inline SelectSmem select_layout(int E) {
  SelectSmem l;
  l.cand = 0;
  l.words = align16(sizeof(int) * (size_t)E);
  l.sel = l.words + sizeof(unsigned long long) * (size_t)E;
  l.total = l.sel + sizeof(int) * 2 * kMaxTopK;
  return l;
}

__host__ __device__ inline FinishSmem finish_layout(int E) {
  FinishSmem f;
  f.lrow = 0;
  f.tokmask = 0;
  f.uidx = f.tokmask + align16(sizeof(unsigned long long) * (size_t)E);
  f.poff = f.uidx + align16(sizeof(int) * (size_t)E);
  f.sidx = f.poff + align16(sizeof(int) * (size_t)E);
  f.sw = f.sidx + align16(sizeof(int) * kMaxTokens * kMaxTopK);
  f.misc = f.sw + align16(sizeof(float) * kMaxTokens * kMaxTopK);
  f.total = f.misc + sizeof(unsigned long long) * 64;
  return f;
}

// Block-wide exclusive scan of (a, b) pairs, kSelThreads threads; returns totals.
__device__ void block_scan2(int& a, int& b, int& tot_a, int& tot_b, int* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int ia = a, ib = b;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int va = __shfl_up_sync(0xffffffffu, ia, o), vb = __shfl_up_sync(0xffffffffu, ib, o);
    if (lane >= o) { ia += va; ib += vb; }
  }
  constexpr int nw = kSelThreads / 32;
  if (lane == 31) { scratch[warp] = ia; scratch[nw + warp] = ib; }
  __syncthreads();
  int wa = 0, wb = 0, ta = 0, tb = 0;
  for (int w = 0; w < nw; ++w) {
    if (w < warp) { wa += scratch[w]; wb += scratch[nw + w]; }
    ta += scratch[w];
    tb += scratch[nw + w];
  }
  a = wa + ia - a;
  b = wb + ib - b;
  tot_a = ta;
  tot_b = tb;
  __syncthreads();
}

// The last CTA of route_select_kernel: the step counter, the union of the
// selected experts and the (token, expert) pairs grouped by expert.
__device__ void route_finish(const LayerArgs& a, unsigned char* smem) {
  const int tid = threadIdx.x;
  const int E = a.E, k = a.k, T = a.T;
  const FinishSmem f = finish_layout(E);
  unsigned long long* tokmask = reinterpret_cast<unsigned long long*>(smem + f.tokmask);
  int* uidx = reinterpret_cast<int*>(smem + f.uidx);
  int* poff = reinterpret_cast<int*>(smem + f.poff);
  int* sidx = reinterpret_cast<int*>(smem + f.sidx);
  float* sw = reinterpret_cast<float*>(smem + f.sw);
  unsigned long long* misc = reinterpret_cast<unsigned long long*>(smem + f.misc);
  __shared__ uint32_t s_seq;
  __shared__ int s_nunion;

  if (tid == 0) {
    a.st->ticket = 0;
    s_seq = a.st->step + 1;
    a.st->step = s_seq;
  }
  for (int e = tid; e < E; e += kSelThreads) tokmask[e] = 0ull;
  __syncthreads();
  const uint32_t seq = s_seq;
  // keep the fused decode path's gate/up counters of the next step at zero
  for (int i = tid; i < a.cnt_stride / kCntPad; i += kSelThreads)
    a.counters[(size_t)((seq + 1u) & 1u) * a.cnt_stride + (size_t)i * kCntPad] = 0u;

  // ---- the tokens' selections (route_select_kernel), ascending expert index
  for (int p = tid; p < T * k; p += kSelThreads) {
    const int e = __ldcg(a.topk_idx + p);
    sidx[p] = e;
    sw[p] = __ldcg(a.topk_w + p);
    atomicOr(&tokmask[e], 1ull << (p / k));
  }
  __syncthreads();

  // ---- union of selected experts (ascending) and pair offsets
  const int per = (E + kSelThreads - 1) / kSelThreads;
  const int e0 = tid * per;
  int fl = 0, cn = 0;
  for (int e = e0; e < e0 + per && e < E; ++e) {
    int c = __popcll(tokmask[e]);
    fl += c > 0;
    cn += c;
  }
  int tot_f, tot_c;
  block_scan2(fl, cn, tot_f, tot_c, reinterpret_cast<int*>(misc));
  for (int e = e0; e < e0 + per && e < E; ++e) {
    int c = __popcll(tokmask[e]);
    uidx[e] = fl;
    poff[e] = cn;
    if (c > 0) {
      a.u_expert[fl] = e;
      a.u_off[fl] = cn;
      ++fl;
      cn += c;
    }
  }
  if (tid == 0) {
    a.u_off[tot_f] = tot_c;
    s_nunion = tot_f;
  }
  __syncthreads();
  const int n_union = s_nunion;

  // ---- pairs sorted by (expert, token)
  for (int p = tid; p < T * k; p += kSelThreads) {
    const int t = p / k;
    const int e = sidx[p];
    const int pos = __popcll(tokmask[e] & ((1ull << t) - 1ull));
    const int dst = poff[e] + pos;
    a.pair_token[dst] = t;
    a.pair_w[dst] = sw[p];
    a.tk_u[p] = uidx[e];
    a.tk_pos[p] = pos;
  }

  // ---- every expert resident: slot = expert (pooled layers run the fused path)
  for (int u = tid; u < n_union; u += kSelThreads) a.u_slot[u] = a.u_expert[u];
  if (tid == 0) {
    a.st->n_union = n_union;
    a.st->n_miss = 0;
    a.st->forwards += 1ull;
    a.st->hits += (unsigned long long)n_union;
  }
  __threadfence();
}

__global__ void __launch_bounds__(kRouteThreads) route_kernel(LayerArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = a.H, E = a.E, T = a.T;
  // block = (row pair, block of kRouteTokBlock tokens): more blocks, fewer
  // dependent L2 round trips for x per warp
  const int nrb = (E + kRouteRows - 1) / kRouteRows;
  const int rb = blockIdx.x % nrb, tb = blockIdx.x / nrb;
  const int t_lo = tb * kRouteTokBlock, t_hi = min(T, t_lo + kRouteTokBlock);
  const int row = rb * kRouteRows + (warp >> 2);
  const int q = warp & 3;
  const int n4 = H / 16;  // float4 groups per quarter row
  const bool row_ok = row < E;

  // Router rows do not depend on the previous kernel: load them first.
  float4 w[kRouteVec];
  const float4* wq = reinterpret_cast<const float4*>(a.W_r + (size_t)(row_ok ? row : 0) * H + q * (H / 4));
#pragma unroll
  for (int i = 0; i < kRouteVec; ++i) {
    const int j = lane + 32 * i;
    w[i] = (row_ok && j < n4) ? __ldg(wq + j) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  pdl_wait();

  // x (bf16) -> x16: fp16 in B-fragment order, for the expert kernels
  {
    const int oct = T * H / 8;
    int bad = 0;
    for (int o = blockIdx.x * kRouteThreads + tid; o < oct; o += gridDim.x * kRouteThreads) {
      const int t = o / (H / 8), k8 = (o % (H / 8)) * 8;
      const uint4 v = *reinterpret_cast<const uint4*>(a.x + (size_t)t * H + k8);
      const uint32_t vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float f0 = __uint_as_float(vv[i] << 16), f1 = __uint_as_float(vv[i] & 0xFFFF0000u);
        bad |= !(fabsf(f0) < 65504.f) | !(fabsf(f1) < 65504.f);
        const __half2 h = __floats2half2_rn(f0, f1);
        *reinterpret_cast<__half2*>(a.x16 + (size_t)t * H + frag_pos(k8 + 2 * i)) = h;
      }
    }
    if (bad) set_error(a, MOE_ERR_DEVICE);
  }

  float* red = reinterpret_cast<float*>(smem);  // [warps][T] quarter partials
  // the row's Euclidean norm (for the select kernel's error bound)
  {
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < kRouteVec; ++i)
      ss = fmaf(w[i].x, w[i].x, fmaf(w[i].y, w[i].y, fmaf(w[i].z, w[i].z, fmaf(w[i].w, w[i].w, ss))));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) red[warp] = ss;
    __syncthreads();
    if (tb == 0 && tid < kRouteRows && rb * kRouteRows + tid < E) {
      const float* r4 = red + 4 * tid;
      a.wnorm[rb * kRouteRows + tid] = sqrtf(((r4[0] + r4[1]) + r4[2]) + r4[3]) * 1.001f;
    }
    __syncthreads();
  }
  // Plain fp32 partials, the quarter row held in registers and x read from
  // L2 four tokens at a time (every load of the four issued before the
  // arithmetic).  At most kRouteVec*4 + 5 + 3 roundings per logit; the
  // select kernel recomputes, exactly, every expert this bound leaves in doubt.
  const uint2* xq = reinterpret_cast<const uint2*>(a.x + q * (H / 4));
  for (int t0 = t_lo; t0 < t_hi; t0 += kRouteTok) {
    uint2 xv[kRouteTok][kRouteVec];
#pragma unroll
    for (int u = 0; u < kRouteTok; ++u)
#pragma unroll
      for (int i = 0; i < kRouteVec; ++i) {
        const int j = lane + 32 * i;
        xv[u][i] = (t0 + u < t_hi && j < n4) ? __ldcg(xq + (size_t)(t0 + u) * (H / 4) + j) : make_uint2(0u, 0u);
      }
    float d[kRouteTok];
#pragma unroll
    for (int u = 0; u < kRouteTok; ++u) {
      d[u] = 0.f;
#pragma unroll
      for (int i = 0; i < kRouteVec; ++i) {
        const uint2 v = xv[u][i];
        d[u] = fmaf(w[i].x, bf_lo(v.x), fmaf(w[i].y, bf_hi(v.x), fmaf(w[i].z, bf_lo(v.y), fmaf(w[i].w, bf_hi(v.y), d[u]))));
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
      for (int u = 0; u < kRouteTok; ++u) d[u] += __shfl_xor_sync(0xffffffffu, d[u], o);
    if (lane == 0) {
#pragma unroll
      for (int u = 0; u < kRouteTok; ++u)
        if (t0 + u < t_hi) red[warp * kMaxTokens + t0 + u] = d[u];
    }
  }
  __syncthreads();
  const int nt = t_hi - t_lo;
  for (int i = tid; i < kRouteRows * nt; i += kRouteThreads) {
    const int r = i / nt, t = t_lo + i % nt;
    const int e = rb * kRouteRows + r;
    if (e < E) {
      const float* pr = red + (4 * r) * kMaxTokens + t;
      a.logits[(size_t)t * E + e] =
          (((pr[0] + pr[kMaxTokens]) + pr[2 * kMaxTokens]) + pr[3 * kMaxTokens]) + (a.bias ? __ldg(a.bias + e) : 0.f);
    }
  }
  pdl_trigger();
}

// The canonical compensated router's rank word of expert e for one token,
// computed by one warp: the four quarter partials in lane-strided float4
// groups, each reduced by the xor butterfly, then summed with the bias
// (the fused decode kernel's arithmetic, so its keys bit for bit).  The
// next quarter's loads are issued before the current quarter's arithmetic.
__device__ __forceinline__ uint64_t exact_rank_word(const float* W_r, const float* bias, const uint16_t* x, int H,
                                                    int e, int lane) {
  const int n4 = H / 16;
  const float4* wr = reinterpret_cast<const float4*>(W_r + (size_t)e * H);
  const uint2* xr = reinterpret_cast<const uint2*>(x);
  float4 wv[2][kRouteVec];
  uint2 xv[2][kRouteVec];
  auto load = [&](int q, int b) {
#pragma unroll
    for (int i = 0; i < kRouteVec; ++i) {
      const int j = lane + 32 * i;
      if (j < n4) {
        wv[b][i] = __ldg(wr + q * n4 + j);
        xv[b][i] = __ldcg(xr + q * n4 + j);
      }
    }
  };
  DF q4[4];
  load(0, 0);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    if (q < 3) load(q + 1, (q + 1) & 1);
    DF d{0.f, 0.f};
#pragma unroll
    for (int i = 0; i < kRouteVec; ++i) {
      const int j = lane + 32 * i;
      if (j < n4) {
        const uint2 v = xv[q & 1][i];
        dot2_acc4(d, wv[q & 1][i], make_float4(bf_lo(v.x), bf_hi(v.x), bf_lo(v.y), bf_hi(v.y)));
      }
    }
    q4[q] = warp_sum_df(d);
  }
  return rank_word(logit_key(q4[0], q4[1], q4[2], q4[3], bias ? __ldg(bias + e) : 0.f), e);
}

// CTA per token: the k selected experts from the fp32 logits, made exact.
// An fp32 logit here is within delta_t = 4e-6 (max_e |W_r[e]| |x_t| + max|b|)
// of its exact value (at most 41 roundings of partial sums bounded by
// sum |w x| + |b|).  Every expert whose fp32 logit is not below the
// (k+1)-th largest minus 2 delta_t is a candidate; the others provably rank
// below k experts.  The CTA's warps recompute the candidates with the
// canonical compensated router (exact_rank_word), which gives the fused
// decode kernel's keys bit for bit; the k best exact keys are the selection
// and their weights come from those keys, so a batched token is routed
// exactly as it would be alone.  The last CTA then groups the pairs.
template <int CPL>
__global__ void __launch_bounds__(kSelThreads) route_select_kernel(LayerArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = a.E, k = a.k, H = a.H;
  const int t = blockIdx.x;
  const SelectSmem L = select_layout(E);
  int* cand = reinterpret_cast<int*>(smem + L.cand);
  unsigned long long* words = reinterpret_cast<unsigned long long*>(smem + L.words);
  int* sel = reinterpret_cast<int*>(smem + L.sel);
  float* selv = reinterpret_cast<float*>(sel + kMaxTopK);
  __shared__ unsigned int s_wmax, s_bmax;
  __shared__ float s_kth, s_xs;
  __shared__ int s_ncand;
  if (tid == 0) { s_wmax = 0u; s_bmax = 0u; s_ncand = 0; s_kth = -INFINITY; }
  const uint16_t* xt = a.x + (size_t)t * H;
  pdl_wait();
  __syncthreads();
  {
    unsigned int wm = 0u, bm = 0u;
    for (int e = tid; e < E; e += kSelThreads) {
      wm = max(wm, __float_as_uint(__ldcg(a.wnorm + e)));
      if (a.bias) bm = max(bm, __float_as_uint(fabsf(__ldg(a.bias + e))));
    }
    atomicMax(&s_wmax, wm);
    atomicMax(&s_bmax, bm);
  }
  const float* lt = a.logits + (size_t)t * E;
  if (warp == 0 && k < E) {
    // the (k+1)-th largest fp32 logit (k + 1 rounds of a warp maximum)
    constexpr int kRegs = CPL > 0 ? CPL : 1;
    float lv[kRegs];
#pragma unroll
    for (int i = 0; i < kRegs; ++i) lv[i] = (CPL > 0 && lane + 32 * i < E) ? __ldcg(lt + lane + 32 * i) : -FLT_MAX;
    uint32_t taken[kMaxExperts / 1024] = {};
    float thr = -INFINITY;
    for (int r = 0; r <= k; ++r) {
      float bv = -FLT_MAX;
      int bi = INT_MAX;
      if (CPL > 0) {
#pragma unroll
        for (int i = 0; i < kRegs; ++i) {
          const int e = lane + 32 * i;
          if (e < E && !((taken[0] >> i) & 1u) && (lv[i] > bv || (lv[i] == bv && e < bi))) { bv = lv[i]; bi = e; }
        }
      } else {
        for (int e = lane, i = 0; e < E; e += 32, ++i) {
          if ((taken[i >> 5] >> (i & 31)) & 1u) continue;
          const float v = __ldcg(lt + e);
          if (v > bv || (v == bv && e < bi)) { bv = v; bi = e; }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
      }
      // none left above -FLT_MAX (the rest -inf or NaN): every logit is a candidate
      if (bi == INT_MAX) { thr = -INFINITY; break; }
      if (lane == (bi & 31)) {
        if (CPL > 0) taken[0] |= 1u << ((bi >> 5) & 31);
        else taken[(bi >> 5) >> 5] |= 1u << ((bi >> 5) & 31);
      }
      thr = bv;
    }
    if (lane == 0) s_kth = thr;
  } else if (warp == 1) {
    float xs = 0.f;
    const uint32_t* xw = reinterpret_cast<const uint32_t*>(xt);
    for (int i = lane; i < H / 2; i += 32) {
      const uint32_t v = __ldcg(xw + i);
      xs = fmaf(bf_lo(v), bf_lo(v), fmaf(bf_hi(v), bf_hi(v), xs));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) xs += __shfl_xor_sync(0xffffffffu, xs, o);
    if (lane == 0) s_xs = xs;
  }
  __syncthreads();
  {
    const float delta = 4e-6f * (__uint_as_float(s_wmax) * sqrtf(s_xs) * 1.001f + __uint_as_float(s_bmax)) + 1e-30f;
    const float thr = s_kth - 2.f * delta;  // -inf: every expert (k = E, or too few finite logits)
    // NaN logits are candidates too (their exact keys rank them last)
    for (int e = tid; e < E; e += kSelThreads) {
      const float v = __ldcg(lt + e);
      if (!(v < thr)) cand[atomicAdd(&s_ncand, 1)] = e;
    }
  }
  __syncthreads();
  const int n = s_ncand;
  for (int c = warp; c < n; c += kSelThreads / 32) {
    const uint64_t w = exact_rank_word(a.W_r, a.bias, xt, H, cand[c], lane);
    if (lane == 0) words[c] = w;
  }
  __syncthreads();
  if (warp == 0) {
    // the k best exact words (all nonzero and distinct; n >= k)
    for (int r = 0; r < k; ++r) {
      uint64_t best = 0ull;
      int bpos = -1;
      for (int c = lane; c < n; c += 32) {
        const uint64_t v = words[c];
        if (v > best) { best = v; bpos = c; }
      }
      const uint64_t m = warp_max_u64(best);
      if (best == m && bpos >= 0) words[bpos] = 0ull;
      if (lane == 0) {
        sel[r] = word_expert(m);
        selv[r] = key_value(word_key(m));
      }
      __syncwarp();
    }
    if (lane == 0) softmax_ascending(sel, selv, k, a.topk_idx + t * k, a.topk_w + t * k);
  }
  __threadfence();
  __syncthreads();
  __shared__ uint32_t s_ticket;
  if (tid == 0) s_ticket = atomicAdd(&a.st->ticket, 1u);
  __syncthreads();
  if (s_ticket != gridDim.x - 1) return;
  __threadfence();
  pdl_trigger();
  route_finish(a, smem);
}

// ------------------------------------------------------------------ gate/up

constexpr int kGuThreads = 128;  // 4 warps split the K = H reduction of a strip, as in the fused path
constexpr int kGuWarpsPerTask = kGuThreads / 32;

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
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
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Batched gate/up: one (expert, 16-row strip) task per iteration; the strip
// (gate and up rows, all of K) arrives in shared memory with one bulk copy.
// One stage per block keeps the block small, so four blocks share an SM and
// one block's copy flies while the others multiply.  The task's tokens are
// taken two 8-token groups (two mma N tiles) per pass over the strip; the
// activation fragments of a warp's next super-tile are loaded from L2 while
// the current one is multiplied.  The four warps split K as the fused decode
// kernel does (super-tiles st = warp, warp + 4, ...; partial sums added in
// warp order), so a token's h does not depend on its batch.
struct GuTask {
  const uint8_t* strip;
  int cnt, poff, sh;
};
__device__ __forceinline__ GuTask gu_task(const LayerArgs& a, int task, int NS) {
  const int gu = task / NS, s = task % NS;
  GuTask r;
  r.sh = gu < a.n_shared;
  const uint8_t* base;
  if (r.sh) {
    base = a.shared;
    r.cnt = a.T;
    r.poff = a.T * a.k;
  } else {
    const int u = gu - a.n_shared;
    base = a.arena + (int64_t)__ldcg(a.u_slot + u) * a.blob;
    r.poff = __ldcg(a.u_off + u);
    r.cnt = __ldcg(a.u_off + u + 1) - r.poff;
  }
  r.strip = base + (int64_t)s * gu_strip_bytes(a.H);
  return r;
}

__device__ __forceinline__ bool mbar_wait_bounded(const LayerArgs& a, uint64_t* bar, uint32_t parity,
                                                  uint64_t deadline) {
  int spins = 0;
  while (!mbar_try_wait(bar, parity)) {
    if (((++spins) & 63) == 0 && global_ns() > deadline) {
      set_error(a, MOE_ERR_TIMEOUT);
      return false;
    }
  }
  return true;
}

constexpr int kGuGroups = 2;  // 8-token groups per pass over a strip

__global__ void __launch_bounds__(kGuThreads, 4) gateup_kernel(LayerArgs a) {
  extern __shared__ __align__(128) unsigned char gsm[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int H = a.H, I = a.I;
  const int NS = I / 16, nst = H / 64;
  const uint32_t sbytes = (uint32_t)gu_strip_bytes(H);
  const size_t pitch = (sbytes + 127) & ~127u;
  unsigned char* stage = gsm;
  float* red = reinterpret_cast<float*>(gsm + pitch);  // [4 warps][kGuGroups][32 lanes][8]
  __shared__ __align__(8) uint64_t full;
  if (tid == 0) {
    mbar_init(&full, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  const int n_union = ld_cg_i32(&a.st->n_union);
  const int n_tasks = (a.n_shared + n_union) * NS;
  if (dev_error(a)) return;
  const uint64_t deadline = global_ns() + 2000000000ull;
  int it = 0;
  for (int task = blockIdx.x; task < n_tasks; task += gridDim.x, ++it) {
    // the stage was released by the barrier that ended the last task
    if (tid == 0) {
      mbar_expect_tx(&full, sbytes);
      bulk_g2s(stage, gu_task(a, task, NS).strip, sbytes, &full);
    }
    const GuTask tk = gu_task(a, task, NS);
    const int s = task % NS;
    const int ng = (tk.cnt + 7) >> 3;
    int tok[kGuGroups];
    const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(a, &full, it & 1, deadline));
    if (ng == 0) __syncthreads();  // (no pass below) release the stage all the same
    for (int qb = 0; qb < ng; qb += kGuGroups) {
#pragma unroll
      for (int q = 0; q < kGuGroups; ++q) {
        const int i = (qb + q) * 8 + g;
        tok[q] = (i < tk.cnt) ? (tk.sh ? i : __ldcg(a.pair_token + tk.poff + i)) : 0;
      }
      const int nq = min(kGuGroups, ng - qb);
      float accg[kGuGroups][4], accu[kGuGroups][4];
#pragma unroll
      for (int q = 0; q < kGuGroups; ++q)
#pragma unroll
        for (int c = 0; c < 4; ++c) accg[q][c] = accu[q][c] = 0.f;
      if (ok) {
        uint4 bx[kGuGroups][2];
        auto load_x = [&](int st) {
#pragma unroll
          for (int q = 0; q < kGuGroups; ++q)
            if (q < nq && st < nst) {
              const uint4* xr = reinterpret_cast<const uint4*>(a.x16 + (size_t)tok[q] * H + st * 64 + t4 * 16);
              bx[q][0] = __ldcg(xr);
              bx[q][1] = __ldcg(xr + 1);
            }
        };
        load_x(warp);
        for (int st = warp; st < nst; st += kGuWarpsPerTask) {
          uint4 cx[kGuGroups][2];
#pragma unroll
          for (int q = 0; q < kGuGroups; ++q) { cx[q][0] = bx[q][0]; cx[q][1] = bx[q][1]; }
          load_x(st + kGuWarpsPerTask);
          const SupertileA ag = dequant_supertile(*reinterpret_cast<const uint4*>(stage + st * 512 + lane * 16),
                                                  *reinterpret_cast<const uint2*>(stage + 8 * H + st * 64 + g * 8));
          const SupertileA au = dequant_supertile(*reinterpret_cast<const uint4*>(stage + 9 * H + st * 512 + lane * 16),
                                                  *reinterpret_cast<const uint2*>(stage + 17 * H + st * 64 + g * 8));
#pragma unroll
          for (int q = 0; q < kGuGroups; ++q)
            if (q < nq) {
              supertile_mma_pre(accg[q], ag, cx[q][0], cx[q][1]);
              supertile_mma_pre(accu[q], au, cx[q][0], cx[q][1]);
            }
        }
      }
#pragma unroll
      for (int q = 0; q < kGuGroups; ++q) {
        float4* dst = reinterpret_cast<float4*>(red + (((warp * kGuGroups) + q) * 32 + lane) * 8);
        dst[0] = make_float4(accg[q][0], accg[q][1], accg[q][2], accg[q][3]);
        dst[1] = make_float4(accu[q][0], accu[q][1], accu[q][2], accu[q][3]);
      }
      __syncthreads();
      // warp q reduces group q over the four warps, in warp order
      if (warp < nq) {
        const int q = warp;
        float gs[4] = {0.f, 0.f, 0.f, 0.f}, us[4] = {0.f, 0.f, 0.f, 0.f};
        for (int w = 0; w < kGuWarpsPerTask; ++w) {
          const float4* src = reinterpret_cast<const float4*>(red + (((w * kGuGroups) + q) * 32 + lane) * 8);
          const float4 p = src[0], r = src[1];
          gs[0] += p.x; gs[1] += p.y; gs[2] += p.z; gs[3] += p.w;
          us[0] += r.x; us[1] += r.y; us[2] += r.z; us[3] += r.w;
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int rowin = (c < 2) ? g : g + 8;
          const int i = (qb + q) * 8 + 2 * t4 + (c & 1);
          if (i < tk.cnt)
            a.h16[(size_t)(tk.poff + i) * I + frag_pos(s * 16 + rowin)] = __float2half_rn(silu(gs[c]) * us[c]);
        }
      }
      __syncthreads();  // red (and, after the last pass, the stage) is free again
    }
  }
}

// ------------------------------------------------------------------ down + combine

// Batched down with the combine folded in: CTA r owns the 16-row output
// strip r.  The work items are (expert entry, 8-token group) pairs, numbered
// expert by expert, and warp w takes items w, w + nw, ...: a hot expert's
// groups land on different warps.  Each item's expert strip (16 rows, all of
// K = I) is streamed into the warp's own two-stage ring by a bulk copy (the
// next item's copy issued before this one's products), and the h rows of
// its tokens are read from L2 with every load of the item in flight
// together.  Each pair's 16 outputs land in shared memory as fp32; after a
// block barrier every (token, row) is combined as
// y = sum_j w_j z_j (ascending expert) + z_shared, the fused decode kernel's
// fma chain, and rounded once to bf16.
constexpr int kDnThreads = 512;
constexpr int kDnMaxWarps = kDnThreads / 32;
constexpr int kDnChunk = 8;  // super-tiles whose h fragments are loaded together
constexpr int kDnMaxEntries = kMaxTokens * kMaxTopK + 2;

__host__ __device__ inline size_t down_z_bytes(int T, int k, int n_shared) {
  return align16(sizeof(float) * 16 * ((size_t)T * k + (size_t)n_shared * T));
}
__host__ __device__ inline size_t down_stage_pitch(int I) { return ((size_t)down_strip_bytes(I) + 127) & ~size_t(127); }

__global__ void __launch_bounds__(kDnThreads, 1) down_kernel(LayerArgs a, int nw) {
  extern __shared__ __align__(128) unsigned char dsm[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int H = a.H, I = a.I, T = a.T, k = a.k;
  const int r = blockIdx.x;
  float* zb = reinterpret_cast<float*>(dsm);  // [pair][16 rows]
  const size_t pitch = down_stage_pitch(I);
  const uint32_t sbytes = (uint32_t)down_strip_bytes(I);
  unsigned char* ring = dsm + down_z_bytes(T, k, a.n_shared) + (size_t)warp * 2 * pitch;
  __shared__ __align__(8) uint64_t bar[kDnMaxWarps][2];
  __shared__ int s_item[kDnMaxEntries + 1];  // first item of each expert entry; [n_ex] = total
  if (warp < nw && lane == 0) {
    mbar_init(&bar[warp][0], 1);
    mbar_init(&bar[warp][1], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  pdl_wait();
  pdl_trigger();
  const int n_union = ld_cg_i32(&a.st->n_union);
  const int n_ex = n_union + a.n_shared;
  const int nst = I / 64;
  if (dev_error(a)) return;
  if (warp == 0) {  // items per entry (its 8-token groups), scanned
    int carry = 0;
    for (int b0 = 0; b0 < n_ex; b0 += 32) {
      const int xi = b0 + lane;
      int v = 0;
      if (xi < n_ex) {
        const int cnt = xi >= n_union ? T : __ldcg(a.u_off + xi + 1) - __ldcg(a.u_off + xi);
        v = (cnt + 7) >> 3;
      }
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
      }
      if (xi < n_ex) s_item[xi] = carry + incl - v;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) s_item[n_ex] = carry;
  }
  __syncthreads();
  const int n_items = s_item[n_ex];
  const uint64_t deadline = global_ns() + 2000000000ull;
  auto entry_of = [&](int i) {  // the entry whose items include i
    int lo = 0, hi = n_ex - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_item[mid] <= i) lo = mid; else hi = mid - 1;
    }
    return lo;
  };
  auto strip_of = [&](int xi) -> const uint8_t* {
    const uint8_t* base = xi >= n_union ? a.shared : a.arena + (int64_t)__ldcg(a.u_slot + xi) * a.blob;
    return base + down_base(H, I) + (int64_t)r * sbytes;
  };
  if (warp < nw) {
    int pending[2] = {0, 0};  // per stage: 1 + the parity of a copy not yet waited for, else 0
    if (lane == 0 && warp < n_items) {
      mbar_expect_tx(&bar[warp][0], sbytes);
      bulk_g2s(ring, strip_of(entry_of(warp)), sbytes, &bar[warp][0]);
      pending[0] = 1;
    }
    int it = 0;
    for (int i = warp; i < n_items; i += nw, ++it) {
      const int sb = it & 1;
      // stage sb ^ 1 held the previous item, whose products this warp finished
      if (lane == 0 && i + nw < n_items) {
        mbar_expect_tx(&bar[warp][sb ^ 1], sbytes);
        bulk_g2s(ring + (sb ^ 1) * pitch, strip_of(entry_of(i + nw)), sbytes, &bar[warp][sb ^ 1]);
        pending[sb ^ 1] = 1 + (((it + 1) >> 1) & 1);
      }
      const int xi = entry_of(i), q = i - s_item[xi];
      const bool sh = xi >= n_union;
      const int poff = sh ? T * k : __ldcg(a.u_off + xi);
      const int cnt = sh ? T : __ldcg(a.u_off + xi + 1) - poff;
      const int col0 = 8 * q;
      const int ti = col0 + g;
      const __half* hrow = a.h16 + (size_t)(poff + (ti < cnt ? ti : 0)) * I + t4 * 16;
      bool ok = true;
      if (lane == 0) {
        ok = mbar_wait_bounded(a, &bar[warp][sb], (it >> 1) & 1, deadline);
        if (ok) pending[sb] = 0;
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      const unsigned char* sp = ring + sb * pitch;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      for (int st0 = 0; st0 < nst && ok; st0 += kDnChunk) {
        uint4 bh[kDnChunk][2];
#pragma unroll
        for (int b = 0; b < kDnChunk; ++b)
          if (st0 + b < nst) {
            bh[b][0] = __ldcg(reinterpret_cast<const uint4*>(hrow + (st0 + b) * 64));
            bh[b][1] = __ldcg(reinterpret_cast<const uint4*>(hrow + (st0 + b) * 64 + 8));
          }
#pragma unroll
        for (int b = 0; b < kDnChunk; ++b)
          if (st0 + b < nst) {
            const int st = st0 + b;
            const SupertileA ad = dequant_supertile(*reinterpret_cast<const uint4*>(sp + st * 512 + lane * 16),
                                                    *reinterpret_cast<const uint2*>(sp + 8 * I + st * 64 + g * 8));
            supertile_mma_pre(acc, ad, bh[b][0], bh[b][1]);
          }
      }
      // lane (g, t4) holds rows g, g + 8 of the group's columns 2 t4, 2 t4 + 1
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int row = (c < 2) ? g : g + 8;
        const int col = col0 + 2 * t4 + (c & 1);
        if (col < cnt) zb[(size_t)(poff + col) * 16 + row] = acc[c];
      }
      __syncwarp();
    }
    // a copy whose wait ran out may still be in flight: wait for it again
    // (bounded) so that nothing lands in shared memory after the block exits
    if (lane == 0)
      for (int b = 0; b < 2; ++b)
        if (pending[b]) (void)mbar_wait_bounded(a, &bar[warp][b], (uint32_t)(pending[b] - 1), global_ns() + 2000000000ull);
  }
  __syncthreads();
  for (int q = tid; q < T * 16; q += kDnThreads) {
    const int t = q >> 4, row = q & 15;
    float v = 0.f;
    for (int j = 0; j < k; ++j) {
      const int p = __ldcg(a.u_off + __ldcg(a.tk_u + t * k + j)) + __ldcg(a.tk_pos + t * k + j);
      v = fmaf(__ldcg(a.topk_w + t * k + j), zb[(size_t)p * 16 + row], v);
    }
    if (a.n_shared) v += zb[(size_t)(T * k + t) * 16 + row];
    a.y[(size_t)t * H + r * 16 + row] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
  }
}

// ------------------------------------------------------------------ residual + RMSNorm

__global__ void __launch_bounds__(kNormThreads) residual_rmsnorm_kernel(const uint16_t* x, const uint16_t* y, int H,
                                                                          float eps, uint16_t* x_out, uint16_t* xhat) {
  extern __shared__ __align__(16) uint4 xs4[];  // [H / 8] bf16 chunks of x + y
  __shared__ float part[kNormThreads / 32];
  const int t = blockIdx.x, tid = threadIdx.x;
  constexpr int kC = kMaxHidden / 8 / kNormThreads;  // chunks per thread
  const int n8 = H / 8;
  // programmatic dependent launch: let the next kernel start its prologue,
  // then wait for the work that wrote x and y
  pdl_trigger();
  pdl_wait();
  const uint4* x4 = reinterpret_cast<const uint4*>(x + (size_t)t * H);
  const uint4* y4 = y ? reinterpret_cast<const uint4*>(y + (size_t)t * H) : nullptr;
  uint4 xv[kC], yv[kC];  // every load of the thread first
#pragma unroll
  for (int c = 0; c < kC; ++c) {
    const int i = tid + kNormThreads * c;
    xv[c] = i < n8 ? x4[i] : make_uint4(0u, 0u, 0u, 0u);
    yv[c] = (y4 && i < n8) ? y4[i] : make_uint4(0u, 0u, 0u, 0u);
  }
  float ss = 0.f;
#pragma unroll
  for (int c = 0; c < kC; ++c) {
    const int i = tid + kNormThreads * c;
    if (i < n8) xs4[i] = resid_chunk(xv[c], yv[c], y4 != nullptr, ss);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((tid & 31) == 0) part[tid >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
  for (int w = 0; w < kNormThreads / 32; ++w) tot += part[w];
  const float inv = 1.0f / sqrtf(tot / (float)H + eps);
#pragma unroll
  for (int c = 0; c < kC; ++c) {
    const int i = tid + kNormThreads * c;
    if (i < n8) {
      if (x_out) reinterpret_cast<uint4*>(x_out + (size_t)t * H)[i] = xs4[i];
      reinterpret_cast<uint4*>(xhat + (size_t)t * H)[i] = scale_chunk(xs4[i], inv);
    }
  }
}

template <typename K>
cudaError_t launch(K kernel, int grid, int block, size_t smem, cudaStream_t s, bool pdl, const LayerArgs& a) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, a);
}

size_t gateup_smem(int H) {
  const size_t pitch = ((size_t)gu_strip_bytes(H) + 127) & ~size_t(127);
  return pitch + sizeof(float) * kGuWarpsPerTask * kGuGroups * 32 * 8;
}

}  // namespace

namespace {
size_t g_down_smem = 0;  // dynamic shared memory down_kernel may use (set by configure_kernels)
}  // namespace

size_t route_smem_bytes(int H, int E) {
  (void)E;
  (void)H;
  return sizeof(float) * (kRouteThreads / 32) * kMaxTokens;
}

size_t select_smem_bytes(int E) {
  const size_t a = select_layout(E).total;
  const size_t b = finish_layout(E).total;
  return a > b ? a : b;
}

cudaError_t configure_kernels(int H, int E) {
  cudaError_t e = cudaFuncSetAttribute(route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)route_smem_bytes(kMaxHidden, kMaxExperts));
  if (e != cudaSuccess) return e;
  const void* sel[7] = {(const void*)route_select_kernel<1>, (const void*)route_select_kernel<2>,
                        (const void*)route_select_kernel<4>, (const void*)route_select_kernel<8>,
                        (const void*)route_select_kernel<16>, (const void*)route_select_kernel<32>,
                        (const void*)route_select_kernel<0>};
  for (const void* f : sel) {
    e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)select_smem_bytes(kMaxExperts));
    if (e != cudaSuccess) return e;
  }
  e = cudaFuncSetAttribute(gateup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gateup_smem(kMaxHidden));
  if (e != cudaSuccess) return e;
  {
    int dev = 0, optin = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, down_kernel);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, optin - (int)fa.sharedSizeBytes);
    if (e != cudaSuccess) return e;
    g_down_smem = (size_t)optin - fa.sharedSizeBytes;
  }
  e = cudaFuncSetAttribute(residual_rmsnorm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)(2 * kMaxHidden));
  (void)H;
  (void)E;
  return e;
}

int gateup_max_blocks_per_sm(int H) {
  int n = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, gateup_kernel, kGuThreads, gateup_smem(H));
  return n > 0 ? n : 1;
}

// Warps of down_kernel that stream expert strips: as many two-stage rings as
// fit next to the pairs' outputs in the opt-in shared memory, at most 16.
int down_warps(int T, int k, int n_shared, int I) {
  const size_t avail = g_down_smem;
  const size_t z = down_z_bytes(T, k, n_shared), per = 2 * down_stage_pitch(I);
  if (avail < z + per) return 0;
  const size_t n = (avail - z) / per;
  return n < (size_t)kDnMaxWarps ? (int)n : kDnMaxWarps;
}

cudaError_t launch_route(const LayerArgs& a, cudaStream_t s, bool pdl) {
  const int grid = (a.E + kRouteRows - 1) / kRouteRows * ((a.T + kRouteTokBlock - 1) / kRouteTokBlock);
  cudaError_t e = launch(route_kernel, grid, kRouteThreads, route_smem_bytes(a.H, a.E), s, pdl, a);
  if (e != cudaSuccess) return e;
  const int sg = a.T;  // one CTA per token
  const size_t sm = select_smem_bytes(a.E);
  if (a.E <= 32) return launch(route_select_kernel<1>, sg, kSelThreads, sm, s, true, a);
  if (a.E <= 64) return launch(route_select_kernel<2>, sg, kSelThreads, sm, s, true, a);
  if (a.E <= 128) return launch(route_select_kernel<4>, sg, kSelThreads, sm, s, true, a);
  if (a.E <= 256) return launch(route_select_kernel<8>, sg, kSelThreads, sm, s, true, a);
  if (a.E <= 512) return launch(route_select_kernel<16>, sg, kSelThreads, sm, s, true, a);
  if (a.E <= 1024) return launch(route_select_kernel<32>, sg, kSelThreads, sm, s, true, a);
  return launch(route_select_kernel<0>, sg, kSelThreads, sm, s, true, a);
}

cudaError_t launch_gateup(const LayerArgs& a, cudaStream_t s, bool pdl, int grid) {
  return launch(gateup_kernel, grid, kGuThreads, gateup_smem(a.H), s, pdl, a);
}

cudaError_t launch_down(const LayerArgs& a, cudaStream_t s, bool pdl, int nw) {
  const size_t smem = down_z_bytes(a.T, a.k, a.n_shared) + (size_t)nw * 2 * down_stage_pitch(a.I);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.H / 16);
  cfg.blockDim = dim3(kDnThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, down_kernel, a, nw);
}

cudaError_t launch_residual_rmsnorm(const uint16_t* x, const uint16_t* y, int T, int H, float eps, uint16_t* x_out,
                                    uint16_t* xhat, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(T);
  cfg.blockDim = dim3(kNormThreads);
  cfg.dynamicSmemBytes = 2 * (size_t)H;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, residual_rmsnorm_kernel, x, y, H, eps, x_out, xhat);
}

}  // namespace moe
