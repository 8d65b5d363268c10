// Decode-path kernels of the quantized MoE FFN layer (sm_103a).
//
// One moe_forward = three stream-ordered kernels chained with programmatic
// dependent launch (griddepcontrol), so each grid is already resident when
// its predecessor finishes:
//   route_kernel   router GEMV (compensated fp32, four warps per expert row,
//                  the canonical order of moe_route.cuh), then in the
//                  last-arriving CTA: top-k per token, softmax weights and
//                  grouping of (token, expert) pairs by expert.
//   gateup_kernel  per (expert, 16-row strip): 4-bit gate and up rows
//                  dequantized in registers into mma.m16n8k16 fragments,
//                  fp32 accumulation with exact per-block scaling, then
//                  h = silu(g) * u stored as fp16.
//   down_kernel    per 16-row output strip: every selected expert's down rows,
//                  then the routing-weighted combine in ascending expert
//                  order (shared expert last) and one bf16 rounding.
// These kernels serve layers whose experts are all resident (slot = expert);
// a layer with a slot pool runs the fused decode kernel, which holds the
// hit check (Betelgeuse news page, section 机制: 调度 and 显存 rows).
#include <cfloat>
#include <climits>

#include "moe.h"
#include "moe_internal.h"
#include "moe_mma.cuh"
#include "moe_route.cuh"

namespace moe {
namespace {

// ------------------------------------------------------------------ PTX helpers

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ uint4 ld_cg4(const void* p) {
  uint4 r;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}
__device__ __forceinline__ uint2 ld_cg2(const void* p) {
  uint2 r;
  asm volatile("ld.global.cg.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
  return r;
}
__device__ __forceinline__ int ld_cg_i32(const int* p) {
  int r;
  asm volatile("ld.global.cg.s32 %0, [%1];" : "=r"(r) : "l"(p));
  return r;
}
__device__ __forceinline__ float ld_cg_f32(const float* p) {
  float r;
  asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(r) : "l"(p));
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
constexpr int kRouteChunk = 8;       // tokens staged in shared memory at a time
constexpr int kRouteVec = kMaxHidden / 512;  // float4 per lane per quarter row

struct FinishSmem {
  size_t lrow, tokmask, uidx, poff, sidx, sw, misc, total;
};

__host__ __device__ inline size_t align16(size_t v) { return (v + 15) & ~size_t(15); }

// Warps of the last CTA that select top-k (each stages one token's E rank
// words in shared memory).
__host__ __device__ inline int topk_warps(int E) { return E <= 2048 ? 8 : 4; }

__host__ __device__ inline FinishSmem finish_layout(int E) {
  FinishSmem f;
  f.lrow = 0;
  f.tokmask = f.lrow + align16(sizeof(unsigned long long) * topk_warps(E) * (size_t)E);
  f.uidx = f.tokmask + align16(sizeof(unsigned long long) * (size_t)E);
  f.poff = f.uidx + align16(sizeof(int) * (size_t)E);
  f.sidx = f.poff + align16(sizeof(int) * (size_t)E);
  f.sw = f.sidx + align16(sizeof(int) * kMaxTokens * kMaxTopK);
  f.misc = f.sw + align16(sizeof(float) * kMaxTokens * kMaxTopK);
  f.total = f.misc + sizeof(unsigned long long) * 64;
  return f;
}

// Block-wide exclusive scan of (a, b) pairs, 256 threads; returns totals.
__device__ void block_scan2(int& a, int& b, int& tot_a, int& tot_b, int* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int ia = a, ib = b;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int va = __shfl_up_sync(0xffffffffu, ia, o), vb = __shfl_up_sync(0xffffffffu, ib, o);
    if (lane >= o) { ia += va; ib += vb; }
  }
  if (lane == 31) { scratch[warp] = ia; scratch[8 + warp] = ib; }
  __syncthreads();
  int wa = 0, wb = 0, ta = 0, tb = 0;
  for (int w = 0; w < 8; ++w) {
    if (w < warp) { wa += scratch[w]; wb += scratch[8 + w]; }
    ta += scratch[w];
    tb += scratch[8 + w];
  }
  a = wa + ia - a;
  b = wb + ib - b;
  tot_a = ta;
  tot_b = tb;
  __syncthreads();
}

// The last CTA: top-k, grouping, hit check, LRU, doorbell.
__device__ void route_finish(const LayerArgs& a, unsigned char* smem) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = a.E, k = a.k, T = a.T;
  const FinishSmem f = finish_layout(E);
  float* lrow = reinterpret_cast<float*>(smem + f.lrow);
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
  for (int e = tid; e < E; e += kRouteThreads) tokmask[e] = 0ull;
  __syncthreads();
  const uint32_t seq = s_seq;
  // keep the fused decode path's gate/up counters of the next step at zero
  for (int i = tid; i < a.cnt_stride; i += kRouteThreads) a.counters[(size_t)((seq + 1u) & 1u) * a.cnt_stride + i] = 0u;

  // ---- top-k per token (warp per token), ties to the lower index
  const int nw = topk_warps(E);
  if (warp < nw)
    for (int t = warp; t < T; t += nw) {
      unsigned long long* lr = reinterpret_cast<unsigned long long*>(lrow) + (size_t)warp * E;
      for (int e = lane; e < E; e += 32) lr[e] = rank_word(__ldcg(&a.keys[(size_t)t * E + e]), e);
      __syncwarp();
      int sel[kMaxTopK];
      float selv[kMaxTopK];
      warp_select_k(lr, E, k, sel, selv);
      if (lane == 0) {
        // ascending expert index, weights renormalised over the selection
        softmax_ascending(sel, selv, k, a.topk_idx + t * k, a.topk_w + t * k);
        for (int j = 0; j < k; ++j) {
          sidx[t * k + j] = sel[j];
          sw[t * k + j] = a.topk_w[t * k + j];
          atomicOr(&tokmask[sel[j]], 1ull << t);
        }
      }
      __syncwarp();
    }
  __syncthreads();

  // ---- union of selected experts (ascending) and pair offsets
  const int per = (E + kRouteThreads - 1) / kRouteThreads;
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
  for (int p = tid; p < T * k; p += kRouteThreads) {
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
  for (int u = tid; u < n_union; u += kRouteThreads) a.u_slot[u] = a.u_expert[u];
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
  const int row = blockIdx.x * kRouteRows + (warp >> 2);
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

  float* xs = reinterpret_cast<float*>(smem);                  // [chunk][H]
  DF* red = reinterpret_cast<DF*>(xs + kRouteChunk * H);        // [8 warps][chunk]
  for (int t0 = 0; t0 < T; t0 += kRouteChunk) {
    const int nt = min(kRouteChunk, T - t0);
    __syncthreads();
    stage_x_f32<kRouteThreads>(a.x + (size_t)t0 * H, nt * H, xs, tid);
    __syncthreads();
    for (int tt = 0; tt < nt; ++tt) {
      // the canonical compensated order (moe_route.cuh): lane-strided float4
      // groups of this quarter, then the xor butterfly
      const float4* xr = reinterpret_cast<const float4*>(xs + tt * H + q * (H / 4));
      DF d{0.f, 0.f};
#pragma unroll
      for (int i = 0; i < kRouteVec; ++i) {
        const int j = lane + 32 * i;
        if (j < n4) dot2_acc4(d, w[i], xr[j]);
      }
      d = warp_sum_df(d);
      if (lane == 0) red[warp * kRouteChunk + tt] = d;
    }
    __syncthreads();
    if (tid < kRouteRows * nt) {
      const int r = tid / nt, tt = tid % nt;
      const int e = blockIdx.x * kRouteRows + r;
      if (e < E) {
        const DF* pr = red + (4 * r) * kRouteChunk + tt;
        a.keys[(size_t)(t0 + tt) * E + e] = logit_key(pr[0], pr[kRouteChunk], pr[2 * kRouteChunk],
                                                      pr[3 * kRouteChunk], a.bias ? __ldg(a.bias + e) : 0.f);
      }
    }
  }
  __threadfence();
  __syncthreads();
  pdl_trigger();
  __shared__ uint32_t s_ticket;
  if (tid == 0) s_ticket = atomicAdd(&a.st->ticket, 1u);
  __syncthreads();
  if (s_ticket != gridDim.x - 1) return;
  __threadfence();
  route_finish(a, smem);
}

// ------------------------------------------------------------------ gate/up

constexpr int kGuThreads = 128;  // 4 warps split the K = H reduction of a strip, as in the fused path
constexpr int kGuWarpsPerTask = kGuThreads / 32;
constexpr int kGuBatch = 2;      // super-tiles per warp with loads in flight together

template <int NG>
__global__ void __launch_bounds__(kGuThreads) gateup_kernel(LayerArgs a) {
  extern __shared__ __align__(16) float red[];  // [4 warps][NG][32 lanes][8]
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int H = a.H, I = a.I;
  const int NS = I / 16, nst = H / 64;
  const int n_union = ld_cg_i32(&a.st->n_union);
  const int n_tasks = (a.n_shared + n_union) * NS;
  __shared__ int s_go;
  for (int task = blockIdx.x; task < n_tasks; task += gridDim.x) {
    const int gu = task / NS, s = task % NS;
    const bool sh = gu < a.n_shared;
    const uint8_t* base;
    int cnt, poff;
    if (sh) {
      base = a.shared;
      cnt = a.T;
      poff = a.T * a.k;
    } else {
      const int u = gu - a.n_shared;
      base = a.arena + (int64_t)ld_cg_i32(&a.u_slot[u]) * a.blob;
      poff = ld_cg_i32(&a.u_off[u]);
      cnt = ld_cg_i32(&a.u_off[u + 1]) - poff;
    }
    // one thread decides for the block whether the layer still runs
    if (tid == 0) s_go = dev_error(a) == 0;
    __syncthreads();
    if (!s_go) return;
    const uint8_t* strip = base + (int64_t)s * gu_strip_bytes(H);
    const int ng = (cnt + 7) >> 3;
    int tok[NG];
#pragma unroll
    for (int q = 0; q < NG; ++q) {
      const int i = q * 8 + g;
      tok[q] = (i < cnt) ? (sh ? i : ld_cg_i32(&a.pair_token[poff + i])) : 0;
    }
    float accg[NG][4], accu[NG][4];
#pragma unroll
    for (int q = 0; q < NG; ++q)
#pragma unroll
      for (int c = 0; c < 4; ++c) accg[q][c] = accu[q][c] = 0.f;

    for (int st0 = warp; st0 < nst; st0 += kGuWarpsPerTask * kGuBatch) {
      uint4 ngw[kGuBatch], nuw[kGuBatch];
      uint2 gsc[kGuBatch], usc[kGuBatch];
#pragma unroll
      for (int b = 0; b < kGuBatch; ++b) {
        const int st = st0 + kGuWarpsPerTask * b;
        if (st < nst) {
          ngw[b] = __ldcg(reinterpret_cast<const uint4*>(strip + st * 512 + lane * 16));
          gsc[b] = __ldcg(reinterpret_cast<const uint2*>(strip + 8 * H + st * 64 + g * 8));
          nuw[b] = __ldcg(reinterpret_cast<const uint4*>(strip + 9 * H + st * 512 + lane * 16));
          usc[b] = __ldcg(reinterpret_cast<const uint2*>(strip + 17 * H + st * 64 + g * 8));
        }
      }
#pragma unroll
      for (int b = 0; b < kGuBatch; ++b) {
        const int st = st0 + kGuWarpsPerTask * b;
        if (st < nst) {
          // every token group's activation fragments first (plain loads the
          // compiler may overlap), then the weights dequantized once and
          // multiplied against each group
          uint4 bx[NG][2];
#pragma unroll
          for (int q = 0; q < NG; ++q)
            if (q < ng) {
              const uint4* xr = reinterpret_cast<const uint4*>(a.x16 + (size_t)tok[q] * H + st * 64 + t4 * 16);
              bx[q][0] = __ldcg(xr);
              bx[q][1] = __ldcg(xr + 1);
            }
          const SupertileA ag = dequant_supertile(ngw[b], gsc[b]);
          const SupertileA au = dequant_supertile(nuw[b], usc[b]);
#pragma unroll
          for (int q = 0; q < NG; ++q) {
            if (q < ng) {
              supertile_mma_pre(accg[q], ag, bx[q][0], bx[q][1]);
              supertile_mma_pre(accu[q], au, bx[q][0], bx[q][1]);
            }
          }
        }
      }
    }
#pragma unroll
    for (int q = 0; q < NG; ++q) {
      float4* dst = reinterpret_cast<float4*>(red + (((warp * NG) + q) * 32 + lane) * 8);
      dst[0] = make_float4(accg[q][0], accg[q][1], accg[q][2], accg[q][3]);
      dst[1] = make_float4(accu[q][0], accu[q][1], accu[q][2], accu[q][3]);
    }
    __syncthreads();
    for (int q = warp; q < ng; q += kGuWarpsPerTask) {
      float gs[4] = {0.f, 0.f, 0.f, 0.f}, us[4] = {0.f, 0.f, 0.f, 0.f};
      for (int w = 0; w < kGuWarpsPerTask; ++w) {
        const float4* src = reinterpret_cast<const float4*>(red + (((w * NG) + q) * 32 + lane) * 8);
        const float4 p = src[0], r = src[1];
        gs[0] += p.x; gs[1] += p.y; gs[2] += p.z; gs[3] += p.w;
        us[0] += r.x; us[1] += r.y; us[2] += r.z; us[3] += r.w;
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int rowin = (c < 2) ? g : g + 8;
        const int col = 2 * t4 + (c & 1);
        const int i = q * 8 + col;
        if (i < cnt) {
          const int hrow = poff + i;
          a.h16[(size_t)hrow * I + frag_pos(s * 16 + rowin)] = __float2half_rn(silu(gs[c]) * us[c]);
        }
      }
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------------ down + combine

constexpr int kDnThreads = 256;  // 8 warps, one expert each per batch
constexpr int kDnWarps = kDnThreads / 32;
constexpr int kDnBatch1 = 8;     // super-tiles with loads in flight together (one token group)
constexpr int kDnBatch8 = 2;     // the same with eight token groups (registers)

template <int NG>
__global__ void __launch_bounds__(kDnThreads) down_kernel(LayerArgs a) {
  extern __shared__ __align__(16) float dsm[];
  float* zbuf = dsm;                                   // [warps][NG][32 lanes][4]
  float* yacc = dsm + kDnWarps * NG * 32 * 4;          // [T][16]
  int* m_u = reinterpret_cast<int*>(yacc + a.T * 16);  // [T][k] union index of (t, j)
  int* m_pos = m_u + a.T * a.k;                        // [T][k] its place among the expert's pairs
  float* m_w = reinterpret_cast<float*>(m_pos + a.T * a.k);  // [T][k] routing weight
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int H = a.H, I = a.I, T = a.T, k = a.k;
  const int n_union = ld_cg_i32(&a.st->n_union);
  const int n_ex = n_union + a.n_shared;
  const int nst = I / 64;
  // the combine's per-pair metadata, read once
  for (int i = tid; i < T * k; i += kDnThreads) {
    m_u[i] = __ldcg(a.tk_u + i);
    m_pos[i] = __ldcg(a.tk_pos + i);
    m_w[i] = __ldcg(a.topk_w + i);
  }
  __syncthreads();
  constexpr int kDnBatch = NG > 1 ? kDnBatch8 : kDnBatch1;
  for (int r = blockIdx.x; r < H / 16; r += gridDim.x) {
    for (int q = tid; q < T * 16; q += kDnThreads) yacc[q] = 0.f;
    for (int b0 = 0; b0 < n_ex; b0 += kDnWarps) {
      const int xi = b0 + warp;
      if (xi < n_ex) {
        const bool sh = xi >= n_union;
        const uint8_t* base;
        int cnt, poff;
        if (sh) {
          base = a.shared;
          cnt = T;
          poff = T * k;
        } else {
          base = a.arena + (int64_t)ld_cg_i32(&a.u_slot[xi]) * a.blob;
          poff = ld_cg_i32(&a.u_off[xi]);
          cnt = ld_cg_i32(&a.u_off[xi + 1]) - poff;
        }
        const uint8_t* strip = base + down_base(H, I) + (int64_t)r * down_strip_bytes(I);
        const int ng = (cnt + 7) >> 3;
        int hrow[NG];
#pragma unroll
        for (int q = 0; q < NG; ++q) {
          const int i = q * 8 + g;
          hrow[q] = poff + ((i < cnt) ? i : 0);
        }
        float acc[NG][4];
#pragma unroll
        for (int q = 0; q < NG; ++q) acc[q][0] = acc[q][1] = acc[q][2] = acc[q][3] = 0.f;
        for (int st0 = 0; st0 < nst; st0 += kDnBatch) {
          uint4 nw[kDnBatch];
          uint2 sc[kDnBatch];
#pragma unroll
          for (int b = 0; b < kDnBatch; ++b) {
            const int st = st0 + b;
            if (st < nst) {
              nw[b] = __ldcg(reinterpret_cast<const uint4*>(strip + st * 512 + lane * 16));
              sc[b] = __ldcg(reinterpret_cast<const uint2*>(strip + 8 * I + st * 64 + g * 8));
            }
          }
#pragma unroll
          for (int b = 0; b < kDnBatch; ++b) {
            const int st = st0 + b;
            if (st < nst) {
              uint4 bh[NG][2];  // every group's h fragments first, then the products
#pragma unroll
              for (int q = 0; q < NG; ++q)
                if (q < ng) {
                  const uint4* hr = reinterpret_cast<const uint4*>(a.h16 + (size_t)hrow[q] * I + st * 64 + t4 * 16);
                  bh[q][0] = __ldcg(hr);
                  bh[q][1] = __ldcg(hr + 1);
                }
              const SupertileA ad = dequant_supertile(nw[b], sc[b]);  // once for every token group
#pragma unroll
              for (int q = 0; q < NG; ++q)
                if (q < ng) supertile_mma_pre(acc[q], ad, bh[q][0], bh[q][1]);
            }
          }
        }
#pragma unroll
        for (int q = 0; q < NG; ++q)
          *reinterpret_cast<float4*>(zbuf + ((warp * NG + q) * 32 + lane) * 4) =
              make_float4(acc[q][0], acc[q][1], acc[q][2], acc[q][3]);
      }
      __syncthreads();
      // combine this batch: token t, output row; ascending expert order
      for (int q = tid; q < T * 16; q += kDnThreads) {
        const int t = q >> 4, row = q & 15;
        float v = yacc[q];
        for (int j = 0; j < k; ++j) {
          const int u = m_u[t * k + j];
          if (u >= b0 && u < b0 + kDnWarps) {
            const int pos = m_pos[t * k + j];
            const int grp = pos >> 3, col = pos & 7;
            const int lz = (row & 7) * 4 + (col >> 1), rz = (row >> 3) * 2 + (col & 1);
            v = fmaf(m_w[t * k + j], zbuf[(((u - b0) * NG + grp) * 32 + lz) * 4 + rz], v);
          }
        }
        if (a.n_shared && n_union >= b0 && n_union < b0 + kDnWarps) {
          const int grp = t >> 3, col = t & 7;
          const int lz = (row & 7) * 4 + (col >> 1), rz = (row >> 3) * 2 + (col & 1);
          v += zbuf[(((n_union - b0) * NG + grp) * 32 + lz) * 4 + rz];
        }
        yacc[q] = v;
      }
      __syncthreads();
    }
    for (int q = tid; q < T * 16; q += kDnThreads) {
      const int t = q >> 4, row = q & 15;
      a.y[(size_t)t * H + r * 16 + row] = __bfloat16_as_ushort(__float2bfloat16_rn(yacc[q]));
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------------ residual + RMSNorm

__global__ void __launch_bounds__(256) residual_rmsnorm_kernel(const uint16_t* x, const uint16_t* y, int H, float eps,
                                                                 uint16_t* x_out, uint16_t* xhat) {
  extern __shared__ float xs[];  // [H]
  __shared__ float part[8];
  const int t = blockIdx.x, tid = threadIdx.x;
  // programmatic dependent launch: let the next kernel start its prologue,
  // then wait for the work that wrote x and y
  pdl_trigger();
  pdl_wait();
  float ss = 0.f;
  for (int i = tid; i < H; i += 256) {
    float v = __uint_as_float((uint32_t)x[(size_t)t * H + i] << 16);
    if (y) v += __uint_as_float((uint32_t)y[(size_t)t * H + i] << 16);
    const __nv_bfloat16 b = __float2bfloat16_rn(v);
    const float vr = __bfloat162float(b);
    xs[i] = vr;
    ss = fmaf(vr, vr, ss);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((tid & 31) == 0) part[tid >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
  for (int w = 0; w < 8; ++w) tot += part[w];
  const float inv = 1.0f / sqrtf(tot / (float)H + eps);
  for (int i = tid; i < H; i += 256) {
    if (x_out) x_out[(size_t)t * H + i] = __bfloat16_as_ushort(__float2bfloat16_rn(xs[i]));
    xhat[(size_t)t * H + i] = __bfloat16_as_ushort(__float2bfloat16_rn(xs[i] * inv));
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

size_t gateup_smem(int NG) { return sizeof(float) * kGuWarpsPerTask * NG * 32 * 8; }
size_t down_smem(int NG, int T) { return sizeof(float) * (kDnWarps * NG * 32 * 4 + T * 16 + 3 * T * kMaxTopK); }

}  // namespace

size_t route_smem_bytes(int H, int E) {
  size_t a = sizeof(float) * kRouteChunk * (size_t)H + sizeof(DF) * 8 * kRouteChunk;
  size_t b = finish_layout(E).total;
  return a > b ? a : b;
}

cudaError_t configure_kernels(int H, int E) {
  cudaError_t e = cudaFuncSetAttribute(route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)route_smem_bytes(kMaxHidden, kMaxExperts));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(gateup_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gateup_smem(8));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(down_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)down_smem(8, kMaxTokens));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(residual_rmsnorm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)(sizeof(float) * kMaxHidden));
  (void)H;
  (void)E;
  return e;
}

int gateup_max_blocks_per_sm(int T) {
  int n = 0;
  if (T <= 8)
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, gateup_kernel<1>, kGuThreads, gateup_smem(1));
  else
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, gateup_kernel<8>, kGuThreads, gateup_smem(8));
  return n > 0 ? n : 1;
}

int down_max_blocks_per_sm(int T) {
  int n = 0;
  if (T <= 8)
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, down_kernel<1>, kDnThreads, down_smem(1, 8));
  else
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, down_kernel<8>, kDnThreads, down_smem(8, kMaxTokens));
  return n > 0 ? n : 1;
}

cudaError_t launch_route(const LayerArgs& a, cudaStream_t s, bool pdl) {
  const int grid = (a.E + kRouteRows - 1) / kRouteRows;
  return launch(route_kernel, grid, kRouteThreads, route_smem_bytes(a.H, a.E), s, pdl, a);
}

cudaError_t launch_gateup(const LayerArgs& a, cudaStream_t s, bool pdl, int grid) {
  if (a.T <= 8) return launch(gateup_kernel<1>, grid, kGuThreads, gateup_smem(1), s, pdl, a);
  return launch(gateup_kernel<8>, grid, kGuThreads, gateup_smem(8), s, pdl, a);
}

cudaError_t launch_down(const LayerArgs& a, cudaStream_t s, bool pdl, int grid) {
  if (a.T <= 8) return launch(down_kernel<1>, grid, kDnThreads, down_smem(1, a.T), s, pdl, a);
  return launch(down_kernel<8>, grid, kDnThreads, down_smem(8, a.T), s, pdl, a);
}

cudaError_t launch_residual_rmsnorm(const uint16_t* x, const uint16_t* y, int T, int H, float eps, uint16_t* x_out,
                                    uint16_t* xhat, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(T);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = sizeof(float) * H;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, residual_rmsnorm_kernel, x, y, H, eps, x_out, xhat);
}

}  // namespace moe
