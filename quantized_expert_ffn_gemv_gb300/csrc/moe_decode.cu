// Fused decode kernel (T <= 8 tokens per call): the whole MoE layer in one
// cooperative launch of one CTA per SM, 16 warps.  Consecutive launches are
// chained by programmatic dependent launch: the prologue below runs before
// the wait for the previous grid, everything else after it.
//
// Weights stream through shared-memory rings filled with 1-D TMA bulk copies
// (cp.async.bulk + mbarrier); lane 0 of warp 15 is the producer and keeps
// refilling the rings whenever it would otherwise wait.
//
//   prologue   this CTA's router rows, its shared-expert gate/up strip and
//              down strip start loading; x -> fp16 in B-fragment order.
//   router     compensated (double-float) dot products, four warps per row;
//              each logit's 52-bit order key is stored with a 12-bit call tag
//              in one 64-bit word; each CTA then adds one relaxed count on
//              the layer's publication counter, and one lane per CTA waits for
//              all of them before the block reads the keys once.
//   routing    every CTA redundantly: each warp ranks its range of experts
//              (one 64-bit compare orders by logit, then index) and keeps its
//              k best; entries below a threshold taken from the lists' heads
//              cannot be selected; the survivors are ranked against each
//              other, giving the k in rank order.  One token: the union is
//              that order and the experts start at once while a spare warp
//              computes the softmax weights and the combine mapping.  More
//              tokens: ascending expert order, softmax renormalised over the
//              k, the union and the (expert, token) pair lists.  Then the slot
//              hit check and LRU victims (double-buffered pool state, its
//              tables copied to shared memory during the routing; CTA 0 rings
//              the host doorbell).  Betelgeuse news page, section 机制, 调度
//              row: the hit check runs in-stream on the GPU.
//   misses     by default the consuming warps read a missed expert's strips
//              from the mapped pinned master copy themselves (and write them
//              back to its slot); otherwise they wait for the slot's ready
//              flag, set by the host copy server after its copy.
//   gate/up    four warps per 16-row strip (K split four ways), one strip per
//              ring stage at once; h = silu(g) * u rounded to fp16.  One
//              resident token: h goes out as 64-bit words tagged with the
//              call (two values each) and a relaxed count per 64-wide chunk
//              of I says when to look; otherwise h rows go out as fp16 and a
//              per-expert counter is bumped with a release reduction
//              (counters double-buffered by step parity, one cache line each).
//   down       warp w handles selected experts w, w + ds, ...: one resident
//              token: the chunks whose count is complete are read straight
//              into the MMA fragments once every word carries the call's tag,
//              while later strips are still being computed; otherwise the
//              expert's counter, then its h staged in shared memory with
//              cp.async.  z = W_d h for this CTA's 16 output rows; then
//              y = sum_j w_j z_j (ascending expert) + z_shared in fp32,
//              rounded once to bf16.
#include <cfloat>
#include <climits>

#include "moe.h"
#include "moe_internal.h"
#include "moe_mma.cuh"
#include "moe_norm.cuh"
#include "moe_route.cuh"

namespace moe {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = 16;
constexpr int kGroupWarps = 4;             // warps per gate/up strip
constexpr int kProdWarp = 15;
constexpr int kMaxT = 8;
constexpr int kMaxE = 1024;
constexpr int kMaxGuStages = 4;
constexpr int kMaxDnStages = 16;
constexpr int kListStride = kMaxTopK + 1;  // (key, e) entries per warp's top-k list: odd, no bank conflicts

// ------------------------------------------------------------------ PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
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
// Weights are read once per call: their lines are marked first to evict, so
// streaming them through L2 does not push out the kernel's code, the
// activations, logits and counters that the next call reuses.
__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(evict_first_policy())
      : "memory");
}
// 16-byte copy global -> shared through L2 only (data other CTAs wrote in this call)
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ int ld_cg_i32(const int* p) {
  int r;
  asm volatile("ld.global.cg.s32 %0, [%1];" : "=r"(r) : "l"(p));
  return r;
}
__device__ __forceinline__ uint32_t ld_acquire_sys(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.sys.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t ld_acquire_gpu_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void red_release_add(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void red_relaxed_add(uint32_t* p, uint32_t v) {
  asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void named_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ void set_error(const LayerArgs& a, int code) {
  atomicCAS(&a.st->error, 0, code);
  volatile int32_t* m = &a.hm->error;
  if (*m == 0) *m = code;
  __threadfence_system();
}
__device__ __forceinline__ int dev_error(const LayerArgs& a) { return ld_cg_i32(&a.st->error); }
__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

// ------------------------------------------------------------------ shared memory plan

struct Plan {
  int rows_max, umax, gu_stages, dn_stages;
  size_t bars, x16, xraw, regA, gu, dn, red, lists, pooltab, total;
};

__host__ __device__ inline size_t al128(size_t v) { return (v + 127) & ~size_t(127); }

__host__ __device__ inline Plan plan_with(int H, int I, int E, int k, int T, int G, int gs, int ds, bool pool) {
  Plan p;
  p.rows_max = (E + G - 1) / G;
  p.umax = E < T * k ? E : T * k;
  p.gu_stages = gs;
  p.dn_stages = ds;
  size_t o = 0;
  p.bars = o;
  o += al128(8 * (2 * kMaxGuStages + 2 * kMaxDnStages + 2));
  p.x16 = o;
  o += al128((size_t)T * H * 2);
  p.xraw = o;
  o += al128((size_t)T * H * 2);
  // region A: router rows (prologue), routing scratch, then down results
  const size_t router = (size_t)p.rows_max * H * 4;
  // tokmask [E], then the top-k scratch (TopkScratch, at most
  // 4 * kWarps * kMaxTopK words); then the pool scratch (owner, stamp, key per slot, S <= E)
  const size_t routing = al128((size_t)E * 8) + (size_t)4 * kWarps * kMaxTopK * 8 + (size_t)E * 16 + 16 +
                         (size_t)(p.umax + 2) * 8;
  const size_t zbuf = (size_t)(p.umax + 1) * 32 * 4 * 4;
  size_t ra = router > routing ? router : routing;
  ra = ra > zbuf ? ra : zbuf;
  p.regA = o;
  o += al128(ra);
  p.gu = o;
  o += (size_t)gs * al128((size_t)gu_strip_bytes(H));
  p.dn = o;
  o += (size_t)ds * al128((size_t)down_strip_bytes(I));
  p.red = o;
  o += al128((size_t)kWarps * 32 * 8 * 4);
  p.lists = o;
  o += al128((size_t)T * k * 4 * 5 + (size_t)(p.umax + 2) * 4 * 4 + 64 * 8);
  // a pooled call's slot table, slot owners and stamps (S <= E), loaded
  // while the router and the top-k run
  p.pooltab = o;
  if (pool) o += al128((size_t)E * 12);
  p.total = o;
  return p;
}

__host__ __device__ inline Plan make_plan(int H, int I, int E, int k, int T, int G, size_t limit, bool pool) {
  const int nex = (E < T * k ? E : T * k) + 1;
  const int want_dn = nex < kMaxDnStages ? nex : kMaxDnStages;
  const int gs_opts[4] = {3, 2, 2, 1};
  const int ds_opts[4] = {want_dn, want_dn < 8 ? want_dn : 8, want_dn < 4 ? want_dn : 4, want_dn < 2 ? want_dn : 2};
  Plan p = plan_with(H, I, E, k, T, G, gs_opts[0], ds_opts[0], pool);
  for (int i = 1; i < 4 && p.total > limit; ++i) p = plan_with(H, I, E, k, T, G, gs_opts[i], ds_opts[i], pool);
  return p;
}

struct Lists {
  int* s_idx;
  float* s_w;
  int* tk_u;
  int* tk_pos;
  int* pair_token;
  int* u_expert;
  int* u_slot;
  uint32_t* u_wait;
  int* u_off;
  unsigned long long* misc;
};

__device__ inline Lists carve_lists(unsigned char* base, int T, int k, int umax) {
  Lists l;
  int* p = reinterpret_cast<int*>(base);
  const int P = T * k;
  l.s_idx = p;
  l.s_w = reinterpret_cast<float*>(p + P);
  l.tk_u = p + 2 * P;
  l.tk_pos = p + 3 * P;
  l.pair_token = p + 4 * P;
  l.u_expert = p + 5 * P;
  l.u_slot = l.u_expert + (umax + 2);
  l.u_wait = reinterpret_cast<uint32_t*>(l.u_slot + (umax + 2));
  l.u_off = reinterpret_cast<int*>(l.u_wait + (umax + 2));
  size_t off = (size_t)(5 * P + 4 * (umax + 2)) * 4;
  off = (off + 7) & ~size_t(7);
  l.misc = reinterpret_cast<unsigned long long*>(base + off);
  return l;
}

// Expert list index xi: 0 = shared expert (when present), then routed u.
struct Task {
  const uint8_t* base;  // the expert in its slot
  const uint8_t* src;   // pulled misses: the expert in the host master copy, else null
  int cnt, poff, slot;
  uint32_t wait_seq;
};

__device__ __forceinline__ Task task_of(const LayerArgs& a, const Lists& L, int xi, int n_shared) {
  Task t;
  t.src = nullptr;
  if (xi < n_shared) {
    t.base = a.shared;
    t.cnt = a.T;
    t.poff = a.T * a.k;
    t.wait_seq = 0u;
    t.slot = 0;
  } else {
    const int u = xi - n_shared;
    t.slot = L.u_slot[u];
    t.base = a.arena + (int64_t)t.slot * a.blob;
    t.poff = L.u_off[u];
    t.cnt = L.u_off[u + 1] - t.poff;
    t.wait_seq = L.u_wait[u];
    if (t.wait_seq && a.pull) {  // a miss the kernel reads from host memory itself
      t.src = a.master + (int64_t)L.u_expert[u] * a.blob;
      t.wait_seq = 0u;
    }
  }
  return t;
}

// ------------------------------------------------------------------ producer

struct Ring {
  uint64_t *full_gu, *empty_gu, *full_dn, *empty_dn;
  unsigned char *gu, *dn;
  size_t gu_pitch, dn_pitch, gu_bytes, dn_bytes;
  int gs, ds;
};

// Producer state (lane 0 of warp 15): next gate/up task and down entry to issue.
struct Producer {
  int m, d, n_gu, n_dn;
  bool routed;
  uint64_t t_wait0;  // when the producer started waiting for a slot copy (0: not waiting)
};

struct Ctx {
  const LayerArgs* a;
  const Ring* R;
  const Lists* L;
  int c, G, NS, NSh, H, I;
};

// Time spent waiting for slot copies, counted once (by CTA 0's producer).
__device__ __forceinline__ void note_wait_end(Producer& P, const Ctx& x) {
  if (P.t_wait0) {
    if (x.c == 0) atomicAdd(&x.a->st->wait_ns, (unsigned long long)(global_ns() - P.t_wait0));
    P.t_wait0 = 0;
  }
}

// Issue every copy whose ring stage is free; never blocks.  A missed expert
// is only issued once the copy server has published its slot.
__device__ void pump(Producer& P, const Ctx& x) {
  if (!P.routed) return;
  const LayerArgs& a = *x.a;
  const Ring& R = *x.R;
  while (P.m < P.n_gu) {
    const int s = P.m % R.gs;
    const int t = x.c + x.G * P.m;
    const Task tk = task_of(a, *x.L, t / x.NS, x.NSh);
    if (tk.src) {  // pulled by the consuming group itself
      ++P.m;
      continue;
    }
    if (P.m >= R.gs && !mbar_try_wait(&R.empty_gu[s], ((P.m / R.gs) - 1) & 1)) break;
    if (tk.wait_seq) {
      const uint32_t v = ld_acquire_sys(&a.ready[tk.slot]);
      if (v == (tk.wait_seq | kReadyError)) { set_error(a, MOE_ERR_COPY); P.m = P.n_gu; P.d = P.n_dn; return; }
      if (v != tk.wait_seq) {  // copy still in flight
        if (!P.t_wait0) P.t_wait0 = global_ns();
        break;
      }
      note_wait_end(P, x);
    }
    mbar_expect_tx(&R.full_gu[s], (uint32_t)R.gu_bytes);
    bulk_g2s(R.gu + s * R.gu_pitch, tk.base + (size_t)(t % x.NS) * R.gu_bytes, (uint32_t)R.gu_bytes, &R.full_gu[s]);
    ++P.m;
  }
  while (P.d < P.n_dn) {
    const int s = P.d % R.ds;
    const Task tk = task_of(a, *x.L, P.d, x.NSh);
    if (tk.src) {  // pulled by the consuming warp itself
      ++P.d;
      continue;
    }
    if (P.d >= R.ds && !mbar_try_wait(&R.empty_dn[s], ((P.d / R.ds) - 1) & 1)) break;
    if (tk.wait_seq) {
      const uint32_t v = ld_acquire_sys(&a.ready[tk.slot]);
      if (v == (tk.wait_seq | kReadyError)) { set_error(a, MOE_ERR_COPY); P.m = P.n_gu; P.d = P.n_dn; return; }
      if (v != tk.wait_seq) {
        if (!P.t_wait0) P.t_wait0 = global_ns();
        break;
      }
      note_wait_end(P, x);
    }
    mbar_expect_tx(&R.full_dn[s], (uint32_t)R.dn_bytes);
    bulk_g2s(R.dn + s * R.dn_pitch, tk.base + down_base(x.H, x.I) + (size_t)x.c * R.dn_bytes, (uint32_t)R.dn_bytes,
             &R.full_dn[s]);
    ++P.d;
  }
}

// A missed expert's strip read by the threads that need it, straight from the
// pinned host master copy (coherent over the host link), into the ring
// stage: every 16-byte copy of a thread is in flight at once (one round trip
// over the link), then the thread writes the chunks it fetched back to the
// expert's slot for later calls.  The caller then completes the stage's full
// phase.
__device__ __forceinline__ void pull_strip(const uint8_t* src, uint8_t* slot_dst, unsigned char* stage, size_t bytes,
                                           int tid, int nthreads) {
  for (size_t o = (size_t)tid * 16; o < bytes; o += (size_t)nthreads * 16) cp_async16(stage + o, src + o);
  cp_async_wait_all();
  for (size_t o = (size_t)tid * 16; o < bytes; o += (size_t)nthreads * 16)
    *reinterpret_cast<uint4*>(slot_dst + o) = *reinterpret_cast<const uint4*>(stage + o);
}

// Bounded wait on an mbarrier phase; the producer lane keeps pumping while it
// waits, so no warp ever waits on a copy that only it could issue.
__device__ bool wait_full(uint64_t* bar, uint32_t parity, uint64_t deadline, bool is_prod, Producer& P,
                          const Ctx& x) {
  int spins = 0;
  while (!mbar_try_wait(bar, parity)) {
    if (is_prod) pump(P, x);
    if (((++spins) & 31) == 0) {
      if (global_ns() > deadline) { set_error(*x.a, MOE_ERR_TIMEOUT); return false; }
      if (dev_error(*x.a)) return false;
    }
  }
  return true;
}


// ------------------------------------------------------------------ top-k

constexpr uint32_t kTagMask = 0xFFFu;  // call tag in the low 12 bits of a published logit word

// Poll one published logit until it carries this call's tag; returns its key.
__device__ __forceinline__ uint64_t wait_key(const unsigned long long* p, uint32_t tag, const LayerArgs& a,
                                             uint64_t deadline) {
  unsigned long long v = ld_relaxed_u64(p);
  int spins = 0;
  while (((uint32_t)v & kTagMask) != tag) {
    if (((++spins) & 63) == 0 && global_ns() > deadline) {
      set_error(a, MOE_ERR_TIMEOUT);
      break;
    }
    v = ld_relaxed_u64(p);
  }
  return (uint64_t)v >> 12;
}

// Routing scratch of one CTA (region A after the token masks).
struct TopkScratch {
  unsigned long long* list;  // [kWarps][kListStride] each warp's best, in rank order
  unsigned long long* sel;   // [kMaxT][kMaxTopK] each token's k best, in rank order
  unsigned long long* surv;  // survivors: token t's at t * wpt * kMaxTopK (wpt warps per token, wpt * T <= kWarps)
  int* len;                  // [kWarps] entries in each warp's list
  int* nsurv;                // [kMaxT] survivors per token
};
constexpr int kSurvTotal = kWarps * kMaxTopK;  // every list entry of every warp

__device__ inline TopkScratch carve_topk(unsigned char* base) {
  TopkScratch s;
  s.list = reinterpret_cast<unsigned long long*>(base);
  s.sel = s.list + kWarps * kListStride;
  s.surv = s.sel + kMaxT * kMaxTopK;
  s.len = reinterpret_cast<int*>(s.surv + kSurvTotal);
  s.nsurv = s.len + kWarps;
  return s;
}
constexpr size_t kTopkScratchBytes =
    8 * (kWarps * kListStride + kMaxT * kMaxTopK + kSurvTotal) + 4 * (kWarps + kMaxT);
// the shared-memory plan reserves 4 * kWarps * kMaxTopK words for it
static_assert(kTopkScratchBytes <= (size_t)4 * kWarps * kMaxTopK * 8, "routing scratch");

// Level 1: the k best of this warp's range [base, base + range) of one
// token's experts, in rank order, into list[0..len).  One key per lane: each lane's rank from 32 compares.  Several keys per
// lane: k rounds of a warp maximum.
template <int CPL>
__device__ void warp_best(const unsigned long long* words, int E, int k, int base, int range, uint32_t tag,
                          unsigned long long* list, int* len, const LayerArgs& a,
                          uint64_t deadline) {
  const int lane = threadIdx.x & 31;
  uint64_t w[CPL];
#pragma unroll
  for (int j = 0; j < CPL; ++j) {
    const int e = base + lane + 32 * j;
    w[j] = (lane + 32 * j < range && e < E) ? rank_word(wait_key(words + e, tag, a, deadline), e) : 0ull;
  }
  if (CPL == 1) {
    int r = 0;
#pragma unroll 4
    for (int i = 0; i < 32; ++i) {
      const uint64_t wi = ((uint64_t)__shfl_sync(0xffffffffu, (uint32_t)(w[0] >> 32), i) << 32) |
                          __shfl_sync(0xffffffffu, (uint32_t)w[0], i);
      r += wi > w[0];
    }
    const int n = __popc(__ballot_sync(0xffffffffu, w[0] != 0ull));
    if (w[0] != 0ull && r < k) list[r] = w[0];
    if (lane == 0) len[0] = n < k ? n : k;
    return;
  }
  uint32_t taken = 0u;
  int nl = 0;
  for (int r = 0; r < k; ++r) {
    uint64_t my = 0ull;
    int myj = -1;
#pragma unroll
    for (int j = 0; j < CPL; ++j)
      if (!((taken >> j) & 1u) && w[j] > my) { my = w[j]; myj = j; }
    const uint64_t m = warp_max_u64(my);
    if (m == 0ull) break;
    if (my == m) taken |= 1u << myj;  // words are distinct: one lane wins
    if (lane == 0) list[r] = m;
    ++nl;
  }
  if (lane == 0) len[0] = nl;
}

// Level 2, step 1 (warp w of token t's wpt warps): a threshold beta with at
// least k of the token's keys at or above it, the k-th best of the top
// 32 / wpt entries of each of the token's lists (32 keys, one per lane; each
// warp computes it, no barrier); the entries of list w not below beta (every
// selected expert is among them) are appended to the token's survivors.
__device__ __forceinline__ void keep_survivors(const TopkScratch& S, int t, int w, int wpt, int k) {
  const int lane = threadIdx.x & 31;
  const int m = 32 / wpt, li = t * wpt + lane / m, ei = lane % m;
  const uint64_t v = ei < S.len[li] ? S.list[li * kListStride + ei] : 0ull;
  int r = 0;
#pragma unroll 4
  for (int i = 0; i < 32; ++i) {
    const uint64_t vi = ((uint64_t)__shfl_sync(0xffffffffu, (uint32_t)(v >> 32), i) << 32) |
                        __shfl_sync(0xffffffffu, (uint32_t)v, i);
    r += vi > v;
  }
  const unsigned kb = __ballot_sync(0xffffffffu, v != 0ull && r == k - 1);
  const int src = kb ? __ffs(kb) - 1 : 0;
  uint64_t beta = ((uint64_t)__shfl_sync(0xffffffffu, (uint32_t)(v >> 32), src) << 32) |
                  __shfl_sync(0xffffffffu, (uint32_t)v, src);
  if (!kb) beta = 0ull;  // fewer than k keys in the sample: keep every entry
  const int n = S.len[w];
  const uint64_t e = lane < n ? S.list[w * kListStride + lane] : 0ull;
  const bool keep = e != 0ull && e >= beta;
  const unsigned b = __ballot_sync(0xffffffffu, keep);
  int base = 0;
  if (lane == 0 && b) base = atomicAdd(&S.nsurv[t], __popc(b));
  base = __shfl_sync(0xffffffffu, base, 0);
  if (keep) S.surv[t * wpt * kMaxTopK + base + __popc(b & ((1u << lane) - 1u))] = e;
}

// Level 2, step 2 (thread i of token t's wpt * 32 threads): survivor i's
// rank among the token's survivors; the k best land in sel in rank order.
__device__ __forceinline__ void rank_survivors(const TopkScratch& S, int t, int wpt, int i, int k) {
  const int n = S.nsurv[t];
  if (i >= n) return;
  const unsigned long long* sv = S.surv + t * wpt * kMaxTopK;
  const uint64_t me = sv[i];
  int r = 0;
  for (int j = 0; j < n; ++j) r += sv[j] > me;
  if (r < k) S.sel[t * kMaxTopK + r] = me;
}

// One warp per token: the k selected (in rank order in sel) reported in
// ascending expert order with softmax weights renormalised over the k (the
// sum taken in ascending expert order, as on the batched path); marks the
// token in tokmask.  With rank_union (one token) the union entries are in
// rank order and the combine mapping is written here.  sel is reused as
// scratch.
__device__ __forceinline__ void finish_topk(unsigned long long* sel, int k, const Lists& L, unsigned long long* tokmask,
                                            int t, bool write_out, const LayerArgs& a, bool rank_union = false) {
  const int lane = threadIdx.x & 31;
  const uint64_t me = (lane < k) ? sel[lane] : 0ull;
  const int my_e = (lane < k) ? word_expert(me) : INT_MAX;
  const float v = (lane < k) ? key_value(word_key(me)) : 0.f;
  const float m = __shfl_sync(0xffffffffu, v, 0);  // rank 0 holds the largest logit
  int pos = 0;
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {
    const int ej = __shfl_sync(0xffffffffu, my_e, j);
    pos += (int)((j < k) & (ej < my_e));
  }
  const float ex = (lane < k) ? expf(v - m) : 0.f;
  float* ex_sorted = reinterpret_cast<float*>(sel);
  __syncwarp();
  if (lane < k) ex_sorted[pos] = ex;
  __syncwarp();
  float exs[kMaxTopK];  // all loads first, then the sum in ascending expert order
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) exs[j] = (j < k) ? ex_sorted[j] : 0.f;
  float z = 0.f;
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j)
    if (j < k) z += exs[j];
  if (lane < k) {
    const float wj = ex / z;
    L.s_idx[t * k + pos] = my_e;
    L.s_w[t * k + pos] = wj;
    if (rank_union) {  // one token, union in rank order: the expert at position pos is union entry lane
      L.tk_u[pos] = lane;
      L.tk_pos[pos] = 0;
    }
    if (write_out) {
      a.topk_idx[t * k + pos] = my_e;
      a.topk_w[t * k + pos] = wj;
    }
    atomicOr(reinterpret_cast<unsigned int*>(&tokmask[my_e]), 1u << t);  // low word: t < 8
  }
}

// ------------------------------------------------------------------ the kernel

// ONE: the variant for one token with every expert resident and at most
// 512 experts (the decode of a resident stack), compiled without the batch
// loops, the slot-pool code and the wider top-k shapes so that the code one
// launch runs stays small.
// FMT: the weight format (0 linear, 1 codebook), fixed at compile time so the
// linear format's inner loop carries no format test.
template <bool ONE, int FMT>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(LayerArgs a, unsigned long long* tagged_logits,
                                                             int32_t* pool_state, size_t smem_limit) {
  extern __shared__ __align__(128) unsigned char sm[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int G = gridDim.x, c = blockIdx.x;
  const int H = a.H, I = a.I, E = a.E, k = a.k, T = ONE ? 1 : a.T, NS = I / 16, NSh = a.n_shared;
  constexpr int fmt = FMT;
  const uint32_t lut = FMT == 1 ? codebook_lut(threadIdx.x & 31) : 0u;
  const Plan PL = make_plan(H, I, E, k, T, G, smem_limit, !ONE && a.pool);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + PL.bars);
  Ring R;
  R.full_gu = bars;
  R.empty_gu = bars + kMaxGuStages;
  R.full_dn = bars + 2 * kMaxGuStages;
  R.empty_dn = bars + 2 * kMaxGuStages + kMaxDnStages;
  uint64_t* full_rt = bars + 2 * kMaxGuStages + 2 * kMaxDnStages;
  R.gu = sm + PL.gu;
  R.dn = sm + PL.dn;
  R.gu_bytes = (size_t)gu_strip_bytes(H);
  R.dn_bytes = (size_t)down_strip_bytes(I);
  R.gu_pitch = al128(R.gu_bytes);
  R.dn_pitch = al128(R.dn_bytes);
  R.gs = PL.gu_stages;
  R.ds = PL.dn_stages;
  __half* x16 = reinterpret_cast<__half*>(sm + PL.x16);
  uint16_t* xraw = reinterpret_cast<uint16_t*>(sm + PL.xraw);
  float* wrows = reinterpret_cast<float*>(sm + PL.regA);
  float* red = reinterpret_cast<float*>(sm + PL.red);
  const Lists L = carve_lists(sm + PL.lists, T, k, PL.umax);
  __shared__ uint32_t s_seq;
  __shared__ int s_nunion, s_nmiss;
  const bool is_prod = (warp == kProdWarp && lane == 0);
  const Ctx X{&a, &R, &L, c, G, NS, NSh, H, I};
  Producer P;
  P.m = 0;
  P.d = 0;
  P.n_gu = 0;
  P.n_dn = 0;
  P.routed = false;
  P.t_wait0 = 0;

  const int r0 = (int)((long long)c * E / G), r1 = (int)((long long)(c + 1) * E / G);
  const int nrows = r1 - r0;
  const bool has_dn = c < H / 16;
  const bool pre_gu = NSh && c < NS;  // task 0 of this CTA is a shared-expert strip, loaded early

  // Programmatic dependent launch: the next kernel in the stream may be
  // scheduled now.  Its CTAs take an SM only when one of ours leaves it, run
  // their prologue (read-only weights into shared memory) and then wait for
  // this grid to complete before touching anything it writes.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // this thread's router bias (read-only; thread i publishes row i / kMaxT)
  const float bias_v = (a.bias && tid < nrows * kMaxT) ? __ldg(a.bias + r0 + tid / kMaxT) : 0.f;
  if (tid == 0) {
    for (int s = 0; s < R.gs; ++s) { mbar_init(&R.full_gu[s], 1); mbar_init(&R.empty_gu[s], kGroupWarps); }
    for (int s = 0; s < R.ds; ++s) { mbar_init(&R.full_dn[s], 1); mbar_init(&R.empty_dn[s], 1); }
    mbar_init(full_rt, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  // ---- prologue: weights that do not depend on this call's input
  if (is_prod) {
    if (nrows > 0) {
      mbar_expect_tx(full_rt, (uint32_t)(nrows * H * 4));
      bulk_g2s(wrows, a.W_r + (size_t)r0 * H, (uint32_t)(nrows * H * 4), full_rt);
    }
    if (pre_gu) {
      mbar_expect_tx(&R.full_gu[0], (uint32_t)R.gu_bytes);
      bulk_g2s(R.gu, a.shared + (size_t)c * R.gu_bytes, (uint32_t)R.gu_bytes, &R.full_gu[0]);
      P.m = 1;
    }
    if (NSh && has_dn) {
      mbar_expect_tx(&R.full_dn[0], (uint32_t)R.dn_bytes);
      bulk_g2s(R.dn, a.shared + down_base(H, I) + (size_t)c * R.dn_bytes, (uint32_t)R.dn_bytes, &R.full_dn[0]);
      P.d = 1;
    }
  }
  // Everything below may read or write memory that earlier work in the
  // stream touches (x, the step counter, pool state, counters, logits,
  // outputs): wait for that work to complete (a no-op without a programmatic
  // dependency).  The deadline of every bounded wait starts here.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const uint64_t deadline = global_ns() + a.wait_timeout_ns;
  const uint32_t step0 = (tid == 0) ? (uint32_t)ld_cg_i32(reinterpret_cast<const int*>(&a.st->step)) : 0u;
  const uint32_t dstep0 = (tid == 0) ? (uint32_t)ld_cg_i32(reinterpret_cast<const int*>(&a.st->dstep)) : 0u;
  __shared__ uint32_t s_dseq;
  __shared__ float s_inv[kMaxT];
  if (a.resid) {
    // Fused pre-norm: xs = bf16(resid + y_prev) into xraw, and each token's
    // sum of squares in residual_rmsnorm_kernel's order (moe_norm.cuh: 256
    // threads per token over 8-element chunks), so the result is
    // bit-identical to that kernel's.
    float* part = red;  // [kMaxT][8]
    constexpr int kC = kMaxHidden / 8 / kNormThreads;
    const int n8 = H / 8;
    for (int t0 = 0; t0 < T; t0 += kThreads / kNormThreads) {
      const int t = t0 + tid / kNormThreads, vt = tid % kNormThreads;
      float ss = 0.f;
      if (t < T) {
        const uint4* x4 = reinterpret_cast<const uint4*>(a.resid + (size_t)t * H);
        const uint4* y4 = a.y_prev ? reinterpret_cast<const uint4*>(a.y_prev + (size_t)t * H) : nullptr;
        uint4 xv[kC], yv[kC];  // every load first: one round trip
#pragma unroll
        for (int cc = 0; cc < kC; ++cc) {
          const int i = vt + kNormThreads * cc;
          xv[cc] = i < n8 ? x4[i] : make_uint4(0u, 0u, 0u, 0u);
          yv[cc] = (y4 && i < n8) ? y4[i] : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int cc = 0; cc < kC; ++cc) {
          const int i = vt + kNormThreads * cc;
          if (i < n8) reinterpret_cast<uint4*>(xraw + (size_t)t * H)[i] = resid_chunk(xv[cc], yv[cc], y4 != nullptr, ss);
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      if (lane == 0 && t < T) part[t * 8 + vt / 32] = ss;
    }
    __syncthreads();
    if (tid < T) {
      float tot = 0.f;
      for (int w = 0; w < 8; ++w) tot += part[tid * 8 + w];
      s_inv[tid] = 1.0f / sqrtf(tot / (float)H + a.eps);
    }
    __syncthreads();
  }
  // x -> fp16 in B-fragment order (this CTA's own copy)
  {
    int bad = 0;
    for (int o = tid; o < T * H / 8; o += kThreads) {
      const int t = o / (H / 8), k8 = (o % (H / 8)) * 8;
      uint4 v;
      if (a.resid) {
        // xhat = bf16(xs * inv); this CTA writes its share of xs and xhat out
        const uint4 xs = *reinterpret_cast<const uint4*>(xraw + t * H + k8);
        v = scale_chunk(xs, s_inv[t]);
        if (o % G == c) {
          if (a.x_out) *reinterpret_cast<uint4*>(a.x_out + (size_t)t * H + k8) = xs;
          *reinterpret_cast<uint4*>(a.xhat_out + (size_t)t * H + k8) = v;
        }
      } else {
        v = *reinterpret_cast<const uint4*>(a.x + (size_t)t * H + k8);
      }
      *reinterpret_cast<uint4*>(xraw + t * H + k8) = v;
      const uint32_t vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float f0 = __uint_as_float(vv[i] << 16), f1 = __uint_as_float(vv[i] & 0xFFFF0000u);
        bad |= !(fabsf(f0) < 65504.f) | !(fabsf(f1) < 65504.f);
        *reinterpret_cast<__half2*>(x16 + t * H + frag_pos(k8 + 2 * i)) = __floats2half2_rn(f0, f1);
      }
    }
    if (bad) set_error(a, MOE_ERR_DEVICE);
  }
  if (tid == 0) {
    s_seq = step0 + 1u;
    s_dseq = dstep0 + 1u;
  }
  __syncthreads();
  const uint32_t seq = s_seq;
  const uint32_t tag = s_dseq & kTagMask;  // this call's tag on the published logits
  const uint32_t htag_v = s_dseq;          // this call's tag on one-token h words
  // One token, every expert resident: h goes through tagged words and the
  // down product runs chunk by chunk as they complete.  Otherwise (pooled,
  // or several tokens): h rows and one release-ordered counter per expert;
  // the chunked form was measured slower in the pooled kernel.
  constexpr bool tagged = ONE;
  // Pooled call: this step's slot table, owners and stamps start for shared
  // memory now (written by the previous call, complete at the wait above);
  // the hit check after the top-k then needs no round trip to L2.
  int* slot_s = reinterpret_cast<int*>(sm + PL.pooltab);
  int* own_s = slot_s + E;
  uint32_t* stp_s = reinterpret_cast<uint32_t*>(own_s + a.n_slots);
  if (!ONE && a.pool) {
    const int32_t* pre = pool_state + (size_t)(seq & 1u) * (E + 2 * a.n_slots);
    for (int i = tid; i < E + 2 * a.n_slots; i += kThreads) cp_async4(slot_s + i, pre + i);
    cp_async_commit();
  }
  uint32_t* cnt_cur = a.counters + (size_t)(seq & 1u) * a.cnt_stride;
  uint32_t* cnt_next = a.counters + (size_t)((seq + 1u) & 1u) * a.cnt_stride;

  // ---- router: four warps per row (one per quarter of H) in the canonical
  // compensated order; bf16 x read exactly (shared-memory copy)
  {
    DF* part = reinterpret_cast<DF*>(red);  // [rows_max <= 8][4 quarters][kMaxT]
    if (nrows > 0) {
      int spins = 0;
      while (!mbar_try_wait(full_rt, 0)) {
        if (((++spins) & 31) == 0 && global_ns() > deadline) { set_error(a, MOE_ERR_TIMEOUT); break; }
      }
    }
    const int q = warp & 3, n4 = H / 16;
    for (int row = warp >> 2; row < nrows; row += kWarps / 4) {
      const float* wq = wrows + (size_t)row * H + q * (H / 4);
      for (int t = 0; t < T; ++t) {
        const DF d = warp_sum_df(quarter_partial_bf16(wq, xraw + t * H + q * (H / 4), n4, lane));
        if (lane == 0) part[(row * 4 + q) * kMaxT + t] = d;
      }
    }
    __syncthreads();
    if (tid < nrows * kMaxT) {
      // every row of the kMaxT-token table is published each call (rows past
      // T with no key), so an unread row never keeps a tag older than the
      // previous call's
      const int rr = tid / kMaxT, t = tid % kMaxT, e = r0 + rr;
      uint64_t key = 0ull;
      if (t < T) {
        const DF* pr = part + rr * 4 * kMaxT + t;
        key = logit_key(pr[0], pr[kMaxT], pr[2 * kMaxT], pr[3 * kMaxT], bias_v);
      }
      // key and call tag in one 64-bit word: a reader that sees this call's
      // tag sees this call's key
      st_relaxed_u64(&tagged_logits[(size_t)t * E + e], (unsigned long long)((key << 12) | tag));
    }
    // one count per CTA once its rows are out: readers wait for all G counts
    // of this call on one counter (one polling lane per CTA) and then read
    // every key once, instead of every lane polling its keys' lines (which
    // slowed some CTAs' loads by microseconds).  The count carries no release
    // ordering (a fence here cost about 0.5 us per call): it only says when
    // to read, and a reader that gets ahead of a key sees the previous
    // call's tag in the word and reads it again.
    __syncthreads();
    if (tid == 0) red_relaxed_add(a.pub, 1u);
  }

  // ---- gate/up of one strip by a group of four warps (K split four ways)
  auto gateup_task = [&](int m) {
    const int grp = warp / kGroupWarps, wg = warp % kGroupWarps;
    const int s = m % R.gs;
    const int t_gu = c + G * m;
    const int xi = t_gu / NS, strip = t_gu % NS;
    const Task tk = task_of(a, L, xi, NSh);
    const int col_tok = (g < tk.cnt) ? (xi < NSh ? g : L.pair_token[tk.poff + g]) : 0;
    if (!ONE && tk.src) {  // a missed expert read from host memory by this group
      const size_t off = (size_t)strip * R.gu_bytes;
      pull_strip(tk.src + off, const_cast<uint8_t*>(tk.base) + off, R.gu + s * R.gu_pitch, R.gu_bytes,
                 wg * 32 + lane, kGroupWarps * 32);
      named_sync(1 + grp, kGroupWarps * 32);
      if (wg == 0 && lane == 0) mbar_arrive(&R.full_gu[s]);
    }
    // warp-uniform: the codebook dequantization shuffles across all 32 lanes
    const bool ok = __all_sync(0xffffffffu, wait_full(&R.full_gu[s], (m / R.gs) & 1, deadline, is_prod, P, X));
    float accg[4] = {0.f, 0.f, 0.f, 0.f}, accu[4] = {0.f, 0.f, 0.f, 0.f};
    const int nst = H / 64;
    if (ok) {
      const unsigned char* sb = R.gu + s * R.gu_pitch;
      for (int st = wg; st < nst; st += kGroupWarps) {
        const __half* xr = x16 + col_tok * H + st * 64 + t4 * 16;
        const uint4 b01 = *reinterpret_cast<const uint4*>(xr);
        const uint4 b23 = *reinterpret_cast<const uint4*>(xr + 8);
        const uint4 ng4 = *reinterpret_cast<const uint4*>(sb + st * 512 + lane * 16);
        const uint2 gsc = *reinterpret_cast<const uint2*>(sb + 8 * H + st * 64 + g * 8);
        const uint4 nu4 = *reinterpret_cast<const uint4*>(sb + 9 * H + st * 512 + lane * 16);
        const uint2 usc = *reinterpret_cast<const uint2*>(sb + 17 * H + st * 64 + g * 8);
        supertile_mma(accg, ng4, gsc, b01, b23, fmt, lut);
        supertile_mma(accu, nu4, usc, b01, b23, fmt, lut);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&R.empty_gu[s]);
    float4* dst = reinterpret_cast<float4*>(red + (warp * 32 + lane) * 8);
    dst[0] = make_float4(accg[0], accg[1], accg[2], accg[3]);
    dst[1] = make_float4(accu[0], accu[1], accu[2], accu[3]);
    named_sync(1 + grp, kGroupWarps * 32);
    if (wg == 0) {
      float gsum[4] = {0.f, 0.f, 0.f, 0.f}, usum[4] = {0.f, 0.f, 0.f, 0.f};
      for (int w = 0; w < kGroupWarps; ++w) {
        const float4* src = reinterpret_cast<const float4*>(red + ((grp * kGroupWarps + w) * 32 + lane) * 8);
        const float4 p = src[0], q = src[1];
        gsum[0] += p.x; gsum[1] += p.y; gsum[2] += p.z; gsum[3] += p.w;
        usum[0] += q.x; usum[1] += q.y; usum[2] += q.z; usum[3] += q.w;
      }
      if (tagged) {
        // one token (column 0: lanes with t4 = 0 hold rows g and g + 8): rows
        // g, g + 1, g + 8, g + 9 sit at B-fragment positions p .. p + 3 (g
        // even), written as two tagged words; the relaxed chunk count below
        // tells the readers when to look, the tags what they may take
        const uint32_t q0 = __half_as_ushort(__float2half_rn(silu(gsum[0]) * usum[0]));
        const uint32_t q2 = __half_as_ushort(__float2half_rn(silu(gsum[2]) * usum[2]));
        const uint32_t q1 = __shfl_down_sync(0xffffffffu, q0, 4), q3 = __shfl_down_sync(0xffffffffu, q2, 4);
        if (t4 == 0 && (g & 1) == 0) {
          unsigned long long* dst = a.htag + (size_t)xi * (I / 2) + frag_pos(strip * 16 + g) / 2;
          const unsigned long long tg = (unsigned long long)htag_v << 32;
          st_relaxed_u64(dst, tg | (q1 << 16) | q0);
          st_relaxed_u64(dst + 1, tg | (q3 << 16) | q2);
        }
        // a count per 64-wide chunk of I tells the readers when to look; it
        // carries no release ordering (no fence here): a reader that gets
        // ahead of the words sees an older tag and reads them again
        __syncwarp();
        if (lane == 0) red_relaxed_add(&cnt_cur[((size_t)xi * (NS / 4) + strip / 4) * kCntPad], 1u);
      } else {
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const int rowin = (cc < 2) ? g : g + 8;
          const int col = 2 * t4 + (cc & 1);
          if (col < tk.cnt)
            a.h16[(size_t)(tk.poff + col) * I + frag_pos(strip * 16 + rowin)] =
                __float2half_rn(silu(gsum[cc]) * usum[cc]);
        }
        // the warp's h stores happen before lane 0's release through the warp
        // barrier (no per-thread fence: the release covers them); one count
        // per strip on the expert's counter
        __syncwarp();
        if (lane == 0) red_release_add(&cnt_cur[(size_t)xi * (NS / 4) * kCntPad], 1u);
      }
    }
    named_sync(1 + grp, kGroupWarps * 32);
  };



  // ---- routing, redundantly in every CTA
  unsigned long long* tokmask = reinterpret_cast<unsigned long long*>(sm + PL.regA);
  const TopkScratch TS = carve_topk(sm + PL.regA + al128((size_t)E * 8));
  unsigned long long* sel = TS.sel;  // [T][kMaxTopK] selections in rank order
  // Early path (one token, every expert resident): the experts start right
  // after the selection; a warp with no gate/up or down role finishes the
  // softmax, the combine mapping and the statistics meanwhile.
  const bool early = ONE || T == 1;
  const int fin_warp = R.gs < kMaxGuStages ? R.gs * kGroupWarps : 0;
  for (int e = tid; e < E; e += kThreads) tokmask[e] = 0ull;
  if (tid < kMaxT) TS.nsurv[tid] = 0;
  if (c == 0)  // the other parity's counters, for the next call
    for (int i = tid; i < a.cnt_stride / kCntPad; i += kThreads) cnt_next[(size_t)i * kCntPad] = 0u;
  if (tid == 0) {
    // all G CTAs of this call published: the counter reaches call * G
    // (it only grows; the comparison survives wrap-around)
    const uint32_t want = s_dseq * (uint32_t)G;
    int spins = 0;
    while ((int32_t)(ld_relaxed_u32(a.pub) - want) < 0) {
      if (((++spins) & 63) == 0 && global_ns() > deadline) {
        set_error(a, MOE_ERR_TIMEOUT);
        break;
      }
    }
  }
  __syncthreads();
  {
    // warps per token: 16, 8, 4 or 2 for T = 1, 2, 3-4, 5-8; each warp takes a
    // contiguous range of E / wpt experts, cpl per lane (e = base + lane + 32 j)
    const int wpt = T == 1 ? 16 : (T == 2 ? 8 : (T <= 4 ? 4 : 2));
    const int t = warp / wpt, wt = warp % wpt;
    const int range = (E + wpt - 1) / wpt;
    const int cpl = (range + 31) / 32;
    const int base = wt * range;
    if (t < T) {
      const unsigned long long* words = tagged_logits + (size_t)t * E;
      unsigned long long* lw = TS.list + warp * kListStride;
      if (ONE || cpl == 1)
        warp_best<1>(words, E, k, base, range, tag, lw, TS.len + warp, a, deadline);
      else if (cpl <= 2)
        warp_best<2>(words, E, k, base, range, tag, lw, TS.len + warp, a, deadline);
      else if (cpl <= 4)
        warp_best<4>(words, E, k, base, range, tag, lw, TS.len + warp, a, deadline);
      else if (cpl <= 8)
        warp_best<8>(words, E, k, base, range, tag, lw, TS.len + warp, a, deadline);
      else
        warp_best<16>(words, E, k, base, range, tag, lw, TS.len + warp, a, deadline);
    }
    __syncthreads();
    if (t < T) keep_survivors(TS, t, warp, wpt, k);
    __syncthreads();
    if (t < T) rank_survivors(TS, t, wpt, wt * 32 + lane, k);
    __syncthreads();
    if (warp < T && !early) finish_topk(sel + warp * kMaxTopK, k, L, tokmask, warp, c == 0, a);
  }
  __syncthreads();
  // union of the selected experts (ascending) and pair offsets, from the
  // T*k selected pairs: entry p is the first of its expert when no earlier
  // token selected it.  One token: the union is the selection itself (in rank
  // order on the early path, known as soon as the merge ends).
  if (early) {
    if (tid < k) {
      const int e = word_expert(sel[tid]);
      L.u_expert[tid] = e;
      L.u_off[tid] = tid;
      L.u_slot[tid] = e;
      L.u_wait[tid] = 0u;
      L.pair_token[tid] = 0;
    }
    if (tid == 0) {
      L.u_off[k] = k;
      s_nunion = k;
      s_nmiss = 0;
    }
  } else if (!ONE && T == 1) {
    if (tid < k) {
      const int e = L.s_idx[tid];
      L.u_expert[tid] = e;
      L.u_off[tid] = tid;
      L.u_slot[tid] = e;  // all-resident slot; the pool path overwrites it
      L.u_wait[tid] = 0u;
      L.pair_token[tid] = 0;
      L.tk_u[tid] = tid;
      L.tk_pos[tid] = 0;
    }
    if (tid == 0) {
      L.u_off[k] = k;
      s_nunion = k;
    }
  } else if (!ONE) {
    const int P = T * k;
    int first = 0, ue = 0, po = 0, pos = 0, e = 0, t = 0;
    if (tid < P) {
      e = L.s_idx[tid];
      t = tid / k;
      const unsigned long long below = tokmask[e] & ((1ull << t) - 1ull);
      first = below == 0ull;
      pos = __popcll(below);
      for (int q = 0; q < P; ++q) {
        const int eq = L.s_idx[q];
        if (eq < e) {
          ++po;
          ue += (tokmask[eq] & ((1ull << (q / k)) - 1ull)) == 0ull;
        }
      }
    }
    const int n_u = __syncthreads_count(first);
    if (tid < P) {
      if (first) {
        L.u_expert[ue] = e;
        L.u_off[ue] = po;
        L.u_slot[ue] = e;
        L.u_wait[ue] = 0u;
      }
      L.pair_token[po + pos] = t;
      L.tk_u[tid] = ue;
      L.tk_pos[tid] = pos;
    }
    if (tid == 0) {
      L.u_off[n_u] = P;
      s_nunion = n_u;
    }
  }
  __syncthreads();
  const int n_union = s_nunion;
  // slot hit check: identity when every expert is resident, else LRU on the
  // double-buffered pool state (every CTA derives the same victims)
  const int S = a.n_slots;
  int32_t* nxt_slot = pool_state + (size_t)((seq + 1u) & 1u) * (E + 2 * S);
  int32_t* nxt_owner = nxt_slot + E;
  uint32_t* nxt_stamp = reinterpret_cast<uint32_t*>(nxt_owner + S);
  if (ONE || !a.pool) {
    if (tid == 0 && !early) s_nmiss = 0;  // the early path set it before the barrier above
  } else {
    // pool scratch in region A after the routing lists: per slot owner, stamp
    // and candidate key; per union entry its miss number; the ranked victims
    // the step's tables (slot_s, own_s, stp_s) arrived during the routing;
    // region A after the routing lists holds the candidate keys, each union
    // entry's miss number and the ranked victims
    unsigned long long* key_s = reinterpret_cast<unsigned long long*>(
        sm + PL.regA + al128((size_t)E * 8) + (size_t)4 * kWarps * kMaxTopK * 8);
    int* miss_no = reinterpret_cast<int*>(key_s + S);
    int* victim = miss_no + PL.umax + 2;
    __shared__ int s_ncand;
    cp_async_wait_all();
    __syncthreads();
    // this CTA's slice of the next state starts as a copy of the current one
    // (read now, stored after the decision)
    const int e0 = (int)((long long)c * E / G), e1 = (int)((long long)(c + 1) * E / G);
    const int q0 = (int)((long long)c * S / G), q1 = (int)((long long)(c + 1) * S / G);
    const int ce = e0 + tid, cq = q0 + tid;
    const int cp_slot = ce < e1 ? slot_s[ce] : 0;
    const int cp_owner = cq < q1 ? own_s[cq] : 0;
    const int cp_stamp = cq < q1 ? (int)stp_s[cq] : 0;
    for (int u = tid; u < n_union; u += kThreads) {
      L.u_slot[u] = slot_s[L.u_expert[u]];
      L.u_wait[u] = 0u;
    }
    if (tid == 0) s_ncand = 0;
    __syncthreads();
    // misses in ascending expert order get numbers 0, 1, ... (the union is
    // in that order, except for one token, whose union is in rank order)
    if (warp == 0) {
      if (early) {  // n_union = k <= 32: one entry per lane
        const bool m = lane < n_union && L.u_slot[lane] < 0;
        const int me = lane < n_union ? L.u_expert[lane] : INT_MAX;
        const unsigned b = __ballot_sync(0xffffffffu, m);
        int r = 0;
        for (int j = 0; j < n_union; ++j) r += ((b >> j) & 1u) && L.u_expert[j] < me;
        if (m) miss_no[lane] = r;
        if (lane == 0) s_nmiss = __popc(b);
      } else {
        int base = 0;
        for (int u0 = 0; u0 < n_union; u0 += 32) {
          const int u = u0 + lane;
          const bool m = u < n_union && L.u_slot[u] < 0;
          const unsigned b = __ballot_sync(0xffffffffu, m);
          if (m) miss_no[u] = base + __popc(b & ((1u << lane) - 1u));
          base += __popc(b);
        }
        if (lane == 0) s_nmiss = base;
      }
    }
    __syncthreads();
    const int nm = s_nmiss;
    if (nm > 0) {
      // candidates: empty slots first (ascending), then slots whose expert this
      // call does not use, least recently used first, ties to the lower slot
      for (int q = tid; q < S; q += kThreads) {
        const int ow = own_s[q];
        const uint32_t stp = stp_s[q];
        // the token masks are filled later on the one-token path: there the
        // union (k entries) says which experts this call uses
        bool used = false;
        if (early) {
          for (int j = 0; j < n_union; ++j) used |= L.u_expert[j] == ow;
        } else {
          used = ow >= 0 && tokmask[ow] != 0ull;
        }
        const bool elig = ow < 0 || !used;
        key_s[q] = elig ? (((unsigned long long)(ow >= 0) << 44) | ((unsigned long long)stp << 12) | (unsigned long long)q)
                        : ~0ull;
        if (elig) atomicAdd(&s_ncand, 1);
      }
      __syncthreads();
      // the i-th best candidate slot is the i-th miss's victim
      for (int q = tid; q < S; q += kThreads) {
        const unsigned long long kq = key_s[q];
        if (kq == ~0ull) continue;
        int r = 0;
        for (int j = 0; j < S; ++j) r += key_s[j] < kq;
        if (r < PL.umax) victim[r] = q;
      }
      __syncthreads();
      if (nm > s_ncand && tid == 0) set_error(a, MOE_ERR_STATE);  // configure forbids this
      for (int u = tid; u < n_union; u += kThreads)
        if (L.u_slot[u] < 0) {
          const int i = miss_no[u];
          L.u_slot[u] = (i < s_ncand) ? victim[i] : 0;  // 0 keeps addresses in bounds on error
          L.u_wait[u] = seq;
        }
      __syncthreads();
      // CTA 0 rings the host doorbell as soon as the misses are placed
      if (c == 0 && tid == 0) {
        const uint32_t head0 = a.st->ring_head;
        for (int u = 0; u < n_union; ++u)
          if (L.u_wait[u] != 0u) {  // entries in ascending expert order
            volatile RingEntry* re = &a.hm->ring[(head0 + (uint32_t)miss_no[u]) % kRingSize];
            re->seq = seq;
            re->expert = L.u_expert[u];
            re->slot = L.u_slot[u];
            re->served = a.pull ? 1u : 0u;
          }
        __threadfence_system();
        a.st->ring_head = head0 + (uint32_t)nm;
        *reinterpret_cast<volatile uint32_t*>(&a.hm->head) = head0 + (uint32_t)nm;
        __threadfence_system();
      }
    }
    // next state: every CTA writes its slice (copy, then this step's changes)
    if (ce < e1) nxt_slot[ce] = cp_slot;
    if (cq < q1) {
      nxt_owner[cq] = cp_owner;
      nxt_stamp[cq] = (uint32_t)cp_stamp;
    }
    __syncthreads();
    for (int u = tid; u < n_union; u += kThreads) {
      const int e = L.u_expert[u], q = L.u_slot[u];
      if (q >= q0 && q < q1) nxt_stamp[q] = seq;
      if (L.u_wait[u] != 0u) {
        const int old = own_s[q];  // an evicted expert is never selected now
        if (old >= e0 && old < e1) nxt_slot[old] = -1;
        if (q >= q0 && q < q1) nxt_owner[q] = e;
        if (e >= e0 && e < e1) nxt_slot[e] = q;
      }
    }
  }
  if (c == 0 && tid == (early ? fin_warp * 32 : 0)) {
    // stores and reductions only: nothing here waits for the (possibly cold) counters
    a.st->step = seq;
    a.st->dstep = s_dseq;
    a.st->n_union = n_union;
    a.st->n_miss = s_nmiss;
    atomicAdd(&a.st->forwards, 1ull);
    atomicAdd(&a.st->hits, (unsigned long long)(n_union - s_nmiss));
    atomicAdd(&a.st->misses, (unsigned long long)s_nmiss);
  }
  if (!early) __syncthreads();  // the early path's union was published by the barrier above
  if (early && warp == fin_warp) finish_topk(sel, k, L, tokmask, 0, c == 0, a, true);

  // ---- experts
  const int n_ex = NSh + n_union;
  const int n_gu_tasks = n_ex * NS;
  const int n_my = c < n_gu_tasks ? (n_gu_tasks - c + G - 1) / G : 0;
  if (is_prod) {
    P.n_gu = n_my;
    P.n_dn = has_dn ? n_ex : 0;
    P.routed = true;
    pump(P, X);
  }
  // gate/up: group grp owns ring stage grp and takes this CTA's tasks
  // m = grp, grp + gs, ... in order (a stage's uses are consumed in order by
  // one group, so parity waits never alias a later use)
  {
    const int grp = warp / kGroupWarps;
    if (grp < R.gs)
      for (int m = grp; m < n_my; m += R.gs) gateup_task(m);
  }
  // Missed experts read from host memory: the warps with no gate/up group
  // (and no producer lane) pull this CTA's down strips of the first ds
  // entries now, while the gate/up phase runs; the down strips do not
  // depend on h, so the host-link round trip leaves the down phase.
  const int pw0 = R.gs * kGroupWarps, npw = kProdWarp - pw0;
  if (!ONE && has_dn && a.pull && warp >= pw0 && warp < kProdWarp) {
    for (int xi = warp - pw0; xi < n_ex && xi < R.ds; xi += npw) {
      const Task tk = task_of(a, L, xi, NSh);
      if (!tk.src) continue;
      const size_t off = (size_t)down_base(H, I) + (size_t)c * R.dn_bytes;
      pull_strip(tk.src + off, const_cast<uint8_t*>(tk.base) + off, R.dn + xi * R.dn_pitch, R.dn_bytes, lane, 32);
      __syncwarp();
      if (lane == 0) mbar_arrive(&R.full_dn[xi]);
    }
  }
  // every gate/up copy must be issued before the block barrier below: a
  // group may still be waiting for one that only the producer can issue
  if (is_prod) {
    int spins = 0;
    while (P.m < P.n_gu) {
      pump(P, X);
      if (((++spins) & 31) == 0 && (global_ns() > deadline || dev_error(a))) break;
    }
  }
  // down: warp w takes expert entries w, w + 16, ...
  float* zbuf = reinterpret_cast<float*>(sm + PL.regA);  // [xi][32 lanes][4]
  __syncthreads();  // region A holds routing scratch until here
  // This CTA's gate/up weights are consumed and HBM idles through the rest
  // of the layer: warm L2 with what the next layer's kernel loads first (its
  // router rows and shared-expert strips for this CTA's index) and with this
  // CTA's share of the next layer's listed hot experts.
  if (a.nx_W_r && tid == kThreads - 1) {
    if (nrows > 0) prefetch_l2(a.nx_W_r + (size_t)r0 * H, (uint32_t)(nrows * H * 4));
    if (a.nx_shared) {
      if (c < NS) prefetch_l2(a.nx_shared + (size_t)c * R.gu_bytes, (uint32_t)R.gu_bytes);
      if (has_dn) prefetch_l2(a.nx_shared + down_base(H, I) + (size_t)c * R.dn_bytes, (uint32_t)R.dn_bytes);
    }
    const int parts = NS + H / 16;
    const int32_t* table = nullptr;
    if (a.nx_pool_state) {
      const uint32_t nseq = (uint32_t)ld_cg_i32(reinterpret_cast<const int*>(&a.nx_st->step)) + 1u;
      table = a.nx_pool_state + (size_t)(nseq & 1u) * (E + 2 * a.nx_S);
    }
    for (int u = c; u < a.nx_n_hot * parts; u += G) {
      const int e = __ldg(a.nx_hot + u / parts), pt = u % parts;
      const int slot = table ? ld_cg_i32(table + e) : e;
      if (slot < 0) continue;
      const uint8_t* base = a.nx_arena + (int64_t)slot * a.blob;
      if (pt < NS)
        prefetch_l2(base + (size_t)pt * R.gu_bytes, (uint32_t)R.gu_bytes);
      else
        prefetch_l2(base + down_base(H, I) + (size_t)(pt - NS) * R.dn_bytes, (uint32_t)R.dn_bytes);
    }
  }
  if (has_dn && warp < R.ds) {
    // warp w owns down stage w: entries w, w + ds, ... in order
    const int nst = I / 64;
    // the h rows of an entry are staged in this warp's slice of the (now idle)
    // gate/up ring with one round of 16-byte copies when they fit; rows padded
    // by 16 bytes so the eight token columns fall in different banks
    const int hstride = I + 8;
    const size_t hb_cap = ((size_t)R.gs * R.gu_pitch / (size_t)R.ds) / ((size_t)hstride * 2);
    const int hb_rows = hb_cap < (size_t)T ? (int)hb_cap : T;
    __half* hbuf = reinterpret_cast<__half*>(R.gu + (size_t)warp * hb_rows * hstride * 2);
    for (int xi = warp; xi < n_ex; xi += R.ds) {
      const Task tk = task_of(a, L, xi, NSh);
      const int s = xi % R.ds;
      if (!tagged) {
        // more tokens: the expert's counter first (its strips stream in
        // meanwhile), then every chunk at once below
        const uint32_t* cnt_x = cnt_cur + (size_t)xi * nst * kCntPad;
        if (lane == 0) {
          int spins = 0;
          while (ld_acquire_gpu_u32(&cnt_x[0]) < (uint32_t)NS) {
            if (is_prod) pump(P, X);
            if (((++spins) & 15) == 0) {
              if (global_ns() > deadline) { set_error(a, MOE_ERR_TIMEOUT); break; }
              if (dev_error(a)) break;
            }
            // no __nanosleep here: a sleeping warp was measured to wake up
            // microseconds late now and then, which delayed the whole layer
          }
        }
        __syncwarp();
      }
      if (!ONE && tk.src && !(xi < R.ds && npw > 0)) {  // a miss not pulled early: read it now
        const size_t off = (size_t)down_base(H, I) + (size_t)c * R.dn_bytes;
        pull_strip(tk.src + off, const_cast<uint8_t*>(tk.base) + off, R.dn + s * R.dn_pitch, R.dn_bytes, lane, 32);
        __syncwarp();
        if (lane == 0) mbar_arrive(&R.full_dn[s]);
      }
      const bool staged = !tagged && tk.cnt <= hb_rows;
      if (staged) {  // all of h, one round of copies, before the strip wait
        const int per_row = I / 8;
        for (int o = lane; o < tk.cnt * per_row; o += 32) {
          const int r = o / per_row, cc = o - r * per_row;
          cp_async16(hbuf + r * hstride + cc * 8, a.h16 + (size_t)(tk.poff + r) * I + cc * 8);
        }
        cp_async_wait_all();
        __syncwarp();
      }
      const bool ok = __all_sync(0xffffffffu, wait_full(&R.full_dn[s], (xi / R.ds) & 1, deadline, is_prod, P, X));
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      const unsigned char* sb = R.dn + s * R.dn_pitch;
      const int gsel = (g < tk.cnt) ? g : 0;
      if (!tagged && ok) {
        if (staged) {
          const __half* hb = hbuf + gsel * hstride + t4 * 16;
#pragma unroll 4
          for (int st = 0; st < nst; ++st) {
            const uint4 b01 = *reinterpret_cast<const uint4*>(hb + st * 64);
            const uint4 b23 = *reinterpret_cast<const uint4*>(hb + st * 64 + 8);
            const uint4 nb = *reinterpret_cast<const uint4*>(sb + st * 512 + lane * 16);
            const uint2 scv = *reinterpret_cast<const uint2*>(sb + 8 * I + st * 64 + g * 8);
            supertile_mma(acc, nb, scv, b01, b23, fmt, lut);
          }
        } else {
          const int hrow = tk.poff + gsel;
#pragma unroll 2
          for (int st = 0; st < nst; ++st) {
            const __half* hr = a.h16 + (size_t)hrow * I + st * 64 + t4 * 16;
            const uint4 b01 = __ldcg(reinterpret_cast<const uint4*>(hr));
            const uint4 b23 = __ldcg(reinterpret_cast<const uint4*>(hr + 8));
            const uint4 nb = *reinterpret_cast<const uint4*>(sb + st * 512 + lane * 16);
            const uint2 scv = *reinterpret_cast<const uint2*>(sb + 8 * I + st * 64 + g * 8);
            supertile_mma(acc, nb, scv, b01, b23, fmt, lut);
          }
        }
      }
      if (tagged && ok) {
        // One token: the chunk counters say which 64-wide chunks of h look
        // complete; their words are read with one round trip (lane j holds
        // word j of each chunk) and a chunk counts once all 32 words carry
        // this call's tag.  The down product then runs on the leading valid
        // chunks while later gate/up strips are still being computed
        // elsewhere; each lane's B fragment comes from its 8 words by
        // shuffles.  The accumulation order is one pass over K, as on the
        // other paths.
        constexpr int kBatch = 8;  // chunks read per round trip
        const uint32_t* cnt_x = cnt_cur + (size_t)xi * nst * kCntPad;
        const unsigned long long* hw = a.htag + (size_t)xi * (I / 2) + lane;
        int done = 0, spins = 0;
        while (done < nst) {
          const int ch = done + lane;
          const bool rdy = ch < nst && ld_relaxed_u32(&cnt_x[(size_t)ch * kCntPad]) >= 4u;
          const unsigned m = __ballot_sync(0xffffffffu, rdy);
          int nr = (m == 0xffffffffu) ? 32 : __ffs(~m) - 1;  // chunks counted complete, in order from done
          nr = nr < kBatch ? nr : kBatch;
          int nv = 0;
          if (nr > 0) {
            unsigned long long wv[kBatch];
#pragma unroll
            for (int j = 0; j < kBatch; ++j) wv[j] = (j < nr) ? ld_relaxed_u64(hw + (size_t)(done + j) * 32) : 0ull;
#pragma unroll
            for (int j = 0; j < kBatch; ++j)
              if (j < nr && nv == j && __all_sync(0xffffffffu, (uint32_t)(wv[j] >> 32) == htag_v)) nv = j + 1;
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
              if (j < nv) {
                const uint32_t lo = (uint32_t)wv[j];  // two fp16 values at positions 2 * lane, 2 * lane + 1
                uint4 b01, b23;
                b01.x = __shfl_sync(0xffffffffu, lo, t4 * 8 + 0);
                b01.y = __shfl_sync(0xffffffffu, lo, t4 * 8 + 1);
                b01.z = __shfl_sync(0xffffffffu, lo, t4 * 8 + 2);
                b01.w = __shfl_sync(0xffffffffu, lo, t4 * 8 + 3);
                b23.x = __shfl_sync(0xffffffffu, lo, t4 * 8 + 4);
                b23.y = __shfl_sync(0xffffffffu, lo, t4 * 8 + 5);
                b23.z = __shfl_sync(0xffffffffu, lo, t4 * 8 + 6);
                b23.w = __shfl_sync(0xffffffffu, lo, t4 * 8 + 7);
                const int st = done + j;
                const uint4 nb = *reinterpret_cast<const uint4*>(sb + st * 512 + lane * 16);
                const uint2 scv = *reinterpret_cast<const uint2*>(sb + 8 * I + st * 64 + g * 8);
                supertile_mma(acc, nb, scv, b01, b23, fmt, lut);
              }
            }
            done += nv;
          }
          if (nv == 0) {
            if (is_prod) pump(P, X);
            bool stop = false;
            if (((++spins) & 15) == 0) {
              if (global_ns() > deadline) {
                if (lane == 0) set_error(a, MOE_ERR_TIMEOUT);
                stop = true;
              } else if (dev_error(a)) {
                stop = true;
              }
            }
            // no __nanosleep here: a sleeping warp was measured to wake up
            // microseconds late now and then, which delayed the whole layer
            if (__any_sync(0xffffffffu, stop)) break;
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&R.empty_dn[s]);
      *reinterpret_cast<float4*>(zbuf + (xi * 32 + lane) * 4) = make_float4(acc[0], acc[1], acc[2], acc[3]);
    }
  }
  // no async copy may outlive the CTA: the producer drains what it still owes
  if (is_prod) {
    int spins = 0;
    while (P.m < P.n_gu || P.d < P.n_dn) {
      pump(P, X);
      if (((++spins) & 31) == 0 && (global_ns() > deadline || dev_error(a))) break;
    }
    note_wait_end(P, X);  // a wait cut short by an error or the deadline
  }
  __syncthreads();
  if (has_dn) {
    for (int q = tid; q < T * 16; q += kThreads) {
      const int t = q >> 4, row = q & 15;
      // all loads first, then the fma chain in the selection order (ascending
      // expert index), the same summation order as before
      float wv[kMaxTopK], zv[kMaxTopK];
#pragma unroll
      for (int j = 0; j < kMaxTopK; ++j) {
        wv[j] = 0.f;
        zv[j] = 0.f;
        if (j < k) {
          const int xi = NSh + L.tk_u[t * k + j];
          const int col = L.tk_pos[t * k + j];
          const int lz = (row & 7) * 4 + (col >> 1), rz = (row >> 3) * 2 + (col & 1);
          wv[j] = L.s_w[t * k + j];
          zv[j] = zbuf[(xi * 32 + lz) * 4 + rz];
        }
      }
      float v = 0.f;
#pragma unroll
      for (int j = 0; j < kMaxTopK; ++j)
        if (j < k) v = fmaf(wv[j], zv[j], v);
      if (NSh) {
        const int col = t;
        const int lz = (row & 7) * 4 + (col >> 1), rz = (row >> 3) * 2 + (col & 1);
        v += zbuf[(0 * 32 + lz) * 4 + rz];
      }
      a.y[(size_t)t * H + c * 16 + row] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
    }
  }
}

size_t g_decode_smem_limit = 0;  // dynamic shared memory the kernel may use
bool g_decode_pdl = false;       // the driver takes cooperative launches with programmatic serialization

__global__ void pdl_probe_kernel() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

cudaLaunchConfig_t decode_config(dim3 grid, dim3 block, size_t smem, cudaStream_t s, cudaLaunchAttribute (&attr)[2],
                                 bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cfg;
}

}  // namespace

size_t decode_smem_bytes(int H, int I, int E, int k, int T, int G, bool pool) {
  return make_plan(H, I, E, k, T, G, g_decode_smem_limit, pool).total;
}

cudaError_t decode_configure() {
  int dev = 0, optin = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  cudaFuncAttributes fa;
  const void* variants[3] = {(const void*)decode_kernel<true, 0>, (const void*)decode_kernel<false, 0>,
                             (const void*)decode_kernel<false, 1>};
  size_t st = 0;
  for (const void* f : variants) {
    e = cudaFuncGetAttributes(&fa, f);
    if (e != cudaSuccess) return e;
    st = fa.sharedSizeBytes > st ? fa.sharedSizeBytes : st;
  }
  const size_t limit = (size_t)optin - st;
  for (const void* f : variants) {
    e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)limit);
    if (e != cudaSuccess) return e;
  }
  g_decode_smem_limit = limit;
  // whether a cooperative launch may also carry programmatic serialization:
  // two launches of an empty kernel on a private stream (a refusal is a
  // launch-configuration error, which does not stick to the context)
  static int probed = 0;
  if (!probed) {
    probed = 1;
    cudaStream_t ps;
    e = cudaStreamCreateWithFlags(&ps, cudaStreamNonBlocking);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = decode_config(dim3(1), dim3(32), 0, ps, attr, true);
    bool ok = cudaLaunchKernelEx(&cfg, pdl_probe_kernel) == cudaSuccess;
    ok = ok && cudaLaunchKernelEx(&cfg, pdl_probe_kernel) == cudaSuccess;
    (void)cudaGetLastError();
    e = cudaStreamSynchronize(ps);
    cudaStreamDestroy(ps);
    if (e != cudaSuccess) return e;
    g_decode_pdl = ok;
  }
  return cudaSuccess;
}

bool decode_supported(int H, int I, int E, int k, int T, int G, bool pool) {
  if (T > kMaxT || E > kMaxE || k > kMaxTopK) return false;
  if ((E + G - 1) / G > 8) return false;  // router: two warps per row, 16 warps
  if (H / 16 > G) return false;            // down: one 16-row output strip per CTA
  return g_decode_smem_limit > 0 && decode_smem_bytes(H, I, E, k, T, G, pool) <= g_decode_smem_limit;
}

cudaError_t launch_decode(const LayerArgs& a, unsigned long long* tagged_logits, int32_t* pool_state, int G,
                          cudaStream_t s) {
  // Programmatic serialization only when the kernel waits on nothing outside
  // the stream: a pooled layer whose misses the host copy server serves timed
  // out now and then with it (the wait ran into its deadline), so that case
  // keeps the plain stream order.
  const bool pdl = g_decode_pdl && (!a.pool || a.pull);
  cudaLaunchAttribute attr[2];
  const size_t smem = decode_smem_bytes(a.H, a.I, a.E, a.k, a.T, G, a.pool != 0);
  cudaLaunchConfig_t cfg = decode_config(dim3(G), dim3(kThreads), smem, s, attr, pdl);
  // one token per call, linear weights: one key per lane in top-k
  const bool one = a.T == 1 && !a.pool && a.E <= 16 * 32 && a.fmt == 0;
  if (one) return cudaLaunchKernelEx(&cfg, decode_kernel<true, 0>, a, tagged_logits, pool_state, g_decode_smem_limit);
  if (a.fmt == 1)
    return cudaLaunchKernelEx(&cfg, decode_kernel<false, 1>, a, tagged_logits, pool_state, g_decode_smem_limit);
  return cudaLaunchKernelEx(&cfg, decode_kernel<false, 0>, a, tagged_logits, pool_state, g_decode_smem_limit);
}

}  // namespace moe
