// Routing entry point that allocates nothing (moe_route_noalloc).
//
// Some callers cannot call cudaMalloc: code that runs inside a host
// framework which owns every device allocation through its own pool, code
// loaded into a process whose device memory is fully reserved up front, or
// code called while another component holds the allocator.  This entry
// point gives them the router + top-k step without any allocation: its
// scratch (the T x E router keys and the CTAs' arrival ticket) lives in the
// file-scope device array below, which every GPU that loads this library
// holds until the process exits.  The caller passes only inputs and outputs.
//
// The array is shared by every call on a device and keeps the last call's
// contents; the ticket starts at zero with the module and is reset to zero
// by the last CTA of every call.  Calls that overlap on the GPU (two streams at
// once) race on it: serialize them.
#include <cstdint>
#include <mutex>

#include "moe.h"
#include "moe_internal.h"
#include "moe_route.cuh"

namespace {

constexpr int kNaMaxLogits = 65536;  // T * E limit: 512 KiB of 64-bit router keys
constexpr int kNaTicketWords = 32;   // one 256-byte line for the ticket
constexpr int kNaRows = 2;           // expert rows per CTA: four warps per row, one per quarter of H
constexpr int kNaThreads = 256;
constexpr int kNaChunk = 8;
constexpr int kNaVec = moe::kMaxHidden / 512;
constexpr int kNaMaxDevices = 64;

static __device__ __align__(256) unsigned long long g_noalloc_scratch[kNaTicketWords + kNaMaxLogits];

std::mutex g_setup_mu;
unsigned long long* g_scratch_ptr[kNaMaxDevices] = {};

// Warps of the last CTA that select top-k, each staging one token's E rank
// words in shared memory.
__host__ __device__ inline int na_topk_warps(int E) { return E <= 2048 ? 8 : 4; }

__global__ void __launch_bounds__(kNaThreads) route_noalloc_kernel(const float* __restrict__ W_r,
                                                                   const float* __restrict__ bias,
                                                                   const uint16_t* __restrict__ x, int T, int H,
                                                                   int E, int k, int32_t* topk_idx, float* topk_w,
                                                                   unsigned long long* scratch) {
  extern __shared__ __align__(16) unsigned char sm[];
  unsigned int* ticket = reinterpret_cast<unsigned int*>(scratch);
  unsigned long long* keys = scratch + kNaTicketWords;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int row = blockIdx.x * kNaRows + (warp >> 2), q = warp & 3, n4 = H / 16;
  const bool row_ok = row < E;
  float4 w[kNaVec];
  const float4* wq = reinterpret_cast<const float4*>(W_r + (size_t)(row_ok ? row : 0) * H + q * (H / 4));
#pragma unroll
  for (int i = 0; i < kNaVec; ++i) {
    const int j = lane + 32 * i;
    w[i] = (row_ok && j < n4) ? __ldg(wq + j) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float* xs = reinterpret_cast<float*>(sm);
  moe::DF* red = reinterpret_cast<moe::DF*>(xs + kNaChunk * H);
  for (int t0 = 0; t0 < T; t0 += kNaChunk) {
    const int nt = min(kNaChunk, T - t0);
    __syncthreads();
    moe::stage_x_f32<kNaThreads>(x + (size_t)t0 * H, nt * H, xs, tid);
    __syncthreads();
    for (int tt = 0; tt < nt; ++tt) {
      // the compensated router in the library's canonical order (moe_route.cuh)
      const float4* xr = reinterpret_cast<const float4*>(xs + tt * H + q * (H / 4));
      moe::DF d{0.f, 0.f};
#pragma unroll
      for (int i = 0; i < kNaVec; ++i) {
        const int j = lane + 32 * i;
        if (j < n4) moe::dot2_acc4(d, w[i], xr[j]);
      }
      d = moe::warp_sum_df(d);
      if (lane == 0) red[warp * kNaChunk + tt] = d;
    }
    __syncthreads();
    if (tid < kNaRows * nt) {
      const int r = tid / nt, tt = tid % nt, e = blockIdx.x * kNaRows + r;
      if (e < E) {
        const moe::DF* pr = red + (4 * r) * kNaChunk + tt;
        keys[(size_t)(t0 + tt) * E + e] =
            moe::logit_key(pr[0], pr[kNaChunk], pr[2 * kNaChunk], pr[3 * kNaChunk], bias ? __ldg(bias + e) : 0.f);
      }
    }
  }
  __threadfence();
  __syncthreads();
  __shared__ unsigned int s_ticket;
  if (tid == 0) s_ticket = atomicAdd(ticket, 1u);
  __syncthreads();
  if (s_ticket != gridDim.x - 1) return;
  __threadfence();
  // last CTA: top-k per token (warp per token) by key, ties to the lower
  // index.  Every expert has a key (NaN logits rank below every number), so
  // each token always gets k distinct experts.
  const int nw = na_topk_warps(E);
  if (warp < nw)
    for (int t = warp; t < T; t += nw) {
      unsigned long long* lr = reinterpret_cast<unsigned long long*>(sm) + (size_t)warp * E;
      for (int e = lane; e < E; e += 32) lr[e] = moe::rank_word(__ldcg(&keys[(size_t)t * E + e]), e);
      __syncwarp();
      int sel[moe::kMaxTopK];
      float selv[moe::kMaxTopK];
      moe::warp_select_k(lr, E, k, sel, selv);
      if (lane == 0) moe::softmax_ascending(sel, selv, k, topk_idx + t * k, topk_w + t * k);
      __syncwarp();
    }
  __syncthreads();
  if (tid == 0) *ticket = 0u;  // ready for the next call
}

size_t noalloc_smem(int H, int E) {
  const size_t a = sizeof(float) * (size_t)kNaChunk * H + sizeof(moe::DF) * 8 * kNaChunk;
  const size_t b = sizeof(unsigned long long) * (size_t)na_topk_warps(E) * E;
  return a > b ? a : b;
}

// Once per device, with that device current: resolve the array's device
// address (the host-side symbol is only a stand-in) and raise the kernel's
// shared-memory limit.  Nothing is allocated, and nothing is written: the
// array starts zeroed when the module loads, and every call leaves the
// ticket at zero.
moe_status_t setup_device(int dev, unsigned long long** out) {
  std::lock_guard<std::mutex> g(g_setup_mu);
  if (g_scratch_ptr[dev]) {
    *out = g_scratch_ptr[dev];
    return MOE_OK;
  }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
  size_t most = 0;
  for (int e : {2048, moe::kMaxExperts}) {
    const size_t v = noalloc_smem(moe::kMaxHidden, e);
    most = v > most ? v : most;
  }
  if (cudaFuncSetAttribute(route_noalloc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)most) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  g_scratch_ptr[dev] = (unsigned long long*)p;
  *out = (unsigned long long*)p;
  return MOE_OK;
}

}  // namespace

extern "C" MOE_API moe_status_t moe_route_noalloc(const float* router_w, const float* router_bias, const void* x_bf16,
                                                  int32_t T, int32_t hidden, int32_t n_experts, int32_t top_k,
                                                  int32_t* topk_idx, float* topk_w, void* cuda_stream) {
  if (!router_w || !x_bf16 || !topk_idx || !topk_w) return MOE_ERR_INVALID_ARG;
  if (((uintptr_t)router_w & 15) || ((uintptr_t)x_bf16 & 15) || ((uintptr_t)topk_idx & 3) || ((uintptr_t)topk_w & 3))
    return MOE_ERR_INVALID_ARG;
  if (T < 1 || hidden < 64 || hidden % 64 || n_experts < 1 || top_k < 1 || top_k > n_experts)
    return MOE_ERR_INVALID_ARG;
  if (T > moe::kMaxTokens || hidden > moe::kMaxHidden || n_experts > moe::kMaxExperts || top_k > moe::kMaxTopK ||
      (int64_t)T * n_experts > kNaMaxLogits)
    return MOE_ERR_UNSUPPORTED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNaMaxDevices) return MOE_ERR_CUDA;
  unsigned long long* scratch = nullptr;
  const moe_status_t st = setup_device(dev, &scratch);
  if (st != MOE_OK) return st;
  const int grid = (n_experts + kNaRows - 1) / kNaRows;
  route_noalloc_kernel<<<grid, kNaThreads, noalloc_smem(hidden, n_experts), (cudaStream_t)cuda_stream>>>(
      router_w, router_bias, (const uint16_t*)x_bf16, T, hidden, n_experts, top_k, topk_idx, topk_w, scratch);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
