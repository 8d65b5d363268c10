// Routing entry point that allocates nothing (moe_route_noalloc).
//
// Some callers cannot call cudaMalloc: code that runs inside a host
// framework which owns every device allocation through its own pool, code
// loaded into a process whose device memory is fully reserved up front, or
// code called while another component holds the allocator.  This entry
// point gives them the router + top-k step without any allocation: its
// scratch (the T x E logits and the CTAs' arrival ticket) lives in the
// file-scope device array below, which every GPU that loads this library
// holds until the process exits.  The caller passes only inputs and outputs.
//
// The array is shared by every call on a device and keeps the last call's
// contents; the ticket is cleared once at set-up and reset to zero by the
// last CTA of every call.  Calls that overlap on the GPU (two streams at
// once) race on it: serialize them.
#include <cfloat>
#include <climits>
#include <cstdint>
#include <mutex>

#include "moe.h"
#include "moe_internal.h"

namespace {

constexpr int kNaMaxLogits = 65536;  // T * E limit: 256 KiB of fp32 logits
constexpr int kNaTicketWords = 64;   // one 256-byte line for the ticket
constexpr int kNaRows = 4;
constexpr int kNaThreads = 256;
constexpr int kNaChunk = 8;
constexpr int kNaVec = moe::kMaxHidden / 256;
constexpr int kNaMaxDevices = 64;

static __device__ __align__(256) float g_noalloc_scratch[kNaTicketWords + kNaMaxLogits];

std::mutex g_setup_mu;
float* g_scratch_ptr[kNaMaxDevices] = {};

__global__ void __launch_bounds__(kNaThreads) route_noalloc_kernel(const float* __restrict__ W_r,
                                                                   const float* __restrict__ bias,
                                                                   const uint16_t* __restrict__ x, int T, int H,
                                                                   int E, int k, int32_t* topk_idx, float* topk_w,
                                                                   float* scratch) {
  extern __shared__ __align__(16) float sm[];
  unsigned int* ticket = reinterpret_cast<unsigned int*>(scratch);
  float* logits = scratch + kNaTicketWords;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int row = blockIdx.x * kNaRows + (warp >> 1), half = warp & 1, q4 = H / 8;
  const bool row_ok = row < E;
  float4 w[kNaVec];
  const float4* wrow = reinterpret_cast<const float4*>(W_r + (size_t)(row_ok ? row : 0) * H) + half * q4;
#pragma unroll
  for (int i = 0; i < kNaVec; ++i) {
    const int q = lane + 32 * i;
    w[i] = (row_ok && q < q4) ? __ldg(wrow + q) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float* xs = sm;
  float* red = sm + kNaChunk * H;
  for (int t0 = 0; t0 < T; t0 += kNaChunk) {
    const int nt = min(kNaChunk, T - t0);
    __syncthreads();
    const uint32_t* xsrc = reinterpret_cast<const uint32_t*>(x + (size_t)t0 * H);
    for (int i = tid; i < nt * H / 2; i += kNaThreads) {
      const uint32_t v = xsrc[i];
      xs[2 * i] = __uint_as_float(v << 16);
      xs[2 * i + 1] = __uint_as_float(v & 0xFFFF0000u);
    }
    __syncthreads();
    for (int tt = 0; tt < nt; ++tt) {
      const float4* xr = reinterpret_cast<const float4*>(xs + tt * H) + half * q4;
      float s = 0.f;
#pragma unroll
      for (int i = 0; i < kNaVec; ++i) {
        const int q = lane + 32 * i;
        if (q < q4) {
          const float4 xv = xr[q];
          s = fmaf(w[i].x, xv.x, s);
          s = fmaf(w[i].y, xv.y, s);
          s = fmaf(w[i].z, xv.z, s);
          s = fmaf(w[i].w, xv.w, s);
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      if (lane == 0) red[warp * kNaChunk + tt] = s;
    }
    __syncthreads();
    if (tid < kNaRows * nt) {
      const int r = tid / nt, tt = tid % nt, e = blockIdx.x * kNaRows + r;
      if (e < E)
        logits[(size_t)(t0 + tt) * E + e] =
            (red[(2 * r) * kNaChunk + tt] + red[(2 * r + 1) * kNaChunk + tt]) + (bias ? __ldg(bias + e) : 0.f);
    }
  }
  __threadfence();
  __syncthreads();
  __shared__ unsigned int s_ticket;
  if (tid == 0) s_ticket = atomicAdd(ticket, 1u);
  __syncthreads();
  if (s_ticket != gridDim.x - 1) return;
  __threadfence();
  // last CTA: top-k per token (warp per token), ties to the lower index
  float* lrow = sm;  // [8 warps][E]
  for (int t = warp; t < T; t += kNaThreads / 32) {
    float* lr = lrow + warp * E;
    for (int e = lane; e < E; e += 32) lr[e] = __ldcg(&logits[(size_t)t * E + e]);
    __syncwarp();
    int sel[moe::kMaxTopK];
    float selv[moe::kMaxTopK];
    for (int r = 0; r < k; ++r) {
      float bv = -FLT_MAX;
      int bi = INT_MAX;
      for (int e = lane; e < E; e += 32) {
        const float v = lr[e];
        if (v > bv || (v == bv && e < bi)) { bv = v; bi = e; }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
      }
      if (bi == INT_MAX) bi = 0;
      if (lane == (bi & 31)) lr[bi] = __int_as_float(0x7fc00000);
      sel[r] = bi;
      selv[r] = bv;
      __syncwarp();
    }
    if (lane == 0) {
      const float m = selv[0];
      for (int i = 1; i < k; ++i) {
        const int ki = sel[i];
        const float kv = selv[i];
        int j = i - 1;
        while (j >= 0 && sel[j] > ki) { sel[j + 1] = sel[j]; selv[j + 1] = selv[j]; --j; }
        sel[j + 1] = ki;
        selv[j + 1] = kv;
      }
      float z = 0.f;
      for (int j = 0; j < k; ++j) z += expf(selv[j] - m);
      for (int j = 0; j < k; ++j) {
        topk_idx[t * k + j] = sel[j];
        topk_w[t * k + j] = expf(selv[j] - m) / z;
      }
    }
    __syncwarp();
  }
  if (tid == 0) *ticket = 0u;  // ready for the next call
}

size_t noalloc_smem(int H, int E) {
  const size_t a = sizeof(float) * ((size_t)kNaChunk * H + 8 * kNaChunk);
  const size_t b = sizeof(float) * 8 * (size_t)E;
  return a > b ? a : b;
}

// Once per device, with that device current: resolve the array's device
// address (the host-side symbol is only a stand-in), clear the ticket and
// raise the kernel's shared-memory limit.  Nothing is allocated.
moe_status_t setup_device(int dev, float** out) {
  std::lock_guard<std::mutex> g(g_setup_mu);
  if (g_scratch_ptr[dev]) {
    *out = g_scratch_ptr[dev];
    return MOE_OK;
  }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
  if (cudaMemset(p, 0, sizeof(float) * kNaTicketWords) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaFuncSetAttribute(route_noalloc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)noalloc_smem(moe::kMaxHidden, moe::kMaxExperts)) != cudaSuccess)
    return MOE_ERR_CUDA;
  g_scratch_ptr[dev] = (float*)p;
  *out = (float*)p;
  return MOE_OK;
}

}  // namespace

extern "C" MOE_API moe_status_t moe_route_noalloc(const float* router_w, const float* router_bias, const void* x_bf16,
                                                  int32_t T, int32_t hidden, int32_t n_experts, int32_t top_k,
                                                  int32_t* topk_idx, float* topk_w, void* cuda_stream) {
  if (!router_w || !x_bf16 || !topk_idx || !topk_w) return MOE_ERR_INVALID_ARG;
  if (((uintptr_t)router_w & 15) || ((uintptr_t)x_bf16 & 3) || ((uintptr_t)topk_idx & 3) || ((uintptr_t)topk_w & 3))
    return MOE_ERR_INVALID_ARG;
  if (T < 1 || hidden < 64 || hidden % 64 || n_experts < 1 || top_k < 1 || top_k > n_experts)
    return MOE_ERR_INVALID_ARG;
  if (T > moe::kMaxTokens || hidden > moe::kMaxHidden || n_experts > moe::kMaxExperts || top_k > moe::kMaxTopK ||
      (int64_t)T * n_experts > kNaMaxLogits)
    return MOE_ERR_UNSUPPORTED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNaMaxDevices) return MOE_ERR_CUDA;
  float* scratch = nullptr;
  const moe_status_t st = setup_device(dev, &scratch);
  if (st != MOE_OK) return st;
  const int grid = (n_experts + kNaRows - 1) / kNaRows;
  route_noalloc_kernel<<<grid, kNaThreads, noalloc_smem(hidden, n_experts), (cudaStream_t)cuda_stream>>>(
      router_w, router_bias, (const uint16_t*)x_bf16, T, hidden, n_experts, top_k, topk_idx, topk_w, scratch);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
