// Internal declarations shared by the CUDA library's translation units.
//
// GPU weight layout (a lossless permutation of the canonical blob, built once
// by the host repack, so that every lane's mma.sync A-fragment nibbles and
// block scales are one 16-byte and one 8-byte load):
//
//   expert = [gate/up strip 0 .. I/16-1][down strip 0 .. H/16-1]
//   gate/up strip s (16 intermediate rows, K = H):
//       [gate nibbles 8H B][gate scales H B][up nibbles 8H B][up scales H B]
//   down strip r (16 hidden rows, K = I):
//       [down nibbles 8I B][down scales I B]
//   nibbles of a 16-row strip: super-tiles of 64 k (512 B each), inside one
//     [lane 0..31][k-tile 0..3][u32]; lane = 4g + t holds for k-tile kt
//     (k0 = 64*st + 16*kt; rows g and g+8 of the strip):
//       bits  0- 3 A[g][k0+2t]     bits 16-19 A[g][k0+2t+1]
//       bits  4- 7 A[g][k0+2t+8]   bits 20-23 A[g][k0+2t+9]
//       bits  8-11 A[g+8][k0+2t]   bits 24-27 A[g+8][k0+2t+1]
//       bits 12-15 A[g+8][k0+2t+8] bits 28-31 A[g+8][k0+2t+9]
//     which are exactly the f16 A fragment of mma.m16n8k16 after the
//     magic-exponent dequantization (low nibbles of each half -> a0/a1,
//     high nibbles -> a2/a3).
//   scales of a strip: per super-tile 64 B = [g 0..7][d(g,2st) d(g+8,2st)
//     d(g,2st+1) d(g+8,2st+1)] (binary16), i.e. lane (g, t) reads 8 B.
//
// Activation rows fed to the MMA (x in fp16, h in fp16) use the matching
// B-fragment order inside every 64-element chunk: [t 0..3][kt 0..3]
// [k0+2t, k0+2t+1, k0+2t+8, k0+2t+9].
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace moe {

constexpr int kQBlock = 32;
constexpr int kMaxTokens = 64;
constexpr int kMaxTopK = 16;
constexpr int kMaxExperts = 4096;
constexpr int kMaxHidden = 4096;
constexpr int kMaxInter = 4096;
constexpr int kRingSize = 4096;
constexpr int kCntPad = 32;  // u32 per 128-byte line: each counter has a cache line of its own
constexpr uint32_t kReadyError = 0x80000000u;  // OR-ed into a ready flag when the copy failed

// Byte offsets inside one expert in GPU layout.
__host__ __device__ inline int64_t gu_strip_bytes(int H) { return 18ll * H; }
__host__ __device__ inline int64_t down_strip_bytes(int I) { return 9ll * I; }
__host__ __device__ inline int64_t down_base(int H, int I) { return (int64_t)(I / 16) * gu_strip_bytes(H); }
__host__ __device__ inline int64_t expert_bytes(int H, int I) { return 27ll * H * I / 16; }

// Position of element k of an activation row in the B-fragment order.
__host__ __device__ inline int frag_pos(int k) {
  int chunk = k >> 6, kk = k & 63, kt = kk >> 4, w = kk & 15;
  int hi = w >> 3, t = (w & 7) >> 1, e = w & 1;
  return (chunk << 6) + (t << 4) + (kt << 2) + (hi << 1) + e;
}

// Device-resident per-layer state.
// Three cache lines: the step state (read by every CTA at kernel start and
// written once per call), the sticky error (polled inside bounded waits) and
// the statistics (atomics), so that polling one never contends with writes
// to another.
struct alignas(128) DevState {
  uint32_t step;      // routing steps done; the current step's sequence number after increment
  uint32_t ticket;    // arrival counter of the route kernel's CTAs
  int32_t n_union;    // distinct routed experts of the current step
  int32_t n_miss;     // misses of the current step
  uint32_t ring_head; // doorbell entries written so far
  uint32_t dstep;     // fused decode calls so far (tags the logits they publish)
  int32_t pad0[26];
  int32_t error;      // sticky error (moe_status_t value), 0 = none
  int32_t pad1[31];
  unsigned long long forwards, hits, misses, wait_ns;
  unsigned long long rechecks;  // prefill: experts whose logit was recomputed exactly near the top-k boundary
  unsigned long long pad2[11];
};
static_assert(sizeof(DevState) == 384, "DevState: three 128-byte lines");

struct RingEntry {
  uint32_t seq;
  int32_t expert;
  int32_t slot;
  uint32_t served;  // 1: the kernel read the expert from host memory itself (log only, no copy)
};

// Pinned host memory mapped into the device address space.
struct HostMapped {
  uint32_t head;  // doorbell: number of ring entries published by the device
  uint32_t pad0[31];
  int32_t error;  // mirror of DevState::error for the host
  uint32_t pad1[31];
  RingEntry ring[kRingSize];
};

// Everything a kernel needs, passed by value.
struct LayerArgs {
  int H, E, k, I, n_shared, T;
  int n_slots, pool;  // pool = 0: every expert resident at slot == expert index
  int pull;           // pooled misses: 0 = host copy server, 1 = read by the kernel from the mapped master copy
  int fmt;            // weight format: 0 linear 4-bit, 1 codebook (fused decode kernel only)
  const uint8_t* master;  // device address of the pinned host master copy (GPU layout, expert e at e * blob)
  const float* W_r;
  const float* bias;
  const uint8_t* arena;   // slot s at arena + s * blob
  const uint8_t* shared;  // shared expert, GPU layout
  int64_t blob;
  DevState* st;
  HostMapped* hm;  // device address of the mapped host block
  uint32_t* ready;       // [E] per slot: step whose copy has landed (host copy server)
  float* logits;        // [T][E] tensor-core router output (prefill path)
  float* wnorm;         // [E] router row norms (batched path's error bound)
  __half* x16;          // [T][H] B-fragment order
  int32_t* u_expert;    // [Umax]
  int32_t* u_slot;      // [Umax]
  int32_t* u_off;       // [Umax + 1] pair offsets
  int32_t* pair_token;  // [T*k] pairs sorted by (expert, token)
  float* pair_w;        // [T*k]
  int32_t* tk_u;        // [T*k] union index of (t, j)
  int32_t* tk_pos;      // [T*k] position of (t, j) inside its expert's pairs
  __half* h16;          // [T*k + T][I] B-fragment order; shared expert rows after the routed ones
  // Fused decode of one token with every expert resident: h of expert list
  // entry xi (0 = shared expert when present) as 64-bit words, word j =
  // (call tag << 32) | two fp16 values at B-fragment positions 2j, 2j + 1.
  // Each word is one single-copy-atomic store, so a reader that sees this
  // call's tag in it holds this call's values: the chunk counts that tell
  // readers when to look need no release fence.
  unsigned long long* htag;  // [k + 1][I / 2]
  int32_t* topk_idx;    // [T][k]
  float* topk_w;        // [T][k]
  const uint16_t* x;    // bf16 [T][H]
  uint16_t* y;          // bf16 [T][H]
  // Fused pre-norm (moe_forward_norm, fused decode kernel only): when resid is
  // set the layer input is xhat = bf16(rmsnorm(bf16(resid + y_prev))), formed
  // in the kernel's prologue; x is then unused.
  const uint16_t* resid;   // bf16 [T][H] or null
  const uint16_t* y_prev;  // bf16 [T][H] or null (no residual branch)
  uint16_t* x_out;         // bf16 [T][H] or null: bf16(resid + y_prev)
  uint16_t* xhat_out;      // bf16 [T][H]: the normalised layer input
  float eps;
  unsigned long long wait_timeout_ns;
  uint32_t* pub;        // fused decode: router publications, G per call (own 128-byte line, only grows)
  uint32_t* counters;   // [2][cnt_stride] gate/up strips done per (expert, 64-wide chunk of I), by step parity,
                        // one counter per 128-byte line
  int cnt_stride;       // (max distinct experts per call + 2) * (I / 64) * kCntPad
  // L2 warm-up for the layer that runs next (moe_set_next_layer): its router
  // rows and shared expert, and the listed experts in its resident slots.
  // A cache hint only: results never depend on it.  nx_W_r null = none.
  const float* nx_W_r;
  const uint8_t* nx_shared;
  const uint8_t* nx_arena;        // next layer's slot arena
  const int32_t* nx_pool_state;   // next layer's double-buffered slot tables, or null (all resident: slot = e)
  const DevState* nx_st;          // next layer's state (its step picks the current table)
  int nx_S;                       // next layer's slot count
  const int32_t* nx_hot;          // device [nx_n_hot] expert ids
  int nx_n_hot;
};
constexpr int kMaxHotExperts = 64;

// Launch helpers (moe_kernels.cu).  All return cudaSuccess or the launch error.
cudaError_t launch_route(const LayerArgs& a, cudaStream_t s, bool pdl);
cudaError_t launch_gateup(const LayerArgs& a, cudaStream_t s, bool pdl, int grid);
cudaError_t launch_down(const LayerArgs& a, cudaStream_t s, bool pdl, int nw);
cudaError_t launch_residual_rmsnorm(const uint16_t* x, const uint16_t* y, int T, int H, float eps, uint16_t* x_out,
                                    uint16_t* xhat, cudaStream_t s);
size_t route_smem_bytes(int H, int E);
cudaError_t configure_kernels(int H, int E);
int gateup_max_blocks_per_sm(int H);
int down_warps(int T, int k, int n_shared, int I);

// Fused single-launch decode path (moe_decode.cu), T <= 8.
size_t decode_smem_bytes(int H, int I, int E, int k, int T, int G, bool pool);
bool decode_supported(int H, int I, int E, int k, int T, int G, bool pool);
cudaError_t decode_configure();
cudaError_t launch_decode(const LayerArgs& a, unsigned long long* tagged_logits, int32_t* pool_state, int G,
                          cudaStream_t s);

}  // namespace moe
