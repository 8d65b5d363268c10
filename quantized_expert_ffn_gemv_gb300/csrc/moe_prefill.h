// Prefill path (T > 64): per-call scratch and launch entry (moe_prefill.cu).
#pragma once

#include "moe_internal.h"

namespace moe {

constexpr int kPfN = 128;               // tokens per GEMM chunk (the MMA's N, at most)
constexpr int kMaxPrefillTokens = 8192;  // largest T of one prefill call

// Scratch of the prefill kernels.  Pairs are (token, rank) assignments; the
// shared expert is expert list entry E with all T tokens.
struct PrefillArgs {
  int32_t* counts;      // [E + 1] tokens per routed expert (zeroed each call)
  int32_t* offsets;     // [E + 2] first pair of each expert list entry; [NE] = total
  int32_t* chunk_off;   // [E + 2] first 128-token chunk of each entry; [NE] = total
  int32_t* n_chunks;    // [1]
  int32_t* pair_token;  // [T*k + T] token of each pair, grouped by expert
  int32_t* pair_z;      // [T*k + T] z row of each pair: t*(k+1) + rank (rank k = shared)
  __half* x16p;         // [T][H] fp16 activations, natural order
  __half* h16p;         // [T*k + T][I] fp16 h of each pair, natural order
  __half* z16;          // [T*(k+1)][H] fp16 expert outputs before the weighting
  uint32_t* bitmap;     // [E][ceil(T/32)] bit t of row e: token t selected e (cleared after use)
};

// Bytes of prefill scratch for up to Tm tokens (0 when Tm <= kMaxTokens).
size_t prefill_scratch_bytes(int H, int I, int E, int k, int Tm);
// Carve PrefillArgs from a device block of prefill_scratch_bytes() bytes.
PrefillArgs prefill_carve(void* block, int H, int I, int E, int k, int Tm);
cudaError_t prefill_configure();
cudaError_t launch_prefill(const LayerArgs& a, const PrefillArgs& p, int sm_count, cudaStream_t s);

}  // namespace moe
