// Prefill path (T > 64): per-call scratch, tensor maps and launch entry (moe_prefill.cu).
#pragma once

#include <cuda.h>

#include "moe_internal.h"

namespace moe {

constexpr int kPfN = 256;                // tokens per GEMM chunk (the MMA's N, at most)
constexpr int kSmallN = 16;              // an expert's last chunk of at most this many tokens takes the mma.sync path
constexpr int kMaxPrefillTokens = 8192;  // largest T of one prefill call

// Scratch of the prefill kernels.  Pairs are (token, rank) assignments; the
// shared expert is expert list entry E with all T tokens.
struct PrefillArgs {
  int32_t* counts;      // [E + 1] tokens per routed expert (zeroed each call)
  int32_t* offsets;     // [E + 2] first pair of each expert list entry; [NE] = total
  int32_t* chunk_off;   // [E + 2] first tensor-core chunk of each entry; [NE] = total
  int32_t* n_chunks;    // [2] tensor-core chunks, small chunks
  int4* chunk_rec;      // [max chunks] per tensor-core chunk (more than kSmallN tokens, at most kPfN):
                        //   {expert list entry, first pair, tokens, 0}
  int4* small_rec;      // [E + 1] per small chunk (an entry's last, at most kSmallN tokens): same fields
  int32_t* pair_token;  // [T*k + T] token of each pair, grouped by expert, ascending token
  int32_t* pair_z;      // [T*k + T] z row of each pair: t*(k+1) + rank (rank k = shared)
  uint32_t* bitmap;     // [E][ceil(T/32)] bit t of row e: token t selected e (zeroed each call)
  int32_t* prefix;      // [E][ceil(T/32)] set bits of row e in the words before each word
  uint16_t* w_split;    // [3][E][H] bf16 pieces of the router weights: W = W0 + W1 + W2
  float* wnorm;         // [E] Euclidean norms of the router rows (slightly rounded up)
  float* xnorm;         // [T] Euclidean norms of the call's activation rows (slightly rounded up)
  __half* x16p;         // [T][H] fp16 activations
  __half* h16p;         // [T*k + T][I] fp16 h of each pair
  __half* z16;          // [T*(k+1)][H] fp16 expert outputs before the weighting
  int words;            // ceil(max_tokens / 32): row stride of bitmap and prefix
  // Pooled layers (experts read in waves): per routed expert, where its blob
  // is for the current wave, or null (not in this wave).  Null table: every
  // expert at arena + e * blob (a resident layer).
  const uint8_t** base;
  const uint8_t** base_table;  // [E] storage for that table
  int4* wave_chunk_rec;  // [max chunks] this wave's tensor-core chunks
  int4* wave_small_rec;  // [E + 1] this wave's small chunks
  int32_t* wave_n;       // [2] their counts
};

// TMA descriptors of the router GEMM (128-byte swizzle, bf16, 64-element boxes along K).
struct PrefillMaps {
  CUtensorMap w_split;  // [3][E][H], box 64 x 128 x 1
  CUtensorMap x_bf16;   // the call's x [T][H], box 64 x 128 (encoded per call)
};

typedef CUresult (*TensorMapEncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                      const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                      CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// Bytes of prefill scratch for up to Tm tokens (0 when Tm <= kMaxTokens).
size_t prefill_scratch_bytes(int H, int I, int E, int k, int Tm);
// Carve PrefillArgs from a device block of prefill_scratch_bytes() bytes.
PrefillArgs prefill_carve(void* block, int H, int I, int E, int k, int Tm);
// The fixed tensor maps of the scratch buffers (x_bf16 is left for the call).
bool prefill_encode_maps(TensorMapEncodeFn enc, const PrefillArgs& p, int H, int I, int E, int k, int Tm,
                         PrefillMaps* m);
bool prefill_encode_x(TensorMapEncodeFn enc, const void* x, int H, int T, PrefillMaps* m);
cudaError_t prefill_configure();
cudaError_t launch_prefill(const LayerArgs& a, const PrefillArgs& p, const PrefillMaps& m, int sm_count,
                           cudaStream_t s);
// The same call in three parts, for a pooled layer whose experts come in
// waves: routing and grouping; the expert GEMMs of one wave (the chunks whose
// expert has a base in p.base, the shared expert's in wave 0); the combine.
cudaError_t launch_prefill_route(const LayerArgs& a, const PrefillArgs& p, const PrefillMaps& m, int sm_count,
                                 cudaStream_t s);
cudaError_t launch_prefill_wave(const LayerArgs& a, const PrefillArgs& p, int sm_count, bool wave0, cudaStream_t s);
cudaError_t launch_prefill_combine(const LayerArgs& a, const PrefillArgs& p, cudaStream_t s);

}  // namespace moe
