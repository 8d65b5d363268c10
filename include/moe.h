/*
 * moe.h - C ABI of the GB300 (sm_103a) quantized mixture-of-experts FFN layer.
 *
 * One call of moe_forward runs the MoE FFN layer of Qwen3.8-Flash-Next-style
 * decode on one GPU: router GEMV, softmax and top-k selection, an in-stream
 * check of whether each selected expert is resident in a VRAM expert-slot
 * pool (misses served from pinned host RAM after a host doorbell: read by
 * the kernel itself or copied by a host thread, never dropped), 4-bit
 * block-quantized gate/up/down expert GEMVs with SiLU gating, and the
 * routing-weighted combine.
 *
 * Sources for what the layer is and how residency works:
 *  - Betelgeuse news page ("Betelgeuse: RTX 3060 12GB + 16GB 内存跑 Qwen 3.8
 *    Flash Next, 22 tok/s 不丢专家"), section 机制 (48 layers, 512 routed experts
 *    per layer, 10 routed + 1 shared per token; table rows 显存: VRAM expert
 *    slots, 调度: an in-stream kernel decides hits on the GPU and rings a host
 *    doorbell only on a miss, 内存/盘: misses are served from host RAM) and
 *    section "bit-exact 的确切含义" (top-10 routing never changed; an expert
 *    read/DMA failure is reported as an error instead of continuing with
 *    zero weights).
 *  - Basalt README, section "Memory floors": refuse a memory setting that
 *    does not fit instead of shrinking it.
 *  - halogen-flash-server README, section "Bring your own GGUF": the packed
 *    block-quantized values are repacked losslessly into the kernels' layout.
 *
 * Conventions shared by every call:
 *  - Every call returns a moe_status_t; nothing throws or exits.
 *  - "device" pointers are CUDA device addresses on the layer's device;
 *    "host" pointers are ordinary process memory.
 *  - bf16 tensors are raw IEEE bfloat16 bit patterns, row-major.
 *  - A layer object is not re-entrant: issue its calls from one host thread
 *    and on one stream at a time.
 *  - Asynchronous failures (a slot copy that failed or timed out) are
 *    sticky: the next moe_forward returns MOE_ERR_STATE and moe_get_stats
 *    reports the original code; the affected y is undefined, never silently
 *    zero.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,   /* a pointer, size or shape is invalid */
  MOE_ERR_UNSUPPORTED = 2,   /* valid but outside what this build implements */
  MOE_ERR_OUT_OF_MEMORY = 3, /* an allocation or a caller arena is too small */
  MOE_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed */
  MOE_ERR_COPY = 5,          /* a host->slot expert copy failed */
  MOE_ERR_TIMEOUT = 6,       /* the device gave up waiting for a slot copy */
  MOE_ERR_STATE = 7,         /* the layer holds a sticky error from an earlier call */
  MOE_ERR_DEVICE = 8         /* a device-side check failed (e.g. activation outside fp16 range) */
} moe_status_t;

typedef struct moe_layer moe_layer_t; /* opaque, library-owned */

/*
 * Layer description.  Shapes: H = hidden, E = routed experts, k = routed
 * experts per token, I = expert intermediate size.  Weight format: each
 * expert is one canonical blob [W_gate I x H][W_up I x H][W_down H x I];
 * each R x K matrix is a nibble plane (R*K/2 bytes; element i of a row in
 * byte i/2, low nibble for even i; stored value u = q + 8, q in [-8, 7])
 * followed by a scale plane (R*K/32 binary16 scales, one per block of 32
 * consecutive elements along K).  Weight = scale * (u - 8).
 */
typedef struct {
  int32_t hidden;          /* H: multiple of 64, 64..4096 */
  int32_t n_experts;       /* E: 1..4096 */
  int32_t top_k;           /* k: 1..min(E, 16) */
  int32_t n_shared;        /* 0 or 1 shared expert (weight 1, outside the softmax) */
  int32_t inter;           /* I: multiple of 64, 64..4096 */
  int32_t qblock;          /* quantization block; must be 32 */
  int32_t max_tokens;      /* largest T a moe_forward call may pass: 1..8192 (above 64: H % 128 == 0) */
  int32_t device;          /* CUDA device ordinal */
  const float* router_w;   /* device, fp32 [E][H] row-major; caller-owned, must outlive the layer */
  const float* router_bias;/* device, fp32 [E] (per-expert logit bias), or NULL for none; caller-owned */
  const uint8_t* experts;  /* host, E canonical blobs back to back; read during create only */
  const uint8_t* shared;   /* host, one canonical blob, or NULL when n_shared == 0; read during create only */
  int32_t weight_format;   /* MOE_FMT_LINEAR4 (0) or MOE_FMT_CODEBOOK4 (1), for every blob of the layer */
} moe_layer_desc_t;

/*
 * Weight formats.  Both store, per matrix, the nibble plane and the scale
 * plane described above (one fp16 scale d per block of 32 along K); they
 * differ in what a stored nibble u means:
 *   MOE_FMT_LINEAR4    weight = d * (u - 8)
 *   MOE_FMT_CODEBOOK4  weight = d * C[u], C = {-127, -90, -69, -53, -39, -27,
 *                      -16, -5, 5, 16, 27, 39, 53, 69, 90, 127}: the standard
 *                      normal distribution's quantiles at (u + 1/2) / 16
 *                      scaled to +-127 and rounded, a non-linear 16-entry
 *                      table per block scale (halogen-flash-server README,
 *                      section "Bring your own GGUF", lists such lookup
 *                      formats).  Runs on the fused decode kernel only
 *                      (max_tokens <= 8); its lookups cost more issue slots
 *                      than the linear format's arithmetic decode.
 */
enum { MOE_FMT_LINEAR4 = 0, MOE_FMT_CODEBOOK4 = 1 };

/* Bytes of one expert blob (canonical and repacked sizes are equal). */
MOE_API size_t moe_expert_bytes(int32_t hidden, int32_t inter);

/*
 * The lossless repack between the canonical blob and the GPU layout the
 * kernels stream (halogen-flash-server README, section "Bring your own GGUF":
 * the file's quantized values are moved into the kernels' layout, not
 * requantized).  Host-only; needs no GPU.  Both buffers hold
 * moe_expert_bytes(hidden, inter) bytes; hidden and inter multiples of 64.
 * The GPU layout groups 16 output rows into strips and orders each strip's
 * nibbles and block scales so that every lane of a warp reads its
 * mma.m16n8k16 A-fragment nibbles with one 16-byte load and its two block
 * scales with one 8-byte load; moe_unpack_expert inverts it exactly.
 * Errors: INVALID_ARG.
 */
MOE_API moe_status_t moe_repack_expert(const uint8_t* canonical, int32_t hidden, int32_t inter, uint8_t* gpu_layout);
MOE_API moe_status_t moe_unpack_expert(const uint8_t* gpu_layout, int32_t hidden, int32_t inter, uint8_t* canonical);

/*
 * Create a layer.  Validates the description, repacks every expert blob
 * losslessly into the GPU layout held in a library-owned pinned host master
 * copy (the source of slot copies), uploads the shared expert, and
 * allocates the layer's device scratch.  The layer has no expert slots
 * until moe_slot_pool_configure.
 * Errors: INVALID_ARG (NULL/out-of-range fields, unknown weight format),
 * UNSUPPORTED (qblock != 32, shapes this build does not implement, or the
 * codebook format with max_tokens > 8), OUT_OF_MEMORY, CUDA.
 * On error *out is NULL and nothing stays allocated.
 */
MOE_API moe_status_t moe_layer_create(const moe_layer_desc_t* desc, moe_layer_t** out);

/*
 * Give the layer its VRAM expert-slot pool: n_slots slots of
 * moe_expert_bytes() each, carved from the caller's device arena
 * (e.g. a torch.empty buffer; caller-owned, must outlive the layer or the
 * next configure call, 256-byte aligned).
 *  - n_slots == E: every expert resident.  All blobs are copied into the
 *    arena now (synchronously); no host traffic during moe_forward.
 *  - min(E, min(max_tokens, 8)*k) <= n_slots < E: the pool starts empty (or
 *    as moe_slot_pool_seed sets it); misses are served from the pinned host
 *    master copy (moe_set_miss_service).  Eviction is LRU over forward
 *    calls of at most 8 tokens: the misses of a call are filled in ascending
 *    expert index, taking empty slots first (ascending), then slots whose
 *    expert the call does not use, least recently used first (ties to the
 *    lower slot).
 *    With max_tokens > 64 a prefill call (T > 64) lends the pool's last
 *    slots (Basalt README, section "Prompt chunks"): its scratch occupies the
 *    last ceil(scratch / blob) slots, up to 16 slots below them stage the
 *    touched experts the pool does not hold below the lent range (copied
 *    from the master copy, in waves), and afterwards every lent slot gets
 *    its expert back: the pool's table, stamps and contents are unchanged
 *    and the call does not count as a step.  Such a call synchronizes its
 *    stream once (after routing, to read which experts it touches), so it
 *    cannot be captured in a CUDA graph.  Calls of 9..64 tokens are refused
 *    (UNSUPPORTED).
 * Errors: INVALID_ARG (NULL arena, n_slots out of range), OUT_OF_MEMORY
 * when n_slots * moe_expert_bytes() > arena_bytes, or when a pool cannot
 * lend the prefill scratch plus one staging slot (the request is never
 * shrunk), UNSUPPORTED (n_slots < E on a layer the fused decode kernel does
 * not take: more than 16 x SMs hidden rows, more than min(1024, 8 x SMs)
 * experts, or a shared-memory plan that does not fit; the layer keeps its
 * previous configuration), CUDA.  After a CUDA or OUT_OF_MEMORY failure
 * past the argument checks the layer is unconfigured (moe_forward answers
 * STATE) until a configure succeeds.
 */
MOE_API moe_status_t moe_slot_pool_configure(moe_layer_t* layer, int32_t n_slots, void* arena_dev, size_t arena_bytes);

/*
 * Seed a configured pool from a hot-expert profile (Betelgeuse news page,
 * section 机制: the pool starts from a profile of hot experts instead of
 * cold).  Replaces the pool's contents: experts_host[i] (host int32,
 * distinct, 0 <= e < E) is copied now, synchronously, into slot i, last used
 * before the next call; slots n .. n_slots-1 are empty.  Eviction then
 * proceeds as described above.  Synchronizes the device.
 * Errors: INVALID_ARG (NULL layer, experts NULL with n > 0, n < 0 or
 * n > n_slots, an expert out of range or repeated), STATE (no pool: the
 * layer is unconfigured or every expert is resident; or the layer holds an
 * error), CUDA (the pool is then empty: it is emptied before any slot is
 * overwritten).
 */
MOE_API moe_status_t moe_slot_pool_seed(moe_layer_t* layer, const int32_t* experts_host, int32_t n);

/*
 * y = MoE(x) for T tokens, enqueued on `cuda_stream` (a cudaStream_t; NULL =
 * the legacy default stream).  Stream-ordered and asynchronous; safe to
 * capture in a CUDA graph once the pool is configured.
 *   x_bf16_dev:  device bf16 [T][H], 16-byte aligned (|x| < 65504; larger is MOE_ERR_DEVICE)
 *   y_bf16_dev:  device bf16 [T][H], written (must not alias x)
 *   topk_idx_dev: device int32 [T][k] or NULL: the selected experts of each
 *                token in ascending expert index
 *   topk_w_dev:  device fp32 [T][k] or NULL: their routing weights (softmax
 *                over all E renormalised over the selected k)
 * Selection: the k largest logits (router_w x + router_bias), ties to the
 * lower index.  Logits are compensated (double-float) fp32 dot products,
 * within about 1e-13 of the exact value (bound 5e-10 at H = 2048), so the
 * selection equals a binary64 evaluation's unless two logits lie closer
 * than that; NaN logits rank below every number.  Output: y = sum over the selected experts, in ascending
 * index, of w_j * FFN_j(x), plus FFN_shared(x), accumulated in fp32 and
 * rounded once to bf16 (round to nearest even).
 * Execution by T: T <= 8 one fused kernel (slot pool or all resident) when
 * the layer fits it (see moe_slot_pool_configure), else the three kernels
 * below; 9..64 three kernels (all resident); 65..max_tokens the prefill path
 * (all resident): grouped GEMMs on the tensor cores with fp16 operands
 * (dequantized weights d*q and activations) and fp32 accumulation
 * (halogen-flash-server README, section "Measured": prefill is compute-bound).
 * A token's y depends only on its own x on the first two paths; the prefill
 * path meets the same tolerances but not bit-equality with them.
 * Errors (synchronous): INVALID_ARG (T out of 1..max_tokens, NULL x/y),
 * STATE (no pool configured, or a sticky error), UNSUPPORTED (9 <= T <= 64
 * with a slot pool of fewer than E slots; larger T lend slots, see
 * moe_slot_pool_configure), CUDA (launch failure).
 */
MOE_API moe_status_t moe_forward(moe_layer_t* layer, const void* x_bf16_dev, int32_t T, void* y_bf16_dev,
                                 int32_t* topk_idx_dev, float* topk_w_dev, void* cuda_stream);

/*
 * One layer of a pre-norm stack in one call: residual add and RMSNorm
 * (as moe_residual_rmsnorm below), then y = MoE(xhat) (as moe_forward).
 * The source pages stack 48 such layers but do not spell out the norm; this
 * is the plainest pre-norm: no learned weight, eps from the caller (the
 * stacked workload uses 1e-6).
 *   x_out = bf16(x + y_prev)                      (y_prev may be NULL: x_out = x)
 *   xhat  = bf16(x_out / sqrt(mean(x_out^2) + eps))   (no learned weight)
 *   y     = MoE(xhat)
 * x, y_prev, x_out, xhat: device bf16 [T][H], 16-byte aligned; x_out may be
 * NULL (not written); xhat is always written.  y, topk_idx_dev, topk_w_dev as
 * in moe_forward.  No output may overlap an input or another output.
 * With T <= 8 the residual and the norm run in the fused kernel's prologue
 * (every CTA normalises the T rows itself: no launch between layers), with
 * the same summation order as moe_residual_rmsnorm, so x_out, xhat and y are
 * bit-identical to moe_residual_rmsnorm followed by moe_forward.  Larger T
 * launch exactly that pair.
 * Errors: as moe_forward; INVALID_ARG also for NULL x/xhat, eps < 0 or NaN,
 * misalignment or overlap.
 */
MOE_API moe_status_t moe_forward_norm(moe_layer_t* layer, const void* x_bf16_dev, const void* y_prev_bf16_dev,
                                      int32_t T, float eps, void* x_out_bf16_dev, void* xhat_bf16_dev,
                                      void* y_bf16_dev, int32_t* topk_idx_dev, float* topk_w_dev, void* cuda_stream);

/*
 * Residual + RMSNorm between the layers of a stack (the pre-norm described
 * at moe_forward_norm), enqueued on the stream:
 *   x_out   = bf16(x + y)                 (y may be NULL: x_out = x)
 *   xhat    = bf16(x_out / sqrt(mean(x_out^2) + eps))   (no learned weight)
 * All device bf16 [T][H], 16-byte aligned, H a multiple of 8; x_out may alias
 * x; xhat must not alias the others.  Per token, 256 threads take 8-element
 * chunks (thread v: chunks v, v + 256, ...), accumulate the squares in
 * element order, then a warp butterfly and the 8 warp sums in order.
 * Errors: INVALID_ARG (NULL x/xhat, bad sizes, eps < 0 or NaN, misalignment,
 * aliasing), CUDA.
 */
MOE_API moe_status_t moe_residual_rmsnorm(const void* x_bf16_dev, const void* y_bf16_dev, int32_t T, int32_t hidden,
                                          float eps, void* x_out_bf16_dev, void* xhat_bf16_dev, void* cuda_stream);

typedef struct {
  uint64_t forwards;     /* moe_forward steps the device has completed routing for */
  uint64_t hits;         /* distinct selected experts found resident, summed over steps */
  uint64_t misses;       /* distinct selected experts copied in from host RAM */
  uint64_t h2d_bytes;    /* bytes copied host -> slots */
  uint64_t wait_ns;      /* device time spent waiting for slot copies */
  int32_t n_slots;       /* configured pool size (0 = none) */
  int32_t error;         /* sticky error code (moe_status_t), MOE_OK if none */
  uint64_t rechecks;     /* prefill path: experts whose logit was recomputed exactly because
                            the tensor-core logits put them within the GEMM's error bound of
                            a token's k-th/(k+1)-th boundary, summed over calls */
} moe_stats_t;

/* Synchronize the layer's device and copy stream, then report counters.
 * Returns the sticky error code if one is set (stats still filled). */
MOE_API moe_status_t moe_get_stats(moe_layer_t* layer, moe_stats_t* out);

/*
 * Copy the miss log (one (step, expert, slot) int32 triple per miss, in the
 * order served, step counted from 1 per layer) into out[0 .. 3*max).
 * *n receives the total number logged.  Synchronizes like moe_get_stats.
 */
MOE_API moe_status_t moe_get_miss_log(moe_layer_t* layer, int32_t* out, int64_t max, int64_t* n);

/* Device-side wait limit for a slot copy (default 2 s); 0 restores the default. */
MOE_API moe_status_t moe_set_wait_timeout_ns(moe_layer_t* layer, uint64_t ns);

/*
 * How a pooled layer serves a miss (T <= 8 calls).  Both ring the host
 * doorbell and log the miss (Betelgeuse news page, section 机制, rows 调度
 * and 内存/盘); they differ in who moves the bytes.  Results are
 * bit-identical in both modes.
 *  MOE_MISS_SM_PULL (default): the kernel's own threads read the missed
 *    expert from the pinned master copy over the coherent host link, use it
 *    at once and write it into its slot for later calls; the copy server
 *    only logs the doorbell entry, so nothing in the call waits on the host.
 *  MOE_MISS_COPY_ENGINE: the kernel waits; the copy server copies the
 *    expert into its slot (cudaMemcpyAsync on the layer's copy streams) and
 *    publishes the slot's ready flag with a stream memory operation.  The
 *    copy streams are created at the device's highest priority: streams of
 *    different priorities never share a hardware work queue, so a slot copy
 *    is never queued behind compute work that itself waits for the kernel
 *    that waits for the copy.  The kernel's wait stays bounded
 *    (moe_set_wait_timeout_ns); if it runs out, the call ends with
 *    MOE_ERR_TIMEOUT (no hang, no dropped miss).
 * Applies to calls launched afterwards; a CUDA graph captured earlier keeps
 * the mode it was captured with.  Synchronizes the device.
 * Errors: INVALID_ARG (null layer or unknown mode), CUDA.
 */
enum { MOE_MISS_COPY_ENGINE = 0, MOE_MISS_SM_PULL = 1 };
MOE_API moe_status_t moe_set_miss_service(moe_layer_t* layer, int32_t mode);

/*
 * Name the layer that runs after this one (the next layer of a stack, or
 * the next layer object a caller cycles to), so that every later fused
 * decode call of `layer` (T <= 8) spends the end of its run, when its own
 * weights are consumed and HBM would idle, warming L2 with what the next
 * layer's call loads first: its router rows and shared expert, and the
 * listed experts (hot_experts[0 .. n_hot), e.g. a hot-expert profile, the
 * Betelgeuse news page's section 机制) where they are resident in the next
 * layer's slots.  A cache hint only: outputs, routing and the pool's
 * decisions never depend on it; a listed expert that is not selected costs
 * its bytes of HBM traffic.  next = NULL (and n_hot = 0) removes the link.
 * next must have the layer's shapes and device, and must stay alive while
 * linked; the addresses it warms are those of next's configuration at each
 * call (a CUDA graph keeps those it was captured with: capture again after
 * reconfiguring next).  Synchronizes the device.
 * Errors: INVALID_ARG (null layer, mismatched next, n_hot outside 0..64,
 * an expert out of range), CUDA.
 */
MOE_API moe_status_t moe_set_next_layer(moe_layer_t* layer, moe_layer_t* next, const int32_t* hot_experts,
                                        int32_t n_hot);

/*
 * Host-side fault injection for tests (no GPU fault is ever raised):
 *   fail_copy_n > 0: the n-th copy (counted from 1 after this call) is not
 *                    issued; it is reported to the device as failed, which
 *                    makes the step end with MOE_ERR_COPY.
 *   pause:           nonzero stops the copy server from serving the ring
 *                    (the device wait then times out), zero resumes it.
 */
MOE_API moe_status_t moe_debug_copy_faults(moe_layer_t* layer, int64_t fail_copy_n, int32_t pause);

/* Destroy: synchronizes, stops the copy server, frees library memory. NULL-safe. */
MOE_API void moe_destroy(moe_layer_t* layer);

/*
 * Router + top-k for callers that cannot allocate device memory (no
 * counterpart in the source pages; see moe_noalloc.cu for which callers).
 * Computes, like moe_forward's routing step, the logits router_w x +
 * router_bias, the k largest per token (ties to the lower index) in
 * ascending expert order, and their softmax weights renormalised over the
 * k, writing topk_idx [T][k] (int32) and topk_w [T][k] (fp32), on the
 * current device and the given stream.
 *   router_w: device fp32 [E][H], 16-byte aligned; router_bias: device fp32
 *   [E] or NULL; x_bf16: device bf16 [T][H], 16-byte aligned.
 * The logits are the compensated ones of moe_forward, computed in the same
 * order, so the selection and weights are bit-identical to its routing.
 * Scratch: a fixed 512 KiB device array inside the library (T * E <= 65536
 * 64-bit router keys plus an arrival ticket), shared by every call on a
 * device and kept by it until the process exits.  Nothing is allocated,
 * ever.  The first call on a device sets the array up (resolves its device
 * address and the kernel's shared-memory limit): make that first call
 * before any stream capture.  Calls that overlap on the GPU race on the
 * array: serialize them.
 * Errors: INVALID_ARG (NULL or misaligned pointers, bad shapes),
 * UNSUPPORTED (T > 64, k > 16, H > 4096, E > 4096 or T * E > 65536),
 * CUDA (set-up or launch failure).
 */
MOE_API moe_status_t moe_route_noalloc(const float* router_w, const float* router_bias, const void* x_bf16, int32_t T,
                                       int32_t hidden, int32_t n_experts, int32_t top_k, int32_t* topk_idx,
                                       float* topk_w, void* cuda_stream);

MOE_API const char* moe_status_string(moe_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
