// Host runtime behind include/moe.h: layer objects, the lossless repack into
// the GPU layout, the VRAM expert-slot pool, and the copy server that serves
// misses from the pinned host master copy.
//
// Residency design (Betelgeuse news page, section 机制): every selected
// expert is resolved on the GPU (route kernel); only a miss involves the
// host.  The device appends {seq, expert, slot} to a ring in mapped pinned
// memory and publishes the ring head; this thread polls the head, issues one
// contiguous cudaMemcpyAsync per missed expert on its own stream and then a
// stream write of `seq` into the slot's ready flag, which the expert kernels
// wait on (with a deadline).  A failed or skipped copy is written back as
// seq | kReadyError and surfaces as MOE_ERR_COPY (section "bit-exact 的确切
// 含义": a failed expert read stops with an error rather than using zeros).
#include <cuda.h>

#include <atomic>
#include <chrono>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <thread>
#include <vector>

#include "moe.h"
#include "moe_internal.h"
#include "moe_prefill.h"

using namespace moe;

namespace {

typedef CUresult (*WriteValue32Fn)(CUstream, CUdeviceptr, cuuint32_t, unsigned int);

struct DeviceGuard {
  int prev = -1;
  bool ok = false;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    ok = cudaSetDevice(dev) == cudaSuccess;
  }
  ~DeviceGuard() {
    if (prev >= 0) cudaSetDevice(prev);
  }
};

inline uint8_t nibble_at(const uint8_t* nib, int K, int r, int c) {
  return (uint8_t)((nib[(size_t)r * (K / 2) + c / 2] >> ((c & 1) * 4)) & 15);
}

// Canonical R x K matrix -> GPU-layout strips (see moe_internal.h).
void repack_matrix(const uint8_t* canon, int R, int K, uint8_t* dst, int64_t strip_stride, int64_t nib_off,
                   int64_t sc_off) {
  const uint8_t* nib = canon;
  const uint8_t* sc = canon + (size_t)R * (K / 2);
  for (int s = 0; s < R / 16; ++s) {
    uint8_t* strip = dst + s * strip_stride;
    for (int st = 0; st < K / 64; ++st) {
      for (int lane = 0; lane < 32; ++lane) {
        const int g = lane >> 2, t = lane & 3;
        const int rg = 16 * s + g, rg8 = rg + 8;
        for (int kt = 0; kt < 4; ++kt) {
          const int k0 = 64 * st + 16 * kt;
          uint32_t w = 0;
          w |= (uint32_t)nibble_at(nib, K, rg, k0 + 2 * t) << 0;
          w |= (uint32_t)nibble_at(nib, K, rg, k0 + 2 * t + 8) << 4;
          w |= (uint32_t)nibble_at(nib, K, rg8, k0 + 2 * t) << 8;
          w |= (uint32_t)nibble_at(nib, K, rg8, k0 + 2 * t + 8) << 12;
          w |= (uint32_t)nibble_at(nib, K, rg, k0 + 2 * t + 1) << 16;
          w |= (uint32_t)nibble_at(nib, K, rg, k0 + 2 * t + 9) << 20;
          w |= (uint32_t)nibble_at(nib, K, rg8, k0 + 2 * t + 1) << 24;
          w |= (uint32_t)nibble_at(nib, K, rg8, k0 + 2 * t + 9) << 28;
          std::memcpy(strip + nib_off + st * 512 + lane * 16 + kt * 4, &w, 4);
        }
      }
      for (int g = 0; g < 8; ++g) {
        const int rg = 16 * s + g, rg8 = rg + 8;
        const int b0 = 2 * st, b1 = 2 * st + 1;
        uint8_t* o = strip + sc_off + st * 64 + g * 8;
        std::memcpy(o + 0, sc + ((size_t)rg * (K / 32) + b0) * 2, 2);
        std::memcpy(o + 2, sc + ((size_t)rg8 * (K / 32) + b0) * 2, 2);
        std::memcpy(o + 4, sc + ((size_t)rg * (K / 32) + b1) * 2, 2);
        std::memcpy(o + 6, sc + ((size_t)rg8 * (K / 32) + b1) * 2, 2);
      }
    }
  }
}

// Inverse of repack_matrix.
void unpack_matrix(const uint8_t* src, int R, int K, uint8_t* canon, int64_t strip_stride, int64_t nib_off,
                   int64_t sc_off) {
  uint8_t* nib = canon;
  uint8_t* sc = canon + (size_t)R * (K / 2);
  std::memset(nib, 0, (size_t)R * (K / 2));
  for (int s = 0; s < R / 16; ++s) {
    const uint8_t* strip = src + s * strip_stride;
    for (int st = 0; st < K / 64; ++st) {
      for (int lane = 0; lane < 32; ++lane) {
        const int g = lane >> 2, t = lane & 3;
        const int rg = 16 * s + g, rg8 = rg + 8;
        for (int kt = 0; kt < 4; ++kt) {
          const int k0 = 64 * st + 16 * kt;
          uint32_t w;
          std::memcpy(&w, strip + nib_off + st * 512 + lane * 16 + kt * 4, 4);
          const int rows[8] = {rg, rg, rg8, rg8, rg, rg, rg8, rg8};
          const int cols[8] = {k0 + 2 * t, k0 + 2 * t + 8, k0 + 2 * t, k0 + 2 * t + 8,
                               k0 + 2 * t + 1, k0 + 2 * t + 9, k0 + 2 * t + 1, k0 + 2 * t + 9};
          for (int i = 0; i < 8; ++i) {
            const uint8_t v = (uint8_t)((w >> (4 * i)) & 15);
            nib[(size_t)rows[i] * (K / 2) + cols[i] / 2] |= (uint8_t)(v << ((cols[i] & 1) * 4));
          }
        }
      }
      for (int g = 0; g < 8; ++g) {
        const int rg = 16 * s + g, rg8 = rg + 8;
        const int b0 = 2 * st, b1 = 2 * st + 1;
        const uint8_t* o = strip + sc_off + st * 64 + g * 8;
        std::memcpy(sc + ((size_t)rg * (K / 32) + b0) * 2, o + 0, 2);
        std::memcpy(sc + ((size_t)rg8 * (K / 32) + b0) * 2, o + 2, 2);
        std::memcpy(sc + ((size_t)rg * (K / 32) + b1) * 2, o + 4, 2);
        std::memcpy(sc + ((size_t)rg8 * (K / 32) + b1) * 2, o + 6, 2);
      }
    }
  }
}

inline int64_t mat_bytes(int R, int K) { return (int64_t)R * (K / 2) + (int64_t)R * (K / 32) * 2; }

void repack_expert(const uint8_t* canon, int H, int I, uint8_t* gpu) {
  const int64_t mb = mat_bytes(I, H);
  repack_matrix(canon, I, H, gpu, gu_strip_bytes(H), 0, 8ll * H);
  repack_matrix(canon + mb, I, H, gpu, gu_strip_bytes(H), 9ll * H, 17ll * H);
  repack_matrix(canon + 2 * mb, H, I, gpu + down_base(H, I), down_strip_bytes(I), 0, 8ll * I);
}

void unpack_expert(const uint8_t* gpu, int H, int I, uint8_t* canon) {
  const int64_t mb = mat_bytes(I, H);
  unpack_matrix(gpu, I, H, canon, gu_strip_bytes(H), 0, 8ll * H);
  unpack_matrix(gpu, I, H, canon + mb, gu_strip_bytes(H), 9ll * H, 17ll * H);
  unpack_matrix(gpu + down_base(H, I), H, I, canon + 2 * mb, down_strip_bytes(I), 0, 8ll * I);
}

// Repack n experts on all host cores.
void repack_many(const uint8_t* canon, int64_t n, int H, int I, uint8_t* gpu) {
  const int64_t eb = expert_bytes(H, I);
  unsigned nt = std::thread::hardware_concurrency();
  if (nt == 0) nt = 1;
  if (nt > 32) nt = 32;
  if ((int64_t)nt > n) nt = (unsigned)(n > 0 ? n : 1);
  std::vector<std::thread> th;
  for (unsigned t = 0; t < nt; ++t) {
    const int64_t a = n * t / nt, b = n * (t + 1) / nt;
    auto job = [=] {
      for (int64_t e = a; e < b; ++e) repack_expert(canon + e * eb, H, I, gpu + e * eb);
    };
    try {
      th.emplace_back(job);
    } catch (...) {
      job();
    }
  }
  for (auto& t : th) t.join();
}

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

}  // namespace

struct moe_layer {
  moe_layer_desc_t d{};
  int sm_count = 0;
  int64_t blob = 0;
  uint8_t* master = nullptr;  // pinned host, GPU layout, E experts
  uint8_t* shared_dev = nullptr;
  void* dev_block = nullptr;
  void* pf_block = nullptr;  // prefill scratch (max_tokens > 64, no slot pool)
  PrefillArgs pf{};
  // Prefill on a pooled layer lends the pool's last slots: the scratch
  // occupies slots [S - lend_scratch, S), the experts the call needs that are
  // not resident below lend_first are staged through slots
  // [lend_first, S - lend_scratch) in waves, and every lent slot's expert is
  // copied back from the master copy after the call.
  int lend_first = 0, lend_scratch = 0;
  int32_t* pf_host = nullptr;        // pinned: counts [E + 1], device state, both pool tables
  const uint8_t** pf_tables = nullptr;  // pinned: one [E] base table per wave
  PrefillMaps pf_maps{};
  TensorMapEncodeFn encode_map = nullptr;
  HostMapped* hm_host = nullptr;
  HostMapped* hm_dev = nullptr;
  LayerArgs args{};
  int n_slots = 0;
  uint8_t* arena = nullptr;
  cudaStream_t copy_stream[2] = {nullptr, nullptr};  // misses alternate between two copy engines' queues
  WriteValue32Fn write_value = nullptr;
  uint32_t tail = 0;         // ring entries served (copy-server thread only)
  uint64_t copies = 0;       // copies issued (copy-server thread only)
  bool registered = false;   // polled by the copy server
  std::atomic<bool> paused{false};
  std::atomic<int64_t> fail_copy_n{0};
  std::atomic<int64_t> copies_since_arm{0};
  std::atomic<int> host_error{0};
  std::mutex log_mu;
  std::vector<int32_t> miss_log;
  std::atomic<uint64_t> h2d_bytes{0};
  uint64_t wait_timeout_ns = 2000000000ull;
  unsigned long long* tagged_logits = nullptr;  // fused kernel: [T][E] (step << 32 | logit bits)
  int32_t* pool_state = nullptr;           // fused kernel: double-buffered slot table
  moe_layer* next = nullptr;               // the layer whose weights calls warm in L2 (moe_set_next_layer)
  int32_t* hot_dev = nullptr;              // [kMaxHotExperts] next layer's experts to warm
  int32_t n_hot = 0;
};

namespace {

void serve_entry(moe_layer* L, const RingEntry& e) {
  if (e.served) {  // the kernel read this expert from host memory itself
    L->h2d_bytes += (uint64_t)L->blob;
    std::lock_guard<std::mutex> g(L->log_mu);
    L->miss_log.push_back((int32_t)e.seq);
    L->miss_log.push_back(e.expert);
    L->miss_log.push_back(e.slot);
    return;
  }
  bool fail = false;
  const int64_t n = L->fail_copy_n.load();
  if (n > 0 && ++L->copies_since_arm == n) fail = true;
  if (e.slot < 0 || e.slot >= L->n_slots || e.expert < 0 || e.expert >= L->d.n_experts) fail = true;
  cudaStream_t cs = L->copy_stream[L->copies++ & 1];
  if (!fail) {
    const cudaError_t err = cudaMemcpyAsync(L->arena + (int64_t)e.slot * L->blob, L->master + (int64_t)e.expert * L->blob,
                                            (size_t)L->blob, cudaMemcpyHostToDevice, cs);
    if (err != cudaSuccess) fail = true;
  }
  uint32_t val = e.seq;
  if (fail) {
    val |= kReadyError;
    int expected = 0;
    L->host_error.compare_exchange_strong(expected, MOE_ERR_COPY);
  } else {
    L->h2d_bytes += (uint64_t)L->blob;
  }
  const int slot = (e.slot >= 0 && e.slot < L->n_slots) ? e.slot : 0;
  // published on the same stream after the copy (with a memory barrier)
  L->write_value((CUstream)cs, (CUdeviceptr)(L->args.ready + slot), val, 0);
  std::lock_guard<std::mutex> g(L->log_mu);
  L->miss_log.push_back((int32_t)e.seq);
  L->miss_log.push_back(e.expert);
  L->miss_log.push_back(e.slot);
}

// One copy-server thread for the whole process polls the doorbell rings of
// every layer that has a slot pool.  It spins while doorbells are recent
// (decode rings one every few tens of microseconds) and sleeps in 50 us steps
// after 20 ms without one.
struct CopyServer {
  std::mutex life_mu;  // serializes starting and stopping the thread (taken before mu)
  std::mutex mu;
  std::vector<moe_layer*> layers;
  std::thread th;
  std::atomic<bool> stop{false};
  std::atomic<uint64_t> epoch{0};  // bumped after every poll round
  int device = -1;
};
CopyServer& copy_server() {
  static CopyServer* cs = new CopyServer();  // never destroyed: outlives every layer
  return *cs;
}

bool poll_layer(moe_layer* L) {
  if (L->paused.load(std::memory_order_relaxed)) return false;
  const uint32_t head = __atomic_load_n(&L->hm_host->head, __ATOMIC_ACQUIRE);
  if (head == L->tail) return false;
  while (L->tail != head) {
    RingEntry e;
    const volatile RingEntry* src = &L->hm_host->ring[L->tail % kRingSize];
    e.seq = src->seq;
    e.expert = src->expert;
    e.slot = src->slot;
    e.served = src->served;
    serve_entry(L, e);
    ++L->tail;
  }
  return true;
}

void server_main() {
  CopyServer& S = copy_server();
  cudaStreamCaptureMode mode = cudaStreamCaptureModeRelaxed;
  cudaThreadExchangeStreamCaptureMode(&mode);
  int cur_dev = -1;
  auto last = std::chrono::steady_clock::now();
  std::vector<moe_layer*> snap;
  while (!S.stop.load(std::memory_order_relaxed)) {
    {
      std::lock_guard<std::mutex> g(S.mu);
      snap = S.layers;
    }
    bool any = false;
    for (moe_layer* L : snap) {
      if (L->d.device != cur_dev) {
        cudaSetDevice(L->d.device);
        cur_dev = L->d.device;
      }
      any |= poll_layer(L);
    }
    S.epoch.fetch_add(1, std::memory_order_acq_rel);
    const auto now = std::chrono::steady_clock::now();
    if (any) last = now;
    else if (now - last > std::chrono::milliseconds(20)) std::this_thread::sleep_for(std::chrono::microseconds(50));
  }
}

// At process exit the server stops before the CUDA runtime tears down (its
// exit handler was registered earlier, so it runs later).
void shutdown_server() {
  CopyServer& S = copy_server();
  std::lock_guard<std::mutex> life(S.life_mu);
  S.stop = true;
  if (S.th.joinable()) S.th.join();
}

void register_layer(moe_layer* L) {
  static const bool exit_hook = (std::atexit(shutdown_server), true);
  (void)exit_hook;
  CopyServer& S = copy_server();
  std::lock_guard<std::mutex> life(S.life_mu);
  std::lock_guard<std::mutex> g(S.mu);
  L->tail = __atomic_load_n(&L->hm_host->head, __ATOMIC_ACQUIRE);
  S.layers.push_back(L);
  L->registered = true;
  if (!S.th.joinable()) {
    S.stop = false;
    S.th = std::thread(server_main);
  }
}

// After this returns the server no longer touches L.  Layers created and
// destroyed from several host threads: life_mu keeps a registration from
// slipping in between the decision to stop the thread and the join (which
// would leave a layer with no server) and keeps two joins apart.
void stop_server(moe_layer* L) {
  if (!L->registered) return;
  CopyServer& S = copy_server();
  std::lock_guard<std::mutex> life(S.life_mu);
  bool join = false;
  {
    std::lock_guard<std::mutex> g(S.mu);
    for (size_t i = 0; i < S.layers.size(); ++i)
      if (S.layers[i] == L) {
        S.layers.erase(S.layers.begin() + (long)i);
        break;
      }
    join = S.layers.empty();
    if (join) S.stop = true;
  }
  if (join) {
    if (S.th.joinable()) S.th.join();
    S.stop = false;
  } else {
    // wait for two poll rounds: a round that started before the erase has ended
    const uint64_t e0 = S.epoch.load();
    for (int i = 0; i < 200000 && S.epoch.load() < e0 + 2; ++i) std::this_thread::sleep_for(std::chrono::microseconds(5));
  }
  L->registered = false;
}

int sticky_error(moe_layer* L) {
  int e = L->host_error.load();
  if (e) return e;
  return __atomic_load_n(&L->hm_host->error, __ATOMIC_ACQUIRE);
}

void free_layer(moe_layer* L) {
  if (!L) return;
  stop_server(L);
  for (auto& cs : L->copy_stream)
    if (cs) cudaStreamDestroy(cs);
  if (L->dev_block) cudaFree(L->dev_block);
  if (L->pf_block) cudaFree(L->pf_block);
  if (L->pf_host) cudaFreeHost(L->pf_host);
  if (L->pf_tables) cudaFreeHost(L->pf_tables);
  if (L->shared_dev) cudaFree(L->shared_dev);
  if (L->hm_host) cudaFreeHost(L->hm_host);
  if (L->master) cudaFreeHost(L->master);
  delete L;
}

}  // namespace

extern "C" {

size_t moe_expert_bytes(int32_t hidden, int32_t inter) {
  if (hidden <= 0 || inter <= 0 || hidden % 32 || inter % 32) return 0;
  return (size_t)mat_bytes(inter, hidden) * 3;
}

MOE_API moe_status_t moe_repack_expert(const uint8_t* canon, int32_t hidden, int32_t inter, uint8_t* gpu) {
  if (!canon || !gpu || hidden % 64 || inter % 64 || hidden <= 0 || inter <= 0) return MOE_ERR_INVALID_ARG;
  repack_expert(canon, hidden, inter, gpu);
  return MOE_OK;
}

MOE_API moe_status_t moe_unpack_expert(const uint8_t* gpu, int32_t hidden, int32_t inter, uint8_t* canon) {
  if (!canon || !gpu || hidden % 64 || inter % 64 || hidden <= 0 || inter <= 0) return MOE_ERR_INVALID_ARG;
  unpack_expert(gpu, hidden, inter, canon);
  return MOE_OK;
}

moe_status_t moe_layer_create(const moe_layer_desc_t* desc, moe_layer_t** out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  if (!desc) return MOE_ERR_INVALID_ARG;
  const moe_layer_desc_t& d = *desc;
  if (d.qblock != kQBlock) return MOE_ERR_UNSUPPORTED;
  if (d.hidden <= 0 || d.inter <= 0 || d.n_experts <= 0 || d.top_k <= 0 || d.max_tokens <= 0)
    return MOE_ERR_INVALID_ARG;
  if (d.hidden % 64 || d.inter % 64 || d.hidden > kMaxHidden || d.inter > kMaxInter) return MOE_ERR_UNSUPPORTED;
  if (d.n_experts > kMaxExperts || d.top_k > kMaxTopK || d.top_k > d.n_experts) return MOE_ERR_UNSUPPORTED;
  if (d.max_tokens > kMaxPrefillTokens) return MOE_ERR_UNSUPPORTED;
  if (d.max_tokens > kMaxTokens && d.hidden % 128) return MOE_ERR_UNSUPPORTED;  // prefill M-blocks of 128 rows
  if (d.n_shared != 0 && d.n_shared != 1) return MOE_ERR_UNSUPPORTED;
  if (!d.router_w || !d.experts || (d.n_shared && !d.shared)) return MOE_ERR_INVALID_ARG;
  if (d.weight_format != MOE_FMT_LINEAR4 && d.weight_format != MOE_FMT_CODEBOOK4) return MOE_ERR_INVALID_ARG;
  if (d.weight_format == MOE_FMT_CODEBOOK4 && d.max_tokens > 8) return MOE_ERR_UNSUPPORTED;  // fused kernel only

  DeviceGuard guard(d.device);
  if (!guard.ok) return MOE_ERR_INVALID_ARG;
  moe_layer* L = new (std::nothrow) moe_layer();
  if (!L) return MOE_ERR_OUT_OF_MEMORY;
  L->d = d;
  L->d.experts = nullptr;  // read during create only
  L->d.shared = nullptr;
  L->blob = expert_bytes(d.hidden, d.inter);
  const int E = d.n_experts, H = d.hidden, I = d.inter, k = d.top_k, Tm = d.max_tokens;
  auto fail = [&](moe_status_t s) {
    free_layer(L);
    return s;
  };
  if (cudaDeviceGetAttribute(&L->sm_count, cudaDevAttrMultiProcessorCount, d.device) != cudaSuccess)
    return fail(MOE_ERR_CUDA);
  int cc_major = 0;
  cudaDeviceGetAttribute(&cc_major, cudaDevAttrComputeCapabilityMajor, d.device);
  if (cc_major < 10) return fail(MOE_ERR_UNSUPPORTED);
  if (configure_kernels(H, E) != cudaSuccess) return fail(MOE_ERR_CUDA);

  // stream write for the ready flags (driver entry point; no link-time libcuda)
  {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuStreamWriteValue32", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return fail(MOE_ERR_CUDA);
    L->write_value = (WriteValue32Fn)fn;
  }

  // pinned master copy in GPU layout
  if (cudaHostAlloc((void**)&L->master, (size_t)L->blob * E, cudaHostAllocMapped) != cudaSuccess) {
    L->master = nullptr;
    return fail(MOE_ERR_OUT_OF_MEMORY);
  }
  repack_many(d.experts, E, H, I, L->master);
  void* master_dev = nullptr;
  if (cudaHostGetDevicePointer(&master_dev, L->master, 0) != cudaSuccess) return fail(MOE_ERR_CUDA);

  if (d.n_shared) {
    std::vector<uint8_t> tmp((size_t)L->blob);
    repack_expert(d.shared, H, I, tmp.data());
    if (cudaMalloc((void**)&L->shared_dev, (size_t)L->blob) != cudaSuccess) {
      L->shared_dev = nullptr;
      return fail(MOE_ERR_OUT_OF_MEMORY);
    }
    if (cudaMemcpy(L->shared_dev, tmp.data(), (size_t)L->blob, cudaMemcpyHostToDevice) != cudaSuccess)
      return fail(MOE_ERR_CUDA);
  }

  // mapped host block (doorbell ring + error mirror)
  if (cudaHostAlloc((void**)&L->hm_host, sizeof(HostMapped), cudaHostAllocMapped) != cudaSuccess) {
    L->hm_host = nullptr;
    return fail(MOE_ERR_OUT_OF_MEMORY);
  }
  std::memset(L->hm_host, 0, sizeof(HostMapped));
  if (cudaHostGetDevicePointer((void**)&L->hm_dev, L->hm_host, 0) != cudaSuccess) return fail(MOE_ERR_CUDA);

  // device state + scratch, one allocation
  // the decode and batched paths take T <= kMaxTokens; larger T runs the prefill path
  const int Tb = Tm < kMaxTokens ? Tm : kMaxTokens;
  const int Um = E < Tb * k ? E : Tb * k;
  const size_t P = (size_t)Tb * k;
  size_t off = 0;
  auto carve = [&](size_t bytes) {
    size_t o = off;
    off += align256(bytes);
    return o;
  };
  const int Tl = Tm;                         // fp32 logits: the batched path (any T the fused kernel declines), prefill
  const int Tk = Tb > 8 ? Tb : 8;            // the fused kernel publishes 8 token rows every call
  const size_t o_st = carve(sizeof(DevState)), o_ready = carve(4ull * E), o_logits = carve(4ull * Tl * E),
               o_x16 = carve(2ull * Tb * H), o_uexp = carve(4ull * Um), o_uslot = carve(4ull * Um),
               o_uoff = carve(4ull * (Um + 1)), o_ptok = carve(4 * P),
               o_pw = carve(4 * P), o_tku = carve(4 * P), o_tkpos = carve(4 * P),
               o_h16 = carve(2ull * (P + Tb) * I), o_tki = carve(4ull * Tm * k), o_tkw = carve(4ull * Tm * k),
               o_bar = carve(8ull * Tk * E), o_cnt = carve(8ull * (Um + 2) * (I / 64) * kCntPad), o_pool = carve(4ull * 2 * 3 * E),
               o_hot = carve(4ull * kMaxHotExperts), o_wnorm = carve(4ull * E),
               o_pub = carve(128), o_htag = carve(4ull * (k + 1) * I);
  if (cudaMalloc(&L->dev_block, off) != cudaSuccess) {
    L->dev_block = nullptr;
    return fail(MOE_ERR_OUT_OF_MEMORY);
  }
  uint8_t* b = (uint8_t*)L->dev_block;
  if (cudaMemset(b, 0, off) != cudaSuccess) return fail(MOE_ERR_CUDA);
  LayerArgs& a = L->args;
  a.H = H;
  a.E = E;
  a.k = k;
  a.I = I;
  a.n_shared = d.n_shared;
  a.W_r = d.router_w;
  a.bias = d.router_bias;
  a.shared = L->shared_dev;
  a.blob = L->blob;
  a.st = (DevState*)(b + o_st);
  a.pub = (uint32_t*)(b + o_pub);
  a.hm = L->hm_dev;
  a.ready = (uint32_t*)(b + o_ready);
  a.logits = (float*)(b + o_logits);
  a.wnorm = (float*)(b + o_wnorm);
  a.x16 = (__half*)(b + o_x16);
  a.u_expert = (int32_t*)(b + o_uexp);
  a.u_slot = (int32_t*)(b + o_uslot);
  a.u_off = (int32_t*)(b + o_uoff);
  a.pair_token = (int32_t*)(b + o_ptok);
  a.pair_w = (float*)(b + o_pw);
  a.tk_u = (int32_t*)(b + o_tku);
  a.tk_pos = (int32_t*)(b + o_tkpos);
  a.h16 = (__half*)(b + o_h16);
  a.htag = (unsigned long long*)(b + o_htag);  // zeroed above: tag 0 is never a call's
  a.topk_idx = (int32_t*)(b + o_tki);
  a.topk_w = (float*)(b + o_tkw);
  a.wait_timeout_ns = L->wait_timeout_ns;
  a.master = (const uint8_t*)master_dev;
  a.pull = 1;  // misses read by the kernel from the mapped master copy (moe_set_miss_service)
  a.fmt = d.weight_format;
  L->tagged_logits = (unsigned long long*)(b + o_bar);
  a.counters = (uint32_t*)(b + o_cnt);
  a.cnt_stride = (Um + 2) * (I / 64) * kCntPad;
  L->pool_state = (int32_t*)(b + o_pool);
  L->hot_dev = (int32_t*)(b + o_hot);
  if (decode_configure() != cudaSuccess) return fail(MOE_ERR_CUDA);
  if (const size_t pfb = prefill_scratch_bytes(H, I, E, k, Tm)) {
    if (prefill_configure() != cudaSuccess) return fail(MOE_ERR_CUDA);
    if (cudaMalloc(&L->pf_block, pfb) != cudaSuccess) {
      L->pf_block = nullptr;
      return fail(MOE_ERR_OUT_OF_MEMORY);
    }
    if (cudaMemset(L->pf_block, 0, pfb) != cudaSuccess) return fail(MOE_ERR_CUDA);
    L->pf = prefill_carve(L->pf_block, H, I, E, k, Tm);
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return fail(MOE_ERR_CUDA);
    L->encode_map = (TensorMapEncodeFn)fn;
    if (!prefill_encode_maps(L->encode_map, L->pf, H, I, E, k, Tm, &L->pf_maps)) return fail(MOE_ERR_CUDA);
  }
  // The copy streams take the device's highest priority.  Streams of
  // different priorities never share a hardware work queue, so a slot copy
  // is never queued behind compute work that waits for the decode kernel
  // (which itself waits for the copy): compute streams are created at the
  // default, lowest, priority.
  int prio_least = 0, prio_greatest = 0;
  if (cudaDeviceGetStreamPriorityRange(&prio_least, &prio_greatest) != cudaSuccess) return fail(MOE_ERR_CUDA);
  for (auto& cs : L->copy_stream)
    if (cudaStreamCreateWithPriority(&cs, cudaStreamNonBlocking, prio_greatest) != cudaSuccess) {
      cs = nullptr;
      return fail(MOE_ERR_CUDA);
    }
  *out = L;
  return MOE_OK;
}

// The fused kernel's pool table from a slot map (slot_of [E], owner [E], the
// first n_slots used), every stamp 0 (used before the next step) and every
// ready flag clear.  The device is idle.
bool write_pool_state(moe_layer* L, const std::vector<int32_t>& slot_of, const std::vector<int32_t>& owner) {
  const int E = L->d.n_experts, S = L->n_slots;
  std::vector<uint32_t> zeros(E, 0u);
  // double-buffered: [slot_of E][owner S][stamp S] twice
  std::vector<int32_t> ps((size_t)2 * (E + 2 * S), 0);
  for (int h = 0; h < 2; ++h) {
    int32_t* base = ps.data() + (size_t)h * (E + 2 * S);
    for (int e = 0; e < E; ++e) base[e] = slot_of[e];
    for (int q = 0; q < S; ++q) base[E + q] = owner[q];
  }
  return cudaMemcpy(L->pool_state, ps.data(), ps.size() * 4, cudaMemcpyHostToDevice) == cudaSuccess &&
         cudaMemcpy(L->args.ready, zeros.data(), 4ull * E, cudaMemcpyHostToDevice) == cudaSuccess;
}

}  // extern "C"

namespace {

constexpr int kLendStage = 16;  // slots a pooled prefill stages missing experts through

// Where a layer's prefill scratch lives for its current configuration: its
// own allocation when every expert is resident; the pool's last slots when it
// has a pool (Basalt README, section "Prompt chunks": the prompt path's
// buffers are carved from the expert cache's last slots and the experts in
// them are copied back afterwards).  Refuses a pool too small to lend the
// scratch and one staging slot (Basalt README, section "Memory floors":
// refuse what does not fit instead of shrinking it).
moe_status_t configure_prefill_scratch(moe_layer* L) {
  const int H = L->d.hidden, I = L->d.inter, E = L->d.n_experts, k = L->d.top_k, Tm = L->d.max_tokens;
  const size_t pfb = prefill_scratch_bytes(H, I, E, k, Tm);
  L->lend_first = L->lend_scratch = 0;
  if (!pfb) return MOE_OK;
  const int S = L->n_slots;
  if (L->args.pool) {
    const int n_scr = (int)((pfb + (size_t)L->blob - 1) / (size_t)L->blob);
    const int room = S - n_scr;
    if (room < 1) return MOE_ERR_OUT_OF_MEMORY;
    const int R = room < kLendStage ? room : kLendStage;
    L->lend_scratch = n_scr;
    L->lend_first = S - n_scr - R;
    if (L->pf_block) {
      cudaFree(L->pf_block);
      L->pf_block = nullptr;
    }
    L->pf = prefill_carve(L->arena + (size_t)(S - n_scr) * (size_t)L->blob, H, I, E, k, Tm);
    if (!L->pf_host &&
        cudaHostAlloc((void**)&L->pf_host,
                      sizeof(int32_t) * ((size_t)E + 1 + 2 * (3 * (size_t)E)) + sizeof(DevState) + 128,
                      cudaHostAllocDefault) != cudaSuccess) {
      L->pf_host = nullptr;
      return MOE_ERR_OUT_OF_MEMORY;
    }
    if (!L->pf_tables &&
        cudaHostAlloc((void**)&L->pf_tables, sizeof(uint8_t*) * (size_t)E * ((size_t)E + 1), cudaHostAllocDefault) !=
            cudaSuccess) {  // one table per wave, at most E waves
      L->pf_tables = nullptr;
      return MOE_ERR_OUT_OF_MEMORY;
    }
  } else if (!L->pf_block) {
    if (cudaMalloc(&L->pf_block, pfb) != cudaSuccess) {
      L->pf_block = nullptr;
      return MOE_ERR_OUT_OF_MEMORY;
    }
    if (cudaMemset(L->pf_block, 0, pfb) != cudaSuccess) return MOE_ERR_CUDA;
    L->pf = prefill_carve(L->pf_block, H, I, E, k, Tm);
  }
  if (!prefill_encode_maps(L->encode_map, L->pf, H, I, E, k, Tm, &L->pf_maps)) return MOE_ERR_CUDA;
  return MOE_OK;
}

}  // namespace

extern "C" {

moe_status_t moe_slot_pool_configure(moe_layer_t* L, int32_t n_slots, void* arena_dev, size_t arena_bytes) {
  if (!L || !arena_dev) return MOE_ERR_INVALID_ARG;
  const int E = L->d.n_experts;
  // a pool serves calls of up to 8 tokens in the fused kernel (prefill calls
  // lend slots, below); every distinct expert of one call needs a slot
  const int calls = L->d.max_tokens < 8 ? L->d.max_tokens : 8;
  const int need = E < calls * L->d.top_k ? E : calls * L->d.top_k;
  if (n_slots < need || n_slots > E) return MOE_ERR_INVALID_ARG;
  if (((uintptr_t)arena_dev & 255) != 0) return MOE_ERR_INVALID_ARG;
  if ((size_t)n_slots * (size_t)L->blob > arena_bytes) return MOE_ERR_OUT_OF_MEMORY;
  // only the fused decode kernel serves a pool
  if (n_slots < E && !decode_supported(L->d.hidden, L->d.inter, E, L->d.top_k, 1, L->sm_count, true))
    return MOE_ERR_UNSUPPORTED;
  DeviceGuard guard(L->d.device);
  if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
  stop_server(L);
  L->arena = (uint8_t*)arena_dev;
  L->n_slots = n_slots;
  LayerArgs& a = L->args;
  a.arena = L->arena;
  a.n_slots = n_slots;
  a.pool = n_slots < E;
  // a configure that fails part-way leaves the layer unconfigured (forward
  // answers MOE_ERR_STATE), never half-filled slots behind a valid table
  auto unconfigured = [&](moe_status_t code) {
    L->n_slots = 0;
    a.n_slots = 0;
    a.pool = 0;
    return code;
  };
  std::vector<int32_t> slot_of(E), owner(E, -1);
  if (!a.pool) {
    if (cudaMemcpy(L->arena, L->master, (size_t)L->blob * E, cudaMemcpyHostToDevice) != cudaSuccess)
      return unconfigured(MOE_ERR_CUDA);
    for (int e = 0; e < E; ++e) slot_of[e] = owner[e] = e;
  } else {
    for (int e = 0; e < E; ++e) slot_of[e] = -1;
  }
  if (!write_pool_state(L, slot_of, owner)) return unconfigured(MOE_ERR_CUDA);
  const moe_status_t pf = configure_prefill_scratch(L);
  if (pf != MOE_OK) return unconfigured(pf);
  if (a.pool) {
    try {
      register_layer(L);
    } catch (...) {
      return unconfigured(MOE_ERR_OUT_OF_MEMORY);
    }
  }
  return MOE_OK;
}

moe_status_t moe_slot_pool_seed(moe_layer_t* L, const int32_t* experts, int32_t n) {
  if (!L || n < 0 || (n > 0 && !experts)) return MOE_ERR_INVALID_ARG;
  if (L->n_slots == 0 || !L->args.pool) return MOE_ERR_STATE;
  if (n > L->n_slots) return MOE_ERR_INVALID_ARG;
  if (sticky_error(L)) return MOE_ERR_STATE;
  const int E = L->d.n_experts;
  std::vector<int32_t> slot_of(E, -1), owner(E, -1);
  for (int i = 0; i < n; ++i) {
    const int e = experts[i];
    if (e < 0 || e >= E || slot_of[e] >= 0) return MOE_ERR_INVALID_ARG;
    slot_of[e] = i;
    owner[i] = e;
  }
  DeviceGuard guard(L->d.device);
  if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;  // no call in flight sees the change
  // the pool is marked empty before any slot is overwritten: a copy that
  // fails part-way leaves an empty (consistent) pool, never a table that
  // names an expert whose bytes are no longer in its slot
  const std::vector<int32_t> none(E, -1);
  if (!write_pool_state(L, none, none)) return MOE_ERR_CUDA;
  for (int i = 0; i < n; ++i)
    if (cudaMemcpy(L->arena + (int64_t)i * L->blob, L->master + (int64_t)experts[i] * L->blob, (size_t)L->blob,
                   cudaMemcpyHostToDevice) != cudaSuccess)
      return MOE_ERR_CUDA;
  return write_pool_state(L, slot_of, owner) ? MOE_OK : MOE_ERR_CUDA;
}

namespace {

// The residual + RMSNorm that moe_forward_norm puts in front of the layer.
struct PreNorm {
  const void* x;
  const void* y_prev;
  float eps;
  void* x_out;
  void* xhat;
};

// [p, p + n) and [q, q + n) share a byte (a null pointer shares none).
bool overlap(const void* p, const void* q, size_t n) {
  if (!p || !q) return false;
  const uintptr_t a = (uintptr_t)p, b = (uintptr_t)q;
  return a < b + n && b < a + n;
}

// x is the layer input; with a pre-norm it is the xhat buffer, which the
// fused kernel writes itself and the other paths get from
// residual_rmsnorm_kernel first.
// A prefill call on a pooled layer (Basalt README, section "Prompt chunks").
// The scratch sits in the lent slots; after routing, the host reads which
// experts the call touches and where the pool holds them (one stream
// synchronize), then runs the expert GEMMs in waves: the first with every
// touched expert resident below the lent slots, each wave with up to R
// missing experts copied from the pinned master copy into the staging
// slots.  Afterwards every lent slot gets its own expert back, so the pool
// (table, LRU stamps, contents) is exactly what it was before the call.
moe_status_t prefill_lend(moe_layer* L, const LayerArgs& a, cudaStream_t s) {
  const int E = L->d.n_experts, S = L->n_slots;
  const size_t blob = (size_t)L->blob;
  const int first = L->lend_first, scr0 = S - L->lend_scratch, R = scr0 - first;
  uint8_t* arena = L->arena;
  if (cudaMemsetAsync(arena + (size_t)scr0 * blob, 0, (size_t)L->lend_scratch * blob, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (launch_prefill_route(a, L->pf, L->pf_maps, L->sm_count, s) != cudaSuccess) return MOE_ERR_CUDA;
  int32_t* counts = L->pf_host;
  const size_t ds_off = ((sizeof(int32_t) * ((size_t)E + 1)) + 127) & ~size_t(127);
  DevState* ds = reinterpret_cast<DevState*>(reinterpret_cast<uint8_t*>(L->pf_host) + ds_off);
  int32_t* tabs = reinterpret_cast<int32_t*>(ds + 1);
  if (cudaMemcpyAsync(counts, L->pf.counts, sizeof(int32_t) * (E + 1), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaMemcpyAsync(ds, a.st, sizeof(DevState), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaMemcpyAsync(tabs, L->pool_state, sizeof(int32_t) * 2 * ((size_t)E + 2 * S), cudaMemcpyDeviceToHost, s) !=
          cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  if (ds->error) return MOE_ERR_STATE;
  // the table the next decode call starts from (prefill leaves the step alone)
  const int32_t* slot_of = tabs + (size_t)((ds->step + 1u) & 1u) * ((size_t)E + 2 * S);
  const int32_t* owner = slot_of + E;
  std::vector<int> stage;
  const uint8_t** t0 = L->pf_tables;
  for (int e = 0; e < E; ++e) {
    t0[e] = nullptr;
    if (counts[e] <= 0) continue;
    const int q = slot_of[e];
    if (q >= 0 && q < first)
      t0[e] = arena + (size_t)q * blob;
    else
      stage.push_back(e);
  }
  const int waves = stage.empty() ? 1 : (int)((stage.size() + R - 1) / R);
  uint64_t moved = 0;
  for (int w = 0; w < waves; ++w) {
    const uint8_t** t = L->pf_tables + (size_t)w * E;
    if (w > 0)
      for (int e = 0; e < E; ++e) t[e] = nullptr;
    for (int i = 0; i < R; ++i) {
      const size_t j = (size_t)w * R + i;
      if (j >= stage.size()) break;
      const int e = stage[j];
      uint8_t* dst = arena + (size_t)(first + i) * blob;
      if (cudaMemcpyAsync(dst, L->master + (size_t)e * blob, blob, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return MOE_ERR_CUDA;
      t[e] = dst;
      moved += blob;
    }
    if (cudaMemcpyAsync(L->pf.base_table, t, sizeof(uint8_t*) * E, cudaMemcpyHostToDevice, s) != cudaSuccess)
      return MOE_ERR_CUDA;
    if (launch_prefill_wave(a, L->pf, L->sm_count, w == 0, s) != cudaSuccess) return MOE_ERR_CUDA;
  }
  if (launch_prefill_combine(a, L->pf, s) != cudaSuccess) return MOE_ERR_CUDA;
  for (int q = first; q < S; ++q) {
    const int e = owner[q];
    if (e < 0) continue;
    if (cudaMemcpyAsync(arena + (size_t)q * blob, L->master + (size_t)e * blob, blob, cudaMemcpyHostToDevice, s) !=
        cudaSuccess)
      return MOE_ERR_CUDA;
    moved += blob;
  }
  L->h2d_bytes += moved;
  return MOE_OK;
}

moe_status_t forward_impl(moe_layer_t* L, const void* x, int32_t T, void* y, int32_t* topk_idx, float* topk_w,
                          void* stream, const PreNorm* pn) {
  if (L->n_slots == 0) return MOE_ERR_STATE;
  if (sticky_error(L)) return MOE_ERR_STATE;
  DeviceGuard guard(L->d.device);
  LayerArgs a = L->args;
  a.T = T;
  a.x = (const uint16_t*)x;
  a.y = (uint16_t*)y;
  if (topk_idx) a.topk_idx = topk_idx;
  if (topk_w) a.topk_w = topk_w;
  a.wait_timeout_ns = L->wait_timeout_ns;
  cudaStream_t s = (cudaStream_t)stream;
  if (decode_supported(L->d.hidden, L->d.inter, L->d.n_experts, L->d.top_k, T, L->sm_count, L->args.pool != 0)) {
    if (pn) {
      a.resid = (const uint16_t*)pn->x;
      a.y_prev = (const uint16_t*)pn->y_prev;
      a.x_out = (uint16_t*)pn->x_out;
      a.xhat_out = (uint16_t*)pn->xhat;
      a.eps = pn->eps;
    }
    const moe_layer* nx = L->next;
    if (nx && nx->n_slots > 0) {
      a.nx_W_r = nx->args.W_r;
      a.nx_shared = nx->args.shared;
      a.nx_arena = nx->args.arena;
      a.nx_pool_state = nx->args.pool ? nx->pool_state : nullptr;
      a.nx_st = nx->args.st;
      a.nx_S = nx->args.n_slots;
      a.nx_hot = L->hot_dev;
      a.nx_n_hot = L->n_hot;
    }
    if (launch_decode(a, L->tagged_logits, L->pool_state, L->sm_count, s) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
  }
  // codebook weights: fused path only; a pool: fused path (T <= 8) or a
  // prefill call that lends slots (T > 64)
  if (a.fmt != MOE_FMT_LINEAR4 || (a.pool && T <= kMaxTokens)) return MOE_ERR_UNSUPPORTED;
  if (pn && launch_residual_rmsnorm((const uint16_t*)pn->x, (const uint16_t*)pn->y_prev, T, L->d.hidden, pn->eps,
                                    (uint16_t*)pn->x_out, (uint16_t*)pn->xhat, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (T > kMaxTokens) {
    if (!prefill_encode_x(L->encode_map, x, L->d.hidden, T, &L->pf_maps)) return MOE_ERR_CUDA;
    if (a.pool) return prefill_lend(L, a, s);
    if (launch_prefill(a, L->pf, L->pf_maps, L->sm_count, s) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
  }
  const int Um = L->d.n_experts < T * L->d.top_k ? L->d.n_experts : T * L->d.top_k;
  const int max_tasks = (L->d.n_shared + Um) * (L->d.inter / 16);
  int gu_grid = L->sm_count * gateup_max_blocks_per_sm(L->d.hidden);
  if (gu_grid > max_tasks) gu_grid = max_tasks;
  const int dn_warps = down_warps(T, L->d.top_k, L->d.n_shared, L->d.inter);
  if (dn_warps < 1) return MOE_ERR_UNSUPPORTED;
  if (launch_route(a, s, true) != cudaSuccess) return MOE_ERR_CUDA;
  if (launch_gateup(a, s, true, gu_grid) != cudaSuccess) return MOE_ERR_CUDA;
  if (launch_down(a, s, true, dn_warps) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

}  // namespace

moe_status_t moe_forward(moe_layer_t* L, const void* x, int32_t T, void* y, int32_t* topk_idx, float* topk_w,
                         void* stream) {
  if (!L || !x || !y) return MOE_ERR_INVALID_ARG;
  if (T < 1 || T > L->d.max_tokens) return MOE_ERR_INVALID_ARG;
  if (((uintptr_t)x & 15) || ((uintptr_t)y & 3)) return MOE_ERR_INVALID_ARG;
  return forward_impl(L, x, T, y, topk_idx, topk_w, stream, nullptr);
}

moe_status_t moe_forward_norm(moe_layer_t* L, const void* x, const void* y_prev, int32_t T, float eps, void* x_out,
                              void* xhat, void* y, int32_t* topk_idx, float* topk_w, void* stream) {
  if (!L || !x || !xhat || !y) return MOE_ERR_INVALID_ARG;
  if (T < 1 || T > L->d.max_tokens || !(eps >= 0.f)) return MOE_ERR_INVALID_ARG;
  if ((((uintptr_t)x | (uintptr_t)y_prev | (uintptr_t)x_out | (uintptr_t)xhat) & 15) || ((uintptr_t)y & 3))
    return MOE_ERR_INVALID_ARG;
  const size_t n = (size_t)T * (size_t)L->d.hidden * 2;
  if (overlap(xhat, x, n) || overlap(xhat, y_prev, n) || overlap(xhat, x_out, n) || overlap(xhat, y, n) ||
      overlap(x_out, x, n) || overlap(x_out, y_prev, n) || overlap(x_out, y, n) || overlap(y, x, n) ||
      overlap(y, y_prev, n))
    return MOE_ERR_INVALID_ARG;
  const PreNorm pn{x, y_prev, eps, x_out, xhat};
  return forward_impl(L, xhat, T, y, topk_idx, topk_w, stream, &pn);
}

moe_status_t moe_residual_rmsnorm(const void* x, const void* y, int32_t T, int32_t hidden, float eps, void* x_out,
                                  void* xhat, void* stream) {
  if (!x || !xhat || T < 1 || hidden < 1 || hidden > kMaxHidden || !(eps >= 0.f)) return MOE_ERR_INVALID_ARG;
  if (xhat == x || (y && xhat == y) || (x_out && xhat == x_out)) return MOE_ERR_INVALID_ARG;
  if ((((uintptr_t)x | (uintptr_t)y | (uintptr_t)x_out | (uintptr_t)xhat) & 15) || hidden % 8)
    return MOE_ERR_INVALID_ARG;
  if (launch_residual_rmsnorm((const uint16_t*)x, (const uint16_t*)y, T, hidden, eps, (uint16_t*)x_out,
                              (uint16_t*)xhat, (cudaStream_t)stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status_t moe_get_stats(moe_layer_t* L, moe_stats_t* out) {
  if (!L || !out) return MOE_ERR_INVALID_ARG;
  DeviceGuard guard(L->d.device);
  if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
  DevState ds;
  if (cudaMemcpy(&ds, L->args.st, sizeof(ds), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  std::memset(out, 0, sizeof(*out));
  out->forwards = ds.forwards;
  out->hits = ds.hits;
  out->misses = ds.misses;
  out->h2d_bytes = L->h2d_bytes.load();
  out->wait_ns = ds.wait_ns;
  out->n_slots = L->n_slots;
  int e = L->host_error.load();
  if (!e) e = ds.error;
  out->error = e;
  out->rechecks = ds.rechecks;
  return (moe_status_t)e;
}

moe_status_t moe_get_miss_log(moe_layer_t* L, int32_t* out, int64_t max, int64_t* n) {
  if (!L || !n || (max > 0 && !out)) return MOE_ERR_INVALID_ARG;
  DeviceGuard guard(L->d.device);
  if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
  // the server may still be issuing the last entries: wait until it caught up
  if (L->n_slots < L->d.n_experts) {
    uint32_t head = 0;
    cudaMemcpy(&head, &L->args.st->ring_head, 4, cudaMemcpyDeviceToHost);
    for (int spin = 0; spin < 20000; ++spin) {
      {
        std::lock_guard<std::mutex> g(L->log_mu);
        if (L->miss_log.size() / 3 >= head || L->paused.load()) break;
      }
      std::this_thread::sleep_for(std::chrono::microseconds(100));
    }
  }
  std::lock_guard<std::mutex> g(L->log_mu);
  const int64_t total = (int64_t)(L->miss_log.size() / 3);
  *n = total;
  const int64_t m = total < max ? total : max;
  if (m > 0) std::memcpy(out, L->miss_log.data(), (size_t)m * 3 * sizeof(int32_t));
  return MOE_OK;
}

moe_status_t moe_set_wait_timeout_ns(moe_layer_t* L, uint64_t ns) {
  if (!L) return MOE_ERR_INVALID_ARG;
  L->wait_timeout_ns = ns ? ns : 2000000000ull;
  return MOE_OK;
}

moe_status_t moe_set_miss_service(moe_layer_t* L, int32_t mode) {
  if (!L || (mode != MOE_MISS_COPY_ENGINE && mode != MOE_MISS_SM_PULL)) return MOE_ERR_INVALID_ARG;
  DeviceGuard guard(L->d.device);
  if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;  // no call in flight sees a half-set mode
  L->args.pull = mode == MOE_MISS_SM_PULL ? 1 : 0;
  return MOE_OK;
}

moe_status_t moe_set_next_layer(moe_layer_t* L, moe_layer_t* next, const int32_t* hot_experts, int32_t n_hot) {
  if (!L || n_hot < 0 || n_hot > kMaxHotExperts || (n_hot > 0 && (!hot_experts || !next))) return MOE_ERR_INVALID_ARG;
  if (next && (next->d.hidden != L->d.hidden || next->d.n_experts != L->d.n_experts ||
               next->d.inter != L->d.inter || next->d.n_shared != L->d.n_shared || next->d.device != L->d.device))
    return MOE_ERR_INVALID_ARG;
  for (int i = 0; i < n_hot; ++i)
    if (hot_experts[i] < 0 || hot_experts[i] >= L->d.n_experts) return MOE_ERR_INVALID_ARG;
  DeviceGuard guard(L->d.device);
  if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;  // no call in flight reads the list
  if (n_hot > 0 && cudaMemcpy(L->hot_dev, hot_experts, 4ull * n_hot, cudaMemcpyHostToDevice) != cudaSuccess)
    return MOE_ERR_CUDA;
  L->next = next;
  L->n_hot = n_hot;
  return MOE_OK;
}

moe_status_t moe_debug_copy_faults(moe_layer_t* L, int64_t fail_copy_n, int32_t pause) {
  if (!L || fail_copy_n < 0) return MOE_ERR_INVALID_ARG;
  L->copies_since_arm = 0;
  L->fail_copy_n = fail_copy_n;
  L->paused = pause != 0;
  return MOE_OK;
}

void moe_destroy(moe_layer_t* L) {
  if (!L) return;
  DeviceGuard guard(L->d.device);
  L->paused = false;
  cudaDeviceSynchronize();
  free_layer(L);
}

const char* moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported configuration";
    case MOE_ERR_OUT_OF_MEMORY: return "out of memory";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_COPY: return "expert copy failed";
    case MOE_ERR_TIMEOUT: return "timed out waiting for an expert copy";
    case MOE_ERR_STATE: return "layer not ready or holding an earlier error";
    case MOE_ERR_DEVICE: return "device-side check failed";
  }
  return "unknown status";
}

}  // extern "C"
