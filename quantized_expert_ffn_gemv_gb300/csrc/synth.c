/*
 * Seeded synthetic inputs for the quantized MoE expert-FFN layer.
 *
 * This module only *draws* inputs: Gaussian weights, the 4-bit block
 * quantizer that turns them into the canonical packed expert blob, the
 * per-expert Zipf router bias and the bf16 activations.  It contains none
 * of the layer's arithmetic (no dequantization, routing, FFN or combine);
 * both the CUDA path and the CPU oracle consume what it writes.
 *
 * Everything is counter based: value i of a stream is a pure function of
 * (key, i), so any slice can be generated independently, on any number of
 * threads, and the bytes are identical on x86-64 and aarch64.  To keep them
 * identical the file is compiled with -ffp-contract=off and never calls a
 * libm transcendental: the natural log used by the Gaussian draw and the
 * Zipf bias is evaluated here with an atanh series (basic IEEE operations
 * only), and sqrt is the correctly rounded IEEE square root.
 *
 * Canonical expert blob (one contiguous byte range per expert, so that a
 * miss is one copy; Betelgeuse news page, section 机制, "4KB 对齐的单读 blob"):
 *   [W_gate I x H][W_up I x H][W_down H x I]
 * each matrix R x K (row-major by output row) stored as
 *   nibble plane  R * K/2 bytes: element i of a row in byte i/2,
 *                 low nibble when i is even, stored value u = q + 8
 *   scale plane   R * K/32 IEEE binary16 scales, one per block of 32
 *                 consecutive elements along K (the reduction axis).
 * Quantizer, format 0 (4-bit symmetric, block 32, one fp16 scale):
 *   d = fp16_rn(amax / 7); q = clamp(round_half_even(w / d), -8, 7);
 *   an all-zero block (or one whose scale rounds to 0) stores d = 0, q = 0.
 * Quantizer, format 1 (4-bit codebook, block 32, one fp16 scale; the
 *   non-linear 16-entry lookup formats of the halogen-flash-server README,
 *   section "Bring your own GGUF"): weight = d * C[u] with C the levels of
 *   the standard normal's quantiles (u + 1/2) / 16, scaled to +-127 and
 *   rounded (see kCodebook); d = fp16_rn(amax / 127); u = the level nearest
 *   w / d, ties to the lower u; a zero block stores d = 0 and u = 8.
 */
#include <stdint.h>
#include <string.h>
#include <math.h>
#include <pthread.h>
#include <stdlib.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

/* Output number `ctr` of the splitmix64 stream started at `key`. */
static inline uint64_t draw64(uint64_t key, uint64_t ctr) {
  return mix64(key + (ctr + 1) * GOLDEN);
}

/* Hash a tuple of tags into a stream key. */
uint64_t synth_key(uint64_t seed, uint64_t a, uint64_t b, uint64_t c, uint64_t d) {
  uint64_t k = mix64(seed ^ 0x5EED2026ULL);
  k = mix64(k + a * GOLDEN + 1);
  k = mix64(k + b * GOLDEN + 2);
  k = mix64(k + c * GOLDEN + 3);
  k = mix64(k + d * GOLDEN + 4);
  return k;
}

/* ln(x) for finite x > 0 using only + - * / (atanh series), about 1 ulp. */
static double det_log(double x) {
  uint64_t bits;
  memcpy(&bits, &x, 8);
  int e = (int)((bits >> 52) & 0x7FF);
  if (e == 0) { /* subnormal: scale up by 2^64 */
    x *= 18446744073709551616.0;
    memcpy(&bits, &x, 8);
    e = (int)((bits >> 52) & 0x7FF) - 64;
  }
  e -= 1023;
  bits = (bits & 0x000FFFFFFFFFFFFFULL) | 0x3FF0000000000000ULL;
  double m;
  memcpy(&m, &bits, 8); /* m in [1, 2) */
  if (m > 1.4142135623730951) { m *= 0.5; e += 1; }
  double s = (m - 1.0) / (m + 1.0);
  double s2 = s * s;
  /* 2*atanh(s) = 2 s (1 + s^2/3 + s^4/5 + ...), Horner form; |s| <= 0.172 so
     the first omitted term (s^26/27) is below 1e-21 relative */
  double p = 1.0 / 25.0;
  p = 1.0 / 23.0 + s2 * p;
  p = 1.0 / 21.0 + s2 * p;
  p = 1.0 / 19.0 + s2 * p;
  p = 1.0 / 17.0 + s2 * p;
  p = 1.0 / 15.0 + s2 * p;
  p = 1.0 / 13.0 + s2 * p;
  p = 1.0 / 11.0 + s2 * p;
  p = 1.0 / 9.0 + s2 * p;
  p = 1.0 / 7.0 + s2 * p;
  p = 1.0 / 5.0 + s2 * p;
  p = 1.0 / 3.0 + s2 * p;
  p = 1.0 + s2 * p;
  double sum = s * p;
  return (double)e * 0.6931471805599453 + 2.0 * sum;
}

/* Pair p of standard normals by the Marsaglia polar method. */
static void normal_pair(uint64_t key, uint64_t p, double* n0, double* n1) {
  for (uint64_t a = 0; a < 256; ++a) {
    uint64_t c = (p << 9) | (a << 1);
    double v1 = (double)(draw64(key, c) >> 11) * 0x1.0p-53 * 2.0 - 1.0;
    double v2 = (double)(draw64(key, c | 1) >> 11) * 0x1.0p-53 * 2.0 - 1.0;
    double s = v1 * v1 + v2 * v2;
    if (s > 0.0 && s < 1.0) {
      double f = sqrt(-2.0 * det_log(s) / s);
      *n0 = v1 * f;
      *n1 = v2 * f;
      return;
    }
  }
  *n0 = 0.0;
  *n1 = 0.0;
}

/* Element i of the standard-normal stream `key`. */
static inline double normal_at(uint64_t key, uint64_t i) {
  double a, b;
  normal_pair(key, i >> 1, &a, &b);
  return (i & 1) ? b : a;
}

void synth_normal_f64(uint64_t key, uint64_t start, uint64_t n, double* out) {
  uint64_t i = 0;
  while (i < n) {
    uint64_t g = start + i;
    double a, b;
    normal_pair(key, g >> 1, &a, &b);
    if ((g & 1) == 0) {
      out[i++] = a;
      if (i < n) out[i++] = b;
    } else {
      out[i++] = b;
    }
  }
}

/* ---- rounding helpers (round to nearest even) ---- */

static inline float to_f32(double v) { return (float)v; } /* IEEE RNE */

static uint16_t f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u) return (uint16_t)((u >> 16) | ((u & 0xFFFF) ? 0x40 : 0));
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

/* IEEE binary16, round to nearest even; overflow to inf. */
static uint16_t f64_to_f16(double v) {
  uint16_t sign = 0;
  if (v < 0) { sign = 0x8000; v = -v; }
  if (v != v) return 0x7E00;
  if (v >= 65520.0) return sign | 0x7C00;
  if (v < 0x1.0p-25) return sign; /* rounds to zero (half of min subnormal ties to even 0) */
  int e = 0;
  double m = v;
  /* find e with m = v / 2^e in [1, 2) */
  while (m >= 2.0) { m *= 0.5; ++e; }
  while (m < 1.0) { m *= 2.0; --e; }
  if (e < -14) { /* subnormal: value = k * 2^-24 */
    double k = v * 16777216.0;
    double r = nearbyint(k); /* ties to even under the default mode */
    return sign | (uint16_t)r;
  }
  double frac = (m - 1.0) * 1024.0;
  double r = nearbyint(frac);
  if (r >= 1024.0) { r = 0.0; ++e; }
  if (e > 15) return sign | 0x7C00;
  return sign | (uint16_t)(((e + 15) << 10) | (int)r);
}

static double f16_value(uint16_t h) {
  int e = (h >> 10) & 0x1F, m = h & 0x3FF;
  double v;
  if (e == 0) v = ldexp((double)m, -24);
  else if (e == 31) v = INFINITY;
  else v = ldexp(1024.0 + m, e - 25);
  return (h & 0x8000) ? -v : v;
}

/* ---- quantizer ---- */

/* Quantize R rows of K fp32 weights into a nibble plane and a scale plane. */
void synth_quantize_rows(const float* w, int64_t R, int64_t K, uint8_t* nib, uint16_t* scales) {
  const int64_t nb = K / 32;
  for (int64_t r = 0; r < R; ++r) {
    for (int64_t b = 0; b < nb; ++b) {
      const float* blk = w + r * K + b * 32;
      double amax = 0.0;
      for (int i = 0; i < 32; ++i) {
        double a = fabs((double)blk[i]);
        if (a > amax) amax = a;
      }
      uint16_t d16 = f64_to_f16(amax / 7.0);
      double d = f16_value(d16);
      scales[r * nb + b] = d16;
      uint8_t* out = nib + r * (K / 2) + b * 16;
      for (int i = 0; i < 32; i += 2) {
        int q0 = 0, q1 = 0;
        if (d != 0.0) {
          double t0 = nearbyint((double)blk[i] / d), t1 = nearbyint((double)blk[i + 1] / d);
          q0 = t0 < -8 ? -8 : (t0 > 7 ? 7 : (int)t0);
          q1 = t1 < -8 ? -8 : (t1 > 7 ? 7 : (int)t1);
        }
        out[i / 2] = (uint8_t)((q0 + 8) | ((q1 + 8) << 4));
      }
    }
  }
}

/* The codebook of format 1, ascending. */
static const int kCodebook[16] = {-127, -90, -69, -53, -39, -27, -16, -5, 5, 16, 27, 39, 53, 69, 90, 127};

void synth_quantize_rows_cb(const float* w, int64_t R, int64_t K, uint8_t* nib, uint16_t* scales) {
  const int64_t nb = K / 32;
  for (int64_t r = 0; r < R; ++r) {
    for (int64_t b = 0; b < nb; ++b) {
      const float* blk = w + r * K + b * 32;
      double amax = 0.0;
      for (int i = 0; i < 32; ++i) {
        double a = fabs((double)blk[i]);
        if (a > amax) amax = a;
      }
      uint16_t d16 = f64_to_f16(amax / 127.0);
      double d = f16_value(d16);
      scales[r * nb + b] = d16;
      uint8_t* out = nib + r * (K / 2) + b * 16;
      for (int i = 0; i < 32; i += 2) {
        int u[2] = {8, 8};
        for (int h = 0; h < 2 && d != 0.0; ++h) {
          const double t = (double)blk[i + h] / d;
          double best = fabs(t - kCodebook[0]);
          u[h] = 0;
          for (int c = 1; c < 16; ++c) {
            const double e = fabs(t - kCodebook[c]);
            if (e < best) { best = e; u[h] = c; }
          }
        }
        out[i / 2] = (uint8_t)(u[0] | (u[1] << 4));
      }
    }
  }
}

/* Bytes of one R x K packed matrix / of one expert blob. */
int64_t synth_matrix_bytes(int64_t R, int64_t K) { return R * (K / 2) + R * (K / 32) * 2; }
int64_t synth_expert_bytes(int64_t H, int64_t I) { return 3 * synth_matrix_bytes(I, H); }

/* One R x K matrix of N(0, sigma^2) weights (fp32), quantized into `dst`. */
static void gen_matrix(uint64_t key, int64_t R, int64_t K, double sigma, int fmt, uint8_t* dst, float* rowbuf) {
  uint8_t* nib = dst;
  uint16_t* sc = (uint16_t*)(dst + R * (K / 2));
  for (int64_t r = 0; r < R; ++r) {
    for (int64_t i = 0; i < K; i += 2) {
      double a, b;
      normal_pair(key, (uint64_t)((r * K + i) >> 1), &a, &b);
      rowbuf[i] = to_f32(a * sigma);
      rowbuf[i + 1] = to_f32(b * sigma);
    }
    if (fmt == 1)
      synth_quantize_rows_cb(rowbuf, 1, K, nib + r * (K / 2), sc + r * (K / 32));
    else
      synth_quantize_rows(rowbuf, 1, K, nib + r * (K / 2), sc + r * (K / 32));
  }
}

/* One canonical expert blob; matrix m in {0: gate, 1: up, 2: down} uses key_m. */
void synth_expert_blob(uint64_t key, int64_t H, int64_t I, double sigma, int fmt, uint8_t* blob, float* scratch) {
  const int64_t mb = synth_matrix_bytes(I, H);
  gen_matrix(synth_key(key, 0, 0, 0, 0), I, H, sigma, fmt, blob, scratch);
  gen_matrix(synth_key(key, 1, 0, 0, 0), I, H, sigma, fmt, blob + mb, scratch);
  gen_matrix(synth_key(key, 2, 0, 0, 0), H, I, sigma, fmt, blob + 2 * mb, scratch);
}

typedef struct {
  uint64_t seed, layer, tag;
  int64_t H, I, e0, e1;
  double sigma;
  int fmt;
  uint8_t* out;
} job_t;

static void* expert_worker(void* p) {
  job_t* j = (job_t*)p;
  int64_t K = j->H > j->I ? j->H : j->I;
  float* scratch = (float*)__builtin_alloca((size_t)K * sizeof(float));
  const int64_t eb = synth_expert_bytes(j->H, j->I);
  for (int64_t e = j->e0; e < j->e1; ++e)
    synth_expert_blob(synth_key(j->seed, j->layer, j->tag, (uint64_t)e, 0), j->H, j->I, j->sigma, j->fmt,
                      j->out + (e - j->e0) * eb, scratch);
  return 0;
}

/*
 * Canonical blobs of experts [e0, e1) of `layer` (tag 3 = routed, 4 = shared)
 * in weight format `fmt`, written contiguously to `out`, on up to `threads`
 * threads.
 */
int synth_experts(uint64_t seed, uint64_t layer, uint64_t tag, int64_t H, int64_t I, int64_t e0, int64_t e1,
                  double sigma, int fmt, uint8_t* out, int threads) {
  if (H % 32 || I % 32 || e1 < e0 || fmt < 0 || fmt > 1) return -1;
  int64_t n = e1 - e0;
  if (threads < 1) threads = 1;
  if (threads > 64) threads = 64;
  if (threads > n) threads = (int)(n > 0 ? n : 1);
  pthread_t th[64];
  job_t jobs[64];
  const int64_t eb = synth_expert_bytes(H, I);
  for (int t = 0; t < threads; ++t) {
    int64_t a = e0 + n * t / threads, b = e0 + n * (t + 1) / threads;
    jobs[t] = (job_t){seed, layer, tag, H, I, a, b, sigma, fmt, out + (a - e0) * eb};
  }
  int ok[64] = {0};
  for (int t = 1; t < threads; ++t) ok[t] = pthread_create(&th[t], 0, expert_worker, &jobs[t]) == 0;
  expert_worker(&jobs[0]);
  for (int t = 1; t < threads; ++t) {
    if (ok[t]) pthread_join(th[t], 0);
    else expert_worker(&jobs[t]); /* thread creation failed: do the slice here */
  }
  return 0;
}

/* Router weights: E x H fp32, N(0, 1/H). */
void synth_router(uint64_t seed, uint64_t layer, int64_t E, int64_t H, float* W) {
  uint64_t key = synth_key(seed, layer, 1, 0, 0);
  double sigma = 1.0 / sqrt((double)H);
  for (int64_t i = 0; i < E * H; i += 2) {
    double a, b;
    normal_pair(key, (uint64_t)(i >> 1), &a, &b);
    W[i] = to_f32(a * sigma);
    if (i + 1 < E * H) W[i + 1] = to_f32(b * sigma);
  }
}

/*
 * Per-expert Zipf(s) popularity bias: b_e = -s * ln(1 + pi(e)) where pi is a
 * seeded permutation of 0..E-1 (Fisher-Yates on counter draws).  Adding b to
 * the logits multiplies expert e's softmax mass by rank^-s.
 */
void synth_zipf_bias(uint64_t seed, uint64_t layer, int64_t E, double s, float* bias, int32_t* perm_out) {
  uint64_t key = synth_key(seed, layer, 2, 0, 0);
  int32_t perm[4096];
  if (E > 4096) return;
  for (int64_t i = 0; i < E; ++i) perm[i] = (int32_t)i;
  for (int64_t i = E - 1; i > 0; --i) {
    uint64_t j = draw64(key, (uint64_t)i) % (uint64_t)(i + 1);
    int32_t t = perm[i];
    perm[i] = perm[j];
    perm[j] = t;
  }
  for (int64_t e = 0; e < E; ++e) {
    bias[e] = to_f32(-s * det_log(1.0 + (double)perm[e]));
    if (perm_out) perm_out[e] = perm[e];
  }
}

/*
 * Activations: token t of stream (seed, layer, tag) with resample index
 * sub[t] (0 unless the token was redrawn), H bf16 values of N(0, 1).
 */
void synth_x_bf16(uint64_t seed, uint64_t layer, uint64_t tag, int64_t t0, int64_t T, int64_t H,
                  const int32_t* sub, uint16_t* x) {
  for (int64_t t = 0; t < T; ++t) {
    uint64_t key = synth_key(seed, layer, 5, tag, (uint64_t)(t0 + t) * 1024u + (uint64_t)(sub ? sub[t] : 0));
    for (int64_t i = 0; i < H; i += 2) {
      double a, b;
      normal_pair(key, (uint64_t)(i >> 1), &a, &b);
      x[t * H + i] = f32_to_bf16(to_f32(a));
      x[t * H + i + 1] = f32_to_bf16(to_f32(b));
    }
  }
}

/* Exposed for tests of the generator itself. */
double synth_det_log(double x) { return det_log(x); }
uint16_t synth_f64_to_f16(double v) { return f64_to_f16(v); }
uint16_t synth_f32_to_bf16(float f) { return f32_to_bf16(f); }
