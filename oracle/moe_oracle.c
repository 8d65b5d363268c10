/*
 * CPU oracle for the quantized mixture-of-experts FFN layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this file's library.  The product
 * path never calls it, and it shares no code, header or table with the
 * CUDA library: it reads the canonical packed expert blobs directly and
 * computes everything in IEEE binary64, single-threaded, in the plain order
 * the definition states.
 *
 * What the layer computes (Qwen3.8-Flash-Next MoE FFN as described on the
 * Betelgeuse news page, section 机制 (48 layers, 512 routed experts per layer,
 * 10 routed + 1 shared per token) and section "bit-exact 的确切含义" (the
 * top-10 routing is never altered, no expert is ever dropped)):
 *
 *   logits   l[e]  = sum_h W_r[e,h] * x[h] + b[e]                 (router)
 *   select   S     = the k largest logits, ties to the lower index
 *   weights  w_j   = exp(l_j - m) / sum_{i in S} exp(l_i - m)     (softmax
 *                    over all E renormalised over S; m = max l)
 *   expert   g = W_g x, u = W_u x, h = silu(g) * u, y_e = W_d h
 *            with silu(z) = z / (1 + exp(-z))
 *   output   y = sum_{j in S} w_j y_{e_j} + y_shared              (shared
 *                    expert weight 1, outside the softmax)
 *
 * Weights are 4-bit symmetric blocks of 32 along the reduction axis with one
 * binary16 scale per block, dequantized as w = d * (u - 8) (u the stored
 * nibble).  Readings where the sources are silent (all listed in the design
 * notes): S is reported in ascending expert-index order and the combine runs
 * over S in that order; the shared expert has the routed experts' shape.
 *
 * Also here: RMSNorm + residual for the multi-layer stack, and a simulator
 * of the VRAM expert-slot pool with LRU eviction (Betelgeuse news page,
 * section 机制, 显存/调度 rows: a VRAM slot pool whose hit check runs on the
 * GPU; on a miss the host copies the expert in).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* scalar formats                                                       */
/* ------------------------------------------------------------------ */

/* IEEE binary16 -> binary64 (exact). */
static double half_to_double(uint16_t h) {
  int sign = h >> 15, ex = (h >> 10) & 31, man = h & 1023;
  double v;
  if (ex == 0) v = ldexp((double)man, -24);
  else if (ex == 31) v = man ? NAN : INFINITY;
  else v = ldexp((double)(1024 + man), ex - 25);
  return sign ? -v : v;
}

/* bfloat16 -> binary64 (exact). */
static double bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/*
 * binary64 -> bfloat16, round to nearest, ties to even, in one rounding
 * step (no detour through binary32).  Finite inputs only.
 */
static uint16_t double_to_bf16(double v) {
  if (v == 0.0) return signbit(v) ? 0x8000 : 0;
  uint16_t sign = v < 0 ? 0x8000 : 0;
  double a = fabs(v);
  int e;
  (void)frexp(a, &e);      /* a = m * 2^e, m in [0.5, 1) */
  /* bf16 normal: 8 significant bits; exponent range of binary32 */
  int E = e - 1;            /* a = (2m) * 2^E, 2m in [1, 2) */
  if (E < -126) {           /* subnormal bf16: multiples of 2^-133 */
    double k = nearbyint(ldexp(a, 133));
    return sign | (uint16_t)k;
  }
  double sig = nearbyint(ldexp(a, 7 - E)); /* in [128, 256] */
  if (sig >= 256.0) { sig = 128.0; E += 1; }
  if (E > 127) return sign | 0x7F80;
  return sign | (uint16_t)(((E + 127) << 7) | ((int)sig - 128));
}

/* ------------------------------------------------------------------ */
/* packed matrices                                                      */
/* ------------------------------------------------------------------ */

/* Bytes of one R x K packed matrix: nibble plane then scale plane. */
static int64_t matrix_bytes(int64_t R, int64_t K) { return R * (K / 2) + R * (K / 32) * 2; }

/*
 * Weight formats (the stored 4-bit value u of an element and its block's
 * fp16 scale d give the weight):
 *   0  linear:   w = d * (u - 8)
 *   1  codebook: w = d * C[u], C the 16 levels below: the standard normal
 *      distribution's quantiles at (u + 1/2) / 16, scaled so that the
 *      outermost is 127, rounded to integers (a non-linear 16-entry table
 *      per block scale, the kind of format the halogen-flash-server README
 *      lists under "Bring your own GGUF").
 */
static const double kLevels[16] = {-127, -90, -69, -53, -39, -27, -16, -5, 5, 16, 27, 39, 53, 69, 90, 127};

/* Dequantize row r of an R x K packed matrix of format fmt into out[K]. */
static void dequant_row(const uint8_t* mat, int64_t R, int64_t K, int64_t r, int fmt, double* out) {
  const uint8_t* nib = mat + r * (K / 2);
  const uint8_t* sc = mat + R * (K / 2) + r * (K / 32) * 2;
  for (int64_t c = 0; c < K; ++c) {
    int64_t blk = c / 32;
    uint16_t d16 = (uint16_t)(sc[2 * blk] | (sc[2 * blk + 1] << 8));
    uint8_t byte = nib[c / 2];
    int u = (c % 2 == 0) ? (byte & 15) : (byte >> 4);
    out[c] = half_to_double(d16) * (fmt == 1 ? kLevels[u] : (double)(u - 8));
  }
}

/* Whole matrix, row-major R x K, for tests. */
void oracle_dequant_matrix(const uint8_t* mat, int64_t R, int64_t K, int64_t fmt, double* out) {
  for (int64_t r = 0; r < R; ++r) dequant_row(mat, R, K, r, (int)fmt, out + r * K);
}

/* The codebook of format 1, for tests. */
void oracle_levels(double* out) { memcpy(out, kLevels, sizeof(kLevels)); }

int64_t oracle_expert_bytes(int64_t H, int64_t I) { return 3 * matrix_bytes(I, H); }

/* ------------------------------------------------------------------ */
/* router and selection                                                 */
/* ------------------------------------------------------------------ */

/* l[t*E + e] = sum_h W_r[e*H + h] * x[t*H + h] + b[e]  (b may be NULL). */
void oracle_router_logits(int64_t E, int64_t H, const float* W_r, const float* b, const uint16_t* x,
                          int64_t T, double* l) {
  for (int64_t t = 0; t < T; ++t) {
    for (int64_t e = 0; e < E; ++e) {
      double s = 0.0;
      for (int64_t h = 0; h < H; ++h) s += (double)W_r[e * H + h] * bf16_to_double(x[t * H + h]);
      l[t * E + e] = s + (b ? (double)b[e] : 0.0);
    }
  }
}

/* a ranks before b: larger logit, or equal logit and lower index. */
static int ranks_before(const double* l, int64_t a, int64_t b) {
  return l[a] > l[b] || (l[a] == l[b] && a < b);
}

/*
 * Top-k of one token's E logits.  by_rank[r] (optional) receives the
 * selected experts in rank order (logit descending, index ascending);
 * idx[j] the same set in ascending index order, and w[j] its routing
 * weight.  Returns the gap between the k-th and (k+1)-th ranked logits
 * (+inf when k == E).
 */
double oracle_topk(int64_t E, int64_t k, const double* l, int32_t* idx, double* w, int32_t* by_rank) {
  int32_t* taken = (int32_t*)calloc((size_t)E, sizeof(int32_t));
  int32_t* rank = (int32_t*)malloc((size_t)(k + 1) * sizeof(int32_t));
  int64_t nr = k < E ? k + 1 : k;
  for (int64_t r = 0; r < nr; ++r) {
    int64_t best = -1;
    for (int64_t e = 0; e < E; ++e)
      if (!taken[e] && (best < 0 || ranks_before(l, e, best))) best = e;
    taken[best] = 1;
    rank[r] = (int32_t)best;
  }
  double gap = k < E ? l[rank[k - 1]] - l[rank[k]] : INFINITY;
  if (by_rank)
    for (int64_t r = 0; r < k; ++r) by_rank[r] = rank[r];
  /* ascending index order of the first k */
  int64_t j = 0;
  for (int64_t e = 0; e < E && j < k; ++e) {
    int in = 0;
    for (int64_t r = 0; r < k; ++r) in |= rank[r] == e;
    if (in) idx[j++] = (int32_t)e;
  }
  double m = l[rank[0]], z = 0.0;
  for (int64_t q = 0; q < k; ++q) z += exp(l[idx[q]] - m);
  for (int64_t q = 0; q < k; ++q) w[q] = exp(l[idx[q]] - m) / z;
  free(taken);
  free(rank);
  return gap;
}

/* ------------------------------------------------------------------ */
/* expert FFN and the layer                                             */
/* ------------------------------------------------------------------ */

/*
 * One expert on one token: y[H] = W_d (silu(W_g x) * (W_u x)).
 * blob = canonical expert [W_g I x H][W_u I x H][W_d H x I] in weight format fmt.
 * h_out (optional) receives the I intermediate values.
 */
void oracle_expert(const uint8_t* blob, int64_t H, int64_t I, int64_t fmt, const double* x, double* y,
                   double* h_out) {
  const uint8_t* Wg = blob;
  const uint8_t* Wu = blob + matrix_bytes(I, H);
  const uint8_t* Wd = blob + 2 * matrix_bytes(I, H);
  double* row = (double*)malloc((size_t)(H > I ? H : I) * sizeof(double));
  double* h = (double*)malloc((size_t)I * sizeof(double));
  for (int64_t i = 0; i < I; ++i) {
    double g = 0.0, u = 0.0;
    dequant_row(Wg, I, H, i, (int)fmt, row);
    for (int64_t c = 0; c < H; ++c) g += row[c] * x[c];
    dequant_row(Wu, I, H, i, (int)fmt, row);
    for (int64_t c = 0; c < H; ++c) u += row[c] * x[c];
    h[i] = g / (1.0 + exp(-g)) * u;
  }
  for (int64_t r = 0; r < H; ++r) {
    double s = 0.0;
    dequant_row(Wd, H, I, r, (int)fmt, row);
    for (int64_t i = 0; i < I; ++i) s += row[i] * h[i];
    y[r] = s;
  }
  if (h_out) memcpy(h_out, h, (size_t)I * sizeof(double));
  free(row);
  free(h);
}

/*
 * The layer on T tokens.
 *   experts: E canonical blobs back to back; shared: one blob (or NULL for
 *            a layer without a shared expert)
 *   x:       T x H bf16 (the normalised activations the layer consumes)
 *   y:       T x H binary64
 *   idx, w:  T x k, ascending expert index per token
 *   logits:  T x E (optional), gap: T (optional, k-th minus (k+1)-th logit)
 *   force:   optional T x k expert sets to use instead of the router's
 *            choice (weights still from the logits); for cases where the
 *            router's decision is a near-tie that another summation order
 *            may legitimately resolve the other way.
 *   fmt:     weight format of every blob (0 linear, 1 codebook)
 */
void oracle_moe_forward(int64_t H, int64_t I, int64_t E, int64_t k, const float* W_r, const float* bias,
                        const uint8_t* experts, const uint8_t* shared, const uint16_t* x, int64_t T, double* y,
                        int32_t* idx, double* w, double* logits, double* gap, const int32_t* force, int64_t fmt) {
  const int64_t eb = oracle_expert_bytes(H, I);
  double* l = (double*)malloc((size_t)(T * E) * sizeof(double));
  double* xd = (double*)malloc((size_t)H * sizeof(double));
  double* ye = (double*)malloc((size_t)H * sizeof(double));
  oracle_router_logits(E, H, W_r, bias, x, T, l);
  for (int64_t t = 0; t < T; ++t) {
    const double* lt = l + t * E;
    int32_t* it = idx + t * k;
    double* wt = w + t * k;
    double g = oracle_topk(E, k, lt, it, wt, NULL);
    if (gap) gap[t] = g;
    if (force) {
      /* forced set, ascending order, weights renormalised over it */
      const int32_t* f = force + t * k;
      double m = -INFINITY, z = 0.0;
      for (int64_t j = 0; j < k; ++j) { it[j] = f[j]; if (lt[f[j]] > m) m = lt[f[j]]; }
      for (int64_t j = 0; j < k; ++j) z += exp(lt[it[j]] - m);
      for (int64_t j = 0; j < k; ++j) wt[j] = exp(lt[it[j]] - m) / z;
    }
    for (int64_t c = 0; c < H; ++c) xd[c] = bf16_to_double(x[t * H + c]);
    double* yt = y + t * H;
    for (int64_t c = 0; c < H; ++c) yt[c] = 0.0;
    for (int64_t j = 0; j < k; ++j) {
      oracle_expert(experts + (int64_t)it[j] * eb, H, I, fmt, xd, ye, NULL);
      for (int64_t c = 0; c < H; ++c) yt[c] += wt[j] * ye[c];
    }
    if (shared) {
      oracle_expert(shared, H, I, fmt, xd, ye, NULL);
      for (int64_t c = 0; c < H; ++c) yt[c] += ye[c];
    }
  }
  if (logits) memcpy(logits, l, (size_t)(T * E) * sizeof(double));
  free(l);
  free(xd);
  free(ye);
}

/* ------------------------------------------------------------------ */
/* RMSNorm and residual (multi-layer stack)                             */
/* ------------------------------------------------------------------ */

/*
 * Pre-norm without a learned weight: xhat = bf16(x / sqrt(mean(x^2) + eps)).
 * xhat_f64 (optional) receives the value before the bf16 rounding.
 */
void oracle_rmsnorm(int64_t H, const uint16_t* x, double eps, uint16_t* xhat, double* xhat_f64) {
  double ss = 0.0;
  for (int64_t c = 0; c < H; ++c) {
    double v = bf16_to_double(x[c]);
    ss += v * v;
  }
  double inv = 1.0 / sqrt(ss / (double)H + eps);
  for (int64_t c = 0; c < H; ++c) {
    double v = bf16_to_double(x[c]) * inv;
    if (xhat_f64) xhat_f64[c] = v;
    if (xhat) xhat[c] = double_to_bf16(v);
  }
}

/* x_next = bf16(x + y), both bf16 (the sum is exact in binary64). */
void oracle_residual(int64_t n, const uint16_t* x, const uint16_t* y, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = double_to_bf16(bf16_to_double(x[i]) + bf16_to_double(y[i]));
}

/* binary64 -> bf16 RNE, exposed for tests. */
void oracle_to_bf16(int64_t n, const double* v, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = double_to_bf16(v[i]);
}

/* ------------------------------------------------------------------ */
/* expert-slot pool simulator                                           */
/* ------------------------------------------------------------------ */

/*
 * Replays a trace of steps through an S-slot pool for E experts and lists
 * every miss.  Step n (1-based stamp n) selects the set sel[n*maxsel ..]
 * (any order, -1 padded, duplicates allowed; the union over the step's
 * tokens).  Rules:
 *   - an expert is a hit when the slot table maps it to a slot;
 *   - the step's misses are served in ascending expert index;
 *   - the i-th miss takes the i-th candidate slot, where the candidates are
 *     the empty slots in ascending order, then the occupied slots whose
 *     expert is not selected in this step, by (last-use stamp, slot index)
 *     ascending (least recently used first);
 *   - afterwards every selected expert's slot gets stamp n.
 * init_full != 0 starts with slot e holding expert e (needs S >= E);
 * otherwise the pool starts empty.  seed[0 .. n_seed) (a hot-expert
 * profile, distinct experts, n_seed <= S) then start resident: seed[i] in
 * slot i, last used before the first step (stamp 0).
 * miss_out receives (step, expert, slot) triples.  Returns the number of
 * misses, or -1 if a step selects more distinct experts than the pool can
 * hold, -2 if miss_out is too small, -3 for an invalid seed.
 */
int64_t oracle_pool_sim(int64_t E, int64_t S, int init_full, const int32_t* seed, int64_t n_seed, int64_t n_steps,
                        const int32_t* sel, int64_t maxsel, int32_t* miss_out, int64_t max_miss,
                        int32_t* final_table) {
  int32_t* table = (int32_t*)malloc((size_t)E * sizeof(int32_t));
  int32_t* owner = (int32_t*)malloc((size_t)S * sizeof(int32_t));
  int64_t* stamp = (int64_t*)calloc((size_t)S, sizeof(int64_t));
  uint8_t* used = (uint8_t*)malloc((size_t)E);
  int32_t* cand = (int32_t*)malloc((size_t)S * sizeof(int32_t));
  int64_t n_miss = 0, rc = 0;
  for (int64_t e = 0; e < E; ++e) table[e] = -1;
  for (int64_t s = 0; s < S; ++s) owner[s] = -1;
  if (init_full)
    for (int64_t e = 0; e < E && e < S; ++e) { table[e] = (int32_t)e; owner[e] = (int32_t)e; }
  /* seeding from a hot-expert profile: seed[i] starts resident in slot i,
     last used before the first step (stamp 0) */
  if (n_seed > S) rc = -3;
  for (int64_t i = 0; i < n_seed && rc == 0; ++i) {
    const int32_t e = seed[i];
    if (e < 0 || e >= E || table[e] >= 0 || owner[i] >= 0) { rc = -3; break; }
    table[e] = (int32_t)i;
    owner[i] = e;
  }
  for (int64_t n = 0; n < n_steps && rc == 0; ++n) {
    memset(used, 0, (size_t)E);
    int64_t distinct = 0;
    for (int64_t q = 0; q < maxsel; ++q) {
      int32_t e = sel[n * maxsel + q];
      if (e >= 0 && !used[e]) { used[e] = 1; ++distinct; }
    }
    if (distinct > S) { rc = -1; break; }
    /* candidate victims */
    int64_t nc = 0;
    for (int64_t s = 0; s < S; ++s)
      if (owner[s] < 0) cand[nc++] = (int32_t)s;
    int64_t first_occ = nc;
    for (int64_t s = 0; s < S; ++s)
      if (owner[s] >= 0 && !used[owner[s]]) cand[nc++] = (int32_t)s;
    /* insertion sort of the occupied candidates by (stamp, slot) */
    for (int64_t a = first_occ + 1; a < nc; ++a) {
      int32_t v = cand[a];
      int64_t b = a - 1;
      while (b >= first_occ && (stamp[cand[b]] > stamp[v] || (stamp[cand[b]] == stamp[v] && cand[b] > v))) {
        cand[b + 1] = cand[b];
        --b;
      }
      cand[b + 1] = v;
    }
    int64_t next = 0;
    for (int64_t e = 0; e < E; ++e) {
      if (!used[e] || table[e] >= 0) continue;
      int32_t s = cand[next++];
      if (owner[s] >= 0) table[owner[s]] = -1;
      owner[s] = (int32_t)e;
      table[e] = s;
      if (n_miss >= max_miss) { rc = -2; break; }
      miss_out[3 * n_miss + 0] = (int32_t)(n + 1);
      miss_out[3 * n_miss + 1] = (int32_t)e;
      miss_out[3 * n_miss + 2] = s;
      ++n_miss;
    }
    for (int64_t e = 0; e < E; ++e)
      if (used[e]) stamp[table[e]] = n + 1;
  }
  if (final_table) memcpy(final_table, table, (size_t)E * sizeof(int32_t));
  free(table);
  free(owner);
  free(stamp);
  free(used);
  free(cand);
  return rc ? rc : n_miss;
}
