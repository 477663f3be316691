/*
 * q3a_oracle.c — the CPU oracle of the Qwen3 attention core.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may call, link or load
 * this file: only the tests, the package's smoke check and the benchmark's
 * CPU-baseline leg use it. It shares no code, header, table or helper with the
 * CUDA library.
 *
 * What it computes, in plain fp64 loops on the exact bf16 input values
 * (widened without rounding; no intermediate rounding anywhere):
 *
 *   step 1  QK-Norm of one head row (length d):
 *             ms = (1/d) sum_i x_i^2 ;  y_i = x_i / sqrt(ms + eps) * gamma_i
 *           Source: "7.2 Qwen3 full-scale implementation" (paper.xwysyy.cn),
 *           §7.2.1 RMSNorm: variance = mean(x^2), x * rsqrt(variance + eps),
 *           times scale; no shift. The pages compute it in fp32; here fp64.
 *   step 2  rotate-half RoPE at integer position p:
 *             w_i = theta^(-2i/d), a_i = p * w_i, for i < d/2
 *             y'_i       = y_i cos a_i - y_{i+d/2} sin a_i
 *             y'_{i+d/2} = y_{i+d/2} cos a_i + y_i sin a_i
 *           Source: §7.2.1 compute_rope_params (inv_freq from arange(0,d,2)/d,
 *           angles duplicated to [a, a]) and apply_rope (x*cos + cat(-x2,x1)*sin).
 *           Step 2 is applied to the OUTPUT of step 1 (norm, then RoPE): the
 *           order of §7.2.1's GroupedQueryAttention.forward and of the quoted
 *           transformers Qwen3Attention.forward (llm.rainlin.net "Qwen3" note).
 *   step 3  query head h reads KV group h / g, g = Hq / Hkv
 *           (§7.2.1: keys.repeat_interleave(group_size, dim=1)).
 *   step 4  s_j = qhat . khat_j / sqrt(d), keys j = 0..i only (causal triu mask).
 *   step 5  o = sum_j softmax(s)_j v_j, with the softmax written as
 *           exp(s_j - max s) / sum exp(s_k - max s).
 *           Source: §7.2.1 GroupedQueryAttention.forward (masked_fill with -inf,
 *           softmax(scores / head_dim**0.5), @ values).
 *   chunk   a chunk of Tq new tokens of sequence b at positions start_pos[b]+t:
 *           cached rows 0..start_pos[b]-1 as stored, then the chunk's own keys
 *           (steps 1-2 at their positions) under the causal mask; the same
 *           section of the book.ozine.me chapter (rectangular causal mask from
 *           pos_start).
 *   decode  the new token at p = start_pos: qhat and khat_new from steps 1-2 at
 *           p; keys = cached rows 0..p-1 exactly as stored (never re-normalised
 *           or re-rotated), then khat_new; values = cached rows 0..p-1, then
 *           v_new. Source: "Chapter 20, Qwen3 and Qwen3.5" (book.ozine.me),
 *           §20.3: the new K is rotated at start_pos and concatenated; old K
 *           already carries its position.
 *
 *   rounded  the same prefill with qhat and khat rounded to bf16 (nearest,
 *           ties to even) where a bf16 model rounds them: after step 2 only
 *           (roundings = 1: the tensors a bf16 attention multiplies), or after
 *           step 1 and again after step 2 (roundings = 2: §7.2.1's RMSNorm
 *           returns .to(input_dtype) and apply_rope returns .to(x.dtype)).
 *           Everything else stays fp64. With large gammas the logits are large
 *           and these roundings alone move the output by more than the bf16
 *           output tolerance; this variant is the reference for that regime.
 *
 * Readings where the pages are silent or disagree (kept in the design notes):
 *   - norm BEFORE RoPE (four pages and the quoted transformers code; the
 *     Qwen1->3 blog page says the opposite);
 *   - no rounding of the normalised or rotated values in the plain functions
 *     (the pages' code rounds to the model dtype after each step; the
 *     tolerance of the tests covers it at the workloads' gammas);
 *   - prefill positions start at 0.
 *
 * All entry points return 0 on success and a negative value on a bad argument.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 -> fp64, exact: a bf16 value is the top 16 bits of an fp32. */
static double widen_bf16(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* fp64 -> nearest bf16 value (8 significant bits, ties to even; subnormal
 * spacing 2^-133; beyond the largest finite bf16 -> infinity), as fp64. */
static double round_bf16(double x) {
  if (!isfinite(x) || x == 0.0) return x;
  int e;
  (void)frexp(x, &e); /* |x| = m 2^e, 0.5 <= m < 1 */
  int q = e - 8;      /* spacing of bf16 values at |x| */
  if (q < -133) q = -133;
  double y = ldexp(nearbyint(ldexp(x, -q)), q); /* default mode: ties to even */
  if (fabs(y) > 3.3895313892515355e38) return copysign(INFINITY, x);
  return y;
}

void q3a_oracle_round_bf16(const double* x, long n, double* y) {
  for (long i = 0; i < n; ++i) y[i] = round_bf16(x[i]);
}

static void round_row(double* y, int d) {
  for (int c = 0; c < d; ++c) y[c] = round_bf16(y[c]);
}

static int g_threads = 0; /* 0: OpenMP default */

void q3a_oracle_set_threads(int n) { g_threads = n > 0 ? n : 0; }

int q3a_oracle_threads(void) {
#ifdef _OPENMP
  return g_threads > 0 ? g_threads : omp_get_max_threads();
#else
  return 1;
#endif
}

#ifdef _OPENMP
#define OMP_THREADS (g_threads > 0 ? g_threads : omp_get_max_threads())
#endif

/* step 1 on one row; y may not alias x. */
void q3a_oracle_rmsnorm_row(const uint16_t* x, const uint16_t* gamma, int d, double eps,
                            double* y) {
  double sum_sq = 0.0;
  for (int i = 0; i < d; ++i) {
    double xi = widen_bf16(x[i]);
    sum_sq += xi * xi;
  }
  double mean_sq = sum_sq / (double)d;
  double inv_rms = 1.0 / sqrt(mean_sq + eps);
  for (int i = 0; i < d; ++i) y[i] = widen_bf16(x[i]) * inv_rms * widen_bf16(gamma[i]);
}

/* step 2 on one fp64 row, in place. */
void q3a_oracle_rope_row(double* y, int d, double pos, double theta) {
  int half = d / 2;
  for (int i = 0; i < half; ++i) {
    double w = pow(theta, -(2.0 * (double)i) / (double)d);
    double a = pos * w;
    double c = cos(a), s = sin(a);
    double lo = y[i], hi = y[i + half];
    y[i] = lo * c - hi * s;
    y[i + half] = hi * c + lo * s;
  }
}

/* steps 1 then 2 on every row of x [B, T, H, d]; row (b, t, h) at pos0 + t.
 * out is fp64 [B, T, H, d]. */
int q3a_oracle_qknorm_rope(const uint16_t* x, const uint16_t* gamma, int B, int T, int H,
                           int d, long pos0, double theta, double eps, double* out) {
  if (B < 0 || T < 0 || H < 0 || d <= 0 || (d & 1) || !x || !gamma || !out) return -1;
  long rows = (long)B * T * H;
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(OMP_THREADS)
#endif
  for (long r = 0; r < rows; ++r) {
    long t = (r / H) % T;
    q3a_oracle_rmsnorm_row(x + r * d, gamma, d, eps, out + r * d);
    q3a_oracle_rope_row(out + r * d, d, (double)(pos0 + t), theta);
  }
  return 0;
}

/* Steps 4-5 for one query row against n keys/values given as fp64 rows
 * (keys[j*d..], vals[j*d..]); writes o[d]. */
static void attend_row(const double* qhat, const double* keys, const double* vals, long n,
                       int d, double* scores, double* o) {
  double scale = 1.0 / sqrt((double)d);
  double m = -INFINITY;
  for (long j = 0; j < n; ++j) {
    double s = 0.0;
    for (int c = 0; c < d; ++c) s += qhat[c] * keys[j * d + c];
    s *= scale;
    scores[j] = s;
    if (s > m) m = s;
  }
  double z = 0.0;
  for (long j = 0; j < n; ++j) {
    scores[j] = exp(scores[j] - m);
    z += scores[j];
  }
  for (int c = 0; c < d; ++c) o[c] = 0.0;
  for (long j = 0; j < n; ++j) {
    double p = scores[j] / z;
    for (int c = 0; c < d; ++c) o[c] += p * vals[j * d + c];
  }
}

static int check_shape(int B, int T, int Hq, int Hkv, int d) {
  if (B < 0 || T < 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || (d & 1)) return -1;
  if (Hq % Hkv) return -1;
  return 0;
}

/* steps 1-2 on one row, with the bf16 roundings of the "rounded" variant */
static void norm_rope_rounded(const uint16_t* x, const uint16_t* gamma, int d, double eps,
                              double pos, double theta, int roundings, double* y) {
  q3a_oracle_rmsnorm_row(x, gamma, d, eps, y);
  if (roundings >= 2) round_row(y, d);
  q3a_oracle_rope_row(y, d, pos, theta);
  if (roundings >= 1) round_row(y, d);
}

static int prefill_impl(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                        const uint16_t* q_gamma, const uint16_t* k_gamma, int B, int T, int Hq,
                        int Hkv, int d, double theta, double eps, int roundings, double* out);

/* Full causal prefill. q [B,T,Hq,d], k/v [B,T,Hkv,d] bf16; out fp64 [B,T,Hq,d]. */
int q3a_oracle_prefill(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                       const uint16_t* q_gamma, const uint16_t* k_gamma, int B, int T, int Hq,
                       int Hkv, int d, double theta, double eps, double* out) {
  return prefill_impl(q, k, v, q_gamma, k_gamma, B, T, Hq, Hkv, d, theta, eps, 0, out);
}

/* The prefill with qhat and khat rounded to bf16: roundings = 1 after step 2,
 * roundings = 2 after step 1 and after step 2 (see the header). */
int q3a_oracle_prefill_rounded(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                               const uint16_t* q_gamma, const uint16_t* k_gamma, int B, int T,
                               int Hq, int Hkv, int d, double theta, double eps, int roundings,
                               double* out) {
  if (roundings < 0 || roundings > 2) return -1;
  return prefill_impl(q, k, v, q_gamma, k_gamma, B, T, Hq, Hkv, d, theta, eps, roundings, out);
}

static int prefill_impl(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                        const uint16_t* q_gamma, const uint16_t* k_gamma, int B, int T, int Hq,
                        int Hkv, int d, double theta, double eps, int roundings, double* out) {
  if (check_shape(B, T, Hq, Hkv, d) || !q || !k || !v || !q_gamma || !k_gamma || !out) return -1;
  int g = Hq / Hkv;
  long krows = (long)B * T * Hkv;
  /* khat and v for all (b, t, kv), stored per (b, kv) contiguously over t. */
  double* khat = (double*)malloc(sizeof(double) * (size_t)krows * d);
  double* vals = (double*)malloc(sizeof(double) * (size_t)krows * d);
  if (!khat || !vals) {
    free(khat);
    free(vals);
    return -2;
  }
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(OMP_THREADS)
#endif
  for (long r = 0; r < krows; ++r) {
    long b = r / ((long)T * Hkv), t = (r / Hkv) % T, kv = r % Hkv;
    double* kd = khat + (((b * Hkv + kv) * T) + t) * d;
    double* vd = vals + (((b * Hkv + kv) * T) + t) * d;
    norm_rope_rounded(k + r * d, k_gamma, d, eps, (double)t, theta, roundings, kd);
    for (int c = 0; c < d; ++c) vd[c] = widen_bf16(v[r * d + c]);
  }
  long qrows = (long)B * T * Hq;
  int failed = 0;
#ifdef _OPENMP
#pragma omp parallel num_threads(OMP_THREADS)
#endif
  {
    double* qhat = (double*)malloc(sizeof(double) * d);
    double* scores = (double*)malloc(sizeof(double) * (T > 0 ? T : 1));
    if (!qhat || !scores) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
      failed = 1;
    } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 16)
#endif
      for (long r = 0; r < qrows; ++r) {
        long b = r / ((long)T * Hq), i = (r / Hq) % T, h = r % Hq;
        long kv = h / g;
        norm_rope_rounded(q + r * d, q_gamma, d, eps, (double)i, theta, roundings, qhat);
        const double* kb = khat + (b * Hkv + kv) * (long)T * d;
        const double* vb = vals + (b * Hkv + kv) * (long)T * d;
        attend_row(qhat, kb, vb, i + 1, d, scores, out + r * d);
      }
    }
    free(qhat);
    free(scores);
  }
  free(khat);
  free(vals);
  return failed ? -2 : 0;
}

/* Sampled causal prefill: n rows given by (rb[s], rt[s], rh[s]); each output row
 * is computed from scratch (its keys 0..t normalised and rotated here).
 * out fp64 [n, d]. */
int q3a_oracle_prefill_rows(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                            const uint16_t* q_gamma, const uint16_t* k_gamma, int B, int T,
                            int Hq, int Hkv, int d, double theta, double eps, long n,
                            const int32_t* rb, const int32_t* rt, const int32_t* rh,
                            double* out) {
  if (check_shape(B, T, Hq, Hkv, d) || n < 0 || !out) return -1;
  for (long s = 0; s < n; ++s)
    if (rb[s] < 0 || rb[s] >= B || rt[s] < 0 || rt[s] >= T || rh[s] < 0 || rh[s] >= Hq)
      return -1;
  int g = Hq / Hkv;
  int failed = 0;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(OMP_THREADS)
#endif
  for (long s = 0; s < n; ++s) {
    long b = rb[s], i = rt[s], h = rh[s], kv = h / g;
    long nk = i + 1;
    double* keys = (double*)malloc(sizeof(double) * (size_t)nk * d);
    double* vals = (double*)malloc(sizeof(double) * (size_t)nk * d);
    double* scores = (double*)malloc(sizeof(double) * (size_t)nk);
    double* qhat = (double*)malloc(sizeof(double) * d);
    if (!keys || !vals || !scores || !qhat) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
      failed = 1;
    } else {
      for (long j = 0; j < nk; ++j) {
        long r = ((b * T + j) * Hkv + kv) * d;
        q3a_oracle_rmsnorm_row(k + r, k_gamma, d, eps, keys + j * d);
        q3a_oracle_rope_row(keys + j * d, d, (double)j, theta);
        for (int c = 0; c < d; ++c) vals[j * d + c] = widen_bf16(v[r + c]);
      }
      long rq = ((b * T + i) * Hq + h) * d;
      q3a_oracle_rmsnorm_row(q + rq, q_gamma, d, eps, qhat);
      q3a_oracle_rope_row(qhat, d, (double)i, theta);
      attend_row(qhat, keys, vals, nk, d, scores, out + s * d);
    }
    free(keys);
    free(vals);
    free(scores);
    free(qhat);
  }
  return failed ? -2 : 0;
}

/* Decode of one new token per sequence.
 *   q [B,Hq,d], k_new/v_new [B,Hkv,d] bf16; caches [B,Hkv,S_max,d] bf16 (rows
 *   0..start_pos[b]-1 read as stored); start_pos [B].
 *   out fp64 [B,Hq,d]; k_row fp64 [B,Hkv,d] = the normalised, rotated new key
 *   (the row a decode appends to the cache, before any rounding).
 * Only the sequences with sel[b] != 0 are computed (sel may be NULL: all). */
int q3a_oracle_decode(const uint16_t* q, const uint16_t* k_new, const uint16_t* v_new,
                      const uint16_t* k_cache, const uint16_t* v_cache, const int32_t* start_pos,
                      const uint16_t* q_gamma, const uint16_t* k_gamma, int B, int Hq, int Hkv,
                      int d, long S_max, double theta, double eps, const uint8_t* sel,
                      double* out, double* k_row) {
  if (check_shape(B, 1, Hq, Hkv, d) || S_max <= 0 || !out || !k_row) return -1;
  for (int b = 0; b < B; ++b)
    if (start_pos[b] < 0 || (long)start_pos[b] + 1 > S_max) return -1;
  int g = Hq / Hkv;
  long units = (long)B * Hkv;
  int failed = 0;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(OMP_THREADS)
#endif
  for (long u = 0; u < units; ++u) {
    long b = u / Hkv, kv = u % Hkv;
    if (sel && !sel[b]) continue;
    long p = start_pos[b];
    long nk = p + 1;
    double* keys = (double*)malloc(sizeof(double) * (size_t)nk * d);
    double* vals = (double*)malloc(sizeof(double) * (size_t)nk * d);
    double* scores = (double*)malloc(sizeof(double) * (size_t)nk);
    double* qhat = (double*)malloc(sizeof(double) * d);
    if (!keys || !vals || !scores || !qhat) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
      failed = 1;
    } else {
      const uint16_t* kc = k_cache + (b * Hkv + kv) * S_max * d;
      const uint16_t* vc = v_cache + (b * Hkv + kv) * S_max * d;
      for (long j = 0; j < p; ++j)
        for (int c = 0; c < d; ++c) {
          keys[j * d + c] = widen_bf16(kc[j * d + c]);
          vals[j * d + c] = widen_bf16(vc[j * d + c]);
        }
      double* kn = keys + p * d;
      q3a_oracle_rmsnorm_row(k_new + (b * Hkv + kv) * d, k_gamma, d, eps, kn);
      q3a_oracle_rope_row(kn, d, (double)p, theta);
      for (int c = 0; c < d; ++c) {
        k_row[(b * Hkv + kv) * d + c] = kn[c];
        vals[p * d + c] = widen_bf16(v_new[(b * Hkv + kv) * d + c]);
      }
      for (long h = kv * g; h < (kv + 1) * g; ++h) {
        q3a_oracle_rmsnorm_row(q + (b * Hq + h) * d, q_gamma, d, eps, qhat);
        q3a_oracle_rope_row(qhat, d, (double)p, theta);
        attend_row(qhat, keys, vals, nk, d, scores, out + (b * Hq + h) * d);
      }
    }
    free(keys);
    free(vals);
    free(scores);
    free(qhat);
  }
  return failed ? -2 : 0;
}

/* Chunked prefill against a KV cache ("Chapter 20, Qwen3 and Qwen3.5", §20.3:
 * the model keeps a position counter and builds a rectangular causal mask
 * starting at pos_start; the new keys are rotated at their own positions and
 * concatenated to the cached ones, which are not rotated again).
 *   q [B,Tq,Hq,d], k/v [B,Tq,Hkv,d] bf16: the chunk's projected rows;
 *   caches [B,Hkv,S_max,d] bf16: rows 0..start_pos[b]-1 read as stored;
 *   token t of sequence b sits at position p = start_pos[b] + t and attends
 *   to the cached rows 0..start_pos[b]-1 and the chunk's keys 0..t.
 *   out fp64 [B,Tq,Hq,d]; k_rows fp64 [B,Tq,Hkv,d] = the normalised, rotated
 *   chunk keys (the rows a call appends to the cache, before rounding). */
int q3a_oracle_prefill_chunk(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                             const uint16_t* k_cache, const uint16_t* v_cache,
                             const int32_t* start_pos, const uint16_t* q_gamma,
                             const uint16_t* k_gamma, int B, int Tq, int Hq, int Hkv, int d,
                             long S_max, double theta, double eps, double* out, double* k_rows) {
  if (check_shape(B, Tq, Hq, Hkv, d) || S_max <= 0 || !out || !k_rows) return -1;
  for (int b = 0; b < B; ++b)
    if (start_pos[b] < 0 || (long)start_pos[b] + Tq > S_max) return -1;
  int g = Hq / Hkv;
  long units = (long)B * Hkv;
  int failed = 0;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(OMP_THREADS)
#endif
  for (long u = 0; u < units; ++u) {
    long b = u / Hkv, kv = u % Hkv;
    long p0 = start_pos[b];
    long n_all = p0 + Tq;
    double* keys = (double*)malloc(sizeof(double) * (size_t)(n_all > 0 ? n_all : 1) * d);
    double* vals = (double*)malloc(sizeof(double) * (size_t)(n_all > 0 ? n_all : 1) * d);
    double* scores = (double*)malloc(sizeof(double) * (size_t)(n_all > 0 ? n_all : 1));
    double* qhat = (double*)malloc(sizeof(double) * d);
    if (!keys || !vals || !scores || !qhat) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
      failed = 1;
    } else {
      const uint16_t* kc = k_cache + (b * Hkv + kv) * S_max * d;
      const uint16_t* vc = v_cache + (b * Hkv + kv) * S_max * d;
      for (long j = 0; j < p0; ++j)
        for (int c = 0; c < d; ++c) {
          keys[j * d + c] = widen_bf16(kc[j * d + c]);
          vals[j * d + c] = widen_bf16(vc[j * d + c]);
        }
      for (long t = 0; t < Tq; ++t) {
        long r = ((b * Tq + t) * Hkv + kv) * d;
        double* kn = keys + (p0 + t) * d;
        q3a_oracle_rmsnorm_row(k + r, k_gamma, d, eps, kn);
        q3a_oracle_rope_row(kn, d, (double)(p0 + t), theta);
        for (int c = 0; c < d; ++c) {
          k_rows[r + c] = kn[c];
          vals[(p0 + t) * d + c] = widen_bf16(v[r + c]);
        }
      }
      for (long t = 0; t < Tq; ++t)
        for (long h = kv * g; h < (kv + 1) * g; ++h) {
          long rq = ((b * Tq + t) * Hq + h) * d;
          q3a_oracle_rmsnorm_row(q + rq, q_gamma, d, eps, qhat);
          q3a_oracle_rope_row(qhat, d, (double)(p0 + t), theta);
          attend_row(qhat, keys, vals, p0 + t + 1, d, scores, out + rq);
        }
    }
    free(keys);
    free(vals);
    free(scores);
    free(qhat);
  }
  return failed ? -2 : 0;
}

/* ==========================================================================
 * The gated global-attention layer of Qwen3-Next / Qwen3.5.
 * Sources: "Chapter 20, Qwen3 and Qwen3.5" (book.ozine.me) §20.4 (zero-
 * initialised norm weight used as 1 + w; W_query emitting 2*H*d values that
 * are split into query and gate inside each head; z = Attn(Q,K,V) * sigmoid
 * (gate); Q/K normalised per head, then rotated; partial_rotary_factor:
 * only the first d_r coordinates rotate, with d_r as the denominator of the
 * frequency exponent), and "14. The Qwen family" (niuwancheng.cn), the
 * Qwen3-Next section (q_proj output doubled, half query and half gate;
 * head_dim 256 with RoPE on 64 dims; x_hat * (1 + weight)).
 *
 *   g1  per head h of a token, qg[h*2d .. h*2d+d-1] is the query row and
 *       qg[h*2d+d .. h*2d+2d-1] the gate row;
 *   g2  zero-centred RMSNorm: y_i = x_i / sqrt(mean x^2 + eps) * (1 + w_i);
 *   g3  rotate-half RoPE on y_0..y_{d_r-1} alone (steps 2 with d := d_r, so
 *       w_i = theta^(-2i/d_r) and pairs (i, i + d_r/2)); y_{d_r}.. pass through;
 *   g4  steps 3-5 (GQA map h -> h/g, causal mask, softmax of q.k/sqrt(d), P.V);
 *   g5  z_c = o_c * sigmoid(gate_c), sigmoid(x) = 1 / (1 + exp(-x)).
 * ========================================================================== */

/* g2 on one row; y may not alias x. */
void q3a_oracle_zc_rmsnorm_row(const uint16_t* x, const uint16_t* w, int d, double eps,
                               double* y) {
  double sum_sq = 0.0;
  for (int i = 0; i < d; ++i) {
    double xi = widen_bf16(x[i]);
    sum_sq += xi * xi;
  }
  double inv_rms = 1.0 / sqrt(sum_sq / (double)d + eps);
  for (int i = 0; i < d; ++i) y[i] = widen_bf16(x[i]) * inv_rms * (1.0 + widen_bf16(w[i]));
}

/* g3 on one fp64 row of length d, in place (d is only checked against d_r). */
int q3a_oracle_partial_rope_row(double* y, int d, int d_r, double pos, double theta) {
  if (d_r < 0 || (d_r & 1) || d_r > d) return -1;
  if (d_r > 0) q3a_oracle_rope_row(y, d_r, pos, theta);
  return 0;
}

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

static int check_gated(int B, int T, int Hq, int Hkv, int d, int d_r) {
  if (check_shape(B, T, Hq, Hkv, d)) return -1;
  if (d_r < 0 || (d_r & 1) || d_r > d) return -1;
  return 0;
}

/* The output row of query head h of token i of sequence b (g1-g5), with the
 * keys 0..i normalised and rotated here. out[d]. */
static int gated_row(const uint16_t* qg, const uint16_t* k, const uint16_t* v,
                     const uint16_t* q_w, const uint16_t* k_w, int T, int Hq, int Hkv, int d,
                     int d_r, double theta, double eps, long b, long i, long h, double* out) {
  long kv = h / (Hq / Hkv);
  long nk = i + 1;
  double* keys = (double*)malloc(sizeof(double) * (size_t)nk * d);
  double* vals = (double*)malloc(sizeof(double) * (size_t)nk * d);
  double* scores = (double*)malloc(sizeof(double) * (size_t)nk);
  double* qhat = (double*)malloc(sizeof(double) * d);
  int rc = 0;
  if (!keys || !vals || !scores || !qhat) {
    rc = -2;
  } else {
    for (long j = 0; j < nk; ++j) {
      long r = ((b * T + j) * Hkv + kv) * d;
      q3a_oracle_zc_rmsnorm_row(k + r, k_w, d, eps, keys + j * d);
      q3a_oracle_partial_rope_row(keys + j * d, d, d_r, (double)j, theta);
      for (int c = 0; c < d; ++c) vals[j * d + c] = widen_bf16(v[r + c]);
    }
    const uint16_t* qrow = qg + ((b * T + i) * Hq + h) * 2L * d; /* g1: query half */
    const uint16_t* grow = qrow + d;                              /* g1: gate half */
    q3a_oracle_zc_rmsnorm_row(qrow, q_w, d, eps, qhat);
    q3a_oracle_partial_rope_row(qhat, d, d_r, (double)i, theta);
    attend_row(qhat, keys, vals, nk, d, scores, out);
    for (int c = 0; c < d; ++c) out[c] *= sigmoid(widen_bf16(grow[c]));
  }
  free(keys);
  free(vals);
  free(scores);
  free(qhat);
  return rc;
}

/* Full gated causal prefill. qg [B,T,Hq,2d], k/v [B,T,Hkv,d] bf16, q_w/k_w [d]
 * bf16 (zero-centred weights); out fp64 [B,T,Hq,d]. Keys are normalised and
 * rotated once per (b, t, kv) and shared by the rows that read them. */
int q3a_oracle_gated_prefill(const uint16_t* qg, const uint16_t* k, const uint16_t* v,
                             const uint16_t* q_w, const uint16_t* k_w, int B, int T, int Hq,
                             int Hkv, int d, int d_r, double theta, double eps, double* out) {
  if (check_gated(B, T, Hq, Hkv, d, d_r) || !qg || !k || !v || !q_w || !k_w || !out) return -1;
  int g = Hq / Hkv;
  long krows = (long)B * T * Hkv;
  double* khat = (double*)malloc(sizeof(double) * (size_t)(krows > 0 ? krows : 1) * d);
  double* vals = (double*)malloc(sizeof(double) * (size_t)(krows > 0 ? krows : 1) * d);
  if (!khat || !vals) {
    free(khat);
    free(vals);
    return -2;
  }
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(OMP_THREADS)
#endif
  for (long r = 0; r < krows; ++r) {
    long b = r / ((long)T * Hkv), t = (r / Hkv) % T, kv = r % Hkv;
    double* kd = khat + (((b * Hkv + kv) * T) + t) * d;
    double* vd = vals + (((b * Hkv + kv) * T) + t) * d;
    q3a_oracle_zc_rmsnorm_row(k + r * d, k_w, d, eps, kd);
    q3a_oracle_partial_rope_row(kd, d, d_r, (double)t, theta);
    for (int c = 0; c < d; ++c) vd[c] = widen_bf16(v[r * d + c]);
  }
  long qrows = (long)B * T * Hq;
  int failed = 0;
#ifdef _OPENMP
#pragma omp parallel num_threads(OMP_THREADS)
#endif
  {
    double* qhat = (double*)malloc(sizeof(double) * d);
    double* scores = (double*)malloc(sizeof(double) * (T > 0 ? T : 1));
    if (!qhat || !scores) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
      failed = 1;
    } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 16)
#endif
      for (long r = 0; r < qrows; ++r) {
        long b = r / ((long)T * Hq), i = (r / Hq) % T, h = r % Hq;
        long kv = h / g;
        const uint16_t* qrow = qg + r * 2L * d; /* g1: query half, then gate half */
        const uint16_t* grow = qrow + d;
        q3a_oracle_zc_rmsnorm_row(qrow, q_w, d, eps, qhat);
        q3a_oracle_partial_rope_row(qhat, d, d_r, (double)i, theta);
        attend_row(qhat, khat + (b * Hkv + kv) * (long)T * d,
                   vals + (b * Hkv + kv) * (long)T * d, i + 1, d, scores, out + r * d);
        for (int c = 0; c < d; ++c) out[r * d + c] *= sigmoid(widen_bf16(grow[c]));
      }
    }
    free(qhat);
    free(scores);
  }
  free(khat);
  free(vals);
  return failed ? -2 : 0;
}

/* Sampled gated prefill: n rows (rb[s], rt[s], rh[s]); out fp64 [n, d]. */
int q3a_oracle_gated_prefill_rows(const uint16_t* qg, const uint16_t* k, const uint16_t* v,
                                  const uint16_t* q_w, const uint16_t* k_w, int B, int T,
                                  int Hq, int Hkv, int d, int d_r, double theta, double eps,
                                  long n, const int32_t* rb, const int32_t* rt,
                                  const int32_t* rh, double* out) {
  if (check_gated(B, T, Hq, Hkv, d, d_r) || n < 0 || !out) return -1;
  for (long s = 0; s < n; ++s)
    if (rb[s] < 0 || rb[s] >= B || rt[s] < 0 || rt[s] >= T || rh[s] < 0 || rh[s] >= Hq)
      return -1;
  int failed = 0;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(OMP_THREADS)
#endif
  for (long s = 0; s < n; ++s) {
    if (gated_row(qg, k, v, q_w, k_w, T, Hq, Hkv, d, d_r, theta, eps, rb[s], rt[s], rh[s],
                  out + s * d)) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
      failed = 1;
    }
  }
  return failed ? -2 : 0;
}

/* g2 then g3 on every row of a [B, T, H, stride] bf16 array (the first d
 * elements of each row are the head row; stride = 2d for the query halves of
 * the query/gate projection, d for keys). Row (b, t, h) at position pos0 + t.
 * out fp64 [B, T, H, d]. */
int q3a_oracle_gated_qknorm_rope(const uint16_t* x, long stride, const uint16_t* w, int B, int T,
                                 int H, int d, int d_r, long pos0, double theta, double eps,
                                 double* out) {
  if (B < 0 || T < 0 || H < 0 || d <= 0 || stride < d || d_r < 0 || (d_r & 1) || d_r > d ||
      !x || !w || !out)
    return -1;
  long rows = (long)B * T * H;
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(OMP_THREADS)
#endif
  for (long r = 0; r < rows; ++r) {
    long t = (r / H) % T;
    q3a_oracle_zc_rmsnorm_row(x + r * stride, w, d, eps, out + r * d);
    q3a_oracle_partial_rope_row(out + r * d, d, d_r, (double)(pos0 + t), theta);
  }
  return 0;
}

/* Gated decode: one new token per sequence at p = start_pos[b] (g1-g5 with the
 * KV cache of §20.3): qhat from the query half of qg [B,Hq,2d] at p,
 * khat_new = g3(g2(k_new)) at p; keys = cache rows 0..p-1 as stored, then
 * khat_new; values = cache rows 0..p-1, then v_new; z = o * sigmoid(gate).
 *   caches [B,Hkv,S_max,d]; out fp64 [B,Hq,d]; k_row fp64 [B,Hkv,d]. */
int q3a_oracle_gated_decode(const uint16_t* qg, const uint16_t* k_new, const uint16_t* v_new,
                            const uint16_t* k_cache, const uint16_t* v_cache,
                            const int32_t* start_pos, const uint16_t* q_w, const uint16_t* k_w,
                            int B, int Hq, int Hkv, int d, int d_r, long S_max, double theta,
                            double eps, double* out, double* k_row) {
  if (check_gated(B, 1, Hq, Hkv, d, d_r) || S_max <= 0 || !out || !k_row) return -1;
  for (int b = 0; b < B; ++b)
    if (start_pos[b] < 0 || (long)start_pos[b] + 1 > S_max) return -1;
  int g = Hq / Hkv;
  long units = (long)B * Hkv;
  int failed = 0;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(OMP_THREADS)
#endif
  for (long u = 0; u < units; ++u) {
    long b = u / Hkv, kv = u % Hkv;
    long p = start_pos[b];
    long nk = p + 1;
    double* keys = (double*)malloc(sizeof(double) * (size_t)nk * d);
    double* vals = (double*)malloc(sizeof(double) * (size_t)nk * d);
    double* scores = (double*)malloc(sizeof(double) * (size_t)nk);
    double* qhat = (double*)malloc(sizeof(double) * d);
    if (!keys || !vals || !scores || !qhat) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
      failed = 1;
    } else {
      const uint16_t* kc = k_cache + (b * Hkv + kv) * S_max * d;
      const uint16_t* vc = v_cache + (b * Hkv + kv) * S_max * d;
      for (long j = 0; j < p; ++j)
        for (int c = 0; c < d; ++c) {
          keys[j * d + c] = widen_bf16(kc[j * d + c]);
          vals[j * d + c] = widen_bf16(vc[j * d + c]);
        }
      double* kn = keys + p * d;
      q3a_oracle_zc_rmsnorm_row(k_new + (b * Hkv + kv) * d, k_w, d, eps, kn);
      q3a_oracle_partial_rope_row(kn, d, d_r, (double)p, theta);
      for (int c = 0; c < d; ++c) {
        k_row[(b * Hkv + kv) * d + c] = kn[c];
        vals[p * d + c] = widen_bf16(v_new[(b * Hkv + kv) * d + c]);
      }
      for (long h = kv * g; h < (kv + 1) * g; ++h) {
        const uint16_t* qrow = qg + (b * Hq + h) * 2L * d; /* g1 */
        const uint16_t* grow = qrow + d;
        double* o = out + (b * Hq + h) * d;
        q3a_oracle_zc_rmsnorm_row(qrow, q_w, d, eps, qhat);
        q3a_oracle_partial_rope_row(qhat, d, d_r, (double)p, theta);
        attend_row(qhat, keys, vals, nk, d, scores, o);
        for (int c = 0; c < d; ++c) o[c] *= sigmoid(widen_bf16(grow[c]));
      }
    }
    free(keys);
    free(vals);
    free(scores);
    free(qhat);
  }
  return failed ? -2 : 0;
}

/* Gated chunked prefill against a KV cache (§20.3 protocol on the gated
 * layer): Tq new tokens of sequence b at positions start_pos[b] + t; keys =
 * cache rows 0..start_pos[b]-1 as stored, then the chunk's own keys (g2-g3 at
 * their positions); the causal mask starts at start_pos[b]; z = o * sigmoid(gate).
 *   qg [B,Tq,Hq,2d], k/v [B,Tq,Hkv,d]; caches [B,Hkv,S_max,d];
 *   out fp64 [B,Tq,Hq,d]; k_rows fp64 [B,Tq,Hkv,d] = the chunk's keys. */
int q3a_oracle_gated_prefill_chunk(const uint16_t* qg, const uint16_t* k, const uint16_t* v,
                                   const uint16_t* k_cache, const uint16_t* v_cache,
                                   const int32_t* start_pos, const uint16_t* q_w,
                                   const uint16_t* k_w, int B, int Tq, int Hq, int Hkv, int d,
                                   int d_r, long S_max, double theta, double eps, double* out,
                                   double* k_rows) {
  if (check_gated(B, Tq, Hq, Hkv, d, d_r) || S_max <= 0 || !out || !k_rows) return -1;
  for (int b = 0; b < B; ++b)
    if (start_pos[b] < 0 || (long)start_pos[b] + Tq > S_max) return -1;
  int g = Hq / Hkv;
  long units = (long)B * Hkv;
  int failed = 0;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(OMP_THREADS)
#endif
  for (long u = 0; u < units; ++u) {
    long b = u / Hkv, kv = u % Hkv;
    long p0 = start_pos[b];
    long n_all = p0 + Tq;
    double* keys = (double*)malloc(sizeof(double) * (size_t)(n_all > 0 ? n_all : 1) * d);
    double* vals = (double*)malloc(sizeof(double) * (size_t)(n_all > 0 ? n_all : 1) * d);
    double* scores = (double*)malloc(sizeof(double) * (size_t)(n_all > 0 ? n_all : 1));
    double* qhat = (double*)malloc(sizeof(double) * d);
    if (!keys || !vals || !scores || !qhat) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
      failed = 1;
    } else {
      const uint16_t* kc = k_cache + (b * Hkv + kv) * S_max * d;
      const uint16_t* vc = v_cache + (b * Hkv + kv) * S_max * d;
      for (long j = 0; j < p0; ++j)
        for (int c = 0; c < d; ++c) {
          keys[j * d + c] = widen_bf16(kc[j * d + c]);
          vals[j * d + c] = widen_bf16(vc[j * d + c]);
        }
      for (long t = 0; t < Tq; ++t) {
        long r = ((b * Tq + t) * Hkv + kv) * d;
        double* kn = keys + (p0 + t) * d;
        q3a_oracle_zc_rmsnorm_row(k + r, k_w, d, eps, kn);
        q3a_oracle_partial_rope_row(kn, d, d_r, (double)(p0 + t), theta);
        for (int c = 0; c < d; ++c) {
          k_rows[r + c] = kn[c];
          vals[(p0 + t) * d + c] = widen_bf16(v[r + c]);
        }
      }
      for (long t = 0; t < Tq; ++t)
        for (long h = kv * g; h < (kv + 1) * g; ++h) {
          long rq = (b * Tq + t) * Hq + h;
          const uint16_t* qrow = qg + rq * 2L * d; /* g1 */
          const uint16_t* grow = qrow + d;
          double* o = out + rq * d;
          q3a_oracle_zc_rmsnorm_row(qrow, q_w, d, eps, qhat);
          q3a_oracle_partial_rope_row(qhat, d, d_r, (double)(p0 + t), theta);
          attend_row(qhat, keys, vals, p0 + t + 1, d, scores, o);
          for (int c = 0; c < d; ++c) o[c] *= sigmoid(widen_bf16(grow[c]));
        }
    }
    free(keys);
    free(vals);
    free(scores);
    free(qhat);
  }
  return failed ? -2 : 0;
}
