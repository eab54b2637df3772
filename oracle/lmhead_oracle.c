/*
 * lmhead_oracle.c -- plain, slow, fp64 CPU oracle for the chunked LM-head
 * log-prob + entropy head, forward and exact backward.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package's smoke check
 * and the benchmark's CPU-baseline leg may load or call this file.  It shares
 * no code, header, table, constant or helper with the CUDA implementation,
 * and neither side includes or links the other.
 *
 * What it computes, for every scored token t (mask[t] != 0, or no mask);
 * unscored tokens give zeros everywhere and contribute nothing:
 *
 *   z_v      = (sum_k h[t,k] W[v,k]) / tau                       v = 0..V-1
 *   lse      = log sum_v exp(z_v)
 *   logp     = z_{y'} - lse,         y' = y + V if -V <= y < 0, else y;
 *                                    y' outside [0, V) gives logp = NaN
 *   entropy  = lse - sum_v p_v z_v,  p_v = exp(z_v - lse)
 *
 *   backward, with per-token cotangents g_l (of logp) and g_e (of entropy):
 *   dz_v         = g_l (delta_{v,y'} - p_v) - g_e p_v (z_v - lse + entropy)
 *   d_hidden[t]  = sum_v (dz_v / tau) W[v]
 *   d_weight[v]  = sum_t (dz_{t,v} / tau) h[t]
 *
 * Sources (the method is stated on these pages; this file restates it as
 * plain definitions, evaluated in double precision):
 *  - tunix PR #2913, commit "fused sharded log-prob head
 *    (TUNIX_LOGPS_SHARDED_HEAD=fused)": a chunk's logits give the target
 *    logit (one-hot select), the max and exp-sum, and the entropy from the
 *    same exponentials; section "How the fused log-prob head works": a
 *    log-probability equals the target logit minus (max + log of the shifted
 *    exponential sum); the temperature
 *    divides the logits (tested at 0.7 and 1) and the backward keeps that
 *    division; negative ids wrap and ids are valid in [0, vocab) (review
 *    thread on _target_hit).
 *  - tunix PR #2876 "Compile compute_chunked_logps at chunk_size > 1024",
 *    section "What the new tests check": chunked results agree with a
 *    float64 reference.
 *  - "Long Sequences (SeCO)" guide, section "Efficiency" (the loss per chunk
 *    is chunked cross-entropy) and the exactness table (gradients against an
 *    fp64 ground truth).
 * The entropy cotangent is not printed on the pages (they differentiate it
 * by autodiff); dH/dz_v = -p_v (z_v - lse + H) follows from the definition
 * above and is pinned by finite differences in the tests.
 *
 * The max-shifted evaluation lse = m + log sum exp(z_v - m), m = max_v z_v,
 * is the textbook identity for the same number; it only avoids overflow.
 *
 * Storage: matrices are passed either as double or as raw bfloat16 bit
 * patterns (a bfloat16 is the upper half of an IEEE-754 binary32), which
 * decode exactly to double.  All arithmetic is double.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double bf16_to_double(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Copy row `r` of a [rows, n] matrix into `out` as double. */
static void load_row(const void* m, int is_bf16, int64_t r, int32_t n, double* out) {
  if (is_bf16) {
    const uint16_t* p = (const uint16_t*)m + r * (int64_t)n;
    for (int32_t k = 0; k < n; ++k) out[k] = bf16_to_double(p[k]);
  } else {
    const double* p = (const double*)m + r * (int64_t)n;
    for (int32_t k = 0; k < n; ++k) out[k] = p[k];
  }
}

/* sum_k h[k] * W[v,k], in order k = 0..n-1. */
static double dot_with_row(const double* h, const void* w, int w_bf16, int64_t v, int32_t n) {
  double acc = 0.0;
  if (w_bf16) {
    const uint16_t* p = (const uint16_t*)w + v * (int64_t)n;
    for (int32_t k = 0; k < n; ++k) acc += h[k] * bf16_to_double(p[k]);
  } else {
    const double* p = (const double*)w + v * (int64_t)n;
    for (int32_t k = 0; k < n; ++k) acc += h[k] * p[k];
  }
  return acc;
}

/* Target id after the wrap of negative ids; -1 when it is not a valid id. */
static int64_t wrapped_target(int32_t y, int32_t V) {
  int64_t yy = (int64_t)y;
  if (yy < 0) yy += V;
  return (yy >= 0 && yy < V) ? yy : -1;
}

/* Logits z (length V) of one hidden row h, then lse and entropy. */
static void row_statistics(const double* h, const void* w, int w_bf16, int32_t H, int32_t V,
                           double tau, double* z, double* lse_out, double* ent_out) {
  for (int32_t v = 0; v < V; ++v) z[v] = dot_with_row(h, w, w_bf16, v, H) / tau;
  double m = -INFINITY;
  for (int32_t v = 0; v < V; ++v) m = z[v] > m ? z[v] : m;
  double s = 0.0;
  for (int32_t v = 0; v < V; ++v) s += exp(z[v] - m);
  double lse = m + log(s);
  double spz = 0.0;
  for (int32_t v = 0; v < V; ++v) spz += exp(z[v] - lse) * z[v];
  *lse_out = lse;
  *ent_out = lse - spz;
}

int lmo_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Forward.  Returns 0 on success, -1 on a bad argument, -2 when out of memory. */
int lmo_forward(int64_t T, int32_t H, int32_t V,
                const void* hidden, int hidden_bf16,
                const void* weight, int weight_bf16,
                const int32_t* targets, const uint8_t* mask, double tau,
                double* logp, double* entropy, double* lse) {
  if (T < 0 || H <= 0 || V <= 0 || !(tau > 0.0) || !isfinite(tau)) return -1;
  if (T == 0) return 0;
  if (!hidden || !weight || !targets || !logp || !entropy || !lse) return -1;
  int failed = 0;
#pragma omp parallel
  {
    double* h = (double*)malloc(sizeof(double) * (size_t)H);
    double* z = (double*)malloc(sizeof(double) * (size_t)V);
    if (!h || !z) {
#pragma omp atomic write
      failed = 1;
    }
#pragma omp for schedule(dynamic, 1)
    for (int64_t t = 0; t < T; ++t) {
      if (!h || !z) continue;
      if (mask && !mask[t]) {
        logp[t] = 0.0;
        entropy[t] = 0.0;
        lse[t] = 0.0;
        continue;
      }
      load_row(hidden, hidden_bf16, t, H, h);
      double L, E;
      row_statistics(h, weight, weight_bf16, H, V, tau, z, &L, &E);
      int64_t y = wrapped_target(targets[t], V);
      logp[t] = (y >= 0) ? z[y] - L : NAN;
      entropy[t] = E;
      lse[t] = L;
    }
    free(h);
    free(z);
  }
  return failed ? -2 : 0;
}

/*
 * Backward.  d_hidden [T,H] is overwritten (zero rows for unscored tokens).
 * d_weight [V,H] is overwritten when not NULL.  grad_logp / grad_entropy NULL
 * mean zero cotangents.  The statistics are recomputed from the definition.
 */
int lmo_backward(int64_t T, int32_t H, int32_t V,
                 const void* hidden, int hidden_bf16,
                 const void* weight, int weight_bf16,
                 const int32_t* targets, const uint8_t* mask, double tau,
                 const double* grad_logp, const double* grad_entropy,
                 double* d_hidden, double* d_weight) {
  if (T < 0 || H <= 0 || V <= 0 || !(tau > 0.0) || !isfinite(tau)) return -1;
  if (!weight || (T > 0 && (!hidden || !targets || !d_hidden))) return -1;
  if (d_weight) memset(d_weight, 0, sizeof(double) * (size_t)V * (size_t)H);
  if (T == 0) return 0;

  double* hrows = (double*)malloc(sizeof(double) * (size_t)T * (size_t)H);
  double* lse_t = (double*)malloc(sizeof(double) * (size_t)T);
  double* ent_t = (double*)malloc(sizeof(double) * (size_t)T);
  if (!hrows || !lse_t || !ent_t) {
    free(hrows); free(lse_t); free(ent_t);
    return -2;
  }
  int failed = 0;

  /* Per token: statistics, dz over the whole vocabulary, and d_hidden. */
#pragma omp parallel
  {
    double* z = (double*)malloc(sizeof(double) * (size_t)V);
    double* wrow = (double*)malloc(sizeof(double) * (size_t)H);
    if (!z || !wrow) {
#pragma omp atomic write
      failed = 1;
    }
#pragma omp for schedule(dynamic, 1)
    for (int64_t t = 0; t < T; ++t) {
      double* h = hrows + t * (int64_t)H;
      double* dh = d_hidden + t * (int64_t)H;
      for (int32_t k = 0; k < H; ++k) dh[k] = 0.0;
      for (int32_t k = 0; k < H; ++k) h[k] = 0.0;
      lse_t[t] = 0.0;
      ent_t[t] = 0.0;
      if (!z || !wrow) continue;
      if (mask && !mask[t]) continue;
      load_row(hidden, hidden_bf16, t, H, h);
      double L, E;
      row_statistics(h, weight, weight_bf16, H, V, tau, z, &L, &E);
      lse_t[t] = L;
      ent_t[t] = E;
      double gl = grad_logp ? grad_logp[t] : 0.0;
      double ge = grad_entropy ? grad_entropy[t] : 0.0;
      int64_t y = wrapped_target(targets[t], V);
      for (int32_t v = 0; v < V; ++v) {
        double p = exp(z[v] - L);
        double onehot = (v == y) ? 1.0 : 0.0;
        double dz = gl * (onehot - p) - ge * p * (z[v] - L + E);
        double c = dz / tau;
        load_row(weight, weight_bf16, v, H, wrow);
        for (int32_t k = 0; k < H; ++k) dh[k] += c * wrow[k];
      }
    }
    free(z);
    free(wrow);
  }

  /* d_weight rows: each vocabulary row sums over the scored tokens in order. */
  if (d_weight && !failed) {
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t v = 0; v < V; ++v) {
      double* dw = d_weight + v * (int64_t)H;
      for (int64_t t = 0; t < T; ++t) {
        if (mask && !mask[t]) continue;
        const double* h = hrows + t * (int64_t)H;
        double z = dot_with_row(h, weight, weight_bf16, v, H) / tau;
        double p = exp(z - lse_t[t]);
        double gl = grad_logp ? grad_logp[t] : 0.0;
        double ge = grad_entropy ? grad_entropy[t] : 0.0;
        int64_t y = wrapped_target(targets[t], V);
        double onehot = (v == y) ? 1.0 : 0.0;
        double dz = gl * (onehot - p) - ge * p * (z - lse_t[t] + ent_t[t]);
        double c = dz / tau;
        for (int32_t k = 0; k < H; ++k) dw[k] += c * h[k];
      }
    }
  }
  free(hrows);
  free(lse_t);
  free(ent_t);
  return failed ? -2 : 0;
}

/*
 * Logits-level scoring (for callers that already hold a chunk's logits).
 * The pages test their fused scoring on logits containing infinities and
 * NaNs, including a row without any finite entry, and list the isfinite mask of the
 * cotangent among the parts a test must catch (tunix PR #2913, commit
 * "fused sharded log-prob head": FusedScoringTest), but print no values.
 * This file reads them as follows, with z = logits / tau per row:
 *   - an entry of -inf has probability 0 and contributes nothing (the limit
 *     of the definition); its cotangent is 0 (isfinite mask);
 *   - a NaN or +inf entry anywhere in the row makes lse, logp and entropy
 *     NaN; finite entries' cotangents are then NaN, non-finite ones 0;
 *   - a row with no finite entry has lse = -inf, logp = NaN, entropy = NaN
 *     and an all-zero cotangent;
 *   - otherwise lse, logp, entropy and the cotangent are those of the head
 *     over the finite entries (logp = -inf when the target's logit is -inf).
 * Unscored rows give zeros; invalid targets give logp = NaN (as above).
 */
static int row_has_nan_or_posinf(const double* z, int32_t V) {
  for (int32_t v = 0; v < V; ++v)
    if (isnan(z[v]) || (isinf(z[v]) && z[v] > 0)) return 1;
  return 0;
}

static void logits_row_statistics(const double* z, int32_t V, double* lse_out, double* ent_out) {
  if (row_has_nan_or_posinf(z, V)) {
    *lse_out = NAN;
    *ent_out = NAN;
    return;
  }
  double m = -INFINITY;
  for (int32_t v = 0; v < V; ++v) m = z[v] > m ? z[v] : m;
  if (!isfinite(m)) {  /* no finite entry */
    *lse_out = -INFINITY;
    *ent_out = NAN;
    return;
  }
  double s = 0.0;
  for (int32_t v = 0; v < V; ++v)
    if (isfinite(z[v])) s += exp(z[v] - m);
  double lse = m + log(s);
  double spz = 0.0;
  for (int32_t v = 0; v < V; ++v)
    if (isfinite(z[v])) spz += exp(z[v] - lse) * z[v];
  *lse_out = lse;
  *ent_out = lse - spz;
}

int lmo_logits_forward(int64_t T, int32_t V, const double* logits, const int32_t* targets,
                       const uint8_t* mask, double tau, double* logp, double* entropy,
                       double* lse) {
  if (T < 0 || V <= 0 || !(tau > 0.0) || !isfinite(tau)) return -1;
  if (T == 0) return 0;
  if (!logits || !targets || !logp || !entropy || !lse) return -1;
  int failed = 0;
#pragma omp parallel
  {
    double* z = (double*)malloc(sizeof(double) * (size_t)V);
    if (!z) {
#pragma omp atomic write
      failed = 1;
    }
#pragma omp for schedule(dynamic, 4)
    for (int64_t t = 0; t < T; ++t) {
      if (!z) continue;
      if (mask && !mask[t]) {
        logp[t] = entropy[t] = lse[t] = 0.0;
        continue;
      }
      const double* row = logits + t * (int64_t)V;
      for (int32_t v = 0; v < V; ++v) z[v] = row[v] / tau;
      double L, E;
      logits_row_statistics(z, V, &L, &E);
      int64_t y = wrapped_target(targets[t], V);
      logp[t] = (y >= 0) ? z[y] - L : NAN;
      entropy[t] = E;
      lse[t] = L;
    }
    free(z);
  }
  return failed ? -2 : 0;
}

/* d_logits [T,V] overwritten: d loss / d logits (the 1/tau of z = logits/tau included). */
int lmo_logits_backward(int64_t T, int32_t V, const double* logits, const int32_t* targets,
                        const uint8_t* mask, double tau, const double* grad_logp,
                        const double* grad_entropy, double* d_logits) {
  if (T < 0 || V <= 0 || !(tau > 0.0) || !isfinite(tau)) return -1;
  if (T == 0) return 0;
  if (!logits || !targets || !d_logits) return -1;
  int failed = 0;
#pragma omp parallel
  {
    double* z = (double*)malloc(sizeof(double) * (size_t)V);
    if (!z) {
#pragma omp atomic write
      failed = 1;
    }
#pragma omp for schedule(dynamic, 4)
    for (int64_t t = 0; t < T; ++t) {
      double* dz = d_logits + t * (int64_t)V;
      for (int32_t v = 0; v < V; ++v) dz[v] = 0.0;
      if (!z || (mask && !mask[t])) continue;
      const double* row = logits + t * (int64_t)V;
      for (int32_t v = 0; v < V; ++v) z[v] = row[v] / tau;
      double L, E;
      logits_row_statistics(z, V, &L, &E);
      double gl = grad_logp ? grad_logp[t] : 0.0;
      double ge = grad_entropy ? grad_entropy[t] : 0.0;
      int64_t y = wrapped_target(targets[t], V);
      for (int32_t v = 0; v < V; ++v) {
        if (!isfinite(z[v])) continue;          /* isfinite mask */
        double p = exp(z[v] - L);
        double onehot = (v == y) ? 1.0 : 0.0;
        dz[v] = (gl * (onehot - p) - ge * p * (z[v] - L + E)) / tau;
      }
    }
    free(z);
  }
  return failed ? -2 : 0;
}
