/*
 * Float64 CPU oracle of the fused LM-head scoring, in plain C with OpenMP.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product links, loads or calls
 * this file: only tests/, __graft_entry__ and bench.py's CPU baseline and
 * reference arm use it (through oracle/lmhead_oracle_c.py).  It shares no
 * code, table or constant with the CUDA library.
 *
 * It is a second, independent statement of the definition that
 * oracle/lmhead_oracle.py writes out with numpy: for each given row (every
 * row handed in is a kept row) the whole logit row is materialised in
 * float64 and reduced by plain loops, in the order the definition reads.
 *
 * Sources (web pages; cited by title and section):
 *   [P1] prime-rl pull request #3326, "Don't compute the logprobs and their
 *        gradients for tokens no loss component reads": the vocab matmul
 *        [N, H] x [H, V] is where the work is; kept rows only.
 *   [P2] SkyRL pull request #2374, "feat(megatron): fuse LM-head entropy for
 *        RL": "How it works" (selected-token log-prob and entropy from one
 *        projection; metric-only entropy adds no gradient) and the
 *        gemini-code-assist review (entropy = -(p * log p) summed over the
 *        vocabulary).
 *   [P3] twinkle pull request #283, "Fix three memory defects in the
 *        Megatron path", section 1: log-softmax in float, the softmax
 *        recomputed for the backward.
 *
 * Definition, per row r with hidden h_r and target y_r (natural logs,
 * temperature 1, no bias):
 *   z_v      = sum_k h_r[k] W[v, k]                      (v = 0 .. V-1)
 *   lse      = max_v z_v + log sum_v exp(z_v - max_v z_v)
 *   logp_v   = z_v - lse,   p_v = exp(logp_v)
 *   logprob  = logp_{y_r}
 *   entropy  = -sum_v p_v logp_v
 * and, given gradients g_lp on logprob and g_ent on entropy (g_ent absent:
 * the metric-only entropy of [P2], no entropy term):
 *   dz_v     = g_lp (1[v = y_r] - p_v) - g_ent p_v (logp_v + entropy)
 *   dh_r     = sum_v dz_v W[v, :]
 *   dW[v, :] = sum_r dz_{r,v} h_r        (over the rows handed in)
 * (d entropy / d z_v = -p_v (logp_v + entropy), from entropy = lse -
 * sum_v p_v z_v.)
 *
 * Parity status: pinned by tests/test_oracle_c.py against the numpy oracle
 * (itself pinned by brute force, closed forms and finite differences) and
 * against closed forms of its own (W = 0, V = 1).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* Threads the oracle's parallel loops use. */
int lmhead_oracle_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/*
 * Scores R rows.
 *   h [R, H], W [V, H]: float64, row-major.   y [R]: targets, in [0, V).
 *   g_lp [R], g_ent [R]: gradients on logprob and entropy; g_lp NULL = no
 *       backward (dh, dW untouched); g_ent NULL = metric-only entropy.
 *   lp, ent, lse [R]: outputs.
 *   dh [R, H], dW [V, H]: outputs of the backward (dW is overwritten with the
 *       sum over these R rows).
 * Returns 0; 1 if a target is outside [0, V); 2 if memory ran out; 3 for
 * sizes below 1.
 */
int lmhead_oracle_score_rows(const double* h, const double* W, const int64_t* y,
                             const double* g_lp, const double* g_ent, int64_t R, int64_t H,
                             int64_t V, double* lp, double* ent, double* lse, double* dh,
                             double* dW) {
  if (R < 1 || H < 1 || V < 1) return 3;
  for (int64_t r = 0; r < R; ++r)
    if (y[r] < 0 || y[r] >= V) return 1;
  const int backward = g_lp != NULL;
  /* the logit gradient of every row is kept for the dW sum over rows */
  double* dz = backward ? (double*)malloc(sizeof(double) * (size_t)(R * V)) : NULL;
  if (backward && dz == NULL) return 2;
  int failed = 0;

#pragma omp parallel
  {
    double* z = (double*)malloc(sizeof(double) * (size_t)V);
    if (z == NULL) {
#pragma omp atomic write
      failed = 1;
    }
#pragma omp for schedule(dynamic, 1)
    for (int64_t r = 0; r < R; ++r) {
      if (z == NULL) continue;
      const double* hr = h + r * H;
      /* the logit row */
      for (int64_t v = 0; v < V; ++v) {
        const double* wv = W + v * H;
        double acc = 0.0;
        for (int64_t k = 0; k < H; ++k) acc += hr[k] * wv[k];
        z[v] = acc;
      }
      /* log-sum-exp, shifted by the row maximum */
      double m = z[0];
      for (int64_t v = 1; v < V; ++v)
        if (z[v] > m) m = z[v];
      double s = 0.0;
      for (int64_t v = 0; v < V; ++v) s += exp(z[v] - m);
      const double l = m + log(s);
      /* entropy = -sum p log p */
      double e = 0.0;
      for (int64_t v = 0; v < V; ++v) {
        const double logp = z[v] - l;
        e -= exp(logp) * logp;
      }
      lse[r] = l;
      lp[r] = z[y[r]] - l;
      ent[r] = e;
      if (!backward) continue;
      /* logit gradient */
      double* dzr = dz + r * V;
      const double gl = g_lp[r];
      const double ge = g_ent != NULL ? g_ent[r] : 0.0;
      for (int64_t v = 0; v < V; ++v) {
        const double logp = z[v] - l;
        const double p = exp(logp);
        double g = -gl * p;
        if (v == y[r]) g += gl;
        if (g_ent != NULL) g -= ge * p * (logp + e);
        dzr[v] = g;
      }
      /* hidden gradient of this row: dz W */
      double* dhr = dh + r * H;
      for (int64_t k = 0; k < H; ++k) dhr[k] = 0.0;
      for (int64_t v = 0; v < V; ++v) {
        const double g = dzr[v];
        const double* wv = W + v * H;
        for (int64_t k = 0; k < H; ++k) dhr[k] += g * wv[k];
      }
    }
    free(z);
  }
  if (failed) {
    free(dz);
    return 2;
  }
  if (backward) {
    /* weight gradient: each vocabulary row sums its logit gradients over the
       rows, in row order */
#pragma omp parallel for schedule(static)
    for (int64_t v = 0; v < V; ++v) {
      double* dwv = dW + v * H;
      for (int64_t k = 0; k < H; ++k) dwv[k] = 0.0;
      for (int64_t r = 0; r < R; ++r) {
        const double g = dz[r * V + v];
        const double* hr = h + r * H;
        for (int64_t k = 0; k < H; ++k) dwv[k] += g * hr[k];
      }
    }
    free(dz);
  }
  return 0;
}
