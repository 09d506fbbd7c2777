/*
 * ORACLE -- test infrastructure only.  Plain fp64 CPU attention over an
 * explicitly gathered context.  Only tests/, __graft_entry__.smoke() and
 * bench.py's CPU-baseline leg may load this; the product library never does.
 *
 * Definition followed (no blocking, fusion or reordering beyond it):
 *   "Paged KV cache", How it works, step 3 (attention over the gathered
 *   context with a softmax), and GraniKV Section 2.3 (shared-prefix
 *   attention O_p = softmax(Q K_p^T / sqrt(d)) V_p):
 *     s_i = (q . k_i) * scale,  m = max_i s_i,  Z = sum_i exp(s_i - m),
 *     o   = sum_i exp(s_i - m) v_i / Z,         lse = m + ln Z.
 *   An empty context gives o = 0 and lse = -inf.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* One query row against n keys.  q[d], k[n][d], v[n][d]; o[d]; *lse. */
static void attend_row(int d, int64_t n, const double *q, const double *k, const double *v,
                       double scale, double *s, double *o, double *lse) {
  for (int e = 0; e < d; ++e) o[e] = 0.0;
  if (n == 0) {
    *lse = -INFINITY;
    return;
  }
  double m = -INFINITY;
  for (int64_t i = 0; i < n; ++i) {
    double acc = 0.0;
    for (int e = 0; e < d; ++e) acc += q[e] * k[i * d + e];
    s[i] = acc * scale;
    if (s[i] > m) m = s[i];
  }
  double z = 0.0;
  for (int64_t i = 0; i < n; ++i) {
    double w = exp(s[i] - m);
    z += w;
    for (int e = 0; e < d; ++e) o[e] += w * v[i * d + e];
  }
  for (int e = 0; e < d; ++e) o[e] /= z;
  *lse = m + log(z);
}

/*
 * All query heads of one request.  hkv KV heads, g query heads per KV head
 * (query head qh uses KV head qh / g):
 *   q[hkv*g][d], k[hkv][n][d], v[hkv][n][d] -> o[hkv*g][d], lse[hkv*g].
 * Rows are independent; OpenMP spreads them over the host cores.
 */
int gk_oracle_attend_heads(int hkv, int g, int d, int64_t n, const double *q, const double *k,
                           const double *v, double scale, double *o, double *lse) {
  int bad = 0;
  int rows = hkv * g;
#pragma omp parallel
  {
    double *s = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
#pragma omp for schedule(dynamic, 1)
    for (int r = 0; r < rows; ++r) {
      size_t h = (size_t)(r / g);
      if (!s) {
#pragma omp atomic write
        bad = 1;
        continue;
      }
      attend_row(d, n, q + (size_t)r * d, k + h * (size_t)n * d, v + h * (size_t)n * d, scale, s,
                 o + (size_t)r * d, lse + r);
    }
    free(s);
  }
  return bad;
}

/* Number of threads the OpenMP runtime would use (reported beside CPU timings). */
int gk_oracle_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
