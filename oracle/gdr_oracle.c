/*
 * Gated delta rule oracle: a plain float64 token-by-token recurrence on the CPU.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the checker the CUDA library is compared
 * against; it shares no code with the library and the library never calls it.
 * Only the tests, __graft_entry__.smoke() and bench.py's CPU-baseline leg use it.
 *
 * What it computes (Kev-4B-LiteRT "r15_kernel_test.py", function truth_f64; the same
 * recurrence is stated a second time in DEG "model.py", function delta_rule_reference):
 *
 *   q_hat = q / sqrt(sum(q^2) + 1e-6),  k_hat = k / sqrt(sum(k^2) + 1e-6)
 *   q_til = q_hat * Dk^-0.5
 *   value head h reads key head floor(h / r), r = Hv / Hk  (repeat_interleave order)
 *   S = S0 (or zeros)
 *   for t in 0..L-1:
 *       S     = S * exp(g_t)                (decay first)
 *       kv    = S^T k_hat_t                 (read)
 *       delta = beta_t * (v_t - kv)         (delta)
 *       S     = S + k_hat_t delta^T         (write)
 *       o_t   = S^T q_til_t                 (output reads the updated state)
 *   return o (every position) and S (final state)
 *
 * No blocking, fusion or reordering: each step above is one loop nest below, in the
 * order the pages give. Heads and rows are independent; OpenMP runs them in parallel,
 * which does not change any value (each (row, head) is computed by one thread, in order).
 *
 * Layouts (row-major, contiguous):
 *   q, k  [B, L, Hk, Dk]     v, o  [B, L, Hv, Dv]     g, beta  [B, L, Hv]
 *   S0, S_T  [B, Hv, Dk, Dv]  (S[i][j]: key index i, value index j)
 */
#include <math.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Returns 0 on success, 1 on bad arguments, 2 on allocation failure. */
int gdr_oracle_forward(const double* q, const double* k, const double* v, const double* g,
                       const double* beta, const double* S0, double* o, double* S_T, int B, int L,
                       int Hk, int Hv, int Dk, int Dv, int nthreads) {
  if (!q || !k || !v || !g || !beta || !o) return 1;
  if (B < 1 || L < 0 || Hk < 1 || Hv < 1 || Dk < 1 || Dv < 1 || Hv % Hk != 0) return 1;
  const int r = Hv / Hk;
  int failed = 0;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif

#pragma omp parallel for schedule(dynamic, 1)
  for (int bh = 0; bh < B * Hv; ++bh) {
    const int b = bh / Hv, h = bh % Hv;
    const int hk = h / r; /* interleave: adjacent value heads share a key head */
    double* S = (double*)malloc(sizeof(double) * (size_t)Dk * Dv);
    double* qt = (double*)malloc(sizeof(double) * (size_t)Dk);
    double* kt = (double*)malloc(sizeof(double) * (size_t)Dk);
    double* kv = (double*)malloc(sizeof(double) * (size_t)Dv);
    double* delta = (double*)malloc(sizeof(double) * (size_t)Dv);
    if (!S || !qt || !kt || !kv || !delta) {
#pragma omp atomic write
      failed = 1;
      free(S); free(qt); free(kt); free(kv); free(delta);
      continue;
    }
    if (S0) {
      memcpy(S, S0 + ((size_t)b * Hv + h) * Dk * Dv, sizeof(double) * (size_t)Dk * Dv);
    } else {
      memset(S, 0, sizeof(double) * (size_t)Dk * Dv);
    }
    for (int t = 0; t < L; ++t) {
      const double* qin = q + (((size_t)b * L + t) * Hk + hk) * Dk;
      const double* kin = k + (((size_t)b * L + t) * Hk + hk) * Dk;
      const double* vin = v + (((size_t)b * L + t) * Hv + h) * Dv;
      const double gt = g[((size_t)b * L + t) * Hv + h];
      const double bt = beta[((size_t)b * L + t) * Hv + h];

      /* l2 normalisation, eps inside the square root; q also scaled by Dk^-0.5 */
      double sq = 0.0, sk = 0.0;
      for (int i = 0; i < Dk; ++i) { sq += qin[i] * qin[i]; sk += kin[i] * kin[i]; }
      const double rq = 1.0 / sqrt(sq + 1e-6), rk = 1.0 / sqrt(sk + 1e-6);
      const double scale = 1.0 / sqrt((double)Dk);
      for (int i = 0; i < Dk; ++i) { qt[i] = qin[i] * rq * scale; kt[i] = kin[i] * rk; }

      /* S = S * exp(g) */
      const double decay = exp(gt);
      for (size_t e = 0; e < (size_t)Dk * Dv; ++e) S[e] *= decay;
      /* kv = S^T k_hat */
      for (int j = 0; j < Dv; ++j) kv[j] = 0.0;
      for (int i = 0; i < Dk; ++i)
        for (int j = 0; j < Dv; ++j) kv[j] += S[(size_t)i * Dv + j] * kt[i];
      /* delta = beta (v - kv) */
      for (int j = 0; j < Dv; ++j) delta[j] = (vin[j] - kv[j]) * bt;
      /* S = S + k_hat delta^T */
      for (int i = 0; i < Dk; ++i)
        for (int j = 0; j < Dv; ++j) S[(size_t)i * Dv + j] += kt[i] * delta[j];
      /* o = S^T q_til */
      double* oo = o + (((size_t)b * L + t) * Hv + h) * Dv;
      for (int j = 0; j < Dv; ++j) oo[j] = 0.0;
      for (int i = 0; i < Dk; ++i)
        for (int j = 0; j < Dv; ++j) oo[j] += S[(size_t)i * Dv + j] * qt[i];
    }
    if (S_T) memcpy(S_T + ((size_t)b * Hv + h) * Dk * Dv, S, sizeof(double) * (size_t)Dk * Dv);
    free(S); free(qt); free(kt); free(kv); free(delta);
  }
  return failed ? 2 : 0;
}

/* Number of threads OpenMP would use (for reporting the CPU baseline's core count). */
int gdr_oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
