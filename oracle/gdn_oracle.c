/*
 * Oracle for the Gated DeltaNet forward pass: a plain, slow, fp64 token loop.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path may call this code;
 * only the test suite, the smoke check and the CPU-baseline leg of the
 * benchmark use it. It shares no code, header or constant with the CUDA
 * library.
 *
 * What it computes (per sequence n and head h, state kept in the storage
 * orientation Z = S^T, a d_k x d_v matrix, so that element (i, j) of Z is
 * row j / column i of the d_v x d_k state S used on the illustrated DeltaNet
 * page, "stay-hungry-time.github.io/deltanet", state-shape paragraphs):
 *
 *   variant 1 ("decay, then correct"; that page's GDN paragraph, worked
 *   example old prediction 3, target 5, alpha 0.8, beta 0.5 -> 3.7):
 *       Z~   = alpha_t Z
 *       u_t  = beta_t (v_t - Z~^T k_t)
 *       Z    = Z~ + k_t u_t^T
 *       o_t  = Z^T q_t                       (read after the write)
 *
 *   variant 0 (the recurrence as written on the "GPU parallelisation of
 *   Gated DeltaNet" page, m.lqnn.cn/news/262411, section 1.2):
 *       u_t  = beta_t (v_t - Z^T k_t)
 *       Z    = alpha_t Z + k_t u_t^T
 *       o_t  = Z^T q_t
 *
 *   alpha_t = exp(g_t). Both variants coincide when alpha == 1 (plain
 *   DeltaNet, the delta rule of the illustrated page, "Delta Rule" section:
 *   S_t = S_{t-1} + beta_t (v_t - S_{t-1} k_t) k_t^T, read with o_t = S_t q_t).
 *
 * Layouts (row-major, contiguous):
 *   q, k   [B, T, H, dk]      v, out [B, T, H, dv]      g, beta [B, T, H]
 *   h0, hT [N, H, dk, dv]     (N = B, or the number of packed sequences)
 *   cu_seqlens (optional) int32 [N + 1]: packed sequences; then the tensors
 *   are read as [1, T, H, ...] and B is the number of sequences N.
 *
 * The state never leaves fp64. Work is split over (sequence, head) pairs with
 * OpenMP; each pair is an independent problem.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static void one_sequence_head(const double* q, const double* k, const double* v,
                              const double* g, const double* beta,
                              const double* h0, double* out, double* hT,
                              long t_begin, long t_end, int h, int H, int dk,
                              int dv, int variant, double* Z, double* u) {
  /* Z: dk x dv scratch, u: dv scratch. */
  if (h0)
    memcpy(Z, h0, sizeof(double) * (size_t)dk * dv);
  else
    memset(Z, 0, sizeof(double) * (size_t)dk * dv);

  for (long t = t_begin; t < t_end; ++t) {
    const long row = t * H + h;               /* token-head index */
    const double* qt = q + row * dk;
    const double* kt = k + row * dk;
    const double* vt = v + row * dv;
    const double alpha = exp(g[row]);
    const double b = beta[row];
    double* ot = out + row * dv;

    if (variant == 1) {
      for (long e = 0; e < (long)dk * dv; ++e) Z[e] *= alpha;
    }
    /* prediction Z^T k (with the already-decayed state for variant 1) */
    for (int j = 0; j < dv; ++j) {
      double s = 0.0;
      for (int i = 0; i < dk; ++i) s += Z[(long)i * dv + j] * kt[i];
      u[j] = b * (vt[j] - s);
    }
    if (variant == 0) {
      for (long e = 0; e < (long)dk * dv; ++e) Z[e] *= alpha;
    }
    for (int i = 0; i < dk; ++i)
      for (int j = 0; j < dv; ++j) Z[(long)i * dv + j] += kt[i] * u[j];
    for (int j = 0; j < dv; ++j) {
      double s = 0.0;
      for (int i = 0; i < dk; ++i) s += Z[(long)i * dv + j] * qt[i];
      ot[j] = s;
    }
  }
  if (hT) memcpy(hT, Z, sizeof(double) * (size_t)dk * dv);
}

/* Returns 0 on success, -1 on bad arguments, -2 on allocation failure. */
int gdn_oracle_forward(const double* q, const double* k, const double* v,
                       const double* g, const double* beta, const double* h0,
                       double* out, double* hT, const int32_t* cu_seqlens,
                       int B, int H, int T, int dk, int dv, int variant,
                       int nthreads) {
  if (!q || !k || !v || !g || !beta || !out) return -1;
  if (B < 0 || H <= 0 || T < 0 || dk <= 0 || dv <= 0) return -1;
  if (variant != 0 && variant != 1) return -1;
  const int N = B;
  if (cu_seqlens) {
    if (cu_seqlens[0] != 0 || cu_seqlens[N] != T) return -1;
    for (int n = 0; n < N; ++n)
      if (cu_seqlens[n + 1] < cu_seqlens[n]) return -1;
  }
  const long pairs = (long)N * H;
  int rc = 0;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel
#endif
  {
    double* Z = (double*)malloc(sizeof(double) * (size_t)dk * dv);
    double* u = (double*)malloc(sizeof(double) * (size_t)dv);
    if (!Z || !u) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
      rc = -2;
    } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
      for (long p = 0; p < pairs; ++p) {
        const int n = (int)(p / H), h = (int)(p % H);
        long t0, t1;
        const double *qb = q, *kb = k, *vb = v, *gb = g, *bb = beta;
        double* ob = out;
        if (cu_seqlens) {
          t0 = cu_seqlens[n];
          t1 = cu_seqlens[n + 1];
        } else {
          /* batch n starts at token n*T of the flattened [B*T] token axis */
          t0 = (long)n * T;
          t1 = t0 + T;
        }
        one_sequence_head(qb, kb, vb, gb, bb,
                          h0 ? h0 + p * (long)dk * dv : NULL, ob,
                          hT ? hT + p * (long)dk * dv : NULL, t0, t1, h, H,
                          dk, dv, variant, Z, u);
      }
    }
    free(Z);
    free(u);
  }
  return rc;
}

/* Number of threads the OpenMP runtime would use for the loop above. */
int gdn_oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
