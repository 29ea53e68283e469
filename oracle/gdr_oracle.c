/*
 * gdr_oracle.c -- plain fp64 CPU oracle for the gated delta rule.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header or constant with the CUDA
 * library.
 *
 * What it computes is the definition of the method, token by token, with no
 * chunking, blocking or reordering:
 *
 *   S_t = (I - beta_t k_t k_t^T) Diag(exp g_t) S_{t-1} + beta_t k_t v_t^T
 *   o_t = S_t^T q_t                    (the post-update state, token t included)
 *
 * with S a K x V matrix per (sequence, value head).  The product
 * (I - b k k^T) D S + b k v^T is evaluated as the equivalent rank-1 update
 *   S' = D S;  e = v - S'^T k;  S = S' + k (b e)^T
 * which is the delta-rule "prediction error" form ("FLA 算子内核正确性测试与覆盖矩阵",
 * section 二: the DeltaNet/delta-rule background with the WY representation
 * S^r = P^r S^0 + H^r, P^r a product of generalized Householder factors).
 * The scalar-gate case (GDN) uses D = exp(g_t) I; the per-key-channel case
 * (KDA) uses D = Diag(exp g_t[0..K-1]), scaling row d of S.
 *
 * Readings where the pages leave a step open (each is also listed in the
 * design notes):
 *   - in-kernel L2 norm: x / sqrt(sum x^2 + 1e-6), applied to q and k per
 *     token and head ("use_qk_l2norm_in_kernel" axis, coverage guide section 三);
 *   - grouped value heads: value head hv reads q/k head hv / (HV / H)
 *     (coverage guide section 三: "v's shape expands by HV");
 *   - the state recorded for chunk c of a sequence is the state ENTERING the
 *     chunk, i.e. before token c*C of that sequence is processed
 *     ("flash-linear-attention KCP 精度失效根因排查手册", section on h/dh
 *     cross-rank semantics);
 *   - v_new_t = beta_t * (v_t - (D_t S_{t-1})^T k_t), the per-token write
 *     vector, so that S_t = D_t S_{t-1} + k_t v_new_t^T.
 *
 * Layouts (all row-major, contiguous, fp64):
 *   q, k [B, T, H, K]; v, o, v_new [B, T, HV, V]; g [B, T, HV] or
 *   [B, T, HV, K]; beta [B, T, HV]; h0, ht [N, HV, K, V];
 *   h_chunks [NT, HV, K, V] with NT = sum_n ceil(len_n / C).
 * Dense: N = B and sequence n covers flat tokens [n T, (n+1) T).
 * Varlen (cu_seqlens != NULL): B == 1, sequence n covers [cu[n], cu[n+1]).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_L2_EPS 1e-6

static void l2_normalize(const double *x, double *y, int64_t n, int on) {
  if (!on) {
    memcpy(y, x, (size_t)n * sizeof(double));
    return;
  }
  double ss = 0.0;
  for (int64_t i = 0; i < n; ++i) ss += x[i] * x[i];
  double inv = 1.0 / sqrt(ss + ORACLE_L2_EPS);
  for (int64_t i = 0; i < n; ++i) y[i] = x[i] * inv;
}

/* Returns 0 on success, -1 on bad arguments, -2 on allocation failure. */
int gdr_oracle_fwd(int64_t B, int64_t T, int64_t H, int64_t HV, int64_t K, int64_t V,
                   int gate_per_k, const double *q, const double *k, const double *v,
                   const double *g, const double *beta, const double *h0,
                   const int64_t *cu_seqlens, int64_t N, int use_qk_l2norm,
                   double *o, double *ht, int64_t chunk_size, double *h_chunks,
                   double *v_new, int n_threads) {
  if (B < 0 || T < 0 || H <= 0 || HV <= 0 || K <= 0 || V <= 0) return -1;
  if (HV % H != 0) return -1;
  if (cu_seqlens && B != 1) return -1;
  if (!cu_seqlens) N = B;
  if (h_chunks && chunk_size <= 0) return -1;
  const int64_t G = HV / H;

  /* chunk offsets of each sequence, for recording the chunk-entry states */
  int64_t *chunk_off = (int64_t *)calloc((size_t)N + 1, sizeof(int64_t));
  if (!chunk_off) return -2;
  for (int64_t n = 0; n < N; ++n) {
    int64_t len = cu_seqlens ? cu_seqlens[n + 1] - cu_seqlens[n] : T;
    int64_t nc = chunk_size > 0 ? (len + chunk_size - 1) / chunk_size : 0;
    chunk_off[n + 1] = chunk_off[n] + nc;
  }

  int status = 0;
#ifdef _OPENMP
  if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (int64_t unit = 0; unit < N * HV; ++unit) {
    const int64_t n = unit / HV, hv = unit % HV, hq = hv / G;
    const int64_t t0 = cu_seqlens ? cu_seqlens[n] : n * T;
    const int64_t t1 = cu_seqlens ? cu_seqlens[n + 1] : (n + 1) * T;
    double *S = (double *)malloc((size_t)(K * V) * sizeof(double));
    double *qt = (double *)malloc((size_t)K * sizeof(double));
    double *kt = (double *)malloc((size_t)K * sizeof(double));
    double *e = (double *)malloc((size_t)V * sizeof(double));
    if (!S || !qt || !kt || !e) {
      free(S); free(qt); free(kt); free(e);
#ifdef _OPENMP
#pragma omp atomic write
#endif
      status = -2;
      continue;
    }
    if (h0) memcpy(S, h0 + unit * K * V, (size_t)(K * V) * sizeof(double));
    else memset(S, 0, (size_t)(K * V) * sizeof(double));

    for (int64_t t = t0; t < t1; ++t) {
      const int64_t p = t - t0; /* position within the sequence */
      if (h_chunks && p % chunk_size == 0) {
        const int64_t c = chunk_off[n] + p / chunk_size;
        memcpy(h_chunks + (c * HV + hv) * K * V, S, (size_t)(K * V) * sizeof(double));
      }
      l2_normalize(q + (t * H + hq) * K, qt, K, use_qk_l2norm);
      l2_normalize(k + (t * H + hq) * K, kt, K, use_qk_l2norm);
      const double b = beta[t * HV + hv];
      /* S' = D_t S */
      if (gate_per_k) {
        const double *gt = g + (t * HV + hv) * K;
        for (int64_t d = 0; d < K; ++d) {
          const double a = exp(gt[d]);
          for (int64_t j = 0; j < V; ++j) S[d * V + j] *= a;
        }
      } else {
        const double a = exp(g[t * HV + hv]);
        for (int64_t i = 0; i < K * V; ++i) S[i] *= a;
      }
      /* e = v_t - S'^T k_t */
      const double *vt = v + (t * HV + hv) * V;
      for (int64_t j = 0; j < V; ++j) e[j] = vt[j];
      for (int64_t d = 0; d < K; ++d) {
        const double kd = kt[d];
        for (int64_t j = 0; j < V; ++j) e[j] -= S[d * V + j] * kd;
      }
      /* S = S' + k_t (beta_t e)^T */
      for (int64_t j = 0; j < V; ++j) e[j] *= b;
      if (v_new) memcpy(v_new + (t * HV + hv) * V, e, (size_t)V * sizeof(double));
      for (int64_t d = 0; d < K; ++d) {
        const double kd = kt[d];
        for (int64_t j = 0; j < V; ++j) S[d * V + j] += kd * e[j];
      }
      /* o_t = S_t^T q_t */
      double *ot = o + (t * HV + hv) * V;
      for (int64_t j = 0; j < V; ++j) ot[j] = 0.0;
      for (int64_t d = 0; d < K; ++d) {
        const double qd = qt[d];
        for (int64_t j = 0; j < V; ++j) ot[j] += S[d * V + j] * qd;
      }
    }
    if (ht) memcpy(ht + unit * K * V, S, (size_t)(K * V) * sizeof(double));
    free(S); free(qt); free(kt); free(e);
  }
  free(chunk_off);
  return status;
}

int gdr_oracle_version(void) { return 1; }
