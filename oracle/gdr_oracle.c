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
 * Readings where the pages leave a step open:
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

int gdr_oracle_version(void) { return 2; }

/*
 * ---------------------------------------------------------------------------
 * Reverse recurrence (the gradient of the per-token recurrence above).
 *
 * Given upstream gradients do_t = dL/do_t and dht = dL/dS_T of one sequence,
 * walk the tokens last to first with dS = dL/dS_t, starting from dht:
 *
 *   forward step, recomputed:  S' = D_t S_{t-1};  e = v_t - S'^T k;  u = b e;
 *                              S_t = S' + k u^T;  o_t = S_t^T q
 *   o_t = S_t^T q:             dS += q do_t^T;         dq = S_t do_t
 *   S_t = S' + k u^T:          du = dS^T k;            dk = dS u;   dS' = dS
 *   u = b e:                   dbeta = du . e;         de = b du
 *   e = v - S'^T k:            dv = de;  dk -= S' de;  dS' -= k de^T
 *   S' = D_t S_{t-1}:          dg = sum_j S'_dj dS'_dj (summed over d for the
 *                              scalar gate, since D = exp(g) I);  dS = D_t dS'
 *
 * and at the sequence start dh0 = dS.  With the in-kernel L2 norm x^ = x r,
 * r = (|x|^2 + eps)^-1/2, the chain rule gives dx = r (dx^ - x^ (x^ . dx^)).
 * A q/k head is shared by the HV/H value heads of its group, so its gradient is
 * the sum over them.
 *
 * S_{t-1} is needed for every token in reverse order; it is recomputed from
 * checkpoints of S taken every ORACLE_SEG tokens in one forward sweep, then
 * one segment at a time.  That is storage only: every number is the one the
 * plain forward recurrence produces.
 * ---------------------------------------------------------------------------
 */
#define ORACLE_SEG 64

/* One token's decay and prediction error: S <- D_t S, then e = v_t - S^T k_t. */
static void forward_token(double *S, const double *kt, const double *vt, const double *gt, int gate_per_k,
                          int64_t K, int64_t V, double *e) {
  if (gate_per_k) {
    for (int64_t r = 0; r < K; ++r) {
      const double decay = exp(gt[r]);
      for (int64_t c = 0; c < V; ++c) S[r * V + c] *= decay;
    }
  } else {
    const double decay = exp(gt[0]);
    for (int64_t x = 0; x < K * V; ++x) S[x] *= decay;
  }
  for (int64_t c = 0; c < V; ++c) e[c] = vt[c];
  for (int64_t r = 0; r < K; ++r)
    for (int64_t c = 0; c < V; ++c) e[c] -= S[r * V + c] * kt[r];
}

/* dx = r (dy - y (y . dy)) for y = x r; identity when the norm is off. */
static void l2_normalize_bwd(const double *x, const double *dy, double *dx, int64_t n, int on) {
  if (!on) {
    memcpy(dx, dy, (size_t)n * sizeof(double));
    return;
  }
  double ss = 0.0;
  for (int64_t i = 0; i < n; ++i) ss += x[i] * x[i];
  const double r = 1.0 / sqrt(ss + ORACLE_L2_EPS);
  double ydy = 0.0;
  for (int64_t i = 0; i < n; ++i) ydy += x[i] * r * dy[i];
  for (int64_t i = 0; i < n; ++i) dx[i] = r * (dy[i] - x[i] * r * ydy);
}

/* Returns 0 on success, -1 on bad arguments, -2 on allocation failure.
 * do_ [B,T,HV,V]; dht [N,HV,K,V] or NULL (zero); outputs dq, dk [B,T,H,K],
 * dv [B,T,HV,V], dg shaped like g, dbeta [B,T,HV], dh0 [N,HV,K,V] or NULL. */
int gdr_oracle_bwd(int64_t B, int64_t T, int64_t H, int64_t HV, int64_t K, int64_t V,
                   int gate_per_k, const double *q, const double *k, const double *v,
                   const double *g, const double *beta, const double *h0,
                   const int64_t *cu_seqlens, int64_t N, int use_qk_l2norm,
                   const double *do_, const double *dht, double *dq, double *dk, double *dv,
                   double *dg, double *dbeta, double *dh0, int n_threads) {
  if (B < 0 || T < 0 || H <= 0 || HV <= 0 || K <= 0 || V <= 0) return -1;
  if (HV % H != 0) return -1;
  if (cu_seqlens && B != 1) return -1;
  if (!cu_seqlens) N = B;
  const int64_t G = HV / H;
  const int64_t gw = gate_per_k ? K : 1;
  const int64_t KV = K * V;

  int status = 0;
#ifdef _OPENMP
  if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (int64_t grp = 0; grp < N * H; ++grp) {
    const int64_t n = grp / H, hq = grp % H;
    const int64_t t0 = cu_seqlens ? cu_seqlens[n] : n * T;
    const int64_t t1 = cu_seqlens ? cu_seqlens[n + 1] : (n + 1) * T;
    const int64_t len = t1 - t0;
    const int64_t nseg = (len + ORACLE_SEG - 1) / ORACLE_SEG;
    double *ck = (double *)malloc((size_t)((nseg > 0 ? nseg : 1) * KV) * sizeof(double));
    double *Sprev = (double *)malloc((size_t)(ORACLE_SEG * KV) * sizeof(double));
    double *S = (double *)malloc((size_t)KV * sizeof(double));
    double *dS = (double *)malloc((size_t)KV * sizeof(double));
    double *qn = (double *)malloc((size_t)(len > 0 ? len * K : 1) * sizeof(double));
    double *kn = (double *)malloc((size_t)(len > 0 ? len * K : 1) * sizeof(double));
    double *dqn = (double *)calloc((size_t)(len > 0 ? len * K : 1), sizeof(double));
    double *dkn = (double *)calloc((size_t)(len > 0 ? len * K : 1), sizeof(double));
    double *e = (double *)malloc((size_t)V * sizeof(double));
    double *du = (double *)malloc((size_t)V * sizeof(double));
    if (!ck || !Sprev || !S || !dS || !qn || !kn || !dqn || !dkn || !e || !du) {
      free(ck); free(Sprev); free(S); free(dS); free(qn); free(kn); free(dqn); free(dkn); free(e); free(du);
#ifdef _OPENMP
#pragma omp atomic write
#endif
      status = -2;
      continue;
    }
    for (int64_t p = 0; p < len; ++p) {
      l2_normalize(q + ((t0 + p) * H + hq) * K, qn + p * K, K, use_qk_l2norm);
      l2_normalize(k + ((t0 + p) * H + hq) * K, kn + p * K, K, use_qk_l2norm);
    }
    for (int64_t hv = hq * G; hv < (hq + 1) * G; ++hv) {
      const int64_t unit = n * HV + hv;
      /* forward sweep: checkpoints of the state entering each segment */
      if (h0) memcpy(S, h0 + unit * KV, (size_t)KV * sizeof(double));
      else memset(S, 0, (size_t)KV * sizeof(double));
      for (int64_t p = 0; p < len; ++p) {
        const int64_t t = t0 + p;
        if (p % ORACLE_SEG == 0) memcpy(ck + (p / ORACLE_SEG) * KV, S, (size_t)KV * sizeof(double));
        const double b = beta[t * HV + hv];
        forward_token(S, kn + p * K, v + (t * HV + hv) * V, g + (t * HV + hv) * gw, gate_per_k, K, V, e);
        for (int64_t d = 0; d < K; ++d)
          for (int64_t j = 0; j < V; ++j) S[d * V + j] += kn[p * K + d] * b * e[j];
      }
      /* reverse sweep */
      if (dht) memcpy(dS, dht + unit * KV, (size_t)KV * sizeof(double));
      else memset(dS, 0, (size_t)KV * sizeof(double));
      for (int64_t s = nseg - 1; s >= 0; --s) {
        const int64_t p0 = s * ORACLE_SEG;
        const int64_t p1 = (p0 + ORACLE_SEG < len) ? p0 + ORACLE_SEG : len;
        memcpy(S, ck + s * KV, (size_t)KV * sizeof(double));
        for (int64_t p = p0; p < p1; ++p) {
          const int64_t t = t0 + p;
          memcpy(Sprev + (p - p0) * KV, S, (size_t)KV * sizeof(double));
          const double b = beta[t * HV + hv];
          forward_token(S, kn + p * K, v + (t * HV + hv) * V, g + (t * HV + hv) * gw, gate_per_k, K, V, e);
          for (int64_t d = 0; d < K; ++d)
            for (int64_t j = 0; j < V; ++j) S[d * V + j] += kn[p * K + d] * b * e[j];
        }
        for (int64_t p = p1 - 1; p >= p0; --p) {
          const int64_t t = t0 + p;
          const double *kt = kn + p * K, *qt = qn + p * K;
          const double *dot = do_ + (t * HV + hv) * V;
          const double *gt = g + (t * HV + hv) * gw;
          const double b = beta[t * HV + hv];
          /* S' = D_t S_{t-1} (in place on the stored copy), e = v - S'^T k */
          double *Sd = Sprev + (p - p0) * KV;
          forward_token(Sd, kt, v + (t * HV + hv) * V, gt, gate_per_k, K, V, e);
          /* dS += q do^T */
          for (int64_t d = 0; d < K; ++d)
            for (int64_t j = 0; j < V; ++j) dS[d * V + j] += qt[d] * dot[j];
          /* dq = S_t do = S' do + k (u . do) */
          double udo = 0.0;
          for (int64_t j = 0; j < V; ++j) udo += b * e[j] * dot[j];
          for (int64_t d = 0; d < K; ++d) {
            double acc = kt[d] * udo;
            for (int64_t j = 0; j < V; ++j) acc += Sd[d * V + j] * dot[j];
            dqn[p * K + d] += acc;
          }
          /* du = dS^T k; dk = dS u */
          for (int64_t j = 0; j < V; ++j) du[j] = 0.0;
          for (int64_t d = 0; d < K; ++d)
            for (int64_t j = 0; j < V; ++j) du[j] += dS[d * V + j] * kt[d];
          for (int64_t d = 0; d < K; ++d) {
            double acc = 0.0;
            for (int64_t j = 0; j < V; ++j) acc += dS[d * V + j] * b * e[j];
            dkn[p * K + d] += acc;
          }
          /* dbeta = du . e; de = b du (kept in du); dv = de */
          double db = 0.0;
          for (int64_t j = 0; j < V; ++j) db += du[j] * e[j];
          dbeta[t * HV + hv] = db;
          double *dvt = dv + (t * HV + hv) * V;
          for (int64_t j = 0; j < V; ++j) {
            du[j] *= b;
            dvt[j] = du[j];
          }
          /* dk -= S' de; dS' = dS - k de^T */
          for (int64_t d = 0; d < K; ++d) {
            double acc = 0.0;
            for (int64_t j = 0; j < V; ++j) acc += Sd[d * V + j] * du[j];
            dkn[p * K + d] -= acc;
          }
          for (int64_t d = 0; d < K; ++d)
            for (int64_t j = 0; j < V; ++j) dS[d * V + j] -= kt[d] * du[j];
          /* dg from S' = D S_{t-1}; then dS <- D dS' */
          double *dgt = dg + (t * HV + hv) * gw;
          if (gate_per_k) {
            for (int64_t d = 0; d < K; ++d) {
              double acc = 0.0;
              for (int64_t j = 0; j < V; ++j) acc += Sd[d * V + j] * dS[d * V + j];
              dgt[d] = acc;
              const double a = exp(gt[d]);
              for (int64_t j = 0; j < V; ++j) dS[d * V + j] *= a;
            }
          } else {
            double acc = 0.0;
            for (int64_t i = 0; i < KV; ++i) acc += Sd[i] * dS[i];
            dgt[0] = acc;
            const double a = exp(gt[0]);
            for (int64_t i = 0; i < KV; ++i) dS[i] *= a;
          }
        }
      }
      if (dh0) memcpy(dh0 + unit * KV, dS, (size_t)KV * sizeof(double));
    }
    for (int64_t p = 0; p < len; ++p) {
      l2_normalize_bwd(q + ((t0 + p) * H + hq) * K, dqn + p * K, dq + ((t0 + p) * H + hq) * K, K, use_qk_l2norm);
      l2_normalize_bwd(k + ((t0 + p) * H + hq) * K, dkn + p * K, dk + ((t0 + p) * H + hq) * K, K, use_qk_l2norm);
    }
    free(ck); free(Sprev); free(S); free(dS); free(qn); free(kn); free(dqn); free(dkn); free(e); free(du);
  }
  return status;
}
