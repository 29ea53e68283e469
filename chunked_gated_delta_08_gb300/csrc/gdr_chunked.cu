// gdr_chunked.cu -- the chunked (three-kernel) form of the gated delta rule
// forward, products on warp-level tensor-core MMAs with fp32 accumulation.
//
// Kernel order follows the pages' forward chain (KCP handbook, section on the
// debug-script layout: fwd_intra -> wy -> fwd_h -> o):
//   chunk_index_kernel  cu_seqlens -> (sequence, chunk) map, int64
//   prepare_kernel      per (chunk, value head): L2 norm of k, gate cumsum,
//                       A = tril(beta K K^T * decay, -1), T = (I + A)^-1 by
//                       blocks (tensor cores, 3 x TF32), w and u as products
//                       with T; when given a buffer, also the rows
//                       K * exp(G_C - G) for the state scan
//   fwd_h_kernel        per (sequence, value head, V-tile), sequential over
//                       chunks: h (state entering the chunk), v_new = u - w h,
//                       h <- exp(G_C) h + (K * exp(G_C - G))^T v_new, both
//                       products on tensor cores (gdr_scan.cuh); the rows
//                       K * exp(G_C - G) read as formed by prepare, or formed
//   fwd_o_kernel        per (chunk, value head): o = (q * exp G) h + P v_new
//                       with P = tril(q k^T * decay) (diagonal included),
//                       on tensor cores
//
// Decay factors are always formed as exp(G_i - G_j) with i >= j, so every
// exponent is <= 0 and nothing overflows, whatever the gate values.
//
// Precision by input type: fp32 inputs take every product in 3 x TF32 (close
// to fp32) and the full-precision exponential.  bf16 inputs keep 3 x TF32 for
// the Gram matrices and the solve (T feeds every later product), and take
// the products the fused form also runs in bf16 -- w, u = T [..], v_new = u -
// w h, the state update, q h and P v_new -- as single-pass bf16 warp MMAs
// (m16n8k16, fp32 accumulation), with the hardware exponential.
// All address arithmetic is int64 (coverage guide, section 四).
//
// Pages cited: the coverage guide = "FLA 算子内核正确性测试与覆盖矩阵" (fla/ops correctness-coverage guide);
//   the KCP handbook = "flash-linear-attention KCP 精度失效根因排查手册".
#include <algorithm>

#include "gdr_device.cuh"
#include "gdr_internal.h"
#include "gdr_prep.cuh"
#include "gdr_scan.cuh"

namespace gdr {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kBVh = 32;  // V-tile of the state scan

// --------------------------------------------------------------------------
// chunk index: one block.  Validates cu_seqlens (non-decreasing, cu[0] = 0,
// cu[N] = T); on a violation every offset is -1, every index row is -1 and the
// status word records GDR_ERR_SEQLENS, so the later kernels touch nothing.
// --------------------------------------------------------------------------
__global__ void chunk_index_kernel(const int64_t *__restrict__ cu, int64_t N, int64_t T, int C,
                                   int64_t nt_max, int64_t *__restrict__ chunk_indices,
                                   int64_t *__restrict__ chunk_offsets, int *status) {
  __shared__ long long warp_tot[kThreads / 32];
  __shared__ long long carry_s;
  __shared__ int bad_s;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    carry_s = 0;
    bad_s = 0;
  }
  __syncthreads();
  if (cu) {
    for (int64_t n = tid; n < N; n += blockDim.x)
      if (cu[n + 1] < cu[n]) bad_s = 1;
    if (tid == 0 && (cu[0] != 0 || cu[N] != T)) bad_s = 1;
  }
  __syncthreads();
  if (bad_s) {
    for (int64_t n = tid; n <= N; n += blockDim.x) chunk_offsets[n] = -1;
    if (chunk_indices)
      for (int64_t i = tid; i < 2 * nt_max; i += blockDim.x) chunk_indices[i] = -1;
    if (tid == 0) raise_status(status, GDR_ERR_SEQLENS);
    return;
  }
  for (int64_t base = 0; base < N; base += blockDim.x) {
    const int64_t n = base + tid;
    long long nc = 0;
    if (n < N) {
      const int64_t len = cu ? cu[n + 1] - cu[n] : T;
      nc = (len + C - 1) / C;
    }
    long long x = nc;  // inclusive warp scan
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      long long y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    long long before = 0, total = 0;
    for (int w = 0; w < kWarps; ++w) {
      if (w < warp) before += warp_tot[w];
      total += warp_tot[w];
    }
    const long long excl = carry_s + before + x - nc;
    if (n < N) {
      chunk_offsets[n] = excl;
      if (chunk_indices)
        for (long long j = 0; j < nc; ++j) {
          chunk_indices[2 * (excl + j)] = n;
          chunk_indices[2 * (excl + j) + 1] = j;
        }
    }
    __syncthreads();
    if (tid == 0) carry_s += total;
    __syncthreads();
  }
  const long long nt = carry_s;
  if (tid == 0) chunk_offsets[N] = nt;
  if (chunk_indices)
    for (int64_t i = nt + tid; i < nt_max; i += blockDim.x) {
      chunk_indices[2 * i] = -1;
      chunk_indices[2 * i + 1] = -1;
    }
}

// --------------------------------------------------------------------------
// prepare: grid (nt_max, HV).  Per (chunk, value head), on tensor cores in
// 3 x TF32 wherever the work is a product:
//   Gamma   within-chunk cumsum of g (written to gcum)
//   A_ij    = beta_i sum_d k_id k_jd e^{G_id - G_jd}, i > j.  Scalar gate: the
//             Gram matrix K K^T by tiles, then the decay per entry.  Per-key
//             gate: the diagonal 16 x 16 blocks per entry; a block row a > 0
//             against the rows before it as one product of
//             k_i e^{G_i - G_r} and k_j e^{G_r - G_j}, r = 16 a, so both
//             factors have non-positive exponents (the "safe gate" reading)
//   T       = (I + A)^-1 by blocks (prep::solve_unit_lower)
//   w, u    = T [diag(beta e^G) K | diag(beta) V], 64-column tiles
// smem: ks[C][KL] | gam[C][Kp + 4] or [C] | bet[C] | AT[C][C+1] | Tm[C][C+4] |
//       Bt[C][72] | Xs[16][KL] | Ys[C][KL]   (KL = Kp + 4; Xs, Ys per-key, K <= 128)
// --------------------------------------------------------------------------
constexpr int kBtCols = 64;
constexpr int kBtLd = kBtCols + 8;

__host__ __device__ constexpr int64_t prep_smem_floats(int C, int64_t K, bool per_k) {
  return C * (scan::kpad(K) + 4) + (per_k ? C * (scan::kpad(K) + 4) : C) + C + C * (C + 1) + C * (C + 4) + C * kBtLd +
         prep::gram_scratch_floats(C, K, per_k);
}

// The per-key gate's shared memory allows one block an SM, the scalar gate's two.
template <typename Tin, int C, bool PER_K>
__global__ void __launch_bounds__(kThreads, PER_K ? 1 : 2) prepare_kernel(
    const Tin *__restrict__ k, const Tin *__restrict__ v, const float *__restrict__ g,
    const Tin *__restrict__ beta, const int64_t *__restrict__ cu, const int64_t *__restrict__ chunk_indices,
    int64_t T, int64_t H, int64_t HV, int64_t K, int64_t V, int l2, int beta_logits, float *__restrict__ gcum,
    float *__restrict__ w, float *__restrict__ u,
    float *__restrict__ kb_rows) {
  extern __shared__ float smem[];
  const int64_t Kp = scan::kpad(K), KL = Kp + 4, GL = PER_K ? Kp + 4 : 1;
  constexpr int LA = C + 1, LT = C + 4;
  float *ks = smem;
  float *gam = ks + C * KL;
  float *bet = gam + (PER_K ? C * GL : C);
  float *AT = bet + C;
  float *Tm = AT + C * LA;
  float *Bt = Tm + C * LT;
  float *Xs = Bt + C * kBtLd;
  float *Ys = Xs + 16 * KL;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, gq = lane >> 2, tq = lane & 3;
  const int64_t chunk = blockIdx.x, hv = blockIdx.y;
  int64_t n, j;
  if (!chunk_coords(chunk_indices, chunk, T, C, &n, &j)) return;
  const SeqRange sr = seq_range(cu, n, T);
  const int64_t t0 = sr.bos + j * C;
  const int Lc = (int)(sr.eos - t0 < (int64_t)C ? sr.eos - t0 : (int64_t)C);
  const int64_t hq = hv / (HV / H);
  const int64_t gw = PER_K ? K : 1;
  const int nk = (int)(Kp / 8);
  (void)nk;

  // the chunk's v rows, read tile by tile after the solve: into L2 now
  scan::prefetch_rows_l2(v + (t0 * HV + hv) * V, HV * V * (int64_t)sizeof(Tin), Lc, (int)(V * sizeof(Tin)));
  // ---- k rows (normalized), g, beta
  prep::load_qk_rows<Tin, C>(nullptr, k, t0, Lc, H, hq, K, l2, nullptr, ks, KL);
  prep::tile_to_smem(gam, GL, g + (t0 * HV + hv) * gw, HV * gw, C, (int)gw, Lc, (int)gw);
  for (int i = tid; i < C; i += kThreads) bet[i] = i < Lc ? load_beta(beta, (t0 + i) * HV + hv, beta_logits) : 0.f;
  __syncthreads();
  for (int64_t d = tid; d < gw; d += kThreads) {  // inclusive cumsum down each column
    float acc = 0.f;
    for (int i = 0; i < C; ++i) {
      acc += gam[i * GL + d];
      gam[i * GL + d] = acc;
    }
  }
  __syncthreads();
  for (prep::Walk2D wk(tid, kThreads, (int)gw); wk.r < Lc; wk.next())
    gcum[((t0 + wk.r) * HV + hv) * gw + wk.c] = gam[wk.r * GL + wk.c];
  if (kb_rows)  // k e^{G_L - G} for the state scan, formed once instead of in each of its V-tile blocks
    for (prep::Walk2D wk(tid, kThreads, (int)K); wk.r < Lc; wk.next()) {
      const int i = wk.r, d = wk.c;
      const float gi = PER_K ? gam[i * GL + d] : gam[i], gl = PER_K ? gam[(Lc - 1) * GL + d] : gam[Lc - 1];
      kb_rows[((t0 + i) * HV + hv) * K + d] = ks[i * KL + d] * scan::exp_<scan::kB16<Tin>>(gl - gi);
    }

  // ---- A (strictly lower) into AT
  prep::decayed_gram<C, PER_K, true, scan::kB16<Tin>>(ks, ks, KL, gam, GL, K, Lc, bet, AT, LA, Xs, Ys);

  // ---- T = (I + A)^-1, then dense into Tm (row-major, diagonal 1)
  prep::solve_unit_lower<C>(AT, LA, Bt);
  for (int e = tid; e < C * C; e += kThreads) {
    const int i = e / C, jj = e % C;
    Tm[i * LT + jj] = prep::t_at(AT, LA, i, jj);
  }

  // ---- [w | u] = T [diag(beta e^G) K | diag(beta) V], 64 columns at a time
  const int64_t ncol = K + V;
  for (int64_t c0 = 0; c0 < ncol; c0 += kBtCols) {
    __syncthreads();  // Tm complete; the previous tile's reads of Bt done
    // eight elements per thread in flight: their v loads are issued before any is used
    for (int e0 = tid; e0 < C * kBtCols; e0 += 8 * kThreads) {
      float x[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int e = e0 + q * kThreads, jj = e / kBtCols, cc = e % kBtCols;
        const int64_t col = c0 + cc;
        x[q] = (e < C * kBtCols && jj < Lc && col >= K && col < ncol) ? to_f32(v[((t0 + jj) * HV + hv) * V + (col - K)])
                                                                    : 0.f;
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int e = e0 + q * kThreads, jj = e / kBtCols, cc = e % kBtCols;
        const int64_t col = c0 + cc;
        if (e >= C * kBtCols) break;
        float y = 0.f;
        if (jj < Lc && col < ncol)
          y = col < K ? bet[jj] * scan::exp_<scan::kB16<Tin>>(PER_K ? gam[jj * GL + col] : gam[jj]) * ks[jj * KL + col]
                      : bet[jj] * x[q];
        Bt[jj * kBtLd + cc] = y;
      }
    }
    __syncthreads();
    for (int tix = warp; tix < (C / 16) * (kBtCols / 8); tix += kWarps) {
      const int m0 = 16 * (tix % (C / 16)), n0 = 8 * (tix / (C / 16));
      float d[4];
      if constexpr (scan::kB16<Tin>) prep::tile_b16<false>(d, Tm, LT, Bt, kBtLd, m0, n0, C / 16);
      else prep::tile<false>(d, Tm, LT, Bt, kBtLd, m0, n0, C / 8);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = m0 + gq + 8 * (e >> 1);
        const int64_t col = c0 + n0 + 2 * tq + (e & 1);
        if (i < Lc && col < ncol) {
          if (col < K) w[((t0 + i) * HV + hv) * K + col] = d[e];
          else u[((t0 + i) * HV + hv) * V + (col - K)] = d[e];
        }
      }
    }
  }
}

// --------------------------------------------------------------------------
// fwd_h: one block per (sequence, value head, 32-column V tile), launched
// longest sequence first (seq_of_rank), sequential over the sequence's chunks.
// Each chunk's two products run on tensor cores in 3 x TF32 (gdr_scan.cuh).
// --------------------------------------------------------------------------
// At most 128 registers a thread: two blocks share an SM (the longest sequence's blocks in one wave).
template <typename Tin, int C, bool PER_K>
__global__ void __launch_bounds__(kThreads, 2) fwd_h_kernel(
    const Tin *__restrict__ k, const float *__restrict__ w, const float *__restrict__ u,
    const float *__restrict__ gcum, const float *__restrict__ h0, const int64_t *__restrict__ cu,
    const int64_t *__restrict__ chunk_offsets, int64_t N, int64_t T, int64_t H, int64_t HV, int64_t K,
    int64_t V, int l2, float *__restrict__ h, float *__restrict__ v_new, float *__restrict__ ht,
    const float *__restrict__ kb_rows) {
  extern __shared__ float smem[];
  const scan::Tiles st = scan::carve(smem, C, K);
  if (chunk_offsets && chunk_offsets[N] < 0) return;
  const int tid = threadIdx.x;
  // block b: sequence rank b / (HV * nvt), value head, V tile (rank-major, longest sequences first)
  const int64_t nvt = (V + kBVh - 1) / kBVh, per = HV * nvt;
  const int64_t n = seq_of_rank(cu, N, (int64_t)blockIdx.x / per);
  const int64_t hv = ((int64_t)blockIdx.x % per) / nvt, v0 = ((int64_t)blockIdx.x % nvt) * kBVh;
  const int64_t hq = hv / (HV / H);
  const int64_t Kp = scan::kpad(K);
  const SeqRange sr = seq_range(cu, n, T);
  const int64_t nch = (sr.eos - sr.bos + C - 1) / C;
  const int64_t cbase = chunk_offsets ? chunk_offsets[n] : n * ((T + C - 1) / C);

  for (int64_t e = tid; e < Kp * kBVh; e += kThreads) {
    const int64_t d = e / kBVh, vv = e % kBVh;
    st.hs[d * scan::kHS + vv] = (h0 && d < K && v0 + vv < V) ? h0[((n * HV + hv) * K + d) * V + v0 + vv] : 0.f;
  }
  __syncthreads();

  for (int64_t c = 0; c < nch; ++c) {
    const int64_t t0 = sr.bos + c * C;
    const int Lc = (int)(sr.eos - t0 < (int64_t)C ? sr.eos - t0 : (int64_t)C);
    if (h)
      for (int64_t e = tid; e < K * kBVh; e += kThreads) {
        const int64_t d = e / kBVh, vv = e % kBVh;
        if (v0 + vv < V) h[(((cbase + c) * HV + hv) * K + d) * V + v0 + vv] = st.hs[d * scan::kHS + vv];
      }
    scan::chunk_step<Tin, C, PER_K>(st, k, w, u, gcum, t0, Lc, hv, hq, H, HV, K, V, V, v0, l2, v_new, kb_rows);
  }
  if (ht)
    for (int64_t e = tid; e < K * kBVh; e += kThreads) {
      const int64_t d = e / kBVh, vv = e % kBVh;
      if (v0 + vv < V) ht[((n * HV + hv) * K + d) * V + v0 + vv] = st.hs[d * scan::kHS + vv];
    }
}

// --------------------------------------------------------------------------
// fwd_o: grid (nt_max, HV).  P = tril(q k^T * decay) (diagonal included) by
// prep::decayed_gram, then per 32-column V tile o = (q * e^G) h + P v_new as
// two tensor-core products (3 x TF32).
// smem: qs[C][KL] | ks[C][KL] (then the h tile [Kp][40]) | gam | P[C][C+4] |
//       vn[C][40] | Xs, Ys (per-key gate, K <= 128)
// --------------------------------------------------------------------------
constexpr int kOCols = 32;
constexpr int kOLd = kOCols + 8;

// the ks region also holds the h tile later
__host__ __device__ constexpr int64_t fwd_o_ks_floats(int C, int64_t K) {
  return C * (scan::kpad(K) + 4) > scan::kpad(K) * kOLd ? C * (scan::kpad(K) + 4) : scan::kpad(K) * kOLd;
}

__host__ __device__ constexpr int64_t fwd_o_smem_floats(int C, int64_t K, bool per_k) {
  return C * (scan::kpad(K) + 4) + fwd_o_ks_floats(C, K) + (per_k ? C * (scan::kpad(K) + 4) : C) + C * (C + 4) +
         C * kOLd + prep::gram_scratch_floats(C, K, per_k);
}

// The per-key gate's shared memory allows one block an SM, the scalar gate's two.
template <typename Tin, int C, bool PER_K>
__global__ void __launch_bounds__(kThreads, PER_K ? 1 : 2) fwd_o_kernel(
    const Tin *__restrict__ q, const Tin *__restrict__ k, const float *__restrict__ v_new,
    const float *__restrict__ h, const float *__restrict__ gcum, const int64_t *__restrict__ cu,
    const int64_t *__restrict__ chunk_indices, int64_t T, int64_t H, int64_t HV, int64_t K, int64_t V,
    int l2, Tin *__restrict__ o) {
  extern __shared__ float smem[];
  const int64_t Kp = scan::kpad(K), KL = Kp + 4, GL = PER_K ? Kp + 4 : 1;
  constexpr int LP = C + 4;
  float *qs = smem;
  float *ks = qs + C * KL;
  float *hs = ks;
  float *gam = ks + fwd_o_ks_floats(C, K);
  float *P = gam + (PER_K ? C * GL : C);
  float *vn = P + C * LP;
  float *Xs = vn + C * kOLd;
  float *Ys = Xs + 16 * KL;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, gq = lane >> 2, tq = lane & 3;
  const int64_t chunk = blockIdx.x, hv = blockIdx.y;
  int64_t n, j;
  if (!chunk_coords(chunk_indices, chunk, T, C, &n, &j)) return;
  const SeqRange sr = seq_range(cu, n, T);
  const int64_t t0 = sr.bos + j * C;
  const int Lc = (int)(sr.eos - t0 < (int64_t)C ? sr.eos - t0 : (int64_t)C);
  const int64_t hq = hv / (HV / H);
  const int64_t gw = PER_K ? K : 1;

  prep::load_qk_rows<Tin, C>(q, k, t0, Lc, H, hq, K, l2, qs, ks, KL);
  prep::tile_to_smem(gam, GL, gcum + (t0 * HV + hv) * gw, HV * gw, C, (int)gw, Lc, (int)gw);
  for (int e = tid; e < C * LP; e += kThreads) P[e] = 0.f;  // the product reads P's upper part too
  __syncthreads();
  prep::decayed_gram<C, PER_K, false, scan::kB16<Tin>, scan::kB16<Tin>>(qs, ks, KL, gam, GL, K, Lc, nullptr, P, LP,
                                                                          Xs, Ys);
  // q * e^G in place
  for (prep::Walk2D wk(tid, kThreads, (int)Kp); wk.r < C; wk.next()) {
    const int i = wk.r, d = wk.c;
    if (d < K) qs[i * KL + d] *= scan::exp_<scan::kB16<Tin>>(PER_K ? gam[i * GL + d] : gam[i]);
  }

  auto products = [&](int64_t v0) {
    for (int tix = warp; tix < (C / 16) * (kOCols / 8); tix += kWarps) {
      const int m0 = 16 * (tix % (C / 16)), n0 = 8 * (tix / (C / 16));
      float d1[4], d2[4];
      if constexpr (scan::kB16<Tin>) {
        prep::tile_b16<false>(d1, qs, KL, hs, kOLd, m0, n0, (int)(Kp / 16));
        prep::tile_b16<false>(d2, P, LP, vn, kOLd, m0, n0, C / 16);
      } else {
        prep::tile<false>(d1, qs, KL, hs, kOLd, m0, n0, (int)(Kp / 8));
        prep::tile<false>(d2, P, LP, vn, kOLd, m0, n0, C / 8);
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = m0 + gq + 8 * (e >> 1);
        const int64_t col = v0 + n0 + 2 * tq + (e & 1);
        if (i < Lc && col < V) o[((t0 + i) * HV + hv) * V + col] = from_f32<Tin>(d1[e] + d2[e]);
      }
    }
  };
  const float *hsrc = h + (chunk * HV + hv) * K * V, *vsrc = v_new + (t0 * HV + hv) * V;
  auto vok = [&](int64_t v0) { return (int)(V - v0 < kOCols ? V - v0 : kOCols); };
  if (Kp <= 128) {
    // the next V tile's h and v_new rows load into registers while this tile's products run
    prep::TileRegs<128 * kOCols / kThreads> th;
    prep::TileRegs<C * kOCols / kThreads> tv;
    th.get(hsrc, V, kOCols, (int)K, vok(0));
    tv.get(vsrc, HV * V, kOCols, Lc, vok(0));
    for (int64_t v0 = 0; v0 < V; v0 += kOCols) {
      __syncthreads();  // q * e^G done; the previous tile's reads of hs and vn done
      th.put(hs, kOLd, (int)Kp, kOCols);
      tv.put(vn, kOLd, C, kOCols);
      __syncthreads();
      if (v0 + kOCols < V) {
        th.get(hsrc + v0 + kOCols, V, kOCols, (int)K, vok(v0 + kOCols));
        tv.get(vsrc + v0 + kOCols, HV * V, kOCols, Lc, vok(v0 + kOCols));
      }
      products(v0);
    }
  } else {
    for (int64_t v0 = 0; v0 < V; v0 += kOCols) {
      __syncthreads();  // q * e^G done; the previous tile's reads of hs and vn done
      prep::tile_to_smem(hs, kOLd, hsrc + v0, V, (int)Kp, kOCols, (int)K, vok(v0));
      prep::tile_to_smem(vn, kOLd, vsrc + v0, HV * V, C, kOCols, Lc, vok(v0));
      __syncthreads();
      products(v0);
    }
  }
}

template <typename F>
int launch_checked(F kernel, dim3 grid, size_t smem, cudaStream_t s, const char *name) {
  (void)s;
  if (grid.x == 0 || grid.y == 0 || grid.z == 0) return GDR_OK;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return cuda_error(e, name);
  return GDR_OK;
}

int check_launch(const char *name) {
  count_launch();
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? GDR_OK : cuda_error(e, name);
}

}  // namespace

int launch_chunk_index(const ChunkedArgs &a) {
  chunk_index_kernel<<<1, kThreads, 0, a.stream>>>(a.cu, a.d.N, a.d.T, a.C, a.nt_max, a.chunk_indices,
                                                   a.chunk_offsets, a.status);
  return check_launch("chunk_index_kernel");
}

template <int C_, bool PK_>
struct Cfg {
  static constexpr int C = C_;
  static constexpr bool PK = PK_;
};

// Calls f(Cfg<C, per_k>{}) for the runtime chunk size and gate kind.
template <typename F>
int dispatch_cfg(int C, bool per_k, F &&f) {
  if (C == 64) return per_k ? f(Cfg<64, true>{}) : f(Cfg<64, false>{});
  return per_k ? f(Cfg<32, true>{}) : f(Cfg<32, false>{});
}

template <typename Tin>
static int prepare_t(const ChunkedArgs &a) {
  const int64_t K = a.d.K, V = a.d.V;
  return dispatch_cfg(a.C, a.d.gate == GDR_GATE_PER_K, [&](auto cfg) {
    constexpr int CC = decltype(cfg)::C;
    constexpr bool PK = decltype(cfg)::PK;
    const size_t smem = sizeof(float) * prep_smem_floats(CC, K, PK);
    auto kern = prepare_kernel<Tin, CC, PK>;
    dim3 grid((unsigned)a.nt_max, (unsigned)a.d.HV);
    int rc = launch_checked(kern, grid, smem, a.stream, "prepare_kernel");
    if (rc == GDR_OK && a.nt_max > 0) {
      kern<<<grid, kThreads, smem, a.stream>>>((const Tin *)a.k, (const Tin *)a.v, a.g, (const Tin *)a.beta, a.cu,
                                               a.chunk_indices, a.d.T, a.d.H, a.d.HV, K, V, a.l2,
                                               (a.d.flags & GDR_FLAG_BETA_LOGITS) ? 1 : 0, a.gcum, a.w, a.u, a.kb);
      rc = check_launch("prepare_kernel");
    }
    return rc;
  });
}

template <typename Tin>
static int fwd_h_t(const ChunkedArgs &a) {
  const int64_t K = a.d.K, V = a.d.V;
  return dispatch_cfg(a.C, a.d.gate == GDR_GATE_PER_K, [&](auto cfg) {
    constexpr int CC = decltype(cfg)::C;
    constexpr bool PK = decltype(cfg)::PK;
    const size_t smem = sizeof(float) * scan::smem_floats(CC, K);
    auto kern = fwd_h_kernel<Tin, CC, PK>;
    dim3 grid((unsigned)(a.d.N * a.d.HV * cdiv(V, kBVh)));
    int rc = launch_checked(kern, grid, smem, a.stream, "fwd_h_kernel");
    if (rc == GDR_OK && a.d.N > 0) {
      kern<<<grid, kThreads, smem, a.stream>>>((const Tin *)a.k, a.w, a.u, a.gcum, a.h0, a.cu, a.chunk_offsets,
                                               a.d.N, a.d.T, a.d.H, a.d.HV, K, V, a.l2, a.h, a.v_new, a.ht, a.kb);
      rc = check_launch("fwd_h_kernel");
    }
    return rc;
  });
}

template <typename Tin>
static int fwd_o_t(const ChunkedArgs &a) {
  const int64_t K = a.d.K, V = a.d.V;
  return dispatch_cfg(a.C, a.d.gate == GDR_GATE_PER_K, [&](auto cfg) {
    constexpr int CC = decltype(cfg)::C;
    constexpr bool PK = decltype(cfg)::PK;
    const size_t smem = sizeof(float) * fwd_o_smem_floats(CC, K, PK);
    auto kern = fwd_o_kernel<Tin, CC, PK>;
    dim3 grid((unsigned)a.nt_max, (unsigned)a.d.HV);
    int rc = launch_checked(kern, grid, smem, a.stream, "fwd_o_kernel");
    if (rc == GDR_OK && a.nt_max > 0) {
      kern<<<grid, kThreads, smem, a.stream>>>((const Tin *)a.q, (const Tin *)a.k, a.v_new, a.h, a.gcum, a.cu,
                                               a.chunk_indices, a.d.T, a.d.H, a.d.HV, K, V, a.l2, (Tin *)a.o);
      rc = check_launch("fwd_o_kernel");
    }
    return rc;
  });
}

int launch_chunk_prepare(const ChunkedArgs &a) {
  return a.d.dtype == GDR_BF16 ? prepare_t<__nv_bfloat16>(a) : prepare_t<float>(a);
}
int launch_chunk_fwd_h(const ChunkedArgs &a) {
  return a.d.dtype == GDR_BF16 ? fwd_h_t<__nv_bfloat16>(a) : fwd_h_t<float>(a);
}
int launch_chunk_fwd_o(const ChunkedArgs &a) {
  return a.d.dtype == GDR_BF16 ? fwd_o_t<__nv_bfloat16>(a) : fwd_o_t<float>(a);
}

}  // namespace gdr
