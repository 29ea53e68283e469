// gdr_bwd.cu -- the backward of the chunked gated delta rule.  Products run on
// warp-level tensor-core MMAs with fp32 accumulation: 3 x TF32 for fp32
// inputs; for bf16 inputs the Gram matrices, the solves and the decayed
// products of the gate gradients in 3 x TF32, the rest in one bf16 pass.
//
// The pages give the backward as a chain of chunk kernels (KCP handbook, the
// debug-script layout: bwd_dAu -> bwd_dhu -> bwd_dv -> bwd_o -> bwd_wy ->
// bwd_dqk_intra; coverage guide, section 三, for the gradients graded: dq, dk,
// dv, dg, dbeta, dh0).  This file derives each step from the chunk form of the
// forward.  Per chunk, with Gamma the within-chunk cumsum of g, L the last
// valid row, h the state entering the chunk and dh' = dL/d(state leaving it):
//
//   forward:  v_new = u - w h,  u = T diag(b) V,  w = T diag(b) (K e^G),
//             T = (I + A)^-1,  A_ij = b_i sum_d k_id k_jd e^(G_id - G_jd) (i > j)
//             h' = e^(G_L) h + Kb^T v_new,  Kb = K e^(G_L - G)
//             o  = Qt h + P v_new,  Qt = Q e^G,  P_ri = sum_d q_rd k_id e^(G_rd - G_id) (i <= r)
//   backward: dv_new = P^T do + Kb dh'                      (bwd_dv_local_kernel, bwd_dh_kernel;
//                                                             dv_local also forms the Qt, Kb rows)
//             dh     = Qt^T do + e^(G_L) dh' - w^T dv_new    (bwd_dh_kernel, reverse over chunks)
//             dQt = do h^T,  dW = -dv_new h^T,  dKb = v_new dh'^T,  dP = do v_new^T
//                                                            (bwd_dqkg_kernel)
//             dX = (I + A)^-T dv_new,  dY = (I + A)^-T dW,
//             dA = -(dX u^T + dY w^T) below the diagonal,
//             dv = diag(b) dX,  dbeta = rowsum(dX V + dY K e^G + dA A / b)
//                                                            (bwd_wy_kernel)
//   and dg is the reverse within-chunk cumsum of dGamma; the L2 norm's
//   backward and the sum over the value heads of a q/k group run last
//   (bwd_finalize_kernel).
//
// Every decay factor is e^(G_i - G_j) with i >= j, e^(G_L - G_i) or e^(G_i),
// so no exponent is positive for non-positive gates.  The backward keeps the
// forward's chunk layouts and int64 addressing; it supports K <= 128.
//
// Pages cited: the coverage guide = "FLA 算子内核正确性测试与覆盖矩阵" (fla/ops correctness-coverage guide);
//   the KCP handbook = "flash-linear-attention KCP 精度失效根因排查手册".
#include "gdr_device.cuh"
#include "gdr_internal.h"
#include "gdr_prep.cuh"
#include "gdr_scan.cuh"

namespace gdr {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kBVd = 32;   // V-tile of the dh scan
constexpr int kKmax = 128; // largest K of the backward

struct ChunkPos {
  int64_t t0;  // first token of the chunk
  int Lc;      // valid rows
};

__device__ __forceinline__ bool chunk_pos(const int64_t *cu, const int64_t *chunk_indices, int64_t chunk, int64_t T,
                                          int C, ChunkPos *p) {
  int64_t n, j;
  if (!chunk_coords(chunk_indices, chunk, T, C, &n, &j)) return false;
  const SeqRange sr = seq_range(cu, n, T);
  p->t0 = sr.bos + j * C;
  p->Lc = (int)(sr.eos - p->t0 < (int64_t)C ? sr.eos - p->t0 : (int64_t)C);
  return true;
}

// Gamma of row i, channel d (the scalar gate ignores d).
template <bool PER_K>
__device__ __forceinline__ float gam_at(const float *gam, int i, int64_t d, int64_t K) {
  return PER_K ? gam[i * K + d] : gam[i];
}

// Loads Gamma of the chunk's rows (zero past Lc) from gcum.
template <bool PER_K>
__device__ __forceinline__ void load_gamma(const float *__restrict__ gcum, int64_t t0, int Lc, int C, int64_t HV,
                                           int64_t hv, int64_t K, float *gam, int tid) {
  const int64_t gw = PER_K ? K : 1;
  for (int64_t e = tid; e < C * gw; e += kThreads) {
    const int64_t i = e / gw, d = e % gw;
    gam[e] = i < Lc ? gcum[((t0 + i) * HV + hv) * gw + d] : 0.f;
  }
}

// --------------------------------------------------------------------------
// dv_local: dv_new (local part) = P^T do.  grid (nt_max, HV).  P from
// prep::decayed_gram, then one tensor-core product (3 x TF32) per 32-column
// V tile.
// smem: qs[C][KL] | ks[C][KL] | gam | P[C][C+4] | dos[C][40] | Xs, Ys
// --------------------------------------------------------------------------
constexpr int kDvLd = 40;

__host__ __device__ constexpr int64_t dv_local_smem_floats(int C, int64_t K, bool per_k) {
  return 2 * C * (scan::kpad(K) + 4) + (per_k ? C * (scan::kpad(K) + 4) : C) + C * (C + 4) + C * kDvLd +
         prep::gram_scratch_floats(C, K, per_k);
}

// The per-key gate's shared memory allows one block an SM, the scalar gate's two.
template <typename Tin, int C, bool PER_K>
__global__ void __launch_bounds__(kThreads, PER_K ? 1 : 2) bwd_dv_local_kernel(
    const Tin *__restrict__ q, const Tin *__restrict__ k, const Tin *__restrict__ d_o,
    const float *__restrict__ gcum, const int64_t *__restrict__ cu, const int64_t *__restrict__ chunk_indices,
    int64_t T, int64_t H, int64_t HV, int64_t K, int64_t V, int l2, float *__restrict__ dvn,
    float *__restrict__ qt_rows, float *__restrict__ kb_rows) {
  extern __shared__ float smem[];
  const int64_t Kp = scan::kpad(K), KL = Kp + 4, GL = PER_K ? Kp + 4 : 1;
  constexpr int LP = C + 4;
  float *qs = smem;
  float *ks = qs + C * KL;
  float *gam = ks + C * KL;
  float *P = gam + (PER_K ? C * GL : C);
  float *dos = P + C * LP;
  float *Xs = dos + C * kDvLd;
  float *Ys = Xs + 16 * KL;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, gq = lane >> 2, tq = lane & 3;
  const int64_t hv = blockIdx.y;
  ChunkPos cp;
  if (!chunk_pos(cu, chunk_indices, blockIdx.x, T, C, &cp)) return;
  const int64_t t0 = cp.t0;
  const int Lc = cp.Lc;
  const int64_t hq = hv / (HV / H);
  const int64_t gw = PER_K ? K : 1;

  // the chunk's d_o rows, read tile by tile after the Gram: into L2 now
  scan::prefetch_rows_l2(d_o + (t0 * HV + hv) * V, HV * V * (int64_t)sizeof(Tin), Lc, (int)(V * sizeof(Tin)));
  prep::load_qk_rows<Tin, C>(q, k, t0, Lc, H, hq, K, l2, qs, ks, KL);
  prep::tile_to_smem(gam, GL, gcum + (t0 * HV + hv) * gw, HV * gw, C, (int)gw, Lc, (int)gw);
  for (int e = tid; e < C * LP; e += kThreads) P[e] = 0.f;  // P^T reads the upper part
  __syncthreads();
  // Qt = q e^G and (unless prepare formed them already: kb_rows null) Kb = k e^{G_L - G} of the
  // chunk's rows, read by the reverse state scan
  for (prep::Walk2D wk(tid, kThreads, (int)K); wk.r < Lc; wk.next()) {
    const int i = wk.r, d = wk.c;
    const float gi = PER_K ? gam[i * GL + d] : gam[i];
    const int64_t at = ((t0 + i) * HV + hv) * K + d;
    qt_rows[at] = qs[i * KL + d] * scan::exp_<scan::kB16<Tin>>(gi);
    if (kb_rows) {
      const float gl = PER_K ? gam[(Lc - 1) * GL + d] : gam[Lc - 1];
      kb_rows[at] = ks[i * KL + d] * scan::exp_<scan::kB16<Tin>>(gl - gi);
    }
  }
  // P_ri = sum_d q_rd k_id exp(G_rd - G_id), i <= r < Lc
  prep::decayed_gram<C, PER_K, false, scan::kB16<Tin>, scan::kB16<Tin>>(qs, ks, KL, gam, GL, K, Lc, nullptr, P, LP,
                                                                          Xs, Ys);
  for (int64_t v0 = 0; v0 < V; v0 += 32) {
    __syncthreads();
    prep::tile_to_smem(dos, kDvLd, d_o + (t0 * HV + hv) * V + v0, HV * V, C, 32, Lc,
                       (int)(V - v0 < 32 ? V - v0 : 32));
    __syncthreads();
    for (int tix = warp; tix < (C / 16) * 4; tix += kWarps) {
      const int m0 = 16 * (tix % (C / 16)), n0 = 8 * (tix / (C / 16));
      float d[4] = {0.f, 0.f, 0.f, 0.f};
      prep::tile_acc_t<scan::kB16<Tin>, true, false>(d, P, LP, dos, kDvLd, m0, n0, C / 8);  // A(i, r) = P[r][i]
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = m0 + gq + 8 * (e >> 1);
        const int64_t col = v0 + n0 + 2 * tq + (e & 1);
        if (i < Lc && col < V) dvn[((t0 + i) * HV + hv) * V + col] = d[e];
      }
    }
  }
}

// --------------------------------------------------------------------------
// dh: one block per (sequence, value head, 32-column V tile), launched longest
// sequence first (seq_of_rank), sequential over the sequence's chunks, last
// to first.  Per chunk, on tensor cores (3 x TF32; one bf16 pass for bf16):
//   dv_new += Kb dh'           (C x 32) = (C x K)(K x 32), Kb = k e^{G_L - G}
//   dh = e^{G_L} dh' + Qt^T do - w^T dv_new   (K x 32),      Qt = q e^G
// and dh' (dL/d state leaving the chunk) is recorded per chunk.  Kb and Qt
// rows come formed from bwd_dv_local, so the sequential loop loads rows and
// runs products only.
// smem: the scan tiles (dh in hs, Kb then Qt in kt, w in ws, -dv_new in vn,
//       G_L in gl) | dos[C][40]
// --------------------------------------------------------------------------
// At most 128 registers a thread, so that two blocks share an SM and every block
// of the longest sequence is resident from the start.
template <typename Tin, int C, bool PER_K>
__global__ void __launch_bounds__(kThreads, 2) bwd_dh_kernel(
    const float *__restrict__ qt_rows, const float *__restrict__ kb_rows, const Tin *__restrict__ d_o,
    const float *__restrict__ w, const float *__restrict__ gcum, const float *__restrict__ dht,
    const int64_t *__restrict__ cu, const int64_t *__restrict__ chunk_offsets, int64_t N, int64_t T, int64_t H,
    int64_t HV, int64_t K, int64_t V, int l2, float *__restrict__ dvn, float *__restrict__ dhc,
    float *__restrict__ dh0) {
  extern __shared__ float smem[];
  const scan::Tiles st = scan::carve(smem, C, K);
  float *dos = smem + scan::smem_floats(C, K);
  if (chunk_offsets && chunk_offsets[N] < 0) return;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, gq = lane >> 2, tq = lane & 3;
  // block b: sequence rank b / (HV * nvt), value head, V tile (rank-major, longest sequences first)
  const int64_t nvt = (V + kBVd - 1) / kBVd, per = HV * nvt;
  const int64_t n = seq_of_rank(cu, N, (int64_t)blockIdx.x / per);
  const int64_t hv = ((int64_t)blockIdx.x % per) / nvt, v0 = ((int64_t)blockIdx.x % nvt) * kBVd;
  const int64_t Kp = scan::kpad(K), WL = scan::ws_ld(K), KL = scan::kt_ld(K);
  const SeqRange sr = seq_range(cu, n, T);
  const int64_t nch = (sr.eos - sr.bos + C - 1) / C;
  const int64_t cbase = chunk_offsets ? chunk_offsets[n] : n * ((T + C - 1) / C);
  const int64_t gw = PER_K ? K : 1;
  constexpr int LD = scan::kHS;

  for (int64_t e = tid; e < Kp * kBVd; e += kThreads) {
    const int64_t d = e / kBVd, vv = e % kBVd;
    st.hs[d * LD + vv] = (dht && d < K && v0 + vv < V) ? dht[((n * HV + hv) * K + d) * V + v0 + vv] : 0.f;
  }
  __syncthreads();

  for (int64_t c = nch - 1; c >= 0; --c) {
    const int64_t t0 = sr.bos + c * C;
    const int Lc = (int)(sr.eos - t0 < (int64_t)C ? sr.eos - t0 : (int64_t)C);
    const int64_t tl = t0 + Lc - 1;
    if (c > 0) {  // the previous chunk's rows into L2 while this one runs (it is always whole)
      const int64_t t1 = t0 - C;
      const int vb = (int)((V - v0 < kBVd ? V - v0 : kBVd));
      scan::prefetch_rows_l2(kb_rows + (t1 * HV + hv) * K, HV * K * 4, C, (int)(K * 4));
      scan::prefetch_rows_l2(qt_rows + (t1 * HV + hv) * K, HV * K * 4, C, (int)(K * 4));
      scan::prefetch_rows_l2(w + (t1 * HV + hv) * K, HV * K * 4, C, (int)(K * 4));
      scan::prefetch_rows_l2(gcum + ((t1 + C - 1) * HV + hv) * (PER_K ? K : 1), 4, 1, (int)(4 * (PER_K ? K : 1)));
      scan::prefetch_rows_l2(d_o + (t1 * HV + hv) * V + v0, HV * V * (int64_t)sizeof(Tin), C, vb * (int)sizeof(Tin));
      scan::prefetch_rows_l2(dvn + (t1 * HV + hv) * V + v0, HV * V * 4, C, vb * 4);
    }
    for (int64_t e = tid; e < K * kBVd; e += kThreads) {
      const int64_t d = e / kBVd, vv = e % kBVd;
      if (v0 + vv < V) dhc[(((cbase + c) * HV + hv) * K + d) * V + v0 + vv] = st.hs[d * LD + vv];
    }
    for (int64_t d = tid; d < Kp; d += kThreads)
      st.gl[d] = d < K ? gcum[(tl * HV + hv) * gw + (PER_K ? d : 0)] : 0.f;
    // Kb into kt, w into ws (zero past Lc and past K)
    prep::tile_to_smem(st.kt, KL, kb_rows + (t0 * HV + hv) * K, HV * K, C, (int)Kp, Lc, (int)K);
    prep::tile_to_smem(st.ws, WL, w + (t0 * HV + hv) * K, HV * K, C, (int)Kp, Lc, (int)K);
    __syncthreads();
    // dv_new += Kb dh'; vn keeps -dv_new for the w product below
    for (int tix = warp; tix < (C / 16) * 4; tix += kWarps) {
      const int m0 = 16 * (tix % (C / 16)), n0 = 8 * (tix / (C / 16));
      float d[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = m0 + gq + 8 * (e >> 1);
        const int64_t col = v0 + n0 + 2 * tq + (e & 1);
        d[e] = (i < Lc && col < V) ? dvn[((t0 + i) * HV + hv) * V + col] : 0.f;
      }
      prep::tile_acc_t<scan::kB16<Tin>, false, false>(d, st.kt, KL, st.hs, LD, m0, n0, (int)(Kp / 8));
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = m0 + gq + 8 * (e >> 1), cc = n0 + 2 * tq + (e & 1);
        const int64_t col = v0 + cc;
        if (i < Lc && col < V) dvn[((t0 + i) * HV + hv) * V + col] = d[e];
        st.vn[i * LD + cc] = -d[e];
      }
    }
    __syncthreads();
    // Qt into kt (over Kb), do into dos
    prep::tile_to_smem(st.kt, KL, qt_rows + (t0 * HV + hv) * K, HV * K, C, (int)Kp, Lc, (int)K);
    prep::tile_to_smem(dos, LD, d_o + (t0 * HV + hv) * V + v0, HV * V, C, kBVd, Lc,
                       (int)(V - v0 < kBVd ? V - v0 : kBVd));
    __syncthreads();
    // dh = e^{G_L} dh' + Qt^T do - w^T dv_new
    for (int tix = warp; tix < (int)(Kp / 16) * 4; tix += kWarps) {
      const int m0 = 16 * (tix % (int)(Kp / 16)), n0 = 8 * (tix / (int)(Kp / 16));
      float d[4];
      const float e0 = scan::exp_<scan::kB16<Tin>>(st.gl[PER_K ? m0 + gq : 0]),
                  e1 = scan::exp_<scan::kB16<Tin>>(st.gl[PER_K ? m0 + gq + 8 : 0]);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = m0 + gq + 8 * (e >> 1), cc = n0 + 2 * tq + (e & 1);
        d[e] = st.hs[r * LD + cc] * ((e >> 1) ? e1 : e0);
      }
      prep::tile_acc_t<scan::kB16<Tin>, true, false>(d, st.kt, KL, dos, LD, m0, n0, C / 8);
      prep::tile_acc_t<scan::kB16<Tin>, true, false>(d, st.ws, WL, st.vn, LD, m0, n0, C / 8);
      __syncwarp();
      // every warp reads only its own tiles of hs, so the write-back needs no barrier
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = m0 + gq + 8 * (e >> 1), cc = n0 + 2 * tq + (e & 1);
        st.hs[r * LD + cc] = d[e];
      }
    }
    __syncthreads();
  }
  if (dh0)
    for (int64_t e = tid; e < K * kBVd; e += kThreads) {
      const int64_t d = e / kBVd, vv = e % kBVd;
      if (v0 + vv < V) dh0[((n * HV + hv) * K + d) * V + v0 + vv] = st.hs[d * LD + vv];
    }
}

// --------------------------------------------------------------------------
// dqkg: grid (nt_max, HV).  Accumulates dQt = do h^T, dW = -dv_new h^T (as dv_new h^T, negated when written),
// dKb = v_new dh'^T, dP = do v_new^T over 32-column V tiles on tensor cores
// (3 x TF32, accumulators in registers), then forms the chunk's dq^, dk^ and
// dGamma from the output and state terms on CUDA cores, where thread t owns
// column d = t % 128 and rows i = 2m + t / 128 of every C x K matrix.
// The sums over the other rows of the chunk (sq, sk) come from
// prep::decayed_apply.
// smem: qs, ks [C][Kp+8] | gam[C*K or C] | tiles (do, dv_new, v_new [C][36],
//       h, dh' [Kp][36]; then the staged dQt, dKb [C][Kp]; then sq, sk;
//       sq then the scalar gate's per-element dGamma) | dPs[C][C+4] |
//       colsum[2*128] | gLs[K] | Xs, Ys (per-key gate)
// --------------------------------------------------------------------------
constexpr int kQL = 36;  // row stride of the V tiles (4 mod 32)

__host__ __device__ constexpr int64_t dqkg_region_floats(int C, int64_t K) {
  return (3 * C + 2 * scan::kpad(K)) * kQL > 2 * C * scan::kpad(K) ? (3 * C + 2 * scan::kpad(K)) * kQL
                                                                     : 2 * C * scan::kpad(K);
}

__host__ __device__ constexpr int64_t dqkg_smem_floats(int C, int64_t K, bool per_k) {
  return 2 * C * (scan::kpad(K) + 8) + (per_k ? C * K : C) + dqkg_region_floats(C, K) + C * (C + 4) + 2 * kKmax +
         K + prep::gram_scratch_floats(C, K, per_k);
}

template <typename Tin, int C, bool PER_K>
__global__ void __launch_bounds__(kThreads) bwd_dqkg_kernel(
    const Tin *__restrict__ q, const Tin *__restrict__ k, const Tin *__restrict__ d_o,
    const float *__restrict__ v_new, const float *__restrict__ dvn, const float *__restrict__ h,
    const float *__restrict__ dhc, const float *__restrict__ gcum, const int64_t *__restrict__ cu,
    const int64_t *__restrict__ chunk_indices, int64_t T, int64_t H, int64_t HV, int64_t K, int64_t V, int l2,
    float *__restrict__ dqa, float *__restrict__ dka, float *__restrict__ dga, float *__restrict__ dW) {
  constexpr int MQ = C * kKmax / kThreads;  // rows per thread in the per-element phase
  constexpr int MT = C / 16;                // row tiles
  constexpr int NTW = 16 * MT / 8;          // column tiles of a C x 128 product per warp
  constexpr int NPW = MT * (C / 8) / 8;     // tiles of dP per warp
  extern __shared__ float smem[];
  const int64_t Kp = scan::kpad(K), KQ = Kp + 8;
  constexpr int LP = C + 4;
  float *qs = smem;
  float *ks = qs + C * KQ;
  float *gam = ks + C * KQ;
  float *reg = gam + (PER_K ? C * K : C);
  float *doA = reg, *dvA = doA + C * kQL, *vnA = dvA + C * kQL;
  float *hB = vnA + C * kQL, *dhB = hB + Kp * kQL;
  float *sQ = reg, *sK = reg + C * Kp;  // after the V loop
  float *lo = reg, *up = reg + C * Kp;  // after sQ, sK are read; lo then the scalar gate's dGamma
  float *dPs = reg + dqkg_region_floats(C, K);
  float *colsum = dPs + C * LP;
  float *gLs = colsum + 2 * kKmax;
  float *Xs = gLs + K, *Ys = Xs + 16 * KQ;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, gq = lane >> 2, tq = lane & 3;
  const int64_t chunk = blockIdx.x, hv = blockIdx.y;
  ChunkPos cp;
  if (!chunk_pos(cu, chunk_indices, chunk, T, C, &cp)) return;
  const int64_t t0 = cp.t0;
  const int Lc = cp.Lc;
  const int64_t hq = hv / (HV / H);
  const int d = tid & (kKmax - 1), i_base = tid / kKmax;
  const int ntk = (int)(Kp / 8);  // column tiles of a C x Kp product
  const int m0 = 16 * (warp % MT);
  // the rows of a V tile into L2, one tile ahead of its loads
  auto prefetch_tile = [&](int64_t v0) {
    const int vb = (int)(V - v0 < 32 ? V - v0 : 32);
    const int64_t rs = (t0 * HV + hv) * V + v0, hs0 = (chunk * HV + hv) * K * V + v0;
    scan::prefetch_rows_l2(d_o + rs, HV * V * (int64_t)sizeof(Tin), Lc, vb * (int)sizeof(Tin));
    scan::prefetch_rows_l2(dvn + rs, HV * V * 4, Lc, vb * 4);
    scan::prefetch_rows_l2(v_new + rs, HV * V * 4, Lc, vb * 4);
    scan::prefetch_rows_l2(h + hs0, V * 4, (int)K, vb * 4);
    scan::prefetch_rows_l2(dhc + hs0, V * 4, (int)K, vb * 4);
  };
  prefetch_tile(0);

  prep::load_qk_rows<Tin, C>(q, k, t0, Lc, H, hq, K, l2, qs, ks, KQ);
  prep::tile_to_smem(gam, PER_K ? K : 1, gcum + (t0 * HV + hv) * (PER_K ? K : 1), HV * (PER_K ? K : 1), C,
                     PER_K ? (int)K : 1, Lc, PER_K ? (int)K : 1);
  for (int e = tid; e < 2 * kKmax; e += kThreads) colsum[e] = 0.f;

  float aQ[MQ], aK[MQ];
  float fQ[NTW][4], fW[NTW][4], fK[NTW][4], fP[NPW][4];
#pragma unroll
  for (int s = 0; s < NTW; ++s)
#pragma unroll
    for (int e = 0; e < 4; ++e) fQ[s][e] = fW[s][e] = fK[s][e] = 0.f;
#pragma unroll
  for (int s = 0; s < NPW; ++s)
#pragma unroll
    for (int e = 0; e < 4; ++e) fP[s][e] = 0.f;
  float gLacc = 0.f;

  for (int64_t v0 = 0; v0 < V; v0 += 32) {
    __syncthreads();  // the previous tile's reads are done
    if (v0 + 32 < V) prefetch_tile(v0 + 32);
    {
      // dvA holds +dv_new (dW = -dv_new h^T takes the sign when written)
      const int vok = (int)(V - v0 < 32 ? V - v0 : 32);
      const int64_t rs = (t0 * HV + hv) * V + v0, hs0 = (chunk * HV + hv) * K * V + v0;
      prep::tile_to_smem(doA, kQL, d_o + rs, HV * V, C, 32, Lc, vok);
      prep::tile_to_smem(dvA, kQL, dvn + rs, HV * V, C, 32, Lc, vok);
      prep::tile_to_smem(vnA, kQL, v_new + rs, HV * V, C, 32, Lc, vok);
      prep::tile_to_smem(hB, kQL, h + hs0, V, (int)Kp, 32, (int)K, vok);
      prep::tile_to_smem(dhB, kQL, dhc + hs0, V, (int)Kp, 32, (int)K, vok);
    }
    __syncthreads();
    if (tid < K)
      for (int vv = 0; vv < 32; ++vv) gLacc = fmaf(hB[tid * kQL + vv], dhB[tid * kQL + vv], gLacc);
    if constexpr (scan::kB16<Tin>) {
      // one bf16 pass per k-step of 16 (the operands' rows are float pairs: kQL is even)
#pragma unroll
      for (int k0 = 0; k0 < 32; k0 += 16) {
        uint32_t oa[4], wa[4], na[4];
        {
          const float *ar = doA + (m0 + gq) * kQL + k0 + 2 * tq;
          const float *br = dvA + (m0 + gq) * kQL + k0 + 2 * tq;
          const float *cr = vnA + (m0 + gq) * kQL + k0 + 2 * tq;
          const int offs[4] = {0, 8 * kQL, 8, 8 * kQL + 8};
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            const float2 p0 = *reinterpret_cast<const float2 *>(ar + offs[x]);
            const float2 p1 = *reinterpret_cast<const float2 *>(br + offs[x]);
            const float2 p2 = *reinterpret_cast<const float2 *>(cr + offs[x]);
            oa[x] = scan::bf16x2(p0.x, p0.y);
            wa[x] = scan::bf16x2(p1.x, p1.y);
            na[x] = scan::bf16x2(p2.x, p2.y);
          }
        }
#pragma unroll
        for (int s = 0; s < NTW; ++s) {
          const int tix = warp + 8 * s;
          const int n0 = 8 * (tix / MT);
          if (n0 >= 8 * ntk) continue;
          const float *hb = hB + (n0 + gq) * kQL + k0 + 2 * tq;
          const float *db = dhB + (n0 + gq) * kQL + k0 + 2 * tq;
          const float2 h0v = *reinterpret_cast<const float2 *>(hb), h1v = *reinterpret_cast<const float2 *>(hb + 8);
          const float2 d0v = *reinterpret_cast<const float2 *>(db), d1v = *reinterpret_cast<const float2 *>(db + 8);
          const uint32_t bh0 = scan::bf16x2(h0v.x, h0v.y), bh1 = scan::bf16x2(h1v.x, h1v.y);
          const uint32_t bd0 = scan::bf16x2(d0v.x, d0v.y), bd1 = scan::bf16x2(d1v.x, d1v.y);
          scan::mma_bf16(fQ[s], oa[0], oa[1], oa[2], oa[3], bh0, bh1);
          scan::mma_bf16(fW[s], wa[0], wa[1], wa[2], wa[3], bh0, bh1);
          scan::mma_bf16(fK[s], na[0], na[1], na[2], na[3], bd0, bd1);
        }
#pragma unroll
        for (int s = 0; s < NPW; ++s) {
          const int n0 = 8 * ((warp + 8 * s) / MT);
          const float *vb = vnA + (n0 + gq) * kQL + k0 + 2 * tq;
          const float2 v0v = *reinterpret_cast<const float2 *>(vb), v1v = *reinterpret_cast<const float2 *>(vb + 8);
          scan::mma_bf16(fP[s], oa[0], oa[1], oa[2], oa[3], scan::bf16x2(v0v.x, v0v.y), scan::bf16x2(v1v.x, v1v.y));
        }
      }
    } else {
#pragma unroll
      for (int k0 = 0; k0 < 32; k0 += 8) {
        uint32_t oh[4], ol[4], wh[4], wl[4], nh[4], nl[4];
        {
          const float *ar = doA + (m0 + gq) * kQL + k0 + tq;
          const float *br = dvA + (m0 + gq) * kQL + k0 + tq;
          const float *cr = vnA + (m0 + gq) * kQL + k0 + tq;
          const int offs[4] = {0, 8 * kQL, 4, 8 * kQL + 4};
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            scan::split3(ar[offs[x]], oh[x], ol[x]);
            scan::split3(br[offs[x]], wh[x], wl[x]);
            scan::split3(cr[offs[x]], nh[x], nl[x]);
          }
        }
#pragma unroll
        for (int s = 0; s < NTW; ++s) {
          const int tix = warp + 8 * s;  // m-tile tix % MT (fixed per warp), n-tile tix / MT
          const int n0 = 8 * (tix / MT);
          if (n0 >= 8 * ntk) continue;
          uint32_t bh[2], bl[2], ch[2], cl[2];
          const float *hb = hB + (n0 + gq) * kQL + k0 + tq;
          const float *db = dhB + (n0 + gq) * kQL + k0 + tq;
          scan::split3(hb[0], bh[0], bl[0]);
          scan::split3(hb[4], bh[1], bl[1]);
          scan::split3(db[0], ch[0], cl[0]);
          scan::split3(db[4], ch[1], cl[1]);
          scan::mma3(fQ[s], oh, ol, bh, bl);
          scan::mma3(fW[s], wh, wl, bh, bl);
          scan::mma3(fK[s], nh, nl, ch, cl);
        }
#pragma unroll
        for (int s = 0; s < NPW; ++s) {
          const int n0 = 8 * ((warp + 8 * s) / MT);
          uint32_t bh[2], bl[2];
          const float *vb = vnA + (n0 + gq) * kQL + k0 + tq;
          scan::split3(vb[0], bh[0], bl[0]);
          scan::split3(vb[4], bh[1], bl[1]);
          scan::mma3(fP[s], oh, ol, bh, bl);
        }
      }
    }
  }
  __syncthreads();  // the V tiles are dead: stage dQt and dKb, write dW, stage dP
#pragma unroll
  for (int s = 0; s < NTW; ++s) {
    const int n0 = 8 * ((warp + 8 * s) / MT);
    if (n0 >= 8 * ntk) continue;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int i = m0 + gq + 8 * (e >> 1), dd = n0 + 2 * tq + (e & 1);
      sQ[i * Kp + dd] = fQ[s][e];
      sK[i * Kp + dd] = fK[s][e];
      if (i < Lc && dd < K) dW[((t0 + i) * HV + hv) * K + dd] = -fW[s][e];
    }
  }
#pragma unroll
  for (int s = 0; s < NPW; ++s) {
    const int n0 = 8 * ((warp + 8 * s) / MT);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int r = m0 + gq + 8 * (e >> 1), i = n0 + 2 * tq + (e & 1);
      float val = 0.f;
      if (r < Lc && i <= r) val = PER_K ? fP[s][e] : fP[s][e] * scan::exp_<scan::kB16<Tin>>(gam[r] - gam[i]);
      dPs[r * LP + i] = val;
    }
  }
  __syncthreads();
#pragma unroll
  for (int m = 0; m < MQ; ++m) {
    const int i = 2 * m + i_base;
    aQ[m] = d < K ? sQ[i * Kp + d] : 0.f;
    aK[m] = d < K ? sK[i * Kp + d] : 0.f;
  }
  __syncthreads();  // the staging is dead
  // sq = sum_{j <= i} dP_ij k_j e^{G_i - G_j} (lo), sk = sum_{r >= i} dP_ri q_r e^{G_r - G_i} (up)
  prep::decayed_apply<C, PER_K, false, scan::kB16<Tin>>(dPs, LP, ks, qs, KQ, gam, PER_K ? K : 1, K, Lc, lo, up, Kp,
                                                        Xs, Ys);

  // dW out; dP staged (GDN folds its decay in); column sums of dKb * Kb,
  // each thread's half in a fixed slot so the sum's order is fixed
  if (d < K) {
    float cs = 0.f;
#pragma unroll
    for (int m = 0; m < MQ; ++m) {
      const int i = 2 * m + i_base;
      if (i < Lc) {
        const float gi = gam_at<PER_K>(gam, i, d, K), gL = gam_at<PER_K>(gam, Lc - 1, d, K);
        cs = fmaf(aK[m], ks[i * KQ + d] * scan::exp_<scan::kB16<Tin>>(gL - gi), cs);
      }
    }
    colsum[i_base * kKmax + d] = cs;
  }
  if (tid < K) gLs[tid] = gLacc;
  __syncthreads();

  if (d < K) {
#pragma unroll
    for (int m = 0; m < MQ; ++m) {
      const int i = 2 * m + i_base;
      if (i >= Lc) continue;
      const float gi = gam_at<PER_K>(gam, i, d, K), gL = gam_at<PER_K>(gam, Lc - 1, d, K);
      const float eG = scan::exp_<scan::kB16<Tin>>(gi), eL = scan::exp_<scan::kB16<Tin>>(gL - gi);
      const float qv = qs[i * KQ + d], kv = ks[i * KQ + d];
      float dq = aQ[m] * eG, dk = aK[m] * eL;
      float dgm = aQ[m] * qv * eG - aK[m] * kv * eL;
      const float sq = lo[i * Kp + d], sk = up[i * Kp + d];
      dq += sq;
      dk += sk;
      dgm += qv * sq - kv * sk;
      if (i == Lc - 1) dgm += (colsum[d] + colsum[kKmax + d]) + scan::exp_<scan::kB16<Tin>>(gL) * gLs[d];
      const int64_t row = (t0 + i) * HV + hv;
      dqa[row * K + d] = dq;
      dka[row * K + d] = dk;
      if (PER_K) dga[row * K + d] = dgm;
      else lo[i * Kp + d] = dgm;  // this thread's own entry: read above
    }
  }
  if (!PER_K) {  // scalar gate: dGamma_i = sum_d, one warp per row
    __syncthreads();
    for (int i = warp; i < Lc; i += kWarps) {
      float acc = 0.f;
      for (int64_t dd = lane; dd < K; dd += 32) acc += lo[i * Kp + dd];
      acc = warp_sum(acc);
      if (lane == 0) dga[(t0 + i) * HV + hv] = acc;
    }
  }
}

// --------------------------------------------------------------------------
// wy: grid (nt_max, HV).  The UT transform's backward.  Bm = the decayed Gram
// matrix of k (prep::decayed_gram, strict), A = diag(beta) Bm, T = (I + A)^-1
// by blocks; then on tensor cores (3 x TF32) per 32-column tile
//   dX = T^T dv_new  -> dv = diag(beta) dX, dbeta += rowsum(dX V), dA -= dX u^T
//   dY = T^T dW      -> dA -= dY w^T
// (dA accumulates in register fragments); then dbeta += rowsum(dA Bm) +
// rowsum(dY K e^G), dB = beta_i dA, the k and Gamma terms of the Y and A paths
// on CUDA cores, and dg as the reverse within-chunk cumsum of dGamma.
// smem: ks[C][KL] | gam | bet, dbs, rowacc [C] | AT[C][C+1] (A / T, then dB) |
//       Tm[C][C+4] | Bm[C][C+1] | sY[C][KL] | scratch (gram Xs, Ys; the V
//       tiles; the dW tiles and w; the per-key dGamma)
// --------------------------------------------------------------------------
constexpr int kWt = 32;          // columns per tile
constexpr int kLdB = kWt + 8;    // B operands read [k][n] (8 mod 32)
constexpr int kLdA = kWt + 4;    // A operands / B read [n][k] (4 mod 32)

__host__ __device__ constexpr int64_t wy_scratch_floats(int C, int64_t K, bool per_k) {
  const int64_t KL = scan::kpad(K) + 4;
  const int64_t a = prep::gram_scratch_floats(C, K, per_k);
  const int64_t b = (int64_t)C * (kLdB + 3 * kLdA);
  const int64_t c = (int64_t)C * (kLdB + KL);
  const int64_t m = a > b ? a : b;
  return (m > c ? m : c) > 1536 ? (m > c ? m : c) : 1536;
}

__host__ __device__ constexpr int64_t wy_smem_floats(int C, int64_t K, bool per_k) {
  const int64_t KL = scan::kpad(K) + 4;
  return C * KL + (per_k ? C * (scan::kpad(K) + 4) : C) + 3 * C + C * (C + 1) + C * (C + 4) + C * (C + 1) + 2 * C * KL +
         wy_scratch_floats(C, K, per_k);
}

// Its shared memory allows one block an SM: one block's worth of registers (no cap at 128).
template <typename Tin, int C, bool PER_K>
__global__ void __launch_bounds__(kThreads, 1) bwd_wy_kernel(
    const Tin *__restrict__ k, const Tin *__restrict__ v, const Tin *__restrict__ beta,
    const float *__restrict__ dvn, const float *__restrict__ dW, const float *__restrict__ u,
    const float *__restrict__ w, const float *__restrict__ gcum, const int64_t *__restrict__ cu,
    const int64_t *__restrict__ chunk_indices, int64_t T, int64_t H, int64_t HV, int64_t K, int64_t V, int l2,
    int beta_logits, float *__restrict__ dka, const float *__restrict__ dga, Tin *__restrict__ dv,
    Tin *__restrict__ dbeta, float *__restrict__ dg) {
  constexpr int MQ = C * kKmax / kThreads;
  constexpr int LA = C + 1, LT = C + 4;
  constexpr int MT = C / 16;
  constexpr int NAW = MT * (C / 8) / 8;  // dA tiles per warp
  extern __shared__ float smem[];
  const int64_t Kp = scan::kpad(K), KL = Kp + 4, GL = PER_K ? Kp + 4 : 1;
  float *ks = smem;
  float *gam = ks + C * KL;
  float *bet = gam + (PER_K ? C * GL : C);
  float *dbs = bet + C;
  float *rowacc = dbs + C;
  float *AT = rowacc + C;
  float *Tm = AT + C * LA;
  float *Bm = Tm + C * LT;
  float *sY = Bm + C * LA;
  float *up = sY + C * KL;  // then the per-element dGamma
  float *scr = up + C * KL;
  float *Xs = scr, *Ys = scr + 16 * KL;                                     // gram
  float *dvt = scr, *ut = scr + C * kLdB, *dxt = ut + C * kLdA, *vt = dxt + C * kLdA;  // V tiles
  float *dwt = scr, *wf = scr + C * kLdB;                                   // K tiles, w
  float *gtot = up;
  float *dAs = AT;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, gq = lane >> 2, tq = lane & 3;
  const int64_t hv = blockIdx.y;
  ChunkPos cp;
  if (!chunk_pos(cu, chunk_indices, blockIdx.x, T, C, &cp)) return;
  const int64_t t0 = cp.t0;
  const int Lc = cp.Lc;
  const int64_t hq = hv / (HV / H);
  const int64_t gw = PER_K ? K : 1;
  const int d = tid & (kKmax - 1), i_base = tid / kKmax;
  const int m0 = 16 * (warp % MT);
  // this chunk's rows of the accumulated dk (and dGamma), dW and w are read later: into L2 now;
  // the V tiles one tile ahead of their loads
  scan::prefetch_rows_l2(dka + (t0 * HV + hv) * K, HV * K * 4, Lc, (int)(K * 4));
  if (PER_K) scan::prefetch_rows_l2(dga + (t0 * HV + hv) * K, HV * K * 4, Lc, (int)(K * 4));
  scan::prefetch_rows_l2(dW + (t0 * HV + hv) * K, HV * K * 4, Lc, (int)(K * 4));
  scan::prefetch_rows_l2(w + (t0 * HV + hv) * K, HV * K * 4, Lc, (int)(K * 4));
  auto prefetch_tile = [&](int64_t v0) {
    const int vb = (int)(V - v0 < kWt ? V - v0 : kWt);
    const int64_t rs = (t0 * HV + hv) * V + v0;
    scan::prefetch_rows_l2(dvn + rs, HV * V * 4, Lc, vb * 4);
    scan::prefetch_rows_l2(u + rs, HV * V * 4, Lc, vb * 4);
    scan::prefetch_rows_l2(v + rs, HV * V * (int64_t)sizeof(Tin), Lc, vb * (int)sizeof(Tin));
  };
  prefetch_tile(0);

  prep::load_qk_rows<Tin, C>(nullptr, k, t0, Lc, H, hq, K, l2, nullptr, ks, KL);
  prep::tile_to_smem(gam, GL, gcum + (t0 * HV + hv) * gw, HV * gw, C, (int)gw, Lc, (int)gw);
  for (int i = tid; i < C; i += kThreads) {
    bet[i] = i < Lc ? load_beta(beta, (t0 + i) * HV + hv, beta_logits) : 0.f;
    dbs[i] = 0.f;
    rowacc[i] = 0.f;
  }
  __syncthreads();
  // Bm_ij = sum_d k_id k_jd e^{G_id - G_jd} (i > j); A = diag(beta) Bm
  prep::decayed_gram<C, PER_K, true, scan::kB16<Tin>>(ks, ks, KL, gam, GL, K, Lc, nullptr, Bm, LA, Xs, Ys);
  for (int e = tid; e < C * C; e += kThreads) {
    const int i = e / C, j = e % C;
    if (j < i) AT[i * LA + j] = bet[i] * Bm[i * LA + j];
  }
  __syncthreads();
  prep::solve_unit_lower<C>(AT, LA, scr);
  for (int e = tid; e < C * C; e += kThreads) {
    const int i = e / C, j = e % C;
    Tm[i * LT + j] = prep::t_at(AT, LA, i, j);
  }

  float fA[NAW][4];
#pragma unroll
  for (int s2 = 0; s2 < NAW; ++s2)
#pragma unroll
    for (int e = 0; e < 4; ++e) fA[s2][e] = 0.f;

  // u-path: dX = T^T dv_new per tile; dv; dbeta += rowsum(dX V); acc += dX u^T
  for (int64_t v0 = 0; v0 < V; v0 += kWt) {
    __syncthreads();
    if (v0 + kWt < V) prefetch_tile(v0 + kWt);
    {
      const int vok = (int)(V - v0 < kWt ? V - v0 : kWt);
      prep::tile_to_smem(dvt, kLdB, dvn + (t0 * HV + hv) * V + v0, HV * V, C, kWt, Lc, vok);
      prep::tile_to_smem(ut, kLdA, u + (t0 * HV + hv) * V + v0, HV * V, C, kWt, Lc, vok);
      prep::tile_to_smem(vt, kLdA, v + (t0 * HV + hv) * V + v0, HV * V, C, kWt, Lc, vok);
    }
    __syncthreads();
    for (int tix = warp; tix < MT * (kWt / 8); tix += kWarps) {
      const int mm = 16 * (tix % MT), n0 = 8 * (tix / MT);
      float dd4[4] = {0.f, 0.f, 0.f, 0.f};
      prep::tile_acc_t<scan::kB16<Tin>, true, false>(dd4, Tm, LT, dvt, kLdB, mm, n0, C / 8);  // A(i, j) = T[j][i]
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = mm + gq + 8 * (e >> 1), c = n0 + 2 * tq + (e & 1);
        dxt[i * kLdA + c] = dd4[e];
        if (i < Lc && v0 + c < V) dv[((t0 + i) * HV + hv) * V + v0 + c] = from_f32<Tin>(bet[i] * dd4[e]);
      }
    }
    __syncthreads();
    for (int i = warp; i < Lc; i += kWarps) {  // v rows from the tile (zero past V)
      const float sacc = warp_sum(dxt[i * kLdA + lane] * vt[i * kLdA + lane]);
      if (lane == 0) dbs[i] += sacc;
    }
#pragma unroll
    for (int s2 = 0; s2 < NAW; ++s2) {
      const int n0 = 8 * ((warp + 8 * s2) / MT);
      prep::tile_acc_t<scan::kB16<Tin>, false, true>(fA[s2], dxt, kLdA, ut, kLdA, m0, n0, kWt / 8);  // B(v, j) = u[j][v]
    }
  }
  // w-path: dY = T^T dW into sY, then acc += dY w^T
  for (int64_t d0 = 0; d0 < Kp; d0 += kWt) {
    __syncthreads();
    prep::tile_to_smem(dwt, kLdB, dW + (t0 * HV + hv) * K + d0, HV * K, C, kWt, Lc,
                       (int)(K - d0 < kWt ? (K - d0 > 0 ? K - d0 : 0) : kWt));
    __syncthreads();
    for (int tix = warp; tix < MT * (kWt / 8); tix += kWarps) {
      const int mm = 16 * (tix % MT), n0 = 8 * (tix / MT);
      float dd4[4] = {0.f, 0.f, 0.f, 0.f};
      prep::tile_acc_t<scan::kB16<Tin>, true, false>(dd4, Tm, LT, dwt, kLdB, mm, n0, C / 8);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = mm + gq + 8 * (e >> 1), c = n0 + 2 * tq + (e & 1);
        if (d0 + c < Kp) sY[i * KL + d0 + c] = dd4[e];
      }
    }
  }
  __syncthreads();
  prep::tile_to_smem(wf, KL, w + (t0 * HV + hv) * K, HV * K, C, (int)Kp, Lc, (int)K);
  __syncthreads();
#pragma unroll
  for (int s2 = 0; s2 < NAW; ++s2) {
    const int n0 = 8 * ((warp + 8 * s2) / MT);
    prep::tile_acc_t<scan::kB16<Tin>, false, true>(fA[s2], sY, KL, wf, KL, m0, n0, (int)(Kp / 8));
  }
  __syncthreads();  // AT (T) is dead: dA goes there
#pragma unroll
  for (int s2 = 0; s2 < NAW; ++s2) {
    const int n0 = 8 * ((warp + 8 * s2) / MT);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int i = m0 + gq + 8 * (e >> 1), j = n0 + 2 * tq + (e & 1);
      dAs[i * LA + j] = (j < i && i < Lc) ? -fA[s2][e] : 0.f;
    }
  }
  __syncthreads();
  // dbeta += rowsum(dA Bm) + rowsum(dY K e^G), one warp per row
  for (int i = warp; i < Lc; i += kWarps) {
    float sacc = 0.f;
    for (int j = lane; j < i; j += 32) sacc = fmaf(dAs[i * LA + j], Bm[i * LA + j], sacc);
    for (int64_t dd = lane; dd < K; dd += 32)
      sacc = fmaf(sY[i * KL + dd], ks[i * KL + dd] * scan::exp_<scan::kB16<Tin>>(PER_K ? gam[i * GL + dd] : gam[i]), sacc);
    sacc = warp_sum(sacc);
    if (lane == 0) dbs[i] += sacc;
  }
  __syncthreads();
  // dB = beta_i dA (the scalar gate folds e^{G_i - G_j} in)
  for (int e = tid; e < C * C; e += kThreads) {
    const int i = e / C, j = e % C;
    if (j < i && i < Lc) dAs[i * LA + j] *= bet[i] * (PER_K ? 1.f : scan::exp_<scan::kB16<Tin>>(gam[i] - gam[j]));
  }
  __syncthreads();

  // k^ and Gamma through Y = diag(beta) K e^G and through A:
  // t1 = sum_{j < i} dB_ij k_j e^{G_i - G_j} (lo, over sY), t2 = sum_{r > i} dB_ri k_r e^{G_r - G_i} (up)
  float yv[MQ];
#pragma unroll
  for (int m = 0; m < MQ; ++m) yv[m] = d < K ? sY[(2 * m + i_base) * KL + d] : 0.f;
  __syncthreads();
  float *lo = sY;
  prep::decayed_apply<C, PER_K, true, scan::kB16<Tin>>(dAs, LA, ks, ks, KL, gam, GL, K, Lc, lo, up, KL, scr,
                                                       scr + 16 * KL);
  if (d < K) {
    // the accumulated dk (and per-key dGamma) of this thread's entries, read in two batches so
    // that the loads of a batch are in flight together
#pragma unroll
    for (int hb = 0; hb < 2; ++hb) {
      float ka[MQ / 2], ga[MQ / 2];
#pragma unroll
      for (int mm = 0; mm < MQ / 2; ++mm) {
        const int i = 2 * (hb * (MQ / 2) + mm) + i_base;
        const int64_t row = (t0 + i) * HV + hv;
        ka[mm] = i < Lc ? dka[row * K + d] : 0.f;
        ga[mm] = (PER_K && i < Lc) ? dga[row * K + d] : 0.f;
      }
#pragma unroll
      for (int mm = 0; mm < MQ / 2; ++mm) {
        const int m = hb * (MQ / 2) + mm, i = 2 * m + i_base;
        if (i >= Lc) continue;
        const float gi = PER_K ? gam[i * GL + d] : gam[i];
        const float eG = scan::exp_<scan::kB16<Tin>>(gi), kv = ks[i * KL + d], y = yv[m];
        float dk = bet[i] * y * eG;
        float dgm = dk * kv;
        const float t1 = lo[i * KL + d], t2 = up[i * KL + d];
        dk += t1 + t2;
        dgm += kv * (t1 - t2);
        dka[((t0 + i) * HV + hv) * K + d] = ka[mm] + dk;
        gtot[i * KL + d] = PER_K ? ga[mm] + dgm : dgm;  // this thread's own entry of up
      }
    }
  }
  __syncthreads();
  if (!PER_K) {  // scalar gate: dGamma_i = sum_d, one warp per row
    for (int i = warp; i < Lc; i += kWarps) {
      float acc = 0.f;
      for (int64_t dd = lane; dd < K; dd += 32) acc += gtot[i * KL + dd];
      acc = warp_sum(acc);
      if (lane == 0) rowacc[i] = acc;
    }
    __syncthreads();
  }

  // dg: reverse within-chunk cumsum of dGamma; dbeta out
  if (PER_K) {
    for (int64_t dd = tid; dd < K; dd += kThreads) {
      float run = 0.f;
      for (int i = Lc - 1; i >= 0; --i) {
        run += gtot[i * KL + dd];
        dg[((t0 + i) * HV + hv) * K + dd] = run;
      }
    }
  } else if (tid == 0) {
    float run = 0.f;
    for (int i = Lc - 1; i >= 0; --i) {
      run += rowacc[i] + dga[(t0 + i) * HV + hv];
      dg[(t0 + i) * HV + hv] = run;
    }
  }
  // with logits, dL/dx = dL/dbeta * beta (1 - beta)
  for (int i = tid; i < Lc; i += kThreads)
    dbeta[(t0 + i) * HV + hv] = from_f32<Tin>(beta_logits ? dbs[i] * bet[i] * (1.f - bet[i]) : dbs[i]);
}

// --------------------------------------------------------------------------
// finalize: one warp per (token, q/k head).  Sums dq^, dk^ over the group's
// value heads and applies the L2 norm's backward dx = r (dx^ - x^ (x^ . dx^)).
// --------------------------------------------------------------------------
template <typename Tin>
__global__ void __launch_bounds__(kThreads) bwd_finalize_kernel(
    const Tin *__restrict__ q, const Tin *__restrict__ k, const float *__restrict__ dqa,
    const float *__restrict__ dka, int64_t rows, int64_t H, int64_t HV, int64_t K, int l2, Tin *__restrict__ dq,
    Tin *__restrict__ dk) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (row >= rows * H) return;
  const int64_t t = row / H, hq = row % H, G = HV / H;
#pragma unroll
  for (int which = 0; which < 2; ++which) {
    const Tin *x = which ? k : q;
    const float *acc = which ? dka : dqa;
    Tin *out = which ? dk : dq;
    float dx[kKmax / 32], xv[kKmax / 32];
    float ss = 0.f, dot = 0.f;
#pragma unroll
    for (int m = 0; m < kKmax / 32; ++m) {
      const int64_t d = lane + 32 * m;
      dx[m] = 0.f;
      xv[m] = 0.f;
      if (d < K) {
        for (int64_t g = 0; g < G; ++g) dx[m] += acc[(t * HV + hq * G + g) * K + d];
        xv[m] = to_f32(x[(t * H + hq) * K + d]);
      }
      ss = fmaf(xv[m], xv[m], ss);
    }
    float r = 1.f;
    if (l2) {
      r = rsqrtf(warp_sum(ss) + kL2Eps);
#pragma unroll
      for (int m = 0; m < kKmax / 32; ++m) dot = fmaf(xv[m] * r, dx[m], dot);
      dot = warp_sum(dot);
    }
#pragma unroll
    for (int m = 0; m < kKmax / 32; ++m) {
      const int64_t d = lane + 32 * m;
      if (d < K) out[(t * H + hq) * K + d] = from_f32<Tin>(l2 ? r * (dx[m] - xv[m] * r * dot) : dx[m]);
    }
  }
}

template <typename F>
int set_smem(F kernel, size_t smem, const char *name) {
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  return e == cudaSuccess ? GDR_OK : cuda_error(e, name);
}

int after_launch(const char *name) {
  count_launch();
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? GDR_OK : cuda_error(e, name);
}

template <int C_, bool PK_>
struct Cfg {
  static constexpr int C = C_;
  static constexpr bool PK = PK_;
};

template <typename F>
int dispatch(const BwdArgs &a, F &&f) {
  const bool pk = a.f.d.gate == GDR_GATE_PER_K;
  const bool bf = a.f.d.dtype == GDR_BF16;
  auto by_dtype = [&](auto cfg) {
    return bf ? f(cfg, (__nv_bfloat16 *)nullptr) : f(cfg, (float *)nullptr);
  };
  if (a.f.C == 64) return pk ? by_dtype(Cfg<64, true>{}) : by_dtype(Cfg<64, false>{});
  return pk ? by_dtype(Cfg<32, true>{}) : by_dtype(Cfg<32, false>{});
}

}  // namespace

int launch_bwd_dv_local(const BwdArgs &a) {
  const ChunkedArgs &f = a.f;
  if (f.nt_max == 0) return GDR_OK;
  return dispatch(a, [&](auto cfg, auto tin) {
    using Tin = std::remove_pointer_t<decltype(tin)>;
    constexpr int C = decltype(cfg)::C;
    constexpr bool PK = decltype(cfg)::PK;
    const int64_t K = f.d.K;
    const size_t smem = sizeof(float) * dv_local_smem_floats(C, K, PK);
    auto kern = bwd_dv_local_kernel<Tin, C, PK>;
    int rc = set_smem(kern, smem, "bwd_dv_local_kernel");
    if (rc != GDR_OK) return rc;
    kern<<<dim3((unsigned)f.nt_max, (unsigned)f.d.HV), kThreads, smem, f.stream>>>(
        (const Tin *)f.q, (const Tin *)f.k, (const Tin *)a.d_o, f.gcum, f.cu, f.chunk_indices, f.d.T, f.d.H,
        f.d.HV, K, f.d.V, f.l2, a.dvn, a.dqa, f.kb ? nullptr : a.dka);  // dqa, dka are free until dqkg;
                                                                       // f.kb (== dka) already holds Kb
    return after_launch("bwd_dv_local_kernel");
  });
}

int launch_bwd_dh(const BwdArgs &a) {
  const ChunkedArgs &f = a.f;
  if (f.d.N == 0) return GDR_OK;
  return dispatch(a, [&](auto cfg, auto tin) {
    using Tin = std::remove_pointer_t<decltype(tin)>;
    constexpr int C = decltype(cfg)::C;
    constexpr bool PK = decltype(cfg)::PK;
    const int64_t K = f.d.K;
    const size_t smem = sizeof(float) * (scan::smem_floats(C, K) + C * scan::kHS);
    auto kern = bwd_dh_kernel<Tin, C, PK>;
    int rc = set_smem(kern, smem, "bwd_dh_kernel");
    if (rc != GDR_OK) return rc;
    kern<<<dim3((unsigned)(f.d.N * f.d.HV * cdiv(f.d.V, kBVd))), kThreads, smem, f.stream>>>(
        a.dqa, a.dka, (const Tin *)a.d_o, f.w, f.gcum, a.dht, f.cu, f.chunk_offsets, f.d.N, f.d.T, f.d.H,
        f.d.HV, K, f.d.V, f.l2, a.dvn, a.dhc, a.dh0);  // Qt, Kb rows from bwd_dv_local
    return after_launch("bwd_dh_kernel");
  });
}

int launch_bwd_dqkg(const BwdArgs &a) {
  const ChunkedArgs &f = a.f;
  if (f.nt_max == 0) return GDR_OK;
  return dispatch(a, [&](auto cfg, auto tin) {
    using Tin = std::remove_pointer_t<decltype(tin)>;
    constexpr int C = decltype(cfg)::C;
    constexpr bool PK = decltype(cfg)::PK;
    const int64_t K = f.d.K;
    const size_t smem = sizeof(float) * dqkg_smem_floats(C, K, PK);
    auto kern = bwd_dqkg_kernel<Tin, C, PK>;
    int rc = set_smem(kern, smem, "bwd_dqkg_kernel");
    if (rc != GDR_OK) return rc;
    kern<<<dim3((unsigned)f.nt_max, (unsigned)f.d.HV), kThreads, smem, f.stream>>>(
        (const Tin *)f.q, (const Tin *)f.k, (const Tin *)a.d_o, f.v_new, a.dvn, f.h, a.dhc, f.gcum, f.cu,
        f.chunk_indices, f.d.T, f.d.H, f.d.HV, K, f.d.V, f.l2, a.dqa, a.dka, a.dga, a.dW);
    return after_launch("bwd_dqkg_kernel");
  });
}

int launch_bwd_wy(const BwdArgs &a) {
  const ChunkedArgs &f = a.f;
  if (f.nt_max == 0) return GDR_OK;
  return dispatch(a, [&](auto cfg, auto tin) {
    using Tin = std::remove_pointer_t<decltype(tin)>;
    constexpr int C = decltype(cfg)::C;
    constexpr bool PK = decltype(cfg)::PK;
    const int64_t K = f.d.K;
    const size_t smem = sizeof(float) * wy_smem_floats(C, K, PK);
    auto kern = bwd_wy_kernel<Tin, C, PK>;
    int rc = set_smem(kern, smem, "bwd_wy_kernel");
    if (rc != GDR_OK) return rc;
    kern<<<dim3((unsigned)f.nt_max, (unsigned)f.d.HV), kThreads, smem, f.stream>>>(
        (const Tin *)f.k, (const Tin *)f.v, (const Tin *)f.beta, a.dvn, a.dW, f.u, f.w, f.gcum, f.cu,
        f.chunk_indices, f.d.T, f.d.H, f.d.HV, K, f.d.V, f.l2, (f.d.flags & GDR_FLAG_BETA_LOGITS) ? 1 : 0, a.dka,
        a.dga, (Tin *)a.dv, (Tin *)a.dbeta, a.dg);
    return after_launch("bwd_wy_kernel");
  });
}

int launch_bwd_finalize(const BwdArgs &a) {
  const ChunkedArgs &f = a.f;
  const int64_t rows = f.d.B * f.d.T;
  if (rows == 0) return GDR_OK;
  auto go = [&](auto tin) {
    using Tin = std::remove_pointer_t<decltype(tin)>;
    const int64_t blocks = cdiv(rows * f.d.H, kWarps);
    bwd_finalize_kernel<Tin><<<(unsigned)blocks, kThreads, 0, f.stream>>>(
        (const Tin *)f.q, (const Tin *)f.k, a.dqa, a.dka, rows, f.d.H, f.d.HV, f.d.K, f.l2, (Tin *)a.dq,
        (Tin *)a.dk);
    return after_launch("bwd_finalize_kernel");
  };
  return f.d.dtype == GDR_BF16 ? go((__nv_bfloat16 *)nullptr) : go((float *)nullptr);
}

}  // namespace gdr
