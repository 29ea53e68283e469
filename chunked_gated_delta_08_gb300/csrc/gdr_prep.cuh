// gdr_prep.cuh -- tensor-core building blocks of the chunked form's
// per-chunk preparation: 16 x 8 warp tiles of shared-memory products in
// 3 x TF32 (close to fp32) or one bf16 pass, the decayed Gram and decayed
// products of the per-key gate, and T = (I + A)^-1 of a unit lower-triangular
// C x C matrix by blocks (the UT transform behind the WY representation of
// the coverage guide, section 二).
//
// Fragment layout of mma.sync m16n8k8 (g = lane / 4, t = lane % 4): A (16x8)
// (g, t) (g+8, t) (g, t+4) (g+8, t+4); B (8x8, K x N) (t, g) (t+4, g);
// D (16x8) (g, 2t) (g, 2t+1) (g+8, 2t) (g+8, 2t+1).
//
// Pages cited: the coverage guide = "FLA 算子内核正确性测试与覆盖矩阵" (fla/ops correctness-coverage guide).
#pragma once

#include <type_traits>

#include "gdr_scan.cuh"

namespace gdr {
namespace prep {

// d (16 x 8 tile, rows m0.., cols n0..) = sum over k < 8 nk of A(m, k) B(k, n):
// A(m, k) = a[m lda + k];  B(k, n) = TB ? b[n ldb + k] : b[k ldb + n].
// Conflict-free when lda (and ldb for TB) is 4 mod 32, or ldb 8 mod 32 otherwise.
template <bool TB>
__device__ __forceinline__ void tile(float (&d)[4], const float *a, int64_t lda, const float *b, int64_t ldb,
                                     int m0, int n0, int nk) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int e = 0; e < 4; ++e) d[e] = 0.f;
  for (int ks = 0; ks < nk; ++ks) {
    const int k0 = 8 * ks;
    uint32_t ah[4], al[4], bh[2], bl[2];
    const float *ar = a + (int64_t)(m0 + g) * lda + k0 + t;
    scan::split3(ar[0], ah[0], al[0]);
    scan::split3(ar[8 * lda], ah[1], al[1]);
    scan::split3(ar[4], ah[2], al[2]);
    scan::split3(ar[8 * lda + 4], ah[3], al[3]);
    if (TB) {
      const float *br = b + (int64_t)(n0 + g) * ldb + k0 + t;
      scan::split3(br[0], bh[0], bl[0]);
      scan::split3(br[4], bh[1], bl[1]);
    } else {
      const float *br = b + (int64_t)(k0 + t) * ldb + n0 + g;
      scan::split3(br[0], bh[0], bl[0]);
      scan::split3(br[4 * ldb], bh[1], bl[1]);
    }
    scan::mma3(d, ah, al, bh, bl);
  }
}

// The same product in one bf16 pass (m16n8k16, fp32 accumulation; operands
// rounded to bf16 as they are read), over 16 nk16 values of k, for the bf16
// path's products whose operands the fused form also takes in bf16.  A rows
// and (TB) B rows must start on 8-byte boundaries (even strides and offsets).
template <bool TB>
__device__ __forceinline__ void tile_b16(float (&d)[4], const float *a, int64_t lda, const float *b, int64_t ldb,
                                         int m0, int n0, int nk16) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int e = 0; e < 4; ++e) d[e] = 0.f;
  for (int ks = 0; ks < nk16; ++ks) {
    const int k0 = 16 * ks;
    const float *ar = a + (int64_t)(m0 + g) * lda + k0 + 2 * t;
    const float2 x0 = *reinterpret_cast<const float2 *>(ar), x1 = *reinterpret_cast<const float2 *>(ar + 8 * lda),
                 x2 = *reinterpret_cast<const float2 *>(ar + 8),
                 x3 = *reinterpret_cast<const float2 *>(ar + 8 * lda + 8);
    uint32_t b0, b1;
    if (TB) {
      const float *br = b + (int64_t)(n0 + g) * ldb + k0 + 2 * t;
      const float2 y0 = *reinterpret_cast<const float2 *>(br), y1 = *reinterpret_cast<const float2 *>(br + 8);
      b0 = scan::bf16x2(y0.x, y0.y);
      b1 = scan::bf16x2(y1.x, y1.y);
    } else {
      const float *br = b + (int64_t)(k0 + 2 * t) * ldb + n0 + g;
      b0 = scan::bf16x2(br[0], br[ldb]);
      b1 = scan::bf16x2(br[8 * ldb], br[9 * ldb]);
    }
    scan::mma_bf16(d, scan::bf16x2(x0.x, x0.y), scan::bf16x2(x1.x, x1.y), scan::bf16x2(x2.x, x2.y),
                   scan::bf16x2(x3.x, x3.y), b0, b1);
  }
}

// d += sum over k < 8 nk of A(m, k) B(k, n) on the 16 x 8 tile at (m0, n0):
// A(m, k) = TA ? a[k lda + m] : a[m lda + k];  B(k, n) = TB ? b[n ldb + k] : b[k ldb + n].
template <bool TA, bool TB>
__device__ __forceinline__ void tile_acc(float (&d)[4], const float *a, int64_t lda, const float *b, int64_t ldb,
                                         int m0, int n0, int nk) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  for (int ks = 0; ks < nk; ++ks) {
    const int k0 = 8 * ks;
    uint32_t ah[4], al[4], bh[2], bl[2];
    if (TA) {
      const float *ar = a + (int64_t)(k0 + t) * lda + m0 + g;
      scan::split3(ar[0], ah[0], al[0]);
      scan::split3(ar[8], ah[1], al[1]);
      scan::split3(ar[4 * lda], ah[2], al[2]);
      scan::split3(ar[4 * lda + 8], ah[3], al[3]);
    } else {
      const float *ar = a + (int64_t)(m0 + g) * lda + k0 + t;
      scan::split3(ar[0], ah[0], al[0]);
      scan::split3(ar[8 * lda], ah[1], al[1]);
      scan::split3(ar[4], ah[2], al[2]);
      scan::split3(ar[8 * lda + 4], ah[3], al[3]);
    }
    if (TB) {
      const float *br = b + (int64_t)(n0 + g) * ldb + k0 + t;
      scan::split3(br[0], bh[0], bl[0]);
      scan::split3(br[4], bh[1], bl[1]);
    } else {
      const float *br = b + (int64_t)(k0 + t) * ldb + n0 + g;
      scan::split3(br[0], bh[0], bl[0]);
      scan::split3(br[4 * ldb], bh[1], bl[1]);
    }
    scan::mma3(d, ah, al, bh, bl);
  }
}

// d += the same product in one bf16 pass (m16n8k16, fp32 accumulation) over
// 16 nk16 values of k: A(m, k) = TA ? a[k lda + m] : a[m lda + k];
// B(k, n) = TB ? b[n ldb + k] : b[k ldb + n].  Non-transposed A rows and
// transposed B rows are read as float pairs (even strides and offsets).
template <bool TA, bool TB>
__device__ __forceinline__ void tile_acc_b16(float (&d)[4], const float *a, int64_t lda, const float *b, int64_t ldb,
                                             int m0, int n0, int nk16) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  for (int ks = 0; ks < nk16; ++ks) {
    const int k0 = 16 * ks;
    uint32_t a0, a1, a2, a3, b0, b1;
    if (TA) {
      const float *ar = a + (int64_t)(k0 + 2 * t) * lda + m0 + g;
      a0 = scan::bf16x2(ar[0], ar[lda]);
      a1 = scan::bf16x2(ar[8], ar[lda + 8]);
      a2 = scan::bf16x2(ar[8 * lda], ar[9 * lda]);
      a3 = scan::bf16x2(ar[8 * lda + 8], ar[9 * lda + 8]);
    } else {
      const float *ar = a + (int64_t)(m0 + g) * lda + k0 + 2 * t;
      const float2 x0 = *reinterpret_cast<const float2 *>(ar), x1 = *reinterpret_cast<const float2 *>(ar + 8 * lda),
                   x2 = *reinterpret_cast<const float2 *>(ar + 8),
                   x3 = *reinterpret_cast<const float2 *>(ar + 8 * lda + 8);
      a0 = scan::bf16x2(x0.x, x0.y);
      a1 = scan::bf16x2(x1.x, x1.y);
      a2 = scan::bf16x2(x2.x, x2.y);
      a3 = scan::bf16x2(x3.x, x3.y);
    }
    if (TB) {
      const float *br = b + (int64_t)(n0 + g) * ldb + k0 + 2 * t;
      const float2 y0 = *reinterpret_cast<const float2 *>(br), y1 = *reinterpret_cast<const float2 *>(br + 8);
      b0 = scan::bf16x2(y0.x, y0.y);
      b1 = scan::bf16x2(y1.x, y1.y);
    } else {
      const float *br = b + (int64_t)(k0 + 2 * t) * ldb + n0 + g;
      b0 = scan::bf16x2(br[0], br[ldb]);
      b1 = scan::bf16x2(br[8 * ldb], br[9 * ldb]);
    }
    scan::mma_bf16(d, a0, a1, a2, a3, b0, b1);
  }
}

// The accumulating product for the input type: one bf16 pass for bf16 inputs,
// 3 x TF32 otherwise (nk8 k-steps of 8).
template <bool B16, bool TA, bool TB>
__device__ __forceinline__ void tile_acc_t(float (&d)[4], const float *a, int64_t lda, const float *b, int64_t ldb,
                                           int m0, int n0, int nk8) {
  if constexpr (B16) tile_acc_b16<TA, TB>(d, a, lda, b, ldb, m0, n0, nk8 / 2);
  else tile_acc<TA, TB>(d, a, lda, b, ldb, m0, n0, nk8);
}

// The same with A and B read through functors fa(m, k), fb(k, n) (tile-local
// indices), for the triangular operands of the solve.
template <typename FA, typename FB>
__device__ __forceinline__ void tile_f(float (&d)[4], int nk, FA fa, FB fb) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int e = 0; e < 4; ++e) d[e] = 0.f;
  for (int ks = 0; ks < nk; ++ks) {
    const int k0 = 8 * ks;
    uint32_t ah[4], al[4], bh[2], bl[2];
    scan::split3(fa(g, k0 + t), ah[0], al[0]);
    scan::split3(fa(g + 8, k0 + t), ah[1], al[1]);
    scan::split3(fa(g, k0 + t + 4), ah[2], al[2]);
    scan::split3(fa(g + 8, k0 + t + 4), ah[3], al[3]);
    scan::split3(fb(k0 + t, g), bh[0], bl[0]);
    scan::split3(fb(k0 + t + 4, g), bh[1], bl[1]);
    scan::mma3(d, ah, al, bh, bl);
  }
}

// T[r][s] from the packed array: A strictly below the diagonal of AT (row
// stride lda), T's strict lower part stored transposed above it.
__device__ __forceinline__ float t_at(const float *AT, int lda, int r, int s) {
  return r > s ? AT[s * lda + r] : (r == s ? 1.f : 0.f);
}

// T = (I + A)^-1 for the C x C unit lower-triangular I + A held strictly below
// the diagonal of AT; T's strict lower part is written transposed strictly
// above the diagonal (T_ij at AT[j][i]).  Blocks: 16 x 16 diagonal inverses by
// forward substitution, then [[T1, 0], [T21, T2]] with T21 = -T2 A21 T1 for
// 16 -> 32 and (C = 64) 32 -> 64.  All 256 threads; X is scratch of 1536
// floats.
template <int C>
__device__ void solve_unit_lower(float *AT, int lda, float *X) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  if (warp < C / 16 && lane < 16) {
    const int base = 16 * warp, c = lane;
    float x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float a0 = (i == c) ? 1.f : 0.f, a1 = 0.f;
#pragma unroll
      for (int l = 0; l < i; l += 2) {
        a0 = fmaf(-AT[(base + i) * lda + base + l], x[l], a0);
        if (l + 1 < i) a1 = fmaf(-AT[(base + i) * lda + base + l + 1], x[l + 1], a1);
      }
      x[i] = (i < c) ? 0.f : a0 + a1;
    }
#pragma unroll
    for (int i = 1; i < 16; ++i)
      if (i > c) AT[(base + c) * lda + base + i] = x[i];
  }
  __syncthreads();
  // 16 -> 32: pair p (blocks 2p+1, 2p), n-tile nt; warp = 2p + nt
  if (warp < C / 16) {
    const int p = warp >> 1, nt = warp & 1, r0 = 32 * p + 16, c0 = 32 * p;
    float *Z = X + p * 256;
    float d[4];
    tile_f(d, 2, [&](int r, int k) { return AT[(r0 + r) * lda + c0 + k]; },
           [&](int k, int n) { return t_at(AT, lda, c0 + k, c0 + 8 * nt + n); });
    Z[g * 16 + 8 * nt + 2 * t] = d[0];
    Z[g * 16 + 8 * nt + 2 * t + 1] = d[1];
    Z[(g + 8) * 16 + 8 * nt + 2 * t] = d[2];
    Z[(g + 8) * 16 + 8 * nt + 2 * t + 1] = d[3];
  }
  __syncthreads();
  if (warp < C / 16) {
    const int p = warp >> 1, nt = warp & 1, r0 = 32 * p + 16, c0 = 32 * p;
    const float *Z = X + p * 256;
    float d[4];
    tile_f(d, 2, [&](int r, int k) { return t_at(AT, lda, r0 + r, r0 + k); },
           [&](int k, int n) { return Z[k * 16 + 8 * nt + n]; });
    const int cc = c0 + 8 * nt + 2 * t;
    AT[cc * lda + r0 + g] = -d[0];
    AT[(cc + 1) * lda + r0 + g] = -d[1];
    AT[cc * lda + r0 + g + 8] = -d[2];
    AT[(cc + 1) * lda + r0 + g + 8] = -d[3];
  }
  __syncthreads();
  if (C == 64) {
    // 32 -> 64: Y = A[32:64, 0:32] T[0:32, 0:32]; T[32:64, 0:32] = -T[32:64, 32:64] Y (one 16 x 8 tile per warp)
    const int mt = warp >> 2, nt = warp & 3;
    float *Y = X + 512;
    {
      float d[4];
      tile_f(d, 4, [&](int r, int k) { return AT[(32 + 16 * mt + r) * lda + k]; },
             [&](int k, int n) { return t_at(AT, lda, k, 8 * nt + n); });
      Y[(16 * mt + g) * 32 + 8 * nt + 2 * t] = d[0];
      Y[(16 * mt + g) * 32 + 8 * nt + 2 * t + 1] = d[1];
      Y[(16 * mt + g + 8) * 32 + 8 * nt + 2 * t] = d[2];
      Y[(16 * mt + g + 8) * 32 + 8 * nt + 2 * t + 1] = d[3];
    }
    __syncthreads();
    {
      float d[4];
      tile_f(d, 4, [&](int r, int k) { return t_at(AT, lda, 32 + 16 * mt + r, 32 + k); },
             [&](int k, int n) { return Y[k * 32 + 8 * nt + n]; });
      const int cc = 8 * nt + 2 * t, rr = 32 + 16 * mt + g;
      AT[cc * lda + rr] = -d[0];
      AT[(cc + 1) * lda + rr] = -d[1];
      AT[cc * lda + rr + 8] = -d[2];
      AT[(cc + 1) * lda + rr + 8] = -d[3];
    }
    __syncthreads();
  }
}

// Row and column of element e = start + k * step of a row-major walk with
// `cols` columns, advanced without a division per element (a runtime 64-bit
// division costs dozens of instructions).
struct Walk2D {
  int r, c, dr, dc, cols;
  __device__ __forceinline__ Walk2D(int start, int step, int cols_) : cols(cols_) {
    r = start / cols_;
    c = start - r * cols_;
    dr = step / cols_;
    dc = step - dr * cols_;
  }
  __device__ __forceinline__ void next() {
    r += dr;
    c += dc;
    if (c >= cols) {
      c -= cols;
      ++r;
    }
  }
};

// A rows x cols tile from global memory (row stride lds; fp32 or bf16,
// widened to fp32) into shared memory (row stride ldd), zero past rows_ok rows and cols_ok columns.  Each
// thread has B loads in flight before it stores any, so a tile costs one or
// two memory round trips rather than one per element a thread moves.  All 256
// threads.
template <int B = 16, typename Ts = float>
__device__ __forceinline__ void tile_to_smem(float *dst, int64_t ldd, const Ts *__restrict__ src, int64_t lds,
                                             int rows, int cols, int rows_ok, int cols_ok) {
  Walk2D wk(threadIdx.x, 256, cols);
  for (; wk.r < rows;) {
    float v[B];
    int rr[B], cc[B];
#pragma unroll
    for (int u = 0; u < B; ++u) {
      rr[u] = wk.r;
      cc[u] = wk.c;
      v[u] = (wk.r < rows_ok && wk.c < cols_ok) ? to_f32(src[(int64_t)wk.r * lds + wk.c]) : 0.f;
      wk.next();
    }
#pragma unroll
    for (int u = 0; u < B; ++u)
      if (rr[u] < rows) dst[(int64_t)rr[u] * ldd + cc[u]] = v[u];
  }
}

// A tile like tile_to_smem's held in registers between its loads and its
// stores (N elements per thread, N * 256 >= rows * cols), so the loads of the
// next tile can be in flight while the current one is used.
template <int N>
struct TileRegs {
  float v[N];
  __device__ __forceinline__ void get(const float *__restrict__ src, int64_t lds, int cols, int rows_ok, int cols_ok) {
    Walk2D wk(threadIdx.x, 256, cols);
#pragma unroll
    for (int u = 0; u < N; ++u) {
      v[u] = (wk.r < rows_ok && wk.c < cols_ok) ? src[(int64_t)wk.r * lds + wk.c] : 0.f;
      wk.next();
    }
  }
  __device__ __forceinline__ void put(float *dst, int64_t ldd, int rows, int cols) const {
    Walk2D wk(threadIdx.x, 256, cols);
#pragma unroll
    for (int u = 0; u < N; ++u) {
      if (wk.r < rows) dst[(int64_t)wk.r * ldd + wk.c] = v[u];
      wk.next();
    }
  }
};

// Four consecutive elements of a bf16 or fp32 row as floats (16- or 8-byte load).
template <typename Tin>
__device__ __forceinline__ float4 load4(const Tin *p) {
  if constexpr (std::is_same<Tin, float>::value) {
    return *reinterpret_cast<const float4 *>(p);
  } else {
    const uint2 u = *reinterpret_cast<const uint2 *>(p);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
  }
}

// The rows of load_qk_rows with vector loads, for K % 4 == 0, K <= 128, row
// stride xl % 4 == 0 and q, k aligned to 16 bytes: lane l takes keys 4l ..
// 4l + 3, and all of a warp's rows (C / 8) have their loads in flight at once.
template <typename Tin, int C>
__device__ __forceinline__ void load_qk_rows_vec(const Tin *__restrict__ q, const Tin *__restrict__ k, int64_t t0,
                                                 int Lc, int64_t H, int64_t hq, int64_t K, int l2, float *qs,
                                                 float *ks, int64_t xl) {
  constexpr int kWarps = 8, RPW = C / kWarps;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t width = scan::kpad(K) + 4;
  const int d0 = 4 * lane;
  float4 qv[RPW], kv[RPW];
#pragma unroll
  for (int r = 0; r < RPW; ++r) {
    const int i = warp + kWarps * r;
    const bool ok = i < Lc && d0 < K;
    const int64_t off = ((t0 + i) * H + hq) * K + d0;
    qv[r] = (q && ok) ? load4(q + off) : make_float4(0.f, 0.f, 0.f, 0.f);
    kv[r] = ok ? load4(k + off) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int r = 0; r < RPW; ++r) {
    const int i = warp + kWarps * r;
    // the lane's partial sums in the scan's row loader's order, so both normalize a row alike
    const float sq = fmaf(qv[r].w, qv[r].w, fmaf(qv[r].z, qv[r].z, fmaf(qv[r].y, qv[r].y, fmaf(qv[r].x, qv[r].x, 0.f))));
    const float sk = fmaf(kv[r].w, kv[r].w, fmaf(kv[r].z, kv[r].z, fmaf(kv[r].y, kv[r].y, fmaf(kv[r].x, kv[r].x, 0.f))));
    const float cq = l2 ? rsqrtf(warp_sum(sq) + kL2Eps) : 1.f, ck = l2 ? rsqrtf(warp_sum(sk) + kL2Eps) : 1.f;
    if (d0 < width) {  // zero past K up to the padded width
      if (q) *reinterpret_cast<float4 *>(qs + i * xl + d0) = make_float4(qv[r].x * cq, qv[r].y * cq, qv[r].z * cq, qv[r].w * cq);
      *reinterpret_cast<float4 *>(ks + i * xl + d0) = make_float4(kv[r].x * ck, kv[r].y * ck, kv[r].z * ck, kv[r].w * ck);
    }
    if (lane == 0 && width > 128) {  // the last padding columns past lane 31's keys
      if (q) *reinterpret_cast<float4 *>(qs + i * xl + 128) = make_float4(0.f, 0.f, 0.f, 0.f);
      *reinterpret_cast<float4 *>(ks + i * xl + 128) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
}

// Rows of q (optional) and k, L2-normalized if asked, zero past Lc and past K,
// into qs and ks (row stride xl >= kpad(K) + 4).  Four rows per warp have
// their loads in flight before any row is reduced (all of them, with vector
// loads, where load_qk_rows_vec applies).  All 256 threads.
template <typename Tin, int C>
__device__ __forceinline__ void load_qk_rows(const Tin *__restrict__ q, const Tin *__restrict__ k, int64_t t0,
                                             int Lc, int64_t H, int64_t hq, int64_t K, int l2, float *qs,
                                             float *ks, int64_t xl) {
  if (K <= 128 && K % 4 == 0 && xl % 4 == 0 &&
      ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(qs) |
        reinterpret_cast<uintptr_t>(ks)) & 15u) == 0) {
    load_qk_rows_vec<Tin, C>(q, k, t0, Lc, H, hq, K, l2, qs, ks, xl);
    return;
  }
  constexpr int kWarps = 8;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t width = scan::kpad(K) + 4;
  for (int i0 = warp; i0 < C; i0 += 4 * kWarps) {
    float qv[4][8], kv[4][8];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int i = i0 + kWarps * r;
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const int64_t d = lane + 32 * m;
        const bool ok = i < C && i < Lc && d < K;
        qv[r][m] = (q && ok) ? to_f32(q[((t0 + i) * H + hq) * K + d]) : 0.f;
        kv[r][m] = ok ? to_f32(k[((t0 + i) * H + hq) * K + d]) : 0.f;
      }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int i = i0 + kWarps * r;
      if (i >= C) break;
      float sq = 0.f, sk = 0.f;
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        sq = fmaf(qv[r][m], qv[r][m], sq);
        sk = fmaf(kv[r][m], kv[r][m], sk);
      }
      const float cq = l2 ? rsqrtf(warp_sum(sq) + kL2Eps) : 1.f, ck = l2 ? rsqrtf(warp_sum(sk) + kL2Eps) : 1.f;
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const int64_t d = lane + 32 * m;
        if (d < width) {
          if (q) qs[i * xl + d] = qv[r][m] * cq;
          ks[i * xl + d] = kv[r][m] * ck;
        }
      }
    }
  }
}

// The per-key gate's block-row products need two scaled copies of the rows
// (Xs, Ys); past K = 128 they would not fit, and every entry is formed
// directly instead.
__host__ __device__ constexpr bool gram_factored(int64_t K) { return K <= 128; }

// Floats of scratch (Xs, Ys: 16 + 48 rows at C = 64) decayed_gram and
// decayed_apply need, for row strides up to kpad(K) + 8.
__host__ __device__ constexpr int64_t gram_scratch_floats(int C, int64_t K, bool per_k) {
  return per_k && gram_factored(K) ? C * (scan::kpad(K) + 8) : 0;
}

// out[i][j] = s_i sum_d X_id Y_jd e^{G_id - G_jd} for j < i (STRICT) or
// j <= i, i < Lc; 0 elsewhere (out row stride lo).  X, Y rows have stride xl
// (= kpad(K) + 4, zero past K); gam is G per row (scalar gate, gl = 1) or per
// row and channel (stride gl); s (nullable) is a row scale.  Scalar gate: the
// Gram tiles, then e^{G_i - G_j} per entry.  Per-key gate: diagonal 16 x 16
// blocks entry by entry; block row a > 0 against rows 0 .. 16a-1 as one
// product of X_i e^{G_i - G_r} and Y_j e^{G_r - G_j}, r = 16 a, so no factor
// has a positive exponent for non-positive gates.  FAST takes the hardware
// exponential and B16 one bf16 pass for the tile products (the bf16 path; B16
// only where the result is itself rounded to bf16 next, as P is).  All 256
// threads; ends with a barrier.
template <int C, bool PER_K, bool STRICT, bool FAST = false, bool B16 = false>
__device__ void decayed_gram(const float *X, const float *Y, int64_t xl, const float *gam, int64_t gl, int64_t K,
                             int Lc, const float *s, float *out, int lo, float *Xs, float *Ys) {
  constexpr int kWarps = 8;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, gq = lane >> 2, tq = lane & 3;
  const int64_t Kp = scan::kpad(K);
  const int nk = (int)(Kp / 8);
  auto below = [](int i, int j) { return STRICT ? j < i : j <= i; };
  if (!PER_K) {
    // lower-triangle tiles: row tile a (16 rows) x column tiles 0 .. 2a+1 (8 columns)
    for (int tix = warp; tix < (C / 16) * (C / 16 + 1); tix += kWarps) {
      int a = 0, rem = tix;
      while (rem >= 2 * a + 2) {
        rem -= 2 * a + 2;
        ++a;
      }
      const int m0 = 16 * a, n0 = 8 * rem;
      float d[4];
      if constexpr (B16) tile_b16<true>(d, X, xl, Y, xl, m0, n0, nk / 2);
      else tile<true>(d, X, xl, Y, xl, m0, n0, nk);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = m0 + gq + 8 * (e >> 1), j = n0 + 2 * tq + (e & 1);
        out[i * lo + j] = (below(i, j) && i < Lc) ? (s ? s[i] : 1.f) * scan::exp_<FAST>(gam[i] - gam[j]) * d[e] : 0.f;
      }
    }
    __syncthreads();
    return;
  }
  const bool factored = gram_factored(K);
  const int per_row = factored ? 16 : C;
  if (factored)  // block rows starting past Lc are skipped below: their entries are zero
    for (int e = tid; e < C * C; e += 256) {
      const int i = e / C, j = e % C;
      if (i >= Lc && j < 16 * (i / 16)) out[i * lo + j] = 0.f;
    }
  // one thread per entry: a plain loop over d, no cross-lane reduction
  for (int p = tid; p < C * per_row; p += 256) {
    const int i = p / per_row, j = (factored ? 16 * (i / 16) : 0) + p % per_row;
    float acc = 0.f;
    if (below(i, j) && i < Lc) {
      const float *xr = X + i * xl, *yr = Y + j * xl, *gi = gam + i * gl, *gj = gam + j * gl;
      if (K % 4 == 0 && xl % 4 == 0 && gl % 4 == 0) {  // 16-byte rows: four keys per load
        float a0 = 0.f, a1 = 0.f;
        for (int64_t d = 0; d < K; d += 4) {
          const float4 x = *reinterpret_cast<const float4 *>(xr + d), y = *reinterpret_cast<const float4 *>(yr + d);
          const float4 p = *reinterpret_cast<const float4 *>(gi + d), q = *reinterpret_cast<const float4 *>(gj + d);
          a0 = fmaf(x.x * y.x, scan::exp_<FAST>(p.x - q.x), a0);
          a1 = fmaf(x.y * y.y, scan::exp_<FAST>(p.y - q.y), a1);
          a0 = fmaf(x.z * y.z, scan::exp_<FAST>(p.z - q.z), a0);
          a1 = fmaf(x.w * y.w, scan::exp_<FAST>(p.w - q.w), a1);
        }
        acc = a0 + a1;
      } else {
        for (int64_t d = 0; d < K; ++d) acc = fmaf(xr[d] * yr[d], scan::exp_<FAST>(gi[d] - gj[d]), acc);
      }
      acc *= s ? s[i] : 1.f;
    }
    out[i * lo + j] = acc;
  }
  // 16-byte rows everywhere: the scaled copies move four keys at a time
  const bool vec4 = K % 4 == 0 && xl % 4 == 0 && gl % 4 == 0 &&
                    ((reinterpret_cast<uintptr_t>(X) | reinterpret_cast<uintptr_t>(Y) | reinterpret_cast<uintptr_t>(gam) |
                      reinterpret_cast<uintptr_t>(Xs) | reinterpret_cast<uintptr_t>(Ys)) & 15u) == 0;
  for (int a = 1; factored && a < C / 16 && 16 * a < Lc; ++a) {
    const int r = 16 * a;
    __syncthreads();
    if (vec4) {  // four keys per load and store
      for (Walk2D wk(tid, 256, (int)(Kp / 4)); wk.r < 16 + r; wk.next()) {
        const int row = wk.r;
        const int64_t d = 4 * (int64_t)wk.c;
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
        if (row < 16) {
          const int i = r + row;
          if (d < K && i < Lc) {
            const float4 x = load4(X + i * xl + d), p = load4(gam + i * gl + d), q = load4(gam + r * gl + d);
            o = make_float4(x.x * scan::exp_<FAST>(p.x - q.x), x.y * scan::exp_<FAST>(p.y - q.y),
                            x.z * scan::exp_<FAST>(p.z - q.z), x.w * scan::exp_<FAST>(p.w - q.w));
          }
          *reinterpret_cast<float4 *>(Xs + row * xl + d) = o;
        } else {
          const int jr = row - 16;
          if (d < K) {
            const float4 y = load4(Y + jr * xl + d), p = load4(gam + r * gl + d), q = load4(gam + jr * gl + d);
            o = make_float4(y.x * scan::exp_<FAST>(p.x - q.x), y.y * scan::exp_<FAST>(p.y - q.y),
                            y.z * scan::exp_<FAST>(p.z - q.z), y.w * scan::exp_<FAST>(p.w - q.w));
          }
          *reinterpret_cast<float4 *>(Ys + jr * xl + d) = o;
        }
      }
    } else
    for (Walk2D wk(tid, 256, (int)Kp); wk.r < 16 + r; wk.next()) {
      const int row = wk.r;
      const int64_t d = wk.c;
      if (row < 16) {
        const int i = r + row;
        Xs[row * xl + d] = (d < K && i < Lc) ? X[i * xl + d] * scan::exp_<FAST>(gam[i * gl + d] - gam[r * gl + d]) : 0.f;
      } else {
        const int jr = row - 16;
        Ys[jr * xl + d] = d < K ? Y[jr * xl + d] * scan::exp_<FAST>(gam[r * gl + d] - gam[jr * gl + d]) : 0.f;
      }
    }
    __syncthreads();
    for (int nt = warp; nt < r / 8; nt += kWarps) {
      float d[4];
      if constexpr (B16) tile_b16<true>(d, Xs, xl, Ys, xl, 0, 8 * nt, nk / 2);
      else tile<true>(d, Xs, xl, Ys, xl, 0, 8 * nt, nk);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = r + gq + 8 * (e >> 1), j = 8 * nt + 2 * tq + (e & 1);
        out[i * lo + j] = i < Lc ? (s ? s[i] : 1.f) * d[e] : 0.f;
      }
    }
  }
  __syncthreads();
}

// Both sides of a decayed product with a lower-triangular C x C matrix M
// (row stride lm; zero above the diagonal, and on it when STRICT):
//   lo[i][d] = sum_{j < i (<= i)} M[i][j] Ylo[j][d] e^{G_id - G_jd}
//   up[i][d] = sum_{r > i (>= i)} M[r][i] Yup[r][d] e^{G_rd - G_id}
// for i < Lc, d < kpad(K) (outputs with row stride lw; zero past K; rows past
// Lc are zero or unspecified).  M, Y rows past Lc must be zero; no row past Lc
// enters a decay factor (their G is a placeholder).  Y rows have stride yl
// (zero past K).  Scalar gate: the decay must
// already be folded into M, and lo = M Y, up = M^T Y are plain products.
// Per-key gate: diagonal 16 x 16 blocks term by term; for block row a > 0
// (r0 = 16 a) the block products
//   lo[i] += e^{G_i - G_r0} (M[i, :r0] (Y_j e^{G_r0 - G_j}))        i in block a
//   up[i] += e^{G_r0 - G_i} (M[block a, i]^T (Y_r e^{G_r - G_r0}))  i < r0
// where every exponent is non-positive for non-positive gates.  Xs, Ys:
// scratch of gram_scratch_floats.  FAST takes the hardware exponential (bf16
// inputs); the products stay in 3 x TF32, since the gate gradients sum
// near-cancelling terms.  All 256 threads; ends with a barrier.
template <int C, bool PER_K, bool STRICT, bool FAST = false>
__device__ void decayed_apply(const float *M, int lm, const float *Ylo, const float *Yup, int64_t yl, const float *gam,
                              int64_t gl, int64_t K, int Lc, float *lo, float *up, int64_t lw, float *Xs, float *Ys) {
  constexpr int kWarps = 8;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, gq = lane >> 2, tq = lane & 3;
  const int64_t Kp = scan::kpad(K);
  const int nkt = (int)(Kp / 8);
  if constexpr (!PER_K) {
    {
      for (int tix = warp; tix < (C / 16) * nkt; tix += kWarps) {
        const int m0 = 16 * (tix % (C / 16)), n0 = 8 * (tix / (C / 16));
        float a[4] = {0.f, 0.f, 0.f, 0.f}, b[4] = {0.f, 0.f, 0.f, 0.f};
        tile_acc<false, false>(a, M, lm, Ylo, yl, m0, n0, C / 8);
        tile_acc<true, false>(b, M, lm, Yup, yl, m0, n0, C / 8);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int i = m0 + gq + 8 * (e >> 1), d = n0 + 2 * tq + (e & 1);
          lo[i * lw + d] = a[e];
          up[i * lw + d] = b[e];
        }
      }
    }
    __syncthreads();
  } else {
  if (!gram_factored(K)) {  // per-key gate past K = 128: every term directly
    {
      for (Walk2D wk(tid, 256, (int)Kp); wk.r < C; wk.next()) {
        const int i = wk.r;
        const int64_t d = wk.c;
        float a = 0.f, b = 0.f;
        if (d < K && i < Lc) {
          const float gi = gam[i * gl + d];
          for (int j = 0; j < Lc; ++j) {
            if (STRICT ? j < i : j <= i) a = fmaf(M[i * lm + j] * Ylo[j * yl + d], scan::exp_<FAST>(gi - gam[j * gl + d]), a);
            if (STRICT ? j > i : j >= i) b = fmaf(M[j * lm + i] * Yup[j * yl + d], scan::exp_<FAST>(gam[j * gl + d] - gi), b);
          }
        }
        lo[i * lw + d] = a;
        up[i * lw + d] = b;
      }
    }
    __syncthreads();
    return;
  }
  // diagonal blocks, term by term.  Thread (ib, d) takes column d of blocks ib, ib + RP, ...: it
  // holds the block's gates and Y rows (Ylo for lo, then Yup for up) of that column in registers
  // and forms all 16 rows, with the loops over rows and terms unrolled.
  {
    const int RP = 256 / (int)Kp;  // column groups (Kp <= 128 here)
    const int d = tid % (int)Kp, ib = tid / (int)Kp;
    if (ib < RP) {
      for (int base = 16 * ib; base < C; base += 16 * RP) {
        float yr[16], gg[16];
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
          const int j = base + jj;
          const bool ok = d < K && j < Lc;
          yr[jj] = ok ? Ylo[j * yl + d] : 0.f;
          gg[jj] = ok ? gam[j * gl + d] : 0.f;
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) {  // terms j <= i < Lc
          const int i = base + r;
          float a = 0.f;
          if (d < K && i < Lc) {
#pragma unroll
            for (int jj = 0; jj < (STRICT ? r : r + 1); ++jj)
              a = fmaf(M[i * lm + base + jj] * yr[jj], scan::exp_<FAST>(gg[r] - gg[jj]), a);
          }
          lo[i * lw + d] = a;
        }
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
          const int j = base + jj;
          yr[jj] = d < K && j < Lc ? Yup[j * yl + d] : 0.f;
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) {  // terms j >= i, j < Lc
          const int i = base + r;
          float b = 0.f;
          if (d < K && i < Lc) {
#pragma unroll
            for (int jj = STRICT ? r + 1 : r; jj < 16; ++jj)
              if (base + jj < Lc) b = fmaf(M[(base + jj) * lm + i] * yr[jj], scan::exp_<FAST>(gg[jj] - gg[r]), b);
          }
          up[i * lw + d] = b;
        }
      }
    }
  }
  // 16-byte rows everywhere: the scaled copies move four keys at a time
  const bool vec4 = K % 4 == 0 && yl % 4 == 0 && gl % 4 == 0 &&
                    ((reinterpret_cast<uintptr_t>(Ylo) | reinterpret_cast<uintptr_t>(Yup) | reinterpret_cast<uintptr_t>(gam) |
                      reinterpret_cast<uintptr_t>(Xs) | reinterpret_cast<uintptr_t>(Ys)) & 15u) == 0;
  for (int a = 1; a < C / 16 && 16 * a < Lc; ++a) {
    const int r0 = 16 * a;
    __syncthreads();
    if (vec4) {  // four keys per load and store
      for (Walk2D wk(tid, 256, (int)(Kp / 4)); wk.r < 16 + r0; wk.next()) {
        const int row = wk.r;
        const int64_t d = 4 * (int64_t)wk.c;
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
        if (row < 16) {
          const int r = r0 + row;
          if (d < K && r < Lc) {
            const float4 y = load4(Yup + r * yl + d), p = load4(gam + r * gl + d), q = load4(gam + r0 * gl + d);
            o = make_float4(y.x * scan::exp_<FAST>(p.x - q.x), y.y * scan::exp_<FAST>(p.y - q.y),
                            y.z * scan::exp_<FAST>(p.z - q.z), y.w * scan::exp_<FAST>(p.w - q.w));
          }
          *reinterpret_cast<float4 *>(Xs + row * yl + d) = o;
        } else {
          const int j = row - 16;
          if (d < K) {
            const float4 y = load4(Ylo + j * yl + d), p = load4(gam + r0 * gl + d), q = load4(gam + j * gl + d);
            o = make_float4(y.x * scan::exp_<FAST>(p.x - q.x), y.y * scan::exp_<FAST>(p.y - q.y),
                            y.z * scan::exp_<FAST>(p.z - q.z), y.w * scan::exp_<FAST>(p.w - q.w));
          }
          *reinterpret_cast<float4 *>(Ys + j * yl + d) = o;
        }
      }
    } else
    for (Walk2D wk(tid, 256, (int)Kp); wk.r < 16 + r0; wk.next()) {
      const int row = wk.r;
      const int64_t d = wk.c;
      if (row < 16) {  // Y_r e^{G_r - G_r0}, r in block a (zero past Lc)
        const int r = r0 + row;
        Xs[row * yl + d] = (d < K && r < Lc) ? Yup[r * yl + d] * scan::exp_<FAST>(gam[r * gl + d] - gam[r0 * gl + d]) : 0.f;
      } else {  // Y_j e^{G_r0 - G_j}, j < r0
        const int j = row - 16;
        Ys[j * yl + d] = d < K ? Ylo[j * yl + d] * scan::exp_<FAST>(gam[r0 * gl + d] - gam[j * gl + d]) : 0.f;
      }
    }
    __syncthreads();
    // lo rows r0 .. r0+15: M[r0.., :r0] Ys, scaled by e^{G_i - G_r0}
    for (int nt = warp; nt < nkt; nt += kWarps) {
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      tile_acc<false, false>(acc, M + r0 * lm, lm, Ys, yl, 0, 8 * nt, r0 / 8);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = r0 + gq + 8 * (e >> 1), d = 8 * nt + 2 * tq + (e & 1);
        if (d < K && i < Lc) lo[i * lw + d] += acc[e] * scan::exp_<FAST>(gam[i * gl + d] - gam[r0 * gl + d]);
      }
    }
    // up rows 0 .. r0-1: M[block a, :r0]^T Xs, scaled by e^{G_r0 - G_i}
    for (int tix = warp; tix < (r0 / 16) * nkt; tix += kWarps) {
      const int m0 = 16 * (tix % (r0 / 16)), n0 = 8 * (tix / (r0 / 16));
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      tile_acc<true, false>(acc, M + r0 * lm, lm, Xs, yl, m0, n0, 2);  // A(i, r) = M[r0 + r][i]
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = m0 + gq + 8 * (e >> 1), d = n0 + 2 * tq + (e & 1);
        if (d < K && i < Lc) up[i * lw + d] += acc[e] * scan::exp_<FAST>(gam[r0 * gl + d] - gam[i * gl + d]);
      }
    }
  }
  __syncthreads();
  }
}

}  // namespace prep
}  // namespace gdr
