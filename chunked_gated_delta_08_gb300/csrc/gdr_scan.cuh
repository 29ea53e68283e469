// gdr_scan.cuh -- one chunk of the state scan on a 32-column tile, with both
// of its products on warp-level tensor-core MMAs: 3 x TF32 (close to fp32)
// for fp32 inputs, one bf16 pass (m16n8k16, fp32 accumulation) for bf16.
//
// For the chunk starting at token t0 with Lc valid rows, h the K x 32 state
// tile entering it (shared memory), Gamma the gate cumsum and L the last
// valid row:
//   v_new = u - w h                    (C x 32)  = (C x K)(K x 32)
//   h    <- e^{G_L} h + Kb^T v_new      (K x 32)  = (K x C)(C x 32),  Kb = k e^{G_L - G}
// (the chunk form of the recurrence; the KCP handbook's h is the state
// entering the chunk).  Columns at or past `ucols` take u = 0 (the
// transition columns of the intra-sequence split).
//
// Shared-memory tiles, padded so every fragment load is free of bank
// conflicts (Kp = K rounded up to 16):
//   hs [Kp][kHS]   state tile          ws [C][Kp + 4]  -w
//   kt [C][Kp + 8] Kb                  vn [C][kHS]     v_new
//   gl [Kp]        G_L per key row
//
// Pages cited: the KCP handbook = "flash-linear-attention KCP 精度失效根因排查手册".
#pragma once

#include <type_traits>

#include "gdr_device.cuh"
#include "gdr_sm100.cuh"

namespace gdr {
namespace scan {

constexpr int kCols = 32;      // columns of the state tile
constexpr int kHS = kCols + 8; // row stride of hs and vn (== 8 mod 32)
constexpr int kScanThreads = 256;

__host__ __device__ constexpr int64_t kpad(int64_t K) { return (K + 15) / 16 * 16; }
__host__ __device__ constexpr int64_t ws_ld(int64_t K) { return kpad(K) + 4; }
__host__ __device__ constexpr int64_t kt_ld(int64_t K) { return kpad(K) + 8; }

// floats of shared memory the tiles need
__host__ __device__ constexpr int64_t smem_floats(int C, int64_t K) {
  return kpad(K) * kHS + C * ws_ld(K) + C * kt_ld(K) + C * kHS + kpad(K);
}

struct Tiles {
  float *hs, *ws, *kt, *vn, *gl;
};

__device__ __forceinline__ Tiles carve(float *smem, int C, int64_t K) {
  Tiles t;
  t.hs = smem;
  t.ws = t.hs + kpad(K) * kHS;
  t.kt = t.ws + C * ws_ld(K);
  t.vn = t.kt + C * kt_ld(K);
  t.gl = t.vn + C * kHS;
  return t;
}

__device__ __forceinline__ void split3(float x, uint32_t &hi, uint32_t &lo) { sm100::split_tf32(x, hi, lo); }

// d += A B with A, B split into (hi, lo); the lo * lo term is dropped.
__device__ __forceinline__ void mma3(float (&d)[4], const uint32_t (&ah)[4], const uint32_t (&al)[4],
                                     const uint32_t (&bh)[2], const uint32_t (&bl)[2]) {
  sm100::mma_tf32(d, al[0], al[1], al[2], al[3], bh[0], bh[1]);
  sm100::mma_tf32(d, ah[0], ah[1], ah[2], ah[3], bl[0], bl[1]);
  sm100::mma_tf32(d, ah[0], ah[1], ah[2], ah[3], bh[0], bh[1]);
}

// mma.sync m16n8k16 with bf16 inputs and fp32 accumulation (one pass), for
// products whose operands the bf16 path takes in bf16 anyway (as the fused form
// does).  Each 32-bit register holds two bf16, the lower half the smaller K
// index.  Fragments (g = lane / 4, t = lane % 4): A (16x16) a0 (g, 2t..2t+1)
// a1 (g+8, 2t..) a2 (g, 2t+8..) a3 (g+8, 2t+8..); B (16x8, K x N) b0 (2t..2t+1, g)
// b1 (2t+8.., g); D as for m16n8k8.
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// two fp32 values rounded to a bf16 pair, x0 in the lower half
__device__ __forceinline__ uint32_t bf16x2(float x0, float x1) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(x0, x1);
  return *reinterpret_cast<const uint32_t *>(&v);
}
// e^x: the fast hardware exponential on the bf16 path, the full-precision one otherwise
template <bool FAST>
__device__ __forceinline__ float exp_(float x) {
  return FAST ? __expf(x) : expf(x);
}

// bf16 inputs take the single-pass bf16 products and the fast exponential
template <typename Tin>
constexpr bool kB16 = std::is_same<Tin, __nv_bfloat16>::value;

// Asks L2 for `rows` rows of `row_bytes` bytes, `stride` bytes apart, from p
// (global memory), one 128-byte line per request, spread over the block's
// 256 threads: a sequential scan issues it for the next chunk so that chunk's
// row loads find their lines (and address translations) in L2.
__device__ __forceinline__ void prefetch_rows_l2(const void *p, int64_t stride, int rows, int row_bytes) {
  const int lines = (row_bytes + 127) >> 7;
  for (int e = threadIdx.x; e < rows * lines; e += kScanThreads) {
    const int r = e / lines, l = e - r * lines;
    const char *a = static_cast<const char *>(p) + (int64_t)r * stride + 128 * l;
    asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
  }
}

// Kb rows (L2-normalized k times e^{G_L - G}) into kt and -w into ws, for the
// chunk's rows, zero past Lc and past K.  Warp w takes rows w, w + 8, ...; the
// loads of RB rows (KV values per lane and row) are all issued before any row
// is reduced, so a warp waits on memory once per RB rows.
template <typename Tin, int C, bool PER_K, int KV, int RB>
__device__ __forceinline__ void load_rows(const Tiles &s, const Tin *__restrict__ k, const float *__restrict__ w,
                                          const float *__restrict__ gcum, int64_t t0, int Lc, int64_t hv,
                                          int64_t hq, int64_t H, int64_t HV, int64_t K, int l2) {
  constexpr int kWarps = kScanThreads / 32;
  constexpr int RPW = C / kWarps;  // rows per warp
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t Kp = kpad(K), WL = ws_ld(K), KL = kt_ld(K);
  const int64_t gw = PER_K ? K : 1;
#pragma unroll
  for (int jb = 0; jb < RPW; jb += RB) {
    float kv[RB][KV], gv[RB][KV], wv[RB][KV];
#pragma unroll
    for (int r = 0; r < RB; ++r) {
      const int i = warp + kWarps * (jb + r);
      const bool rok = jb + r < RPW && i < Lc;
      const int64_t tok = t0 + i;
#pragma unroll
      for (int m = 0; m < KV; ++m) {
        const int64_t d = lane + 32 * m;
        const bool ok = rok && d < K;
        kv[r][m] = ok ? to_f32(k[(tok * H + hq) * K + d]) : 0.f;
        gv[r][m] = ok ? gcum[(tok * HV + hv) * gw + (PER_K ? d : 0)] : 0.f;
        wv[r][m] = ok ? w[(tok * HV + hv) * K + d] : 0.f;
      }
    }
#pragma unroll
    for (int r = 0; r < RB; ++r) {
      if (jb + r >= RPW) break;
      const int i = warp + kWarps * (jb + r);
      const bool rok = i < Lc;
      float ss = 0.f;
#pragma unroll
      for (int m = 0; m < KV; ++m) ss = fmaf(kv[r][m], kv[r][m], ss);
      const float sc = l2 ? rsqrtf(warp_sum(ss) + kL2Eps) : 1.f;
#pragma unroll
      for (int m = 0; m < KV; ++m) {
        const int64_t d = lane + 32 * m;
        if (d < Kp) {
          const bool ok = rok && d < K;
          s.kt[i * KL + d] = ok ? kv[r][m] * sc * exp_<kB16<Tin>>(s.gl[d] - gv[r][m]) : 0.f;
          s.ws[i * WL + d] = ok ? -wv[r][m] : 0.f;
        }
      }
    }
  }
}

// The same rows with vector loads, for K % 4 == 0, K <= 128 and 16-byte
// aligned k, w and gcum: lane l takes the four keys 4l .. 4l + 3 of a row (one
// load per row and tensor instead of four), four rows per warp in flight.
// It also loads G_L itself (it does not read s.gl) and writes s.gl, visible to
// the block after the caller's next barrier.
template <typename Tin, int C, bool PER_K>
__device__ __forceinline__ void load_rows_vec(const Tiles &s, const Tin *__restrict__ k, const float *__restrict__ w,
                                              const float *__restrict__ gcum, int64_t t0, int Lc, int64_t hv,
                                              int64_t hq, int64_t H, int64_t HV, int64_t K, int l2) {
  constexpr int kWarps = kScanThreads / 32;
  constexpr int RPW = C / kWarps, RB = 4;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t Kp = kpad(K), WL = ws_ld(K), KL = kt_ld(K);
  const int d0 = 4 * lane;
  const bool lane_in = d0 < K;
  // G at the chunk's last valid row, for this lane's keys (warp 0 also publishes it in s.gl)
  float4 gl = make_float4(0.f, 0.f, 0.f, 0.f);
  {
    const int64_t tl = t0 + Lc - 1;
    if (PER_K) {
      if (lane_in) gl = *reinterpret_cast<const float4 *>(gcum + (tl * HV + hv) * K + d0);
    } else {
      const float x = gcum[tl * HV + hv];
      gl = make_float4(x, x, x, x);
    }
    if (warp == 0 && d0 < Kp) *reinterpret_cast<float4 *>(s.gl + d0) = lane_in ? gl : make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int jb = 0; jb < RPW; jb += RB) {
    float kv[RB][4], gv[RB][4], wv[RB][4];
#pragma unroll
    for (int r = 0; r < RB; ++r) {
      const int i = warp + kWarps * (jb + r);
      const bool ok = lane_in && i < Lc;
      const int64_t tok = t0 + i;
#pragma unroll
      for (int m = 0; m < 4; ++m) kv[r][m] = gv[r][m] = wv[r][m] = 0.f;
      if (ok) {
        if constexpr (kB16<Tin>) {
          const uint2 kk = *reinterpret_cast<const uint2 *>(k + (tok * H + hq) * K + d0);
          const float2 k01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&kk.x));
          const float2 k23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&kk.y));
          kv[r][0] = k01.x;
          kv[r][1] = k01.y;
          kv[r][2] = k23.x;
          kv[r][3] = k23.y;
        } else {
          const float4 kk = *reinterpret_cast<const float4 *>(k + (tok * H + hq) * K + d0);
          kv[r][0] = kk.x;
          kv[r][1] = kk.y;
          kv[r][2] = kk.z;
          kv[r][3] = kk.w;
        }
        const float4 ww = *reinterpret_cast<const float4 *>(w + (tok * HV + hv) * K + d0);
        wv[r][0] = ww.x;
        wv[r][1] = ww.y;
        wv[r][2] = ww.z;
        wv[r][3] = ww.w;
        if constexpr (PER_K) {
          const float4 gg = *reinterpret_cast<const float4 *>(gcum + (tok * HV + hv) * K + d0);
          gv[r][0] = gg.x;
          gv[r][1] = gg.y;
          gv[r][2] = gg.z;
          gv[r][3] = gg.w;
        } else {
          gv[r][0] = gv[r][1] = gv[r][2] = gv[r][3] = gcum[tok * HV + hv];
        }
      }
    }
#pragma unroll
    for (int r = 0; r < RB; ++r) {
      if (jb + r >= RPW) break;
      const int i = warp + kWarps * (jb + r);
      float ss = 0.f;
#pragma unroll
      for (int m = 0; m < 4; ++m) ss = fmaf(kv[r][m], kv[r][m], ss);
      const float sc = l2 ? rsqrtf(warp_sum(ss) + kL2Eps) : 1.f;
      if (d0 < Kp) {
        const bool ok = lane_in && i < Lc;
        float4 kb = make_float4(0.f, 0.f, 0.f, 0.f), nw = kb;
        if (ok) {
          kb = make_float4(kv[r][0] * sc * exp_<kB16<Tin>>(gl.x - gv[r][0]), kv[r][1] * sc * exp_<kB16<Tin>>(gl.y - gv[r][1]),
                           kv[r][2] * sc * exp_<kB16<Tin>>(gl.z - gv[r][2]), kv[r][3] * sc * exp_<kB16<Tin>>(gl.w - gv[r][3]));
          nw = make_float4(-wv[r][0], -wv[r][1], -wv[r][2], -wv[r][3]);
        }
        *reinterpret_cast<float4 *>(s.kt + i * KL + d0) = kb;
        *reinterpret_cast<float4 *>(s.ws + i * WL + d0) = nw;
      }
    }
  }
}

// Kb rows already formed (k e^{G_L - G}, by prepare) and -w, for K % 4 == 0,
// K <= 128 and 16-byte aligned rows: lane l takes keys 4l .. 4l + 3, four rows
// per warp in flight.  Writes G_L per key into s.gl, visible to the block
// after the caller's next barrier.
template <int C, bool PER_K>
__device__ __forceinline__ void load_rows_formed(const Tiles &s, const float *__restrict__ kb,
                                                 const float *__restrict__ w, const float *__restrict__ gcum,
                                                 int64_t t0, int Lc, int64_t hv, int64_t HV, int64_t K) {
  constexpr int kWarps = kScanThreads / 32;
  constexpr int RPW = C / kWarps, RB = 4;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t Kp = kpad(K), WL = ws_ld(K), KL = kt_ld(K);
  const int d0 = 4 * lane;
  const bool lane_in = d0 < K;
  if (warp == 0 && d0 < Kp) {
    const int64_t tl = t0 + Lc - 1;
    float4 gl = make_float4(0.f, 0.f, 0.f, 0.f);
    if (lane_in) {
      if (PER_K) {
        gl = *reinterpret_cast<const float4 *>(gcum + (tl * HV + hv) * K + d0);
      } else {
        const float x = gcum[tl * HV + hv];
        gl = make_float4(x, x, x, x);
      }
    }
    *reinterpret_cast<float4 *>(s.gl + d0) = gl;
  }
#pragma unroll
  for (int jb = 0; jb < RPW; jb += RB) {
    float4 kv[RB], wv[RB];
#pragma unroll
    for (int r = 0; r < RB; ++r) {
      const int i = warp + kWarps * (jb + r);
      const bool ok = lane_in && i < Lc;
      const int64_t off = ((t0 + i) * HV + hv) * K + d0;
      kv[r] = ok ? *reinterpret_cast<const float4 *>(kb + off) : make_float4(0.f, 0.f, 0.f, 0.f);
      wv[r] = ok ? *reinterpret_cast<const float4 *>(w + off) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int r = 0; r < RB; ++r) {
      if (jb + r >= RPW) break;
      const int i = warp + kWarps * (jb + r);
      if (d0 < Kp) {
        *reinterpret_cast<float4 *>(s.kt + i * KL + d0) = kv[r];
        *reinterpret_cast<float4 *>(s.ws + i * WL + d0) = make_float4(-wv[r].x, -wv[r].y, -wv[r].z, -wv[r].w);
      }
    }
  }
}

// The row loader for the shape: vector loads where K % 4 == 0, K <= 128 and
// k, w, gcum are 16-byte aligned (every row then starts on a 16-byte, bf16 k
// an 8-byte, boundary), else the scalar loaders.
template <typename Tin>
__device__ __forceinline__ bool rows_vec_ok(const Tin *k, const float *w, const float *gcum, int64_t K) {
  return K <= 128 && K % 4 == 0 &&
         ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(w) | reinterpret_cast<uintptr_t>(gcum)) & 15u) == 0;
}
template <typename Tin, int C, bool PER_K>
__device__ __forceinline__ void load_rows_auto(const Tiles &s, const Tin *__restrict__ k, const float *__restrict__ w,
                                               const float *__restrict__ gcum, int64_t t0, int Lc, int64_t hv,
                                               int64_t hq, int64_t H, int64_t HV, int64_t K, int l2) {
  if (rows_vec_ok(k, w, gcum, K)) load_rows_vec<Tin, C, PER_K>(s, k, w, gcum, t0, Lc, hv, hq, H, HV, K, l2);
  else if (K <= 128) load_rows<Tin, C, PER_K, 4, 4>(s, k, w, gcum, t0, Lc, hv, hq, H, HV, K, l2);
  else load_rows<Tin, C, PER_K, 8, 2>(s, k, w, gcum, t0, Lc, hv, hq, H, HV, K, l2);
}

// One chunk.  Called by all 256 threads of the block; hs holds the entering
// tile and holds the leaving one on return.  v_new_out (nullable) receives
// v_new for rows < Lc and columns < ucols.  c0col is the tile's first column
// in the scanned matrix.
template <typename Tin, int C, bool PER_K>
__device__ __forceinline__ void chunk_step(const Tiles &s, const Tin *__restrict__ k, const float *__restrict__ w,
                                           const float *__restrict__ u, const float *__restrict__ gcum,
                                           int64_t t0, int Lc, int64_t hv, int64_t hq, int64_t H, int64_t HV,
                                           int64_t K, int64_t V, int64_t ucols, int64_t c0col, int l2,
                                           float *__restrict__ v_new_out, const float *__restrict__ kb_rows = nullptr) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, tq = lane & 3;
  const int64_t Kp = kpad(K), WL = ws_ld(K), KL = kt_ld(K);
  const int64_t gw = PER_K ? K : 1;
  const int64_t tl = t0 + Lc - 1;
  constexpr int kWarps = kScanThreads / 32;
  // u (the start of v_new) for this warp's tile, loaded first so its round trip overlaps the rows'
  const int m0v = 16 * (warp % (C / 16)), n0v = 16 * (warp / (C / 16));
  float acc[2][4];
  if (warp < 2 * (C / 16)) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = m0v + g + 8 * (e >> 1);
        const int64_t col = c0col + n0v + 8 * nt + 2 * tq + (e & 1);
        acc[nt][e] = (i < Lc && col < ucols) ? u[((t0 + i) * HV + hv) * V + col] : 0.f;
      }
  }
  // Kb and -w, zero past Lc and past K; G_L per key into s.gl
  if (kb_rows && rows_vec_ok(kb_rows, w, gcum, K)) {
    load_rows_formed<C, PER_K>(s, kb_rows, w, gcum, t0, Lc, hv, HV, K);
  } else if (rows_vec_ok(k, w, gcum, K)) {
    load_rows_vec<Tin, C, PER_K>(s, k, w, gcum, t0, Lc, hv, hq, H, HV, K, l2);
  } else {
    for (int64_t d = tid; d < Kp; d += kScanThreads)
      s.gl[d] = d < K ? gcum[(tl * HV + hv) * gw + (PER_K ? d : 0)] : 0.f;
    __syncthreads();
    if (K <= 128) load_rows<Tin, C, PER_K, 4, 4>(s, k, w, gcum, t0, Lc, hv, hq, H, HV, K, l2);
    else load_rows<Tin, C, PER_K, 8, 2>(s, k, w, gcum, t0, Lc, hv, hq, H, HV, K, l2);
  }
  __syncthreads();

  // ---- v_new = u - w h: C x 32, warp -> rows 16 (warp & 3) .., columns 16 (warp >> 2) ..
  if (warp < 2 * (C / 16)) {
    const int m0 = m0v, n0 = n0v;
    if constexpr (kB16<Tin>) {
      for (int64_t k0 = 0; k0 < Kp; k0 += 16) {
        const float *a = s.ws + (m0 + g) * WL + k0 + 2 * tq;
        const float2 x0 = *reinterpret_cast<const float2 *>(a), x1 = *reinterpret_cast<const float2 *>(a + 8 * WL),
                     x2 = *reinterpret_cast<const float2 *>(a + 8),
                     x3 = *reinterpret_cast<const float2 *>(a + 8 * WL + 8);
        const uint32_t a0 = bf16x2(x0.x, x0.y), a1 = bf16x2(x1.x, x1.y), a2 = bf16x2(x2.x, x2.y),
                       a3 = bf16x2(x3.x, x3.y);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const float *b = s.hs + (k0 + 2 * tq) * kHS + n0 + 8 * nt + g;
          mma_bf16(acc[nt], a0, a1, a2, a3, bf16x2(b[0], b[kHS]), bf16x2(b[8 * kHS], b[9 * kHS]));
        }
      }
    } else {
      for (int64_t k0 = 0; k0 < Kp; k0 += 8) {
        uint32_t ah[4], al[4];
        const float *a = s.ws + (m0 + g) * WL + k0 + tq;
        split3(a[0], ah[0], al[0]);
        split3(a[8 * WL], ah[1], al[1]);
        split3(a[4], ah[2], al[2]);
        split3(a[8 * WL + 4], ah[3], al[3]);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const float *b = s.hs + (k0 + tq) * kHS + n0 + 8 * nt + g;
          uint32_t bh[2], bl[2];
          split3(b[0], bh[0], bl[0]);
          split3(b[4 * kHS], bh[1], bl[1]);
          mma3(acc[nt], ah, al, bh, bl);
        }
      }
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = m0 + g + 8 * (e >> 1);
        const int cc = n0 + 8 * nt + 2 * tq + (e & 1);
        s.vn[i * kHS + cc] = acc[nt][e];  // zero past Lc (w, u are zero there)
        const int64_t col = c0col + cc;
        if (v_new_out && i < Lc && col < ucols) v_new_out[((t0 + i) * HV + hv) * V + col] = acc[nt][e];
      }
  }
  __syncthreads();

  // ---- h <- e^{G_L} h + Kb^T v_new: Kp x 32, warp -> row tiles warp, warp + 8, ..., all 4 column tiles
  for (int64_t m0 = 16 * warp; m0 < Kp; m0 += 16 * kWarps) {
    float acc[4][4];
    const float e0 = exp_<kB16<Tin>>(s.gl[PER_K ? m0 + g : 0]), e1 = exp_<kB16<Tin>>(s.gl[PER_K ? m0 + g + 8 : 0]);
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int64_t d = m0 + g + 8 * (e >> 1);
        acc[nt][e] = s.hs[d * kHS + 8 * nt + 2 * tq + (e & 1)] * ((e >> 1) ? e1 : e0);
      }
    if constexpr (kB16<Tin>) {
#pragma unroll
      for (int k0 = 0; k0 < C; k0 += 16) {
        const float *a = s.kt + (k0 + 2 * tq) * KL + m0 + g;  // A(d, i) = Kb[i][d]
        const uint32_t a0 = bf16x2(a[0], a[KL]), a1 = bf16x2(a[8], a[KL + 8]), a2 = bf16x2(a[8 * KL], a[9 * KL]),
                       a3 = bf16x2(a[8 * KL + 8], a[9 * KL + 8]);
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
          const float *b = s.vn + (k0 + 2 * tq) * kHS + 8 * nt + g;
          mma_bf16(acc[nt], a0, a1, a2, a3, bf16x2(b[0], b[kHS]), bf16x2(b[8 * kHS], b[9 * kHS]));
        }
      }
    } else {
#pragma unroll
      for (int k0 = 0; k0 < C; k0 += 8) {
        uint32_t ah[4], al[4];
        const float *a = s.kt + (k0 + tq) * KL + m0 + g;  // A(d, i) = Kb[i][d]
        split3(a[0], ah[0], al[0]);
        split3(a[8], ah[1], al[1]);
        split3(a[4 * KL], ah[2], al[2]);
        split3(a[4 * KL + 8], ah[3], al[3]);
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
          const float *b = s.vn + (k0 + tq) * kHS + 8 * nt + g;
          uint32_t bh[2], bl[2];
          split3(b[0], bh[0], bl[0]);
          split3(b[4 * kHS], bh[1], bl[1]);
          mma3(acc[nt], ah, al, bh, bl);
        }
      }
    }
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int64_t d = m0 + g + 8 * (e >> 1);
        s.hs[d * kHS + 8 * nt + 2 * tq + (e & 1)] = acc[nt][e];
      }
  }
  __syncthreads();
}

}  // namespace scan
}  // namespace gdr
