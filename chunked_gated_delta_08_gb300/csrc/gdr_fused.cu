// gdr_fused.cu -- the fused single-pass forward on the sm_103a tensor cores.
//
// One block per (sequence, value head) walks the sequence chunk by chunk with
// the K x V state on chip: it reads q, k, v, g, beta once and writes o and the
// final state once, so nothing of the chunk form (A, T, w, u, h, v_new) goes
// to HBM.  Per chunk of C = 64 tokens, with Gamma the within-chunk cumsum of
// g, r the in-kernel L2-norm scales, L the number of valid rows and h the
// state entering the chunk (the handbook's chunk-start state):
//
//   S     = [K; Q] K^T                               tcgen05, M=128 N=64 K=128
//   A_ij  = beta_i r_i r_j e^{G_i - G_j} (KK^T)_ij, i > j      (CUDA cores)
//   P_rj  = rq_r r_j e^{G_r - G_j} (QK^T)_rj, j <= r           (CUDA cores)
//   T     = (I + A)^-1   blocked 16 x 16 inversion, fp32      (CUDA cores)
//   W'    = T diag(beta e^G r),  U' = T diag(beta)            (bf16 operands)
//   w^T   = K^T W'^T                                  tcgen05, M=128 N=64 K=64
//   vn^T  = V^T U'^T - h^T w^T                        tcgen05 (negated A)
//   o1^T  = h^T Q^T,  o2^T = vn^T P^T                 tcgen05
//   dH    = K^T (vn * r e^{G_L - G})                  tcgen05, M=128 N=128 K=64
//   h'    = e^{G_L} h + dH                            fp32 registers
//   o_r   = rq_r e^{G_r} o1_r + o2_r
//
// Every matrix product has M = 128 (the K or V dimension), so the accumulator
// row is the TMEM lane and each thread of the compute warpgroup owns one lane.
// Tiles arrive by TMA in the 128-byte swizzled layout and are read by the
// tensor cores both K-major and MN-major without any copy.  Every mbarrier
// wait is time-bounded; on expiry the block records GDR_ERR_TIMEOUT in the
// status word, lets its copies in flight land, frees its tensor memory and
// returns.
//
// Supported here: bf16, scalar gate, K = V = 128, C = 64, dense or varlen.
// Other requests return GDR_ERR_UNSUPPORTED so the dispatcher can take the
// chunked form.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <mutex>

#include "gdr_device.cuh"
#include "gdr_internal.h"
#include "gdr_sm100.cuh"

namespace gdr {
namespace {

using namespace sm100;

constexpr int C = 64;
constexpr int DK = 128;
constexpr int DV = 128;
constexpr int kStages = 2;
constexpr int kWG = 128;             // compute warpgroup: warps 0-3, thread t owns TMEM lane t
constexpr int kThreads = kWG + 32;   // + one producer warp
constexpr int kBarWG = 1;            // named barrier of the compute warpgroup
constexpr int LDA = C + 1;           // padded row stride of the fp32 A / T matrices

// shared memory map (offsets from a 1024-byte aligned base)
constexpr uint32_t SZ_QK = 32768;    // [K d0-63 | Q d0-63 | K d64-127 | Q d64-127], each 64 rows x 128 B
constexpr uint32_t SZ_V = 16384;     // [V v0-63 | V v64-127]
constexpr uint32_t STAGE_BYTES = SZ_QK + SZ_V;
constexpr uint32_t OFF_H = kStages * STAGE_BYTES;   // h [d][v] bf16: 2 sub-tiles of 128 rows x 128 B
constexpr uint32_t OFF_WU = OFF_H + 32768;          // W' 8K | U' 8K, later w [i][d] (2 x 8K)
constexpr uint32_t OFF_P = OFF_WU + 16384;          // P [r][j] bf16
constexpr uint32_t OFF_X = OFF_P + 8192;            // A, T fp32 (2 x 64 x 65), later vn^T | vt^T
constexpr uint32_t OFF_VN = OFF_X;                  // vn^T [v][i] bf16 (16K)
constexpr uint32_t OFF_VT = OFF_X + 16384;          // vt^T [v][i] bf16 (16K)
constexpr uint32_t SZ_X = 2 * C * LDA * 4 > 32768 ? 2 * C * LDA * 4 : 32768;
constexpr uint32_t OFF_SMALL = (OFF_X + SZ_X + 1023) & ~1023u;

// TMEM columns
constexpr uint32_t TM_S = 0, TM_W = 64, TM_VN = 128, TM_O1 = 192, TM_O2 = 256, TM_H = 320, TM_COLS = 512;

struct Small {
  float g[kStages][C];
  float beta[kStages][C];
  float gam[C];
  float rq[C], rk[C];
  float sv[C];   // row scale of vt: rk_i e^{G_L - G_i} (0 past the chunk end)
  float so[C];   // row scale of the inter-chunk output: rq_r e^{G_r}
  float X[3 * 256];
  uint64_t full[kStages], empty[kStages], mma;
  uint32_t tmem_slot;
  int err;
  int bad;
};

constexpr uint32_t SMEM_BYTES = OFF_SMALL + sizeof(Small) + 1024;

struct FusedParams {
  const __nv_bfloat16 *beta;
  const float *g, *h0;
  const int64_t *cu;
  __nv_bfloat16 *o;
  float *ht;
  int *status;
  int64_t T, N, H, HV;
  int l2;
  unsigned long long timeout_ns;
};

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t *>(&v);
}

// Writes 8 consecutive bf16 (packed in a uint4) as chunk `chunk` of row `row`
// of a 128-byte swizzled tile.
__device__ __forceinline__ void st_sw128_chunk(uint8_t *tile, uint32_t row, uint32_t chunk, uint4 val) {
  const uint32_t off = (row >> 3) * 1024u + (row & 7u) * 128u + ((chunk ^ (row & 7u)) << 4);
  *reinterpret_cast<uint4 *>(tile + off) = val;
}
__device__ __forceinline__ uint4 ld_sw128_chunk(const uint8_t *tile, uint32_t row, uint32_t chunk) {
  const uint32_t off = (row >> 3) * 1024u + (row & 7u) * 128u + ((chunk ^ (row & 7u)) << 4);
  return *reinterpret_cast<const uint4 *>(tile + off);
}

__device__ __forceinline__ float sumsq_bf16x8(uint4 u) {
  const __nv_bfloat162 *p = reinterpret_cast<const __nv_bfloat162 *>(&u);
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 f = __bfloat1622float2(p[i]);
    s = fmaf(f.x, f.x, s);
    s = fmaf(f.y, f.y, s);
  }
  return s;
}

// T = (I + A)^-1 for a unit lower-triangular 64 x 64 system (A strictly lower),
// by 16 x 16 diagonal-block inversion and block forward substitution:
// T_bj = -T_bb sum_{l=j}^{b-1} A_bl T_lj.  All 128 threads of the warpgroup.
__device__ void solve_unit_lower(const float *A, float *T, float *X, int tid) {
  for (int e = tid; e < C * LDA; e += kWG) T[e] = 0.f;
  named_bar(kBarWG, kWG);
  if (tid < 64) {
    const int b = tid >> 4, c = tid & 15, base = 16 * b;
    float x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float acc = (i == c) ? 1.f : 0.f;
#pragma unroll
      for (int l = 0; l < i; ++l) acc = fmaf(-A[(base + i) * LDA + base + l], x[l], acc);
      x[i] = (i < c) ? 0.f : acc;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) T[(base + i) * LDA + base + c] = x[i];
  }
  named_bar(kBarWG, kWG);
  for (int d = 1; d <= 3; ++d) {
    const int nb = 4 - d;
    for (int o = tid; o < nb * 256; o += kWG) {
      const int bi = o >> 8, b = d + bi, j0 = b - d, i = (o >> 4) & 15, j = o & 15;
      float acc = 0.f;
      for (int l = j0; l < b; ++l) {
#pragma unroll
        for (int m = 0; m < 16; ++m) acc = fmaf(A[(16 * b + i) * LDA + 16 * l + m], T[(16 * l + m) * LDA + 16 * j0 + j], acc);
      }
      X[bi * 256 + i * 16 + j] = acc;
    }
    named_bar(kBarWG, kWG);
    for (int o = tid; o < nb * 256; o += kWG) {
      const int bi = o >> 8, b = d + bi, j0 = b - d, i = (o >> 4) & 15, j = o & 15;
      float acc = 0.f;
#pragma unroll
      for (int m = 0; m < 16; ++m) acc = fmaf(T[(16 * b + i) * LDA + 16 * b + m], X[bi * 256 + m * 16 + j], acc);
      T[(16 * b + i) * LDA + 16 * j0 + j] = -acc;
    }
    named_bar(kBarWG, kWG);
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    gdr_fused_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const FusedParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Small &S = *reinterpret_cast<Small *>(sm + OFF_SMALL);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t unit = blockIdx.x;
  const int64_t n = unit / p.HV, hv = unit % p.HV, hq = hv / (p.HV / p.H);

  // ---- sequence range; every block checks the whole cu_seqlens
  if (tid == 0) {
    S.bad = 0;
    S.err = 0;
  }
  __syncthreads();
  int64_t bos, eos;
  if (p.cu) {
    for (int64_t i = tid; i < p.N; i += kThreads)
      if (p.cu[i + 1] < p.cu[i]) S.bad = 1;
    if (tid == 0 && (p.cu[0] != 0 || p.cu[p.N] != p.T)) S.bad = 1;
    bos = p.cu[n];
    eos = p.cu[n + 1];
  } else {
    bos = n * p.T;
    eos = bos + p.T;
  }
  __syncthreads();
  if (S.bad) {
    if (tid == 0) raise_status(p.status, GDR_ERR_SEQLENS);
    return;
  }
  const int nch = (int)((eos - bos + C - 1) / C);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&S.full[s]), 2);
      mbar_init(smem_u32(&S.empty[s]), 1);
    }
    mbar_init(smem_u32(&S.mma), 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&S.tmem_slot), TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = S.tmem_slot;
  volatile int *err = &S.err;

  if (warp == kWG / 32) {
    // ================================================================ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
    }
    int issued = 0;
    for (int c = 0; c < nch; ++c) {
      const int s = c % kStages, u = c / kStages;
      if (c >= kStages) {
        const bool ok = mbar_wait(smem_u32(&S.empty[s]), (u - 1) & 1, err, p.timeout_ns);
        if (!__all_sync(0xffffffffu, ok)) break;
      }
      const int64_t t0 = bos + (int64_t)c * C;
      const int L = (int)(eos - t0 < C ? eos - t0 : C);
      uint8_t *qk = sm + s * STAGE_BYTES, *vv = qk + SZ_QK;
      if (lane == 0) {
        const uint32_t fb = smem_u32(&S.full[s]);
        mbar_arrive_expect_tx(fb, STAGE_BYTES);
        const int tt = (int)t0;
        tma_load_3d(smem_u32(qk), &tm_k, 0, (int)hq, tt, fb);
        tma_load_3d(smem_u32(qk + 8192), &tm_q, 0, (int)hq, tt, fb);
        tma_load_3d(smem_u32(qk + 16384), &tm_k, 64, (int)hq, tt, fb);
        tma_load_3d(smem_u32(qk + 24576), &tm_q, 64, (int)hq, tt, fb);
        tma_load_3d(smem_u32(vv), &tm_v, 0, (int)hv, tt, fb);
        tma_load_3d(smem_u32(vv + 8192), &tm_v, 64, (int)hv, tt, fb);
      }
      for (int i = lane; i < C; i += 32) {
        S.g[s][i] = i < L ? p.g[(t0 + i) * p.HV + hv] : 0.f;
        S.beta[s][i] = i < L ? __bfloat162float(p.beta[(t0 + i) * p.HV + hv]) : 0.f;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&S.full[s]));
      issued = c + 1;
    }
    // let every copy issued land before the block can exit
    if (lane == 0)
      for (int c = (issued > kStages ? issued - kStages : 0); c < issued; ++c)
        mbar_wait_drain(smem_u32(&S.full[c % kStages]), (c / kStages) & 1, p.timeout_ns);
  } else {
    // ================================================================ compute warpgroup
    const uint32_t lane_addr = tbase + ((uint32_t)(warp * 32) << 16);
    uint8_t *sH = sm + OFF_H, *sWU = sm + OFF_WU, *sP = sm + OFF_P, *sVN = sm + OFF_VN, *sVT = sm + OFF_VT;
    float *sA = reinterpret_cast<float *>(sm + OFF_X);
    float *sT = sA + C * LDA;
    uint32_t mma_phase = 0;

    // state row d = tid in fp32 registers; its bf16 copy in sH (MN-major A operand of h^T)
    float h[DV];
    {
      const float *src = p.h0 ? p.h0 + (unit * DK + tid) * DV : nullptr;
#pragma unroll
      for (int v = 0; v < DV; ++v) h[v] = src ? src[v] : 0.f;
#pragma unroll
      for (int ch = 0; ch < 16; ++ch) {
        uint4 val = make_uint4(pack_bf16(h[8 * ch], h[8 * ch + 1]), pack_bf16(h[8 * ch + 2], h[8 * ch + 3]),
                               pack_bf16(h[8 * ch + 4], h[8 * ch + 5]), pack_bf16(h[8 * ch + 6], h[8 * ch + 7]));
        st_sw128_chunk(sH + (ch >> 3) * 16384, tid, ch & 7, val);
      }
    }
    fence_proxy_async_smem();
    named_bar(kBarWG, kWG);

    // every wait ends in a warpgroup-wide vote, so all 128 threads stop together
    auto wg_wait = [&](uint64_t *bar, uint32_t parity) -> bool {
      const bool ok = mbar_wait(smem_u32(bar), parity, err, p.timeout_ns);
      return named_bar_and(kBarWG, kWG, ok);
    };
    auto wait_mma = [&]() -> bool {
      const bool ok = wg_wait(&S.mma, mma_phase & 1);
      ++mma_phase;
      tc_fence_after();
      return ok;
    };

    for (int c = 0; c < nch; ++c) {
      const int s = c % kStages, u = c / kStages;
      const int64_t t0 = bos + (int64_t)c * C;
      const int L = (int)(eos - t0 < C ? eos - t0 : C);
      if (!wg_wait(&S.full[s], u & 1)) break;
      uint8_t *qk = sm + s * STAGE_BYTES, *vv = qk + SZ_QK;
      const uint32_t aQK = smem_u32(qk), aV = smem_u32(vv);

      // ragged tail: clear rows past the sequence end (they may hold the next sequence)
      if (L < C) {
        for (int e = tid; e < (C - L) * 6 * 8; e += kWG) {
          const int rr = L + e / 48, rest = e % 48, tile = rest / 8, ch = rest % 8;
          uint8_t *base = tile < 4 ? qk + tile * 8192 : vv + (tile - 4) * 8192;
          st_sw128_chunk(base, rr, ch, make_uint4(0, 0, 0, 0));
        }
        fence_proxy_async_smem();
        named_bar(kBarWG, kWG);
      }

      // ---- (1) S = [K; Q] K^T
      if (tid == 0) {
        tc_fence_after();
        constexpr uint32_t id = idesc_bf16(128, 64, 0, 0);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
          mma_bf16(tbase + TM_S, smem_desc(aQK + off, 16, 1024), smem_desc(aQK + off, 16, 1024), id, ks > 0);
        }
        mma_commit(smem_u32(&S.mma));
      }
      // row norms (q rows on threads 0-63, k rows on 64-127) and the gate cumsum
      {
        const int row = tid & 63;
        const uint8_t *t0p = qk + (tid < 64 ? 8192 : 0);
        float ss = 0.f;
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          ss += sumsq_bf16x8(ld_sw128_chunk(t0p, row, ch));
          ss += sumsq_bf16x8(ld_sw128_chunk(t0p + 16384, row, ch));
        }
        const float r = p.l2 ? rsqrtf(ss + kL2Eps) : 1.f;
        if (tid < 64) S.rq[row] = r;
        else S.rk[row] = r;
        if (tid < 64) {
          float x = S.g[s][tid];
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
          }
          S.gam[tid] = x;  // warp 1 adds warp 0's total below
        }
      }
      named_bar(kBarWG, kWG);
      if (tid >= 32 && tid < 64) S.gam[tid] += S.gam[31];
      named_bar(kBarWG, kWG);
      const float gL = S.gam[L - 1];
      if (tid < 64) {
        const float gi = S.gam[tid];
        S.sv[tid] = tid < L ? S.rk[tid] * __expf(gL - gi) : 0.f;
        S.so[tid] = S.rq[tid] * __expf(gi);
      }
      if (!wait_mma()) break;

      // ---- (2) A (rows 0-63) and P (rows 64-127) from S
      {
        float sv[64];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          float r16[16];
          tmem_ld16(lane_addr + TM_S + 16 * q4, r16);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) sv[16 * q4 + j] = r16[j];
        }
        if (tid < 64) {
          const int i = tid;
          const float bi = S.beta[s][i] * S.rk[i], gi = S.gam[i];
#pragma unroll
          for (int j = 0; j < 64; ++j) {
            const float a = (j < i && i < L) ? bi * S.rk[j] * __expf(gi - S.gam[j]) * sv[j] : 0.f;
            sA[i * LDA + j] = a;
          }
        } else {
          const int r = tid - 64;
          const float qr = S.rq[r], gr = S.gam[r];
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {
            float e[8];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
              const int j = 8 * ch + jj;
              e[jj] = (j <= r && r < L) ? qr * S.rk[j] * __expf(gr - S.gam[j]) * sv[j] : 0.f;
            }
            st_sw128_chunk(sP, r, ch,
                           make_uint4(pack_bf16(e[0], e[1]), pack_bf16(e[2], e[3]), pack_bf16(e[4], e[5]),
                                      pack_bf16(e[6], e[7])));
          }
        }
      }
      tc_fence_before();
      named_bar(kBarWG, kWG);

      // ---- (3) T = (I + A)^-1, then W' = T diag(beta e^G rk), U' = T diag(beta)
      solve_unit_lower(sA, sT, S.X, tid);
      {
        const int i = tid >> 1, jh = tid & 1;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          float wv[8], uv[8];
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            const int j = 32 * jh + 8 * cc + jj;
            const float t = sT[i * LDA + j], b = S.beta[s][j];
            uv[jj] = t * b;
            wv[jj] = t * b * __expf(S.gam[j]) * S.rk[j];
          }
          const int ch = 4 * jh + cc;
          st_sw128_chunk(sWU, i, ch, make_uint4(pack_bf16(wv[0], wv[1]), pack_bf16(wv[2], wv[3]),
                                                pack_bf16(wv[4], wv[5]), pack_bf16(wv[6], wv[7])));
          st_sw128_chunk(sWU + 8192, i, ch, make_uint4(pack_bf16(uv[0], uv[1]), pack_bf16(uv[2], uv[3]),
                                                       pack_bf16(uv[4], uv[5]), pack_bf16(uv[6], uv[7])));
        }
      }
      fence_proxy_async_smem();
      named_bar(kBarWG, kWG);

      // ---- (4) w^T = K^T W'^T ; vn^T = V^T U'^T ; o1^T = h^T Q^T
      if (tid == 0) {
        tc_fence_after();
        constexpr uint32_t id_mn = idesc_bf16(128, 64, 1, 0);
        const uint32_t aWU = smem_u32(sWU), aH = smem_u32(sH);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          mma_bf16(tbase + TM_W, smem_desc(aQK + ks * 2048, 16384, 1024), smem_desc(aWU + ks * 32, 16, 1024), id_mn,
                   ks > 0);
          mma_bf16(tbase + TM_VN, smem_desc(aV + ks * 2048, 8192, 1024), smem_desc(aWU + 8192 + ks * 32, 16, 1024),
                   id_mn, ks > 0);
        }
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t qoff = 8192 + (ks >> 2) * 16384 + (ks & 3) * 32;
          mma_bf16(tbase + TM_O1, smem_desc(aH + ks * 2048, 16384, 1024), smem_desc(aQK + qoff, 16, 1024), id_mn,
                   ks > 0);
        }
        mma_commit(smem_u32(&S.mma));
      }
      if (!wait_mma()) break;

      // ---- (5) w [i][d] (K-major B operand) from w^T in TMEM (lane d)
      {
        const int d = tid;
        uint8_t *wt = sWU + (d >> 6) * 8192;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          float r16[16];
          tmem_ld16(lane_addr + TM_W + 16 * q4, r16);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const uint32_t off = sw128_offset(16 * q4 + j, d & 63);
            *reinterpret_cast<__nv_bfloat16 *>(wt + off) = __float2bfloat16_rn(r16[j]);
          }
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      named_bar(kBarWG, kWG);

      // ---- (6) vn^T -= h^T w^T
      if (tid == 0) {
        tc_fence_after();
        constexpr uint32_t id_neg = idesc_bf16(128, 64, 1, 0, 1);
        const uint32_t aWU = smem_u32(sWU), aH = smem_u32(sH);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t woff = (ks >> 2) * 8192 + (ks & 3) * 32;
          mma_bf16(tbase + TM_VN, smem_desc(aH + ks * 2048, 16384, 1024), smem_desc(aWU + woff, 16, 1024), id_neg,
                   1);
        }
        mma_commit(smem_u32(&S.mma));
      }
      if (!wait_mma()) break;

      // ---- (7) vn^T [v][i] and vt^T [v][i] = vn * sv_i (lane v)
      {
        const int v = tid;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          float r16[16];
          tmem_ld16(lane_addr + TM_VN + 16 * q4, r16);
          tmem_ld_wait();
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const int i0 = 16 * q4 + 8 * half;
            const float *x = r16 + 8 * half;
            st_sw128_chunk(sVN, v, i0 >> 3,
                           make_uint4(pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]), pack_bf16(x[4], x[5]),
                                      pack_bf16(x[6], x[7])));
            const float *sc = S.sv + i0;
            st_sw128_chunk(sVT, v, i0 >> 3,
                           make_uint4(pack_bf16(x[0] * sc[0], x[1] * sc[1]), pack_bf16(x[2] * sc[2], x[3] * sc[3]),
                                      pack_bf16(x[4] * sc[4], x[5] * sc[5]), pack_bf16(x[6] * sc[6], x[7] * sc[7])));
          }
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      named_bar(kBarWG, kWG);

      // ---- (8) dH = K^T vt ; o2^T = vn^T P^T
      if (tid == 0) {
        tc_fence_after();
        constexpr uint32_t id_h = idesc_bf16(128, 128, 1, 0);
        constexpr uint32_t id_kk = idesc_bf16(128, 64, 0, 0);
        const uint32_t aVT = smem_u32(sVT), aVN = smem_u32(sVN), aP = smem_u32(sP);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          mma_bf16(tbase + TM_H, smem_desc(aQK + ks * 2048, 16384, 1024), smem_desc(aVT + ks * 32, 16, 1024), id_h,
                   ks > 0);
          mma_bf16(tbase + TM_O2, smem_desc(aVN + ks * 32, 16, 1024), smem_desc(aP + ks * 32, 16, 1024), id_kk,
                   ks > 0);
        }
        mma_commit(smem_u32(&S.mma));
      }
      if (!wait_mma()) break;

      // ---- (9) state update (lane d) and output (lane v)
      {
        const float decay = __expf(gL);
        const int d = tid;
#pragma unroll
        for (int q8 = 0; q8 < 8; ++q8) {
          float r16[16];
          tmem_ld16(lane_addr + TM_H + 16 * q8, r16);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) h[16 * q8 + j] = fmaf(decay, h[16 * q8 + j], r16[j]);
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const float *x = h + 16 * q8 + 8 * half;
            const int ch = 2 * q8 + half;
            st_sw128_chunk(sH + (ch >> 3) * 16384, d, ch & 7,
                           make_uint4(pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]), pack_bf16(x[4], x[5]),
                                      pack_bf16(x[6], x[7])));
          }
        }
        const int v = tid;
        __nv_bfloat16 *orow = p.o + (t0 * p.HV + hv) * DV + v;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          float a16[16], b16[16];
          tmem_ld16(lane_addr + TM_O1 + 16 * q4, a16);
          tmem_ld16(lane_addr + TM_O2 + 16 * q4, b16);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int r = 16 * q4 + j;
            if (r < L) orow[(int64_t)r * p.HV * DV] = __float2bfloat16_rn(fmaf(S.so[r], a16[j], b16[j]));
          }
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      named_bar(kBarWG, kWG);
      if (tid == 0) mbar_arrive(smem_u32(&S.empty[s]));
    }

    if (named_bar_and(kBarWG, kWG, *err == 0) && p.ht) {
      float *dst = p.ht + (unit * DK + tid) * DV;
#pragma unroll
      for (int v = 0; v < DV; v += 4) *reinterpret_cast<float4 *>(dst + v) = make_float4(h[v], h[v + 1], h[v + 2], h[v + 3]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tbase, TM_COLS);
  if (tid == 0 && S.err) raise_status(p.status, GDR_ERR_TIMEOUT);
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 3-D map over a [tokens, heads, D] bf16 tensor, boxes of 64 (D) x 1 x 64 (tokens)
int make_map(CUtensorMap *m, const void *base, int64_t D, int64_t heads, int64_t tokens) {
  auto fn = encode_fn();
  if (!fn) return set_error(GDR_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)heads, (cuuint64_t)tokens};
  cuuint64_t strides[2] = {(cuuint64_t)(D * 2), (cuuint64_t)(heads * D * 2)};
  cuuint32_t box[3] = {64, 1, 64};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return set_error(GDR_ERR_CUDA, "cuTensorMapEncodeTiled failed");
  return GDR_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

int run_fused(const gdr_desc &d, const void *q, const void *k, const void *v, const float *g, const void *beta,
              const float *h0, const int64_t *cu, int Cs, int l2, void *o, float *ht, int *status,
              cudaStream_t stream) {
  if (d.dtype != GDR_BF16 || d.gate != GDR_GATE_SCALAR || d.K != DK || d.V != DV || Cs != C)
    return GDR_ERR_UNSUPPORTED;
  const int64_t tok = d.B * d.T;
  if (tok >= (int64_t)INT32_MAX) return GDR_ERR_UNSUPPORTED;  // TMA coordinates are int32
  if (d.N * d.HV > (int64_t)INT32_MAX) return GDR_ERR_UNSUPPORTED;
  if (tok > 0 && !(aligned16(q) && aligned16(k) && aligned16(v)))
    return set_error(GDR_ERR_ALIGN, "q, k and v must be 16-byte aligned for the fused form");
  if (d.N == 0 || d.HV == 0) return GDR_OK;
  if (tok == 0) {
    // no tokens: the final state is the initial one
    if (ht) {
      cudaError_t e = h0 ? cudaMemcpyAsync(ht, h0, sizeof(float) * d.N * d.HV * DK * DV, cudaMemcpyDeviceToDevice,
                                           stream)
                         : cudaMemsetAsync(ht, 0, sizeof(float) * d.N * d.HV * DK * DV, stream);
      if (e != cudaSuccess) return cuda_error(e, "final state copy");
    }
    return GDR_OK;
  }
  CUtensorMap mq, mk, mv;
  int rc;
  if ((rc = make_map(&mq, q, DK, d.H, tok)) != GDR_OK) return rc;
  if ((rc = make_map(&mk, k, DK, d.H, tok)) != GDR_OK) return rc;
  if ((rc = make_map(&mv, v, DV, d.HV, tok)) != GDR_OK) return rc;
  FusedParams fp;
  fp.beta = (const __nv_bfloat16 *)beta;
  fp.g = g;
  fp.h0 = h0;
  fp.cu = cu;
  fp.o = (__nv_bfloat16 *)o;
  fp.ht = ht;
  fp.status = status;
  fp.T = d.T;
  fp.N = d.N;
  fp.H = d.H;
  fp.HV = d.HV;
  fp.l2 = l2;
  fp.timeout_ns = 2000000000ull;
  cudaError_t e = cudaFuncSetAttribute(gdr_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
  if (e != cudaSuccess) return cuda_error(e, "cudaFuncSetAttribute(gdr_fused_kernel)");
  gdr_fused_kernel<<<(unsigned)(d.N * d.HV), kThreads, SMEM_BYTES, stream>>>(mq, mk, mv, fp);
  count_launch();
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_error(e, "gdr_fused_kernel launch");
  return GDR_OK;
}

}  // namespace gdr
