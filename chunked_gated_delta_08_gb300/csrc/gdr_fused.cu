// gdr_fused.cu -- the fused single-pass forward on the sm_103a tensor cores.
//
// One block per (sequence, value head) walks the sequence chunk by chunk with
// the K x V state on chip: it reads q, k, v, g, beta once and writes o and the
// final state once; nothing of the chunk form (A, T, w, u, h, v_new) goes to
// HBM.  Per chunk of C = 64 tokens, with Gamma the within-chunk cumsum of g,
// r the in-kernel L2-norm scales, L the number of valid rows and h the state
// entering the chunk (the chunk-start state of the KCP handbook):
//
//   S     = [K; Q] K^T                                tcgen05 M=128 N=64  K=128
//   A_ij  = beta_i r_i r_j e^{G_i - G_j} (KK^T)_ij, i > j       (CUDA cores)
//   T     = (I + A)^-1   16 x 16 blocks, then doubling   (CUDA cores, warp MMAs)
//   W'    = T diag(beta e^G r),  U' = T diag(beta)              (bf16 operands)
//   w^T   = K^T W'^T,  vn^T = V^T U'^T                 tcgen05 M=128 N=64  K=64
//   vn^T -= h^T w^T,  o1^T = h^T Q^T                   tcgen05 M=128 N=64  K=128
//   P_rj  = rq_r r_j e^{G_r - G_j} (QK^T)_rj, j <= r            (CUDA cores)
//   dH    = K^T (vn * r e^{G_L - G}),  o2^T = vn^T P^T tcgen05 M=128 N=128/64 K=64
//   h'    = e^{G_L} h + dH                             fp32, in TMEM
//   o_r   = rq_r e^{G_r} o1_r + o2_r
//
// Every product has M = 128 (the K or V dimension), so an accumulator row is a
// TMEM lane and one thread owns it.  q, k, v tiles arrive by TMA in the
// 128-byte swizzle and are read by the tensor cores K-major and MN-major as
// they land.
//
// Warp roles (512 threads):
//   warps 0-3   chain: the state recurrence of chunk c -- the w and v_new
//               epilogues, the decay of the fp32 state held in TMEM (the next
//               MMA adds dH into it), the bf16 copy of the new state -- and
//               the output epilogue of chunk c (staged in the v_new tile,
//               written by two TMA tensor stores);
//   warps 4-11  prep: everything of chunk c that does not need the state
//               (the q and k norms, gate cumsum and scale vectors, A, the
//               solve, W', U', P), so it can start chunk c+1 while the
//               tensor cores turn W', U' into w, u;
//   warp 12     producer: TMA loads of q, k (3-slot ring) and v (1 slot), g, beta;
//   warp 13     MMA issuer: one thread issues every tcgen05.mma in a fixed order.
// Hand-offs are mbarriers, each completing once per chunk.  Every wait is
// bounded (about two seconds of SM clock); on expiry the block records GDR_ERR_TIMEOUT in
// the status word, lets its copies and MMAs in flight finish, frees its
// tensor memory and returns.  A role's decision to stop is uniform across
// its threads.
//
// Supported: bf16, scalar gate, K = V = 128, C = 64, dense or varlen.  Other
// requests return GDR_ERR_UNSUPPORTED so the dispatcher takes the chunked form.
//
// Pages cited: the KCP handbook = "flash-linear-attention KCP 精度失效根因排查手册".
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <mutex>

#include "gdr_device.cuh"
#include "gdr_fused_common.cuh"
#include "gdr_internal.h"
#include "gdr_sm100.cuh"

namespace gdr {
namespace {

using namespace sm100;
using namespace fused;

constexpr int C = 64;
constexpr int DK = 128;
constexpr int DV = 128;
constexpr int kQKSlots = 3;
constexpr int kPrepWarps = 8;
constexpr int kPrepThreads = 32 * kPrepWarps;
constexpr int kProducerWarp = 4 + kPrepWarps;
constexpr int kMmaWarp = kProducerWarp + 1;
constexpr int kThreads = 512;  // 16 warps: the last two only join the final barrier
constexpr int kBarChain = 1;   // named barrier of warps 0-3
constexpr int kBarPrep = 2;    // named barrier of the prep warps
constexpr int LDA = C + 1;     // row stride of the packed fp32 A / T^T matrix
constexpr int kXL = 33;        // row stride of the solve scratch Y [32][kXL]
constexpr int kZL = 18;        // row stride of the solve scratch Z [16][kZL] (two of them)

// shared memory map (offsets from a 1024-byte aligned base)
constexpr uint32_t SZ_QK = 32768;                    // [K d0-63 | Q d0-63 | K d64-127 | Q d64-127]
constexpr uint32_t SZ_V = 16384;                     // [V v0-63 | V v64-127]
constexpr uint32_t OFF_QK = 0;
constexpr uint32_t OFF_V = OFF_QK + kQKSlots * SZ_QK;
constexpr uint32_t OFF_H = OFF_V + SZ_V;             // h [d][v] bf16, 2 sub-tiles of 128 rows: MN-major A of h^T
constexpr uint32_t OFF_WU = OFF_H + 32768;           // W' [i][j] | U' [i][j]; then w [d][i]: MN-major B
constexpr uint32_t OFF_P = OFF_WU + 16384;           // P [r][j]: K-major B
constexpr uint32_t OFF_VN = OFF_P + 8192;            // vn^T [v][i]: K-major A
constexpr uint32_t OFF_VT = OFF_VN + 16384;          // vt^T [v][i]: K-major B
constexpr uint32_t OFF_AT = OFF_VT + 16384;          // fp32 [64][65]: A strictly below, T^T strictly above
constexpr uint32_t OFF_SMALL = (OFF_AT + C * LDA * 4 + 15) & ~15u;

// TMEM columns
// TM_HS holds the fp32 state h; the state-update MMA accumulates dH into it.
constexpr uint32_t TM_S = 0, TM_W = 64, TM_VN = 128, TM_O1 = 192, TM_O2 = 256, TM_HS = 320, TM_COLS = 512;

struct Small {
  float gb[kQKSlots][2][C];     // g, beta of each QK slot (producer)
  // per-chunk scalars, written by the prep warps at the start of their chunk
  // (bw, cw by chunk parity; sv, so, gL by chunk mod 3, which the chain warps
  // read for chunks behind the prep warps')
  float gam[C], rq[C], rk[C];   // gate cumsum and norm scales (0 past the chunk end)
  float bw[2][C];               // beta (0 past the chunk end)
  float ep[C], em[C];           // decay factors e^{G - m}, e^{m - G}
  float cw[2][C];               // column scale of W', beta_j e^{G_j} rk_j
  float sv[3][C];               // chain: row scale of vt, rk_i e^{G_L - G_i} (0 past the end)
  float so[3][C];               // chain: row scale of o1, rq_r e^{G_r}
  float gL[4];                  // chain: G at the chunk's last valid row
  float X[32 * kXL];            // solve scratch
  uint64_t full_qk[kQKSlots], empty_qk[kQKSlots], full_v, empty_v;
  uint64_t b_s, b_sfree, b_prep, b_w, b_wepi, b_pend, b_vn, b_vnepi, b_h, b_state, b_oepi, b_final;
  uint32_t tmem_slot;
  int err;
  int bad;
  int factored;
};

constexpr uint32_t SMEM_BYTES = OFF_SMALL + sizeof(Small) + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

struct FusedParams {
  const __nv_bfloat16 *beta;
  const float *g, *h0;
  const int64_t *cu;
  __nv_bfloat16 *o;
  float *ht;
  int *status;
  int64_t T, N, H, HV;
  int l2;
  int beta_logits;
  unsigned long long timeout_cycles;
};

// T = (I + A)^-1 for a unit lower-triangular 64 x 64 system.  AT holds A
// strictly below the diagonal; T (strictly lower part; its diagonal is 1) is
// written transposed strictly above the diagonal: T_ij at AT[j][i].  The
// inverse is built by doubling the block size, with
// [[T1, 0], [T21, T2]], T21 = -T2 A21 T1 at each step:
//   16 x 16 diagonal blocks by forward substitution (CUDA cores, fp32);
//   16 -> 32 and 32 -> 64 by warp-level tensor-core products in split tf32.
// Threads 0..255 of the prep warps (pw = prep warp 0..7).
__device__ __forceinline__ float t_at(const float *AT, int r, int s) {  // T[r][s]
  return r > s ? AT[s * LDA + r] : (r == s ? 1.f : 0.f);
}

// D (16 x 8 tile at A-rows ar0.., B-cols bc0..) = A_tile(rows, k) * B(k, cols)
// over nk k-steps of 8; A and B read through the functors fa(r, k), fb(k, n).
// The sum over k is order-free, so fragment column t (and t + 4) of k-step ks
// takes k = 2 nk t + 2 ks (+ 1): the four t of a load are 2 nk apart, so the
// fragment loads from the odd-strided AT meet no shared-memory bank conflict at
// nk = 4 and at most two-way ones at nk = 2 (k = t + 4 would be four-way).
// x = hi + lo with hi, lo tf32 bit patterns, by truncation (masking the low 13
// mantissa bits) rather than conversion instructions, which keeps the split on
// the integer and FMA pipes.  |lo| < 2^-10 |x| and lo is truncated in turn, so
// hi*hi + hi*lo + lo*hi misses the product by under 2^-18 of it: fp32-like,
// far below the bf16 rounding W' and U' get next.
__device__ __forceinline__ void split_tf32_trunc(float x, uint32_t &hi, uint32_t &lo) {
  hi = __float_as_uint(x) & 0xffffe000u;
  lo = __float_as_uint(x - __uint_as_float(hi)) & 0xffffe000u;
}

template <typename FA, typename FB>
__device__ __forceinline__ void tile_product(float (&d)[4], int nk, FA fa, FB fb) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int e = 0; e < 4; ++e) d[e] = 0.f;
  for (int ks = 0; ks < nk; ++ks) {
    const int k0 = 2 * nk * t + 2 * ks, k1 = k0 + 1;
    const float a[4] = {fa(g, k0), fa(g + 8, k0), fa(g, k1), fa(g + 8, k1)};
    const float b[2] = {fb(k0, g), fb(k1, g)};
    uint32_t ah[4], al[4], bh[2], bl[2];
#pragma unroll
    for (int e = 0; e < 4; ++e) split_tf32_trunc(a[e], ah[e], al[e]);
#pragma unroll
    for (int e = 0; e < 2; ++e) split_tf32_trunc(b[e], bh[e], bl[e]);
    mma_tf32(d, al[0], al[1], al[2], al[3], bh[0], bh[1]);
    mma_tf32(d, ah[0], ah[1], ah[2], ah[3], bl[0], bl[1]);
    mma_tf32(d, ah[0], ah[1], ah[2], ah[3], bh[0], bh[1]);
  }
}

// Row strides of the solve scratch: Y [32][kXL] and the two Z [16][kZL]; both
// make the B-fragment loads of the permuted k (rows 2 nk apart) bank-conflict free.
__device__ void solve_unit_lower(float *AT, float *X, int pt) {
  const int pw = pt >> 5, lane = pt & 31, g = lane >> 2, t = lane & 3;
  // ---- 16 x 16 diagonal blocks: prep warp b, lane c < 16 solves column c
  if (pw < 4 && lane < 16) {
    const int base = 16 * pw, c = lane;
    float x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float a0 = (i == c) ? 1.f : 0.f, a1 = 0.f;
#pragma unroll
      for (int l = 0; l < i; l += 2) {
        a0 = fmaf(-AT[(base + i) * LDA + base + l], x[l], a0);
        if (l + 1 < i) a1 = fmaf(-AT[(base + i) * LDA + base + l + 1], x[l + 1], a1);
      }
      x[i] = (i < c) ? 0.f : a0 + a1;
    }
#pragma unroll
    for (int i = 1; i < 16; ++i)
      if (i > c) AT[(base + c) * LDA + base + i] = x[i];
  }
  named_bar(kBarPrep, kPrepThreads);
  // ---- 16 -> 32: T_{b,b-1} = -T_bb (A_{b,b-1} T_{b-1,b-1}) for b = 1, 3 (warps 0-3: pair, n-tile)
  if (pw < 4) {
    const int b = 1 + 2 * (pw >> 1), nt = pw & 1, r0 = 16 * b, c0 = 16 * (b - 1);
    float *Z = X + (pw >> 1) * 16 * kZL;  // Z [16][kZL]
    float d[4];
    tile_product(d, 2, [&](int r, int k) { return AT[(r0 + r) * LDA + c0 + k]; },
                 [&](int k, int n) { return t_at(AT, c0 + k, c0 + 8 * nt + n); });
    Z[g * kZL + 8 * nt + 2 * t] = d[0];
    Z[g * kZL + 8 * nt + 2 * t + 1] = d[1];
    Z[(g + 8) * kZL + 8 * nt + 2 * t] = d[2];
    Z[(g + 8) * kZL + 8 * nt + 2 * t + 1] = d[3];
  }
  named_bar(kBarPrep, kPrepThreads);
  if (pw < 4) {
    const int b = 1 + 2 * (pw >> 1), nt = pw & 1, r0 = 16 * b, c0 = 16 * (b - 1);
    const float *Z = X + (pw >> 1) * 16 * kZL;
    float d[4];
    tile_product(d, 2, [&](int r, int k) { return t_at(AT, r0 + r, r0 + k); },
                 [&](int k, int n) { return Z[k * kZL + 8 * nt + n]; });
    const int cc = c0 + 8 * nt + 2 * t;
    AT[cc * LDA + r0 + g] = -d[0];
    AT[(cc + 1) * LDA + r0 + g] = -d[1];
    AT[cc * LDA + r0 + g + 8] = -d[2];
    AT[(cc + 1) * LDA + r0 + g + 8] = -d[3];
  }
  named_bar(kBarPrep, kPrepThreads);
  // ---- 32 -> 64: Y = A[32:64, 0:32] T[0:32, 0:32]; T[32:64, 0:32] = -T[32:64, 32:64] Y (8 warps, one 16 x 8 tile each)
  {
    const int mt = pw >> 2, nt = pw & 3;
    float d[4];
    tile_product(d, 4, [&](int r, int k) { return AT[(32 + 16 * mt + r) * LDA + k]; },
                 [&](int k, int n) { return t_at(AT, k, 8 * nt + n); });
    X[(16 * mt + g) * kXL + 8 * nt + 2 * t] = d[0];
    X[(16 * mt + g) * kXL + 8 * nt + 2 * t + 1] = d[1];
    X[(16 * mt + g + 8) * kXL + 8 * nt + 2 * t] = d[2];
    X[(16 * mt + g + 8) * kXL + 8 * nt + 2 * t + 1] = d[3];
  }
  named_bar(kBarPrep, kPrepThreads);
  {
    const int mt = pw >> 2, nt = pw & 3;
    float d[4];
    tile_product(d, 4, [&](int r, int k) { return t_at(AT, 32 + 16 * mt + r, 32 + k); },
                 [&](int k, int n) { return X[k * kXL + 8 * nt + n]; });
    const int cc = 8 * nt + 2 * t, rr = 32 + 16 * mt + g;
    AT[cc * LDA + rr] = -d[0];
    AT[(cc + 1) * LDA + rr] = -d[1];
    AT[cc * LDA + rr + 8] = -d[2];
    AT[(cc + 1) * LDA + rr + 8] = -d[3];
  }
  named_bar(kBarPrep, kPrepThreads);
}

__global__ void __launch_bounds__(kThreads, 1)
    gdr_fused_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                     const FusedParams p) {
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
    for (int s = 0; s < kQKSlots; ++s) {
      mbar_init(smem_u32(&S.full_qk[s]), 2);
      mbar_init(smem_u32(&S.empty_qk[s]), 1);
    }
    mbar_init(smem_u32(&S.full_v), 1);
    mbar_init(smem_u32(&S.empty_v), 1);
    // the single-arrival hand-off barriers b_s .. b_final are contiguous
    for (uint64_t *b = &S.b_s; b <= &S.b_final; ++b) mbar_init(smem_u32(b), 1);
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
  const uint64_t tmo = p.timeout_cycles;
  uint8_t *const sH = sm + OFF_H, *const sWU = sm + OFF_WU, *const sP = sm + OFF_P, *const sVN = sm + OFF_VN,
                 *const sVT = sm + OFF_VT;

  if (warp < 4) {
    // ================================================================ chain
    const int t = tid;  // TMEM lane: state row d = t, v_new column v = t
    const uint32_t lane_addr = tbase + ((uint32_t)(warp * 32) << 16);
    // one thread polls; the others sleep in the named barrier that shares its verdict
    auto vote_wait = [&](uint64_t *bar, uint32_t parity) -> bool {
      const bool ok = t == 0 ? mbar_wait(smem_u32(bar), parity, err, tmo) : true;
      return named_bar_and(kBarChain, 128, ok);
    };
    // h_0 into TMEM (fp32) and its bf16 copy into sH
    {
      const float *src = p.h0 ? p.h0 + (unit * DK + t) * DV : nullptr;
#pragma unroll
      for (int q8 = 0; q8 < 8; ++q8) {
        float r16[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) r16[j] = src ? src[16 * q8 + j] : 0.f;
        tmem_st16(lane_addr + TM_HS + 16 * q8, r16);
        st_sw128_chunk(sH + (q8 >> 2) * 16384, t, (2 * q8) & 7, pack8(r16));
        st_sw128_chunk(sH + (q8 >> 2) * 16384, t, (2 * q8 + 1) & 7, pack8(r16 + 8));
      }
      tmem_st_wait();
    }
    fence_proxy_async_smem();
    tc_fence_before();
    named_bar(kBarChain, 128);
    if (t == 0) {  // h_0 is ready; D_vn is free
      mbar_arrive(smem_u32(&S.b_state));
      mbar_arrive(smem_u32(&S.b_vnepi));
    }
    bool ok = true;
    for (int c = 0; ok && c < nch; ++c) {
      const uint32_t ph = c & 1;
      const int k3 = c % 3;
      // the next chunk's scalars while the prep warps work on this one
      // the previous output tile in sVN must have been read by its TMA store
      if (t == 0) bulk_wait_read0();
      // w^T of chunk c is in TMEM (its MMAs follow the prep warps' b_prep arrival)
      if (!(ok = vote_wait(&S.b_prep, ph) && vote_wait(&S.b_w, ph))) break;
      tc_fence_after();
      // ---- w [d][i] (MN-major B operand) from w^T in TMEM (lane d, all 64 i)
#pragma unroll
      for (int colh = 0; colh < 2; ++colh) {
        float r32[32];
        tmem_ld32(lane_addr + TM_W + 32 * colh, r32);
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 4; ++q) st_sw128_chunk(sWU, t, 4 * colh + q, pack8(r32 + 8 * q));
      }
      fence_proxy_async_smem();
      tc_fence_before();
      named_bar(kBarChain, 128);
      if (t == 0) mbar_arrive(smem_u32(&S.b_wepi));
      if (!(ok = vote_wait(&S.b_vn, ph))) break;
      tc_fence_after();
      // ---- vn^T [v][i] and vt^T [v][i] = vn * sv_i
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        // every load of this block before any store: the stores could alias them otherwise
        float r32[32], sc[32];
        tmem_ld32(lane_addr + TM_VN + 32 * h2, r32);
        ld_f32x32(S.sv[k3] + 32 * h2, sc);
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int i0 = 32 * h2 + 8 * q;
          const float *x = r32 + 8 * q;
          float y[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) y[e] = x[e] * sc[8 * q + e];
          st_sw128_chunk(sVN, t, i0 >> 3, pack8(x));
          st_sw128_chunk(sVT, t, i0 >> 3, pack8(y));
        }
      }
      // ---- decay the fp32 state in TMEM; the next MMA adds dH into it
      {
        const float decay = __expf(S.gL[k3]);
#pragma unroll
        for (int q8 = 0; q8 < 8; ++q8) {
          float r16[16];
          tmem_ld16(lane_addr + TM_HS + 16 * q8, r16);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) r16[j] *= decay;
          tmem_st16(lane_addr + TM_HS + 16 * q8, r16);
        }
        tmem_st_wait();
      }
      fence_proxy_async_smem();
      tc_fence_before();
      named_bar(kBarChain, 128);
      if (t == 0) mbar_arrive(smem_u32(&S.b_vnepi));
      if (!(ok = vote_wait(&S.b_h, ph))) break;
      tc_fence_after();
      // ---- bf16 copy of the new state for the next chunk's products
#pragma unroll
      for (int h4 = 0; h4 < 4; ++h4) {
        float r32[32];
        tmem_ld32(lane_addr + TM_HS + 32 * h4, r32);
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int ch = 4 * h4 + q;
          st_sw128_chunk(sH + (ch >> 3) * 16384, t, ch & 7, pack8(r32 + 8 * q));
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      named_bar(kBarChain, 128);
      if (t == 0) mbar_arrive(smem_u32(&S.b_state));
      // ---- output of chunk c: o[r][v] = so_r o1[v][r] + o2[v][r] (lane v, all 64 rows).  A whole
      //      chunk goes through sVN (free until the next v_new epilogue) and two TMA tensor stores; a
      //      ragged last chunk is stored element by element so nothing past the sequence end is written.
      {
        const int64_t t0 = bos + (int64_t)c * C;
        const int L = (int)(eos - t0 < C ? eos - t0 : C);
        const int64_t rstride = p.HV * DV;
#pragma unroll 1
        for (int colh = 0; colh < 2; ++colh) {
          float a32[32], b32[32], so[32];
          tmem_ld32(lane_addr + TM_O1 + 32 * colh, a32);
          tmem_ld32(lane_addr + TM_O2 + 32 * colh, b32);
          ld_f32x32(S.so[k3] + 32 * colh, so);
          tmem_ld_wait();
          __nv_bfloat16 ov[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) ov[j] = __float2bfloat16_rn(fmaf(so[j], a32[j], b32[j]));
          if (L == C) {
            uint8_t *tile = sVN + (t >> 6) * 8192;
#pragma unroll
            for (int j = 0; j < 32; ++j)
              *reinterpret_cast<__nv_bfloat16 *>(tile + sw128_offset(32 * colh + j, t & 63)) = ov[j];
          } else {
            __nv_bfloat16 *ocol = p.o + (t0 * p.HV + hv) * DV + t + (int64_t)(32 * colh) * rstride;
            const int nr = L - 32 * colh;
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (j < nr) ocol[(int64_t)j * rstride] = ov[j];
          }
        }
        tc_fence_before();
        if (L == C) fence_proxy_async_smem();
        named_bar(kBarChain, 128);
        if (t == 0) {
          if (L == C) {
            tma_store_3d(&tm_o, smem_u32(sVN), 0, (int)hv, (int)t0);
            tma_store_3d(&tm_o, smem_u32(sVN + 8192), 64, (int)hv, (int)t0);
            bulk_commit();
          }
          mbar_arrive(smem_u32(&S.b_oepi));  // D_o1, D_o2 of chunk c have been read
        }
      }
    }
    if (t == 0) bulk_wait0();  // every output store has landed before the block can exit
    if (named_bar_and(kBarChain, 128, ok && *err == 0) && p.ht) {
      float *dst = p.ht + (unit * DK + t) * DV;
#pragma unroll
      for (int h4 = 0; h4 < 4; ++h4) {
        float r32[32];
        tmem_ld32(lane_addr + TM_HS + 32 * h4, r32);
        tmem_ld_wait();
#pragma unroll
        for (int v = 0; v < 32; v += 4)
          *reinterpret_cast<float4 *>(dst + 32 * h4 + v) = make_float4(r32[v], r32[v + 1], r32[v + 2], r32[v + 3]);
      }
    }
  } else if (warp < 4 + kPrepWarps) {
    // ================================================================ prep
    const int pt = tid - 128;                       // 0..255
    const int quad = warp & 3;                      // TMEM lane quadrant
    const int lrow = quad * 32 + lane;              // TMEM lane of this thread
    const int colh = (warp - 4) >> 2;               // which half of the columns this warp reads
    const uint32_t lane_addr = tbase + ((uint32_t)(quad * 32) << 16);
    float *AT = reinterpret_cast<float *>(sm + OFF_AT);
    auto vote_wait = [&](uint64_t *bar, uint32_t parity) -> bool {
      const bool ok = pt == 0 ? mbar_wait(smem_u32(bar), parity, err, tmo) : true;
      return named_bar_and(kBarPrep, kPrepThreads, ok);
    };
    for (int c = 0; c < nch; ++c) {
      const uint32_t ph = c & 1, php = (c - 1) & 1;
      const int slot = c % kQKSlots;
      const int64_t t0 = bos + (int64_t)c * C;
      const int L = (int)(eos - t0 < C ? eos - t0 : C);
      uint8_t *qk = sm + OFF_QK + slot * SZ_QK;
      if (!vote_wait(&S.b_s, ph)) break;
      tc_fence_after();
      // ragged tail: clear rows past the sequence end (they may hold the next sequence)
      if (L < C) {
        if (!vote_wait(&S.full_v, ph)) break;
        for (int e = pt; e < (C - L) * 48; e += kPrepThreads) {
          const int rr = L + e / 48, rest = e % 48, tile = rest >> 3, ch = rest & 7;
          uint8_t *base = tile < 4 ? qk + tile * 8192 : sm + OFF_V + (tile - 4) * 8192;
          st_sw128_chunk(base, rr, ch, make_uint4(0, 0, 0, 0));
        }
        fence_proxy_async_smem();
      }
      // ---- this chunk's norms, gate cumsum and scale vectors: q row norms (two threads per
      //      row), k row norms from the diagonal of K K^T in TMEM lanes 0-63 (prep warps 4-5),
      //      the gate cumsum (prep warp 0); then one row of each vector per thread of the first
      //      two prep warps
      const int par = c & 1, k3 = c % 3;
      {
        if (pt < 128) {
          const int row = pt >> 1, half = pt & 1;
          const uint8_t *qb = qk + 8192 + half * 16384;
          float ss = 0.f;
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) ss += sumsq_bf16x8(ld_sw128_chunk(qb, row, ch));
          ss += __shfl_xor_sync(0xffffffffu, ss, 1);
          if (half == 0) S.rq[row] = row < L ? (p.l2 ? rsqrtf(ss + kL2Eps) : 1.f) : 0.f;
        }
        if (pt >= 128 && pt < 160) {  // one warp: the inclusive cumsum of g over the chunk
          const int ln = pt - 128;
          float x0 = S.gb[slot][0][ln], x1 = S.gb[slot][0][ln + 32];
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const float y0 = __shfl_up_sync(0xffffffffu, x0, o), y1 = __shfl_up_sync(0xffffffffu, x1, o);
            if (ln >= o) {
              x0 += y0;
              x1 += y1;
            }
          }
          x1 += __shfl_sync(0xffffffffu, x0, 31);
          S.gam[ln] = x0;
          S.gam[ln + 32] = x1;
        }
        if (colh == 0 && quad < 2) {  // TMEM lanes 0-63 of S hold K K^T; its diagonal is |k_i|^2
          const int i = lrow;
          float r32[32];
          tmem_ld32(lane_addr + TM_S + 32 * quad, r32);
          tmem_ld_wait();
          float kk = 0.f;
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (e == (i & 31)) kk = r32[e];
          S.rk[i] = i < L ? (p.l2 ? rsqrtf(kk + kL2Eps) : 1.f) : 0.f;
        }
        named_bar(kBarPrep, kPrepThreads);
        if (pt < 64) {
          const float g0 = S.gam[0], gl = S.gam[L - 1];
          const float m = 0.5f * (g0 + gl);
          const float gi = S.gam[pt];
          S.sv[k3][pt] = pt < L ? S.rk[pt] * __expf(gl - gi) : 0.f;
          S.so[k3][pt] = S.rq[pt] * __expf(gi);
          S.ep[pt] = __expf(gi - m);
          S.em[pt] = __expf(m - gi);
          const float bw = pt < L ? S.gb[slot][1][pt] : 0.f;
          S.bw[par][pt] = bw;
          S.cw[par][pt] = bw * __expf(gi) * S.rk[pt];
          if (pt == 0) {
            S.gL[k3] = gl;
            S.factored = (g0 - gl) <= 160.f;
          }
        }
        named_bar(kBarPrep, kPrepThreads);
      }
      const bool factored = S.factored;
      // ---- A from lanes 0-63 of S: A_ij = beta_i rk_i rk_j e^{G_i - G_j} (k_i . k_j), i > j;
      //      P from lanes 64-127: P_rj = rq_r rk_j e^{G_r - G_j} (q_r . k_j), j <= r, kept packed in
      //      registers until its buffer is free, so S can be overwritten by the next chunk's product.
      uint32_t pk[16];
      {
        const int i = quad < 2 ? lrow : lrow - 64;
        const float bi = quad < 2 ? S.bw[par][i] * S.rk[i] : S.rq[i], epi = S.ep[i], gi = S.gam[i];
#pragma unroll
        for (int h16 = 0; h16 < 2; ++h16) {
          const int j0 = 32 * colh + 16 * h16;
          float r16[16], f[16], rk[16];
          tmem_ld16(lane_addr + TM_S + j0, r16);
          ld_f32x16(S.rk + j0, rk);
          if (factored) {
            ld_f32x16(S.em + j0, f);
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) f[jj] *= epi;
          } else {
            ld_f32x16(S.gam + j0, f);
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) f[jj] = __expf(gi - f[jj]);
          }
          tmem_ld_wait();
          if (quad < 2) {
#pragma unroll
            for (int jj = 0; jj < 16; ++jj)
              if (j0 + jj < i) AT[i * LDA + j0 + jj] = bi * rk[jj] * f[jj] * r16[jj];
          } else {
#pragma unroll
            for (int jj = 0; jj < 16; jj += 2) {
              const float e0 = j0 + jj <= i ? bi * rk[jj] * f[jj] * r16[jj] : 0.f;
              const float e1 = j0 + jj + 1 <= i ? bi * rk[jj + 1] * f[jj + 1] * r16[jj + 1] : 0.f;
              pk[8 * h16 + jj / 2] = pack_bf16(e0, e1);
            }
          }
        }
      }
      tc_fence_before();
      named_bar(kBarPrep, kPrepThreads);
      if (pt == 0) mbar_arrive(smem_u32(&S.b_sfree));  // S may now take the next chunk's product
      // ---- T = (I + A)^-1
      solve_unit_lower(AT, S.X, pt);
      // ---- W' = T diag(beta e^G rk), U' = T diag(beta) into the w region once w(c-1) is consumed
      if (c > 0 && !vote_wait(&S.b_vn, php)) break;
      {
        const int i = pt & 63, j0 = 16 * (pt >> 6);  // row i, columns j0 .. j0 + 15
        float tv[16], bw[16], cw[16];
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) tv[jj] = t_at(AT, i, j0 + jj);
        ld_f32x16(S.bw[par] + j0, bw);
        ld_f32x16(S.cw[par] + j0, cw);
        float wv[16], uv[16];
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
          uv[jj] = tv[jj] * bw[jj];
          wv[jj] = tv[jj] * cw[jj];
        }
        st_sw128_chunk(sWU, i, j0 >> 3, pack8(wv));
        st_sw128_chunk(sWU, i, (j0 >> 3) + 1, pack8(wv + 8));
        st_sw128_chunk(sWU + 8192, i, j0 >> 3, pack8(uv));
        st_sw128_chunk(sWU + 8192, i, (j0 >> 3) + 1, pack8(uv + 8));
      }
      fence_proxy_async_smem();
      named_bar(kBarPrep, kPrepThreads);
      if (pt == 0) mbar_arrive(smem_u32(&S.b_prep));
      // ---- P of chunk c, once MMA_o2(c-1) has consumed P(c-1)
      if (c > 0) {
        if (!vote_wait(&S.b_h, php)) break;
        tc_fence_after();
      }
      if (quad >= 2) {
        const int r = lrow - 64;
        st_sw128_chunk(sP, r, 4 * colh, make_uint4(pk[0], pk[1], pk[2], pk[3]));
        st_sw128_chunk(sP, r, 4 * colh + 1, make_uint4(pk[4], pk[5], pk[6], pk[7]));
        st_sw128_chunk(sP, r, 4 * colh + 2, make_uint4(pk[8], pk[9], pk[10], pk[11]));
        st_sw128_chunk(sP, r, 4 * colh + 3, make_uint4(pk[12], pk[13], pk[14], pk[15]));
      }
      fence_proxy_async_smem();
      tc_fence_before();
      named_bar(kBarPrep, kPrepThreads);
      // b_pend: P(c) is in place
      if (pt == 0) mbar_arrive(smem_u32(&S.b_pend));
    }
    tc_fence_before();
  } else if (warp == kProducerWarp) {
    // ================================================================ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_o);
    }
    int issued_qk = 0, issued_v = 0;
    for (int c = 0; c < nch; ++c) {
      const int slot = c % kQKSlots, u = c / kQKSlots;
      if (c >= kQKSlots) {
        const bool ok = lane == 0 ? mbar_wait(smem_u32(&S.empty_qk[slot]), (u - 1) & 1, err, tmo) : true;
        if (!__all_sync(0xffffffffu, ok)) break;
      }
      const int64_t t0 = bos + (int64_t)c * C;
      const int L = (int)(eos - t0 < C ? eos - t0 : C);
      const int tt = (int)t0;
      uint8_t *qk = sm + OFF_QK + slot * SZ_QK;
      if (lane == 0) {
        const uint32_t fb = smem_u32(&S.full_qk[slot]);
        mbar_arrive_expect_tx(fb, SZ_QK);
        tma_load_3d(smem_u32(qk), &tm_k, 0, (int)hq, tt, fb);
        tma_load_3d(smem_u32(qk + 8192), &tm_q, 0, (int)hq, tt, fb);
        tma_load_3d(smem_u32(qk + 16384), &tm_k, 64, (int)hq, tt, fb);
        tma_load_3d(smem_u32(qk + 24576), &tm_q, 64, (int)hq, tt, fb);
      }
      for (int i = lane; i < C; i += 32) {
        S.gb[slot][0][i] = i < L ? p.g[(t0 + i) * p.HV + hv] : 0.f;
        S.gb[slot][1][i] = i < L ? load_beta(p.beta, (t0 + i) * p.HV + hv, p.beta_logits) : 0.f;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&S.full_qk[slot]));
      issued_qk = c + 1;
      if (c >= 1) {
        const bool ok = lane == 0 ? mbar_wait(smem_u32(&S.empty_v), (c - 1) & 1, err, tmo) : true;
        if (!__all_sync(0xffffffffu, ok)) break;
      }
      if (lane == 0) {
        const uint32_t fb = smem_u32(&S.full_v);
        mbar_arrive_expect_tx(fb, SZ_V);
        tma_load_3d(smem_u32(sm + OFF_V), &tm_v, 0, (int)hv, tt, fb);
        tma_load_3d(smem_u32(sm + OFF_V + 8192), &tm_v, 64, (int)hv, tt, fb);
      }
      issued_v = c + 1;
    }
    // let every copy issued land before the block can exit
    if (lane == 0) {
      for (int c = (issued_qk > kQKSlots ? issued_qk - kQKSlots : 0); c < issued_qk; ++c)
        mbar_wait_drain(smem_u32(&S.full_qk[c % kQKSlots]), (c / kQKSlots) & 1, tmo);
      if (issued_v > 0) mbar_wait_drain(smem_u32(&S.full_v), (issued_v - 1) & 1, tmo);
    }
  } else if (warp == kMmaWarp && lane == 0) {
    // ================================================================ MMA issuer
    constexpr uint32_t id_s = idesc_bf16(128, 64, 0, 0);        // [K;Q] K^T
    constexpr uint32_t id_mnk = idesc_bf16(128, 64, 1, 0);      // A MN-major, B K-major
    constexpr uint32_t id_vn = idesc_bf16(128, 64, 1, 1, 1);    // -h^T w^T, both MN-major
    constexpr uint32_t id_h = idesc_bf16(128, 128, 1, 0);       // K^T vt
    constexpr uint32_t id_kk = idesc_bf16(128, 64, 0, 0);       // vn^T P^T
    const uint32_t aH = smem_u32(sH), aWU = smem_u32(sWU), aP = smem_u32(sP), aVN = smem_u32(sVN),
                   aVT = smem_u32(sVT), aV = smem_u32(sm + OFF_V);
    auto wt = [&](uint64_t *bar, uint32_t parity) { return mbar_wait_spin(smem_u32(bar), parity, err, tmo); };
    // Descriptors are built once: an operand at base + off (off a multiple of 16 bytes, every shared
    // address below 2^18) has the base's descriptor plus off / 16 in its 14-bit address field.
    auto at = [](uint64_t base, uint32_t off) { return base + (uint64_t)(off >> 4); };
    const uint32_t aQK0 = smem_u32(sm + OFF_QK);
    const uint64_t dQK0k = smem_desc(aQK0, 16, 1024), dQK0mn = smem_desc(aQK0, 16384, 1024);
    const uint64_t dWUk = smem_desc(aWU, 16, 1024), dWUmn = smem_desc(aWU, 16384, 1024);
    const uint64_t dVmn = smem_desc(aV, 8192, 1024), dHmn = smem_desc(aH, 16384, 1024);
    const uint64_t dVTk = smem_desc(aVT, 16, 1024), dVNk = smem_desc(aVN, 16, 1024), dPk = smem_desc(aP, 16, 1024);
    auto issue_s = [&](int c) {
      const uint64_t qk = at(dQK0k, (uint32_t)(c % kQKSlots) * SZ_QK);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
        mma_bf16(tbase + TM_S, at(qk, off), at(qk, off), id_s, ks > 0);
      }
      mma_commit(smem_u32(&S.b_s));
    };
    if (nch > 0 && wt(&S.full_qk[0], 0)) {
      tc_fence_after();
      issue_s(0);
      for (int c = 0; c < nch; ++c) {
        const uint32_t ph = c & 1;
        const int slot = c % kQKSlots;
        const uint64_t qkk = at(dQK0k, (uint32_t)slot * SZ_QK), qkmn = at(dQK0mn, (uint32_t)slot * SZ_QK);
        // S of the next chunk as soon as the prep warps have read this one's
        if (c + 1 < nch) {
          if (!(wt(&S.b_sfree, ph) && wt(&S.full_qk[(c + 1) % kQKSlots], ((c + 1) / kQKSlots) & 1))) break;
          tc_fence_after();
          issue_s(c + 1);
        }
        // w^T = K^T W'^T ; vn^T = V^T U'^T
        if (!(wt(&S.b_prep, ph) && wt(&S.full_v, ph) && wt(&S.b_vnepi, ph))) break;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          mma_bf16(tbase + TM_W, at(qkmn, ks * 2048), at(dWUk, ks * 32), id_mnk, ks > 0);
          mma_bf16(tbase + TM_VN, at(dVmn, ks * 2048), at(dWUk, 8192 + ks * 32), id_mnk, ks > 0);
        }
        mma_commit(smem_u32(&S.b_w));
        mma_commit(smem_u32(&S.empty_v));
        // vn^T -= h^T w^T
        if (!(wt(&S.b_wepi, ph) && wt(&S.b_state, ph))) break;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          mma_bf16(tbase + TM_VN, at(dHmn, ks * 2048), at(dWUmn, ks * 2048), id_vn, 1);
        mma_commit(smem_u32(&S.b_vn));
        // o1^T = h^T Q^T, once the chain has read chunk c-1's output accumulators
        if (c > 0 && !wt(&S.b_oepi, (c - 1) & 1)) break;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t qoff = 8192 + (ks >> 2) * 16384 + (ks & 3) * 32;
          mma_bf16(tbase + TM_O1, at(dHmn, ks * 2048), at(qkk, qoff), id_mnk, ks > 0);
        }
        // dH = K^T vt ; o2^T = vn^T P^T
        if (!(wt(&S.b_vnepi, ph ^ 1) && wt(&S.b_pend, ph))) break;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          mma_bf16(tbase + TM_HS, at(qkmn, ks * 2048), at(dVTk, ks * 32), id_h, 1);
          mma_bf16(tbase + TM_O2, at(dVNk, ks * 32), at(dPk, ks * 32), id_kk, ks > 0);
        }
        mma_commit(smem_u32(&S.b_h));
        mma_commit(smem_u32(&S.empty_qk[slot]));
      }
    }
    // wait for every MMA issued so far before the tensor memory is released
    mma_commit(smem_u32(&S.b_final));
    mbar_wait_drain(smem_u32(&S.b_final), 0, tmo);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tbase, TM_COLS);
  if (tid == 0 && S.err) raise_status(p.status, GDR_ERR_TIMEOUT);
}

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

bool aligned16(const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

}  // namespace

int fused_make_map(CUtensorMap *m, const void *base, int64_t D, int64_t heads, int64_t tokens) {
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

int run_fused(const gdr_desc &d, const void *q, const void *k, const void *v, const float *g, const void *beta,
              const float *h0, const int64_t *cu, int Cs, int l2, void *o, float *ht, int *status,
              cudaStream_t stream) {
  if (d.dtype != GDR_BF16 || d.gate != GDR_GATE_SCALAR || d.K != DK || d.V != DV || Cs != C)
    return GDR_ERR_UNSUPPORTED;
  const int64_t tok = d.B * d.T;
  if (tok >= (int64_t)INT32_MAX) return GDR_ERR_UNSUPPORTED;  // TMA coordinates are int32
  if (d.N * d.HV > (int64_t)INT32_MAX) return GDR_ERR_UNSUPPORTED;
  if (tok > 0 && !(aligned16(q) && aligned16(k) && aligned16(v) && aligned16(o)))
    return set_error(GDR_ERR_ALIGN, "q, k, v and o must be 16-byte aligned for the fused form");
  if (d.N == 0) return GDR_OK;
  if (tok == 0) {
    // no tokens: the final state is the initial one
    if (ht) {
      const size_t bytes = sizeof(float) * d.N * d.HV * DK * DV;
      cudaError_t e = h0 ? cudaMemcpyAsync(ht, h0, bytes, cudaMemcpyDeviceToDevice, stream)
                         : cudaMemsetAsync(ht, 0, bytes, stream);
      if (e != cudaSuccess) return cuda_error(e, "final state copy");
    }
    return GDR_OK;
  }
  CUtensorMap mq, mk, mv, mo;
  int rc;
  if ((rc = fused_make_map(&mq, q, DK, d.H, tok)) != GDR_OK) return rc;
  if ((rc = fused_make_map(&mk, k, DK, d.H, tok)) != GDR_OK) return rc;
  if ((rc = fused_make_map(&mv, v, DV, d.HV, tok)) != GDR_OK) return rc;
  if ((rc = fused_make_map(&mo, o, DV, d.HV, tok)) != GDR_OK) return rc;
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
  fp.beta_logits = (d.flags & GDR_FLAG_BETA_LOGITS) ? 1 : 0;
  fp.timeout_cycles = 1ull << 32;  // about two seconds at GB300 clocks
  cudaError_t e = cudaFuncSetAttribute(gdr_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
  if (e != cudaSuccess) return cuda_error(e, "cudaFuncSetAttribute(gdr_fused_kernel)");
  gdr_fused_kernel<<<(unsigned)(d.N * d.HV), kThreads, SMEM_BYTES, stream>>>(mq, mk, mv, mo, fp);
  count_launch();
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_error(e, "gdr_fused_kernel launch");
  return GDR_OK;
}

}  // namespace gdr
