// gdr_recurrent.cu -- the per-token (fused recurrent) form of the gated delta
// rule forward, for decode and other short inputs.
//
// The coverage guide (section 三, the fused_recurrent tests with
// use_qk_l2norm_in_kernel) lists this form beside the chunked one; it is the
// recurrence itself, one token at a time:
//   S <- D_t S;  e = v_t - S^T k_t;  S <- S + beta_t k_t e^T;  o_t = S^T q_t
// with D_t = exp(g_t) (scalar gate) or Diag(exp g_t) (per-key-channel gate).
//
// Layout of the work: one block of 128 threads per (sequence, value head,
// 32-column V tile).  Column j = lane of the tile; warp w holds rows
// [w K/4, (w+1) K/4) of the state in registers, so a decode step reads and
// writes the state exactly once, coalesced.  The two reductions over K per
// token (S^T k and S^T q) combine the four warps' partial sums in shared
// memory.  The state is read from h0 at the start and written to ht at the
// end by the same block, so ht may alias h0 (in-place decode).  With the
// varlen layout, cu_seqlens is first checked by the chunk-index kernel; on a
// violation nothing is written.
//
// Pages cited: the coverage guide = "FLA 算子内核正确性测试与覆盖矩阵" (fla/ops correctness-coverage guide).
#include "gdr_device.cuh"
#include "gdr_internal.h"

namespace gdr {
namespace {

constexpr int kRThreads = 128;  // 4 warps
constexpr int kRCols = 32;      // V columns per block
constexpr int kRMaxRows = 64;   // rows per warp: K <= 256

template <typename Tin, bool PER_K, int ROWS>
__global__ void __launch_bounds__(kRThreads, ROWS <= 32 ? 8 : 4) recurrent_fwd_kernel(
    const Tin *__restrict__ q, const Tin *__restrict__ k, const Tin *__restrict__ v, const float *__restrict__ g,
    const Tin *__restrict__ beta, const float *h0, const int64_t *__restrict__ cu,
    const int64_t *__restrict__ chunk_offsets, int64_t N, int64_t T, int64_t H, int64_t HV, int64_t K, int64_t V,
    int l2, int beta_logits, Tin *__restrict__ o, float *ht) {
  __shared__ float kq[2][256];  // normalized k, q of the current token
  __shared__ float dec[256];    // exp(g) per row (per-key gate) or [0] (scalar)
  __shared__ float red[2][4][kRCols];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t unit = blockIdx.x, n = unit / HV, hv = unit % HV, hq = hv / (HV / H);
  const int64_t col = (int64_t)blockIdx.y * kRCols + lane;
  const bool colok = col < V;
  const int r0 = warp * ROWS;                     // first state row of this warp
  const int nrow = (int)(K - r0 < ROWS ? (K - r0 > 0 ? K - r0 : 0) : ROWS);  // rows < K it holds
  if (chunk_offsets && chunk_offsets[N] < 0) return;  // cu_seqlens rejected by the chunk index
  const SeqRange sr = seq_range(cu, n, T);
  const int64_t state_base = (unit * K + r0) * V + col;  // row r0 of this column

  float S[ROWS];
#pragma unroll
  for (int r = 0; r < ROWS; ++r) S[r] = (h0 && colok && r < nrow) ? h0[state_base + (int64_t)r * V] : 0.f;

  for (int64_t t = sr.bos; t < sr.eos; ++t) {
    // k, q of the token, normalized (warps 0 and 1); decay factors (warps 2, 3)
    if (warp < 2) {
      const Tin *x = (warp == 0 ? k : q) + (t * H + hq) * K;
      float r[8];
      float ss = 0.f;
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const int d = lane + 32 * m;
        r[m] = d < K ? to_f32(x[d]) : 0.f;
        ss = fmaf(r[m], r[m], ss);
      }
      const float sc = l2 ? rsqrtf(warp_sum(ss) + kL2Eps) : 1.f;
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const int d = lane + 32 * m;
        if (d < K) kq[warp][d] = r[m] * sc;
      }
    } else if (PER_K) {
      for (int d = tid - 64; d < K; d += 64) dec[d] = expf(g[(t * HV + hv) * K + d]);
    } else if (tid == 64) {
      dec[0] = expf(g[t * HV + hv]);
    }
    const float b = load_beta(beta, t * HV + hv, beta_logits);
    const float vj = colok ? to_f32(v[(t * HV + hv) * V + col]) : 0.f;
    __syncthreads();
    // S <- D S; partial S^T k  (rows past K hold zero and read zero k)
    const float *kr = kq[0] + r0, *qr = kq[1] + r0, *dr = dec + (PER_K ? r0 : 0);
    float pk = 0.f;
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
      if (r < nrow) {
        S[r] *= PER_K ? dr[r] : dr[0];
        pk = fmaf(S[r], kr[r], pk);
      }
    }
    red[0][warp][lane] = pk;
    __syncthreads();
    const float e = b * (vj - (red[0][0][lane] + red[0][1][lane] + red[0][2][lane] + red[0][3][lane]));
    // S <- S + k (b e)^T; partial S^T q
    float po = 0.f;
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
      if (r < nrow) {
        S[r] = fmaf(kr[r], e, S[r]);
        po = fmaf(S[r], qr[r], po);
      }
    }
    red[1][warp][lane] = po;
    __syncthreads();
    if (warp == 0 && colok)
      o[(t * HV + hv) * V + col] =
          from_f32<Tin>(red[1][0][lane] + red[1][1][lane] + red[1][2][lane] + red[1][3][lane]);
  }
  if (ht && colok) {
#pragma unroll
    for (int r = 0; r < ROWS; ++r)
      if (r < nrow) ht[state_base + (int64_t)r * V] = S[r];
  }
}

template <typename Tin, bool PER_K, int ROWS>
void launch_with(const ChunkedArgs &a, dim3 grid) {
  recurrent_fwd_kernel<Tin, PER_K, ROWS><<<grid, kRThreads, 0, a.stream>>>(
      (const Tin *)a.q, (const Tin *)a.k, (const Tin *)a.v, a.g, (const Tin *)a.beta, a.h0, a.cu, a.chunk_offsets,
      a.d.N, a.d.T, a.d.H, a.d.HV, a.d.K, a.d.V, a.l2, (a.d.flags & GDR_FLAG_BETA_LOGITS) ? 1 : 0, (Tin *)a.o,
      a.ht);
}

template <typename Tin, bool PER_K>
int launch_rows(const ChunkedArgs &a) {
  dim3 grid((unsigned)(a.d.N * a.d.HV), (unsigned)cdiv(a.d.V, kRCols));
  const int64_t rows = cdiv(a.d.K, 4);  // rows per warp
  if (rows <= 8) launch_with<Tin, PER_K, 8>(a, grid);
  else if (rows <= 16) launch_with<Tin, PER_K, 16>(a, grid);
  else if (rows <= 32) launch_with<Tin, PER_K, 32>(a, grid);
  else launch_with<Tin, PER_K, kRMaxRows>(a, grid);
  count_launch();
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? GDR_OK : cuda_error(e, "recurrent_fwd_kernel");
}

}  // namespace

int launch_recurrent_fwd(const ChunkedArgs &a) {
  if (a.d.N == 0) return GDR_OK;
  const bool pk = a.d.gate == GDR_GATE_PER_K;
  if (a.d.dtype == GDR_BF16) return pk ? launch_rows<__nv_bfloat16, true>(a) : launch_rows<__nv_bfloat16, false>(a);
  return pk ? launch_rows<float, true>(a) : launch_rows<float, false>(a);
}

}  // namespace gdr
