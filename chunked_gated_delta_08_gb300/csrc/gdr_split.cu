// gdr_split.cu -- the intra-sequence split of the state scan (one GPU).
//
// The KCP handbook (background and its steps 3-4) splits a sequence into
// segments that run in parallel, each from a zero state, and merges them: a
// segment's chunks map an entering state S_in to
//   S_out = M S_in + S_ext
// where S_ext is the segment's end state from S_in = 0 and M (K x K) is the
// product of the per-chunk transitions.  In the chunk form a chunk maps h to
//   h' = e^(G_L) h + Kb^T (u - w h) = (D_L - Kb^T w) h + Kb^T u,  Kb = K e^(G_L - G),
// so [S_ext | M] is the chunk recurrence run on the augmented K x (V + K)
// matrix X = [0 | I], with u taken as zero in the M columns.
//
// Three launches after the chunked prepare:
//   seg_scan_kernel<.., false>  per (segment, head, 32-column tile of V + K):
//                               X over the segment's chunks -> [S_ext | M]
//   merge_kernel                per (sequence, head, V tile), sequential over the
//                               sequence's segments: S_in(s+1) = M_s S_in(s) + S_ext,s
//   seg_scan_kernel<.., true>   per (segment, head, V tile): the plain chunk
//                               recurrence from S_in(s), writing h per chunk,
//                               v_new and, for a sequence's last segment, ht
// then the chunked fwd_o.  The sequential depth falls from a sequence's chunk
// count to one segment's chunks plus its segment count, at about three times
// the state-scan arithmetic.
//
// Pages cited: the KCP handbook = "flash-linear-attention KCP 精度失效根因排查手册".
#include "gdr_device.cuh"
#include "gdr_internal.h"
#include "gdr_scan.cuh"

namespace gdr {
namespace {

constexpr int kThreads = 256;
constexpr int kTile = 32;  // columns per block

// FINAL = false: columns [0, V + K) of X = [S_ext | M], X starting at [0 | I].
// FINAL = true:  columns [0, V) of the state, starting at S_in of the segment.
// Each chunk is one scan::chunk_step (tensor cores, 3 x TF32).
template <typename Tin, int C, bool PER_K, bool FINAL>
__global__ void __launch_bounds__(kThreads) seg_scan_kernel(
    const Tin *__restrict__ k, const float *__restrict__ w, const float *__restrict__ u,
    const float *__restrict__ gcum, const int64_t *__restrict__ cu, const int64_t *__restrict__ chunk_offsets,
    const int64_t *__restrict__ seg_indices, int S, int64_t T, int64_t H, int64_t HV, int64_t K, int64_t V,
    int l2, float *__restrict__ X, const float *__restrict__ s_in, float *__restrict__ h,
    float *__restrict__ v_new, float *__restrict__ ht) {
  extern __shared__ float smem[];
  const scan::Tiles st = scan::carve(smem, C, K);
  const int tid = threadIdx.x;
  const int64_t seg = blockIdx.x, hv = blockIdx.y, c0col = (int64_t)blockIdx.z * kTile;
  const int64_t ncol = FINAL ? V : V + K;  // width of the scanned matrix
  const int64_t hq = hv / (HV / H);
  const int64_t Kp = scan::kpad(K);
  int64_t n, s;
  if (!chunk_coords(seg_indices, seg, T, C * S, &n, &s)) return;
  const SeqRange sr = seq_range(cu, n, T);
  const int64_t nch = (sr.eos - sr.bos + C - 1) / C;
  const int64_t cbeg = s * S, cend = (cbeg + S < nch) ? cbeg + S : nch;
  const int64_t cbase = chunk_offsets ? chunk_offsets[n] : n * ((T + C - 1) / C);

  for (int64_t e = tid; e < Kp * kTile; e += kThreads) {
    const int64_t d = e / kTile, col = c0col + e % kTile;
    float x = 0.f;
    if (d < K) {
      if (FINAL) {
        if (col < V) x = s_in[((seg * HV + hv) * K + d) * V + col];
      } else if (col >= V && col < ncol) {
        x = (col - V == d) ? 1.f : 0.f;
      }
    }
    st.hs[d * scan::kHS + e % kTile] = x;
  }
  __syncthreads();

  for (int64_t c = cbeg; c < cend; ++c) {
    const int64_t t0 = sr.bos + c * C;
    const int Lc = (int)(sr.eos - t0 < (int64_t)C ? sr.eos - t0 : (int64_t)C);
    if (FINAL && h)
      for (int64_t e = tid; e < K * kTile; e += kThreads) {
        const int64_t d = e / kTile, col = c0col + e % kTile;
        if (col < V) h[(((cbase + c) * HV + hv) * K + d) * V + col] = st.hs[d * scan::kHS + e % kTile];
      }
    scan::chunk_step<Tin, C, PER_K>(st, k, w, u, gcum, t0, Lc, hv, hq, H, HV, K, V, V, c0col, l2,
                                     FINAL ? v_new : nullptr);
  }
  if (FINAL) {
    if (ht && cend == nch)
      for (int64_t e = tid; e < K * kTile; e += kThreads) {
        const int64_t d = e / kTile, col = c0col + e % kTile;
        if (col < V) ht[((n * HV + hv) * K + d) * V + col] = st.hs[d * scan::kHS + e % kTile];
      }
  } else {
    for (int64_t e = tid; e < K * kTile; e += kThreads) {
      const int64_t d = e / kTile, col = c0col + e % kTile;
      if (col < ncol) X[((seg * HV + hv) * K + d) * (V + K) + col] = st.hs[d * scan::kHS + e % kTile];
    }
  }
}

// Per (sequence, head, V tile): S_in(0) = h0; S_in(s+1) = M_s S_in(s) + S_ext,s.
// A sequence with no tokens has no segment: its ht is h0, written here.
// Thread t owns entries e = t + 256 m of the K x 32 tile; M is read from X
// (one row per warp at a time, a broadcast).  smem: st[K*32]
constexpr int kMergePer = 256 * kTile / kThreads;  // entries per thread at K = 256

__global__ void __launch_bounds__(kThreads) merge_kernel(const float *__restrict__ X, const float *__restrict__ h0,
                                                         const int64_t *__restrict__ cu,
                                                         const int64_t *__restrict__ seg_offsets, int64_t N,
                                                         int64_t T, int S, int C, int64_t HV, int64_t K, int64_t V,
                                                         float *__restrict__ s_in, float *__restrict__ ht) {
  extern __shared__ float smem[];
  float *st = smem;
  if (seg_offsets && seg_offsets[N] < 0) return;
  const int tid = threadIdx.x;
  const int64_t n = blockIdx.x, hv = blockIdx.y, v0 = (int64_t)blockIdx.z * kTile;
  const SeqRange sr = seq_range(cu, n, T);
  const int64_t seglen = (int64_t)S * C;
  const int64_t nseg = (sr.eos - sr.bos + seglen - 1) / seglen;
  const int64_t sbase = seg_offsets ? seg_offsets[n] : n * ((T + seglen - 1) / seglen);
  const int64_t ld = V + K;
  for (int64_t e = tid; e < K * kTile; e += kThreads) {
    const int64_t d = e / kTile, col = v0 + e % kTile;
    st[e] = (h0 && col < V) ? h0[((n * HV + hv) * K + d) * V + col] : 0.f;
    if (nseg == 0 && ht && col < V) ht[((n * HV + hv) * K + d) * V + col] = st[e];  // empty sequence: ht = h0
  }
  __syncthreads();
  for (int64_t s = 0; s < nseg; ++s) {
    const int64_t seg = sbase + s;
    const float *xs = X + (seg * HV + hv) * K * ld;
    float acc[kMergePer];
#pragma unroll
    for (int m = 0; m < kMergePer; ++m) {
      const int64_t e = tid + (int64_t)kThreads * m;
      acc[m] = 0.f;
      if (e < K * kTile) {
        const int64_t d = e / kTile, vv = e % kTile, col = v0 + vv;
        if (col < V) s_in[((seg * HV + hv) * K + d) * V + col] = st[e];
        float a = col < V ? xs[d * ld + col] : 0.f;
        const float *mrow = xs + d * ld + V;
        for (int64_t j = 0; j < K; ++j) a = fmaf(__ldg(mrow + j), st[j * kTile + vv], a);
        acc[m] = a;
      }
    }
    __syncthreads();
#pragma unroll
    for (int m = 0; m < kMergePer; ++m) {
      const int64_t e = tid + (int64_t)kThreads * m;
      if (e < K * kTile) st[e] = acc[m];
    }
    __syncthreads();
  }
}

template <int C_, bool PK_>
struct Cfg {
  static constexpr int C = C_;
  static constexpr bool PK = PK_;
};

template <typename F>
int dispatch(const ChunkedArgs &a, F &&f) {
  const bool pk = a.d.gate == GDR_GATE_PER_K;
  const bool bf = a.d.dtype == GDR_BF16;
  auto by_dtype = [&](auto cfg) { return bf ? f(cfg, (__nv_bfloat16 *)nullptr) : f(cfg, (float *)nullptr); };
  if (a.C == 64) return pk ? by_dtype(Cfg<64, true>{}) : by_dtype(Cfg<64, false>{});
  return pk ? by_dtype(Cfg<32, true>{}) : by_dtype(Cfg<32, false>{});
}

int after_launch(const char *name) {
  count_launch();
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? GDR_OK : cuda_error(e, name);
}

template <bool FINAL>
int launch_seg_scan(const ChunkedArgs &a, const SplitArgs &sp) {
  if (sp.nseg_max == 0) return GDR_OK;
  return dispatch(a, [&](auto cfg, auto tin) {
    using Tin = std::remove_pointer_t<decltype(tin)>;
    constexpr int C = decltype(cfg)::C;
    constexpr bool PK = decltype(cfg)::PK;
    const int64_t K = a.d.K, V = a.d.V;
    const int64_t ncol = FINAL ? V : V + K;
    const size_t smem = sizeof(float) * scan::smem_floats(C, K);
    auto kern = seg_scan_kernel<Tin, C, PK, FINAL>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return cuda_error(e, "seg_scan_kernel");
    kern<<<dim3((unsigned)sp.nseg_max, (unsigned)a.d.HV, (unsigned)cdiv(ncol, kTile)), kThreads, smem, a.stream>>>(
        (const Tin *)a.k, a.w, a.u, a.gcum, a.cu, a.chunk_offsets, sp.seg_indices, sp.S, a.d.T, a.d.H, a.d.HV, K, V,
        a.l2, sp.X, sp.s_in, a.h, a.v_new, a.ht);
    return after_launch("seg_scan_kernel");
  });
}

}  // namespace

int launch_split_transitions(const ChunkedArgs &a, const SplitArgs &sp) { return launch_seg_scan<false>(a, sp); }
int launch_split_final(const ChunkedArgs &a, const SplitArgs &sp) { return launch_seg_scan<true>(a, sp); }

int launch_split_merge(const ChunkedArgs &a, const SplitArgs &sp) {
  if (a.d.N == 0) return GDR_OK;
  const size_t smem = sizeof(float) * a.d.K * kTile;
  merge_kernel<<<dim3((unsigned)a.d.N, (unsigned)a.d.HV, (unsigned)cdiv(a.d.V, kTile)), kThreads, smem, a.stream>>>(
      sp.X, a.h0, a.cu, sp.seg_offsets, a.d.N, a.d.T, sp.S, a.C, a.d.HV, a.d.K, a.d.V, sp.s_in, a.ht);
  return after_launch("merge_kernel");
}

}  // namespace gdr
