// gdr_device.cuh -- small device helpers shared by the kernels of libgdr.so.
//
// Pages cited: the coverage guide = "FLA 算子内核正确性测试与覆盖矩阵" (fla/ops correctness-coverage guide).
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace gdr {

// Element conversions for the two input dtypes.
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// L2-norm reading: x / sqrt(sum x^2 + 1e-6), per token and head.
constexpr float kL2Eps = 1e-6f;

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Token range [bos, eos) of sequence n: the varlen layout reads cu_seqlens,
// the dense layout is n*T .. (n+1)*T.  int64 throughout.
struct SeqRange {
  int64_t bos, eos;
};
__device__ __forceinline__ SeqRange seq_range(const int64_t *cu, int64_t n, int64_t T) {
  if (cu) return {cu[n], cu[n + 1]};
  return {n * T, (n + 1) * T};
}

// The sequence a state-scan block takes: blocks are launched in order of rank,
// and rank r is the r-th longest sequence (ties by index), so the longest
// scans start in the first wave instead of waiting for slots behind shorter
// ones.  Ranks are computed in the block for up to kRankedSeqs sequences (one
// thread per sequence counts the longer ones); beyond that, and in the dense
// layout (all sequences equal), rank r is sequence r.  Called by every thread
// of the block (it synchronizes).
constexpr int kRankedSeqs = 256;
__device__ __forceinline__ int64_t seq_of_rank(const int64_t *cu, int64_t N, int64_t r) {
  if (!cu || N > kRankedSeqs || N > (int64_t)blockDim.x) return r;
  __shared__ long long picked;
  if (threadIdx.x == 0) picked = r;
  __syncthreads();
  if ((int64_t)threadIdx.x < N) {
    const int64_t n = threadIdx.x, len = cu[n + 1] - cu[n];
    int64_t rank = 0;
    for (int64_t m = 0; m < N; ++m) {
      const int64_t lm = cu[m + 1] - cu[m];
      rank += (lm > len || (lm == len && m < n)) ? 1 : 0;
    }
    if (rank == r) picked = n;
  }
  __syncthreads();
  return picked;
}

// Maps a chunk row to (sequence, chunk-in-sequence); false if the row is unused.
__device__ __forceinline__ bool chunk_coords(const int64_t *chunk_indices, int64_t chunk, int64_t T, int C,
                                             int64_t *n, int64_t *j) {
  if (chunk_indices) {
    *n = chunk_indices[2 * chunk];
    *j = chunk_indices[2 * chunk + 1];
    return *n >= 0;
  }
  const int64_t ncs = (T + C - 1) / C;
  *n = chunk / ncs;
  *j = chunk % ncs;
  return true;
}

// beta as stored, or the logistic sigmoid of a stored logit (the "raw beta"
// input of the coverage guide, section 三).
template <typename Tin>
__device__ __forceinline__ float load_beta(const Tin *beta, int64_t idx, int logits) {
  const float x = to_f32(beta[idx]);
  return logits ? 1.f / (1.f + expf(-x)) : x;
}

// Records the first problem seen by any kernel into the status word.
__device__ __forceinline__ void raise_status(int *status, int code) {
  if (status) atomicCAS(status, 0, code);
}

}  // namespace gdr
