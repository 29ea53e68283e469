// tmem_probe.cu -- test helper for the tensor-memory conventions of
// gdr_sm100.cuh that the fused kernel relies on beyond shared-memory operands:
//   tmem_a_probe   D = A B^T with A read from tensor memory (written there by
//                  tcgen05.st from a host image of 32-bit words per lane and
//                  column) and B from shared memory (K-major, 128-byte swizzle);
//   ld16_probe     which lane and column each register of a 16x256b.x2 load
//                  holds, from tensor memory filled with (lane, column) tags.
// One CTA of 128 threads; every wait is bounded.
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdr_sm100.cuh"

using namespace gdr::sm100;

struct TaParams {
  int N, nk;
  uint32_t b_lbo, b_sbo;
  uint32_t b_step[16];
  int b_bytes;
};

namespace {

constexpr int kRegion = 64 * 1024;
constexpr uint32_t kACol = 256;  // A image columns in tensor memory

__device__ void alloc512(uint32_t *slot) {
  if ((threadIdx.x >> 5) == 0) {
    tmem_alloc(smem_u32(slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
}

__device__ void free512(uint32_t tbase) {
  tc_fence_before();
  __syncthreads();
  if ((threadIdx.x >> 5) == 0) tmem_dealloc(tbase, 512);
}

// a_words: [128 lanes][nk * 8 columns] 32-bit words; d_out [128][N] fp32.
__global__ void __launch_bounds__(128) tmem_a_kernel(const uint32_t *a_words, const uint4 *b_img, TaParams p,
                                                     float *d_out, int *err) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t mbar;
  __shared__ uint32_t tslot;
  __shared__ int s_err;
  const int tid = threadIdx.x, warp = tid >> 5;
  uint8_t *sb = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  for (int i = tid; i < p.b_bytes / 16; i += 128) reinterpret_cast<uint4 *>(sb)[i] = b_img[i];
  if (tid == 0) {
    s_err = 0;
    mbar_init(smem_u32(&mbar), 1);
    fence_mbar_init();
  }
  fence_proxy_async_smem();
  __syncthreads();
  alloc512(&tslot);
  const uint32_t tbase = tslot, lane_addr = tbase + ((uint32_t)(warp * 32) << 16);
  const int ncol = p.nk * 8;
  for (int c0 = 0; c0 < ncol; c0 += 8) {
    uint32_t u[8];
    for (int j = 0; j < 8; ++j) u[j] = a_words[tid * ncol + c0 + j];
    tmem_st8(lane_addr + kACol + c0, u);
  }
  tmem_st_wait();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0) {
    const uint32_t idesc = idesc_bf16(128, p.N, 0, 0);
    for (int ks = 0; ks < p.nk; ++ks) {
      const uint64_t db = smem_desc(smem_u32(sb) + p.b_step[ks], p.b_lbo, p.b_sbo);
      mma_bf16_ta(tbase, tbase + kACol + 8 * ks, db, idesc, ks > 0 ? 1u : 0u);
    }
    mma_commit(smem_u32(&mbar));
  }
  const bool ok = mbar_wait(smem_u32(&mbar), 0, &s_err, 1000000000ull);
  tc_fence_after();
  if (ok) {
    for (int c0 = 0; c0 < p.N; c0 += 16) {
      float r[16];
      tmem_ld16(lane_addr + (uint32_t)c0, r);
      tmem_ld_wait();
      for (int j = 0; j < 16; ++j) d_out[tid * p.N + c0 + j] = r[j];
    }
  }
  free512(tbase);
  if (tid == 0 && s_err) *err = 1;
}

// Tensor memory lane l, column c holds the tag l * 1000 + c; each warp reads
// its lane quadrant with two 16x256b.x2 loads (lane offsets 0 and 16).
// out[warp][half][thread][reg]
__global__ void __launch_bounds__(128) ld16_kernel(float *out) {
  __shared__ uint32_t tslot;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  alloc512(&tslot);
  const uint32_t tbase = tslot;
  float v[16];
  for (int j = 0; j < 16; ++j) v[j] = (float)(tid * 1000 + j);
  tmem_st16(tbase + ((uint32_t)(warp * 32) << 16), v);
  tmem_st_wait();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  for (int half = 0; half < 2; ++half) {
    float r[8];
    tmem_ld_16x256b_x2(tbase + ((uint32_t)(warp * 32 + 16 * half) << 16), r);
    tmem_ld_wait();
    for (int j = 0; j < 8; ++j) out[((warp * 2 + half) * 32 + lane) * 8 + j] = r[j];
  }
  free512(tbase);
}

}  // namespace

extern "C" int tmem_a_probe(const uint32_t *a_words_host, const void *b_host, const TaParams *p, float *d_host) {
  if (p->N < 16 || p->N > 256 || p->N % 16 || p->nk < 1 || p->nk > 16) return -100;
  if (p->b_bytes > kRegion || p->b_bytes % 16) return -101;
  const size_t a_bytes = sizeof(uint32_t) * 128 * p->nk * 8;
  void *a = nullptr, *b = nullptr;
  float *d = nullptr;
  int *err = nullptr;
  int rc = 0;
  if (cudaMalloc(&a, a_bytes) || cudaMalloc(&b, p->b_bytes) || cudaMalloc((void **)&d, 128 * p->N * 4) ||
      cudaMalloc((void **)&err, 4))
    return -1;
  cudaMemcpy(a, a_words_host, a_bytes, cudaMemcpyHostToDevice);
  cudaMemcpy(b, b_host, p->b_bytes, cudaMemcpyHostToDevice);
  cudaMemset(d, 0, 128 * p->N * 4);
  cudaMemset(err, 0, 4);
  const size_t smem = kRegion + 1024;
  cudaFuncSetAttribute(tmem_a_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  tmem_a_kernel<<<1, 128, smem>>>((const uint32_t *)a, (const uint4 *)b, *p, d, err);
  if (cudaDeviceSynchronize() != cudaSuccess) rc = -2;
  int herr = 0;
  cudaMemcpy(&herr, err, 4, cudaMemcpyDeviceToHost);
  if (herr) rc = -3;
  cudaMemcpy(d_host, d, 128 * p->N * 4, cudaMemcpyDeviceToHost);
  cudaFree(a);
  cudaFree(b);
  cudaFree(d);
  cudaFree(err);
  return rc;
}

extern "C" int ld16_probe(float *out_host) {
  float *d = nullptr;
  const size_t bytes = sizeof(float) * 4 * 2 * 32 * 8;
  if (cudaMalloc((void **)&d, bytes)) return -1;
  cudaMemset(d, 0, bytes);
  ld16_kernel<<<1, 128>>>(d);
  int rc = cudaDeviceSynchronize() == cudaSuccess ? 0 : -2;
  cudaMemcpy(out_host, d, bytes, cudaMemcpyDeviceToHost);
  cudaFree(d);
  return rc;
}
