// umma_probe.cu -- test helper: one CTA runs a chain of tcgen05 MMAs on
// operand images copied verbatim into shared memory, then reads D back from
// tensor memory.  Used by tests/test_gpu_umma_layouts.py to check the
// descriptor and layout conventions of gdr_sm100.cuh against torch.
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdr_sm100.cuh"

using namespace gdr::sm100;

struct ProbeParams {
  int M, N, a_mn, b_mn, neg_a, nk;
  uint32_t a_lbo, a_sbo, b_lbo, b_sbo;
  uint32_t a_step[16], b_step[16];
  int a_bytes, b_bytes;
};

constexpr int kRegion = 96 * 1024;

__global__ void __launch_bounds__(128) umma_probe_kernel(const uint4 *a_img, const uint4 *b_img, ProbeParams p,
                                                         float *d_out, int *err) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t mbar;
  __shared__ uint32_t tslot;
  __shared__ int s_err;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t *sm = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  uint8_t *sa = sm, *sb = sm + kRegion;
  for (int i = tid; i < p.a_bytes / 16; i += 128) reinterpret_cast<uint4 *>(sa)[i] = a_img[i];
  for (int i = tid; i < p.b_bytes / 16; i += 128) reinterpret_cast<uint4 *>(sb)[i] = b_img[i];
  if (tid == 0) {
    s_err = 0;
    mbar_init(smem_u32(&mbar), 1);
    fence_mbar_init();
  }
  fence_proxy_async_smem();
  __syncthreads();
  if (warp == 0) {
    tmem_alloc(smem_u32(&tslot), 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tslot;
  if (tid == 0) {
    const uint32_t idesc = idesc_bf16(p.M, p.N, p.a_mn, p.b_mn, p.neg_a);
    for (int ks = 0; ks < p.nk; ++ks) {
      const uint64_t da = smem_desc(smem_u32(sa) + p.a_step[ks], p.a_lbo, p.a_sbo);
      const uint64_t db = smem_desc(smem_u32(sb) + p.b_step[ks], p.b_lbo, p.b_sbo);
      mma_bf16(tbase, da, db, idesc, ks > 0 ? 1u : 0u);
    }
    mma_commit(smem_u32(&mbar));
  }
  const bool ok = mbar_wait(smem_u32(&mbar), 0, &s_err, 1000000000ull);
  tc_fence_after();
  if (ok) {
    for (int c0 = 0; c0 < p.N; c0 += 16) {
      float r[16];
      tmem_ld16(tbase + ((uint32_t)(warp * 32) << 16) + (uint32_t)c0, r);
      tmem_ld_wait();
      const int row = warp * 32 + lane;
      if (row < p.M)
        for (int j = 0; j < 16; ++j) d_out[row * p.N + c0 + j] = r[j];
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tbase, 256);
  if (tid == 0 && s_err) *err = 1;
}

extern "C" int umma_probe(const void *a_host, const void *b_host, const ProbeParams *p, float *d_host) {
  if (p->M != 128 || p->N < 16 || p->N > 256 || p->N % 16 || p->nk < 1 || p->nk > 16) return -100;
  if (p->a_bytes > kRegion || p->b_bytes > kRegion || p->a_bytes % 16 || p->b_bytes % 16) return -101;
  void *a = nullptr, *b = nullptr;
  float *d = nullptr;
  int *err = nullptr;
  int rc = 0;
  const size_t smem = 2 * kRegion + 1024;
  if (cudaMalloc(&a, p->a_bytes) || cudaMalloc(&b, p->b_bytes) || cudaMalloc((void **)&d, 128 * p->N * 4) ||
      cudaMalloc((void **)&err, 4))
    return -1;
  cudaMemcpy(a, a_host, p->a_bytes, cudaMemcpyHostToDevice);
  cudaMemcpy(b, b_host, p->b_bytes, cudaMemcpyHostToDevice);
  cudaMemset(d, 0, 128 * p->N * 4);
  cudaMemset(err, 0, 4);
  cudaFuncSetAttribute(umma_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  umma_probe_kernel<<<1, 128, smem>>>((const uint4 *)a, (const uint4 *)b, *p, d, err);
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
