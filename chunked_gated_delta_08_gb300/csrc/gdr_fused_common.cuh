// gdr_fused_common.cuh -- helpers of the fused tensor-core kernel: bf16
// packing, 128-byte-swizzled shared-memory tiles, and TMA descriptor setup.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace gdr {
namespace fused {

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ uint4 pack8(const float *x) {
  return make_uint4(pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]), pack_bf16(x[4], x[5]), pack_bf16(x[6], x[7]));
}

// 16-byte chunk `chunk` (8 bf16) of row `row` of a 128-byte-swizzled tile
// (rows of 128 bytes, 8-row atoms of 1024 bytes, chunk index XOR row % 8).
__device__ __forceinline__ uint32_t sw128_chunk_off(uint32_t row, uint32_t chunk) {
  return (row >> 3) * 1024u + (row & 7u) * 128u + ((chunk ^ (row & 7u)) << 4);
}
__device__ __forceinline__ void st_sw128_chunk(uint8_t *tile, uint32_t row, uint32_t chunk, uint4 val) {
  *reinterpret_cast<uint4 *>(tile + sw128_chunk_off(row, chunk)) = val;
}
__device__ __forceinline__ uint4 ld_sw128_chunk(const uint8_t *tile, uint32_t row, uint32_t chunk) {
  return *reinterpret_cast<const uint4 *>(tile + sw128_chunk_off(row, chunk));
}

// Batched vector loads of 8 / 16 / 32 consecutive floats (16-byte aligned).
__device__ __forceinline__ void ld_f32x8(const float *src, float (&d)[8]) {
  const float4 a = reinterpret_cast<const float4 *>(src)[0], b = reinterpret_cast<const float4 *>(src)[1];
  d[0] = a.x;
  d[1] = a.y;
  d[2] = a.z;
  d[3] = a.w;
  d[4] = b.x;
  d[5] = b.y;
  d[6] = b.z;
  d[7] = b.w;
}
__device__ __forceinline__ void ld_f32x16(const float *src, float (&d)[16]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float4 v = reinterpret_cast<const float4 *>(src)[q];
    d[4 * q] = v.x;
    d[4 * q + 1] = v.y;
    d[4 * q + 2] = v.z;
    d[4 * q + 3] = v.w;
  }
}
__device__ __forceinline__ void ld_f32x32(const float *src, float (&d)[32]) {
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const float4 v = reinterpret_cast<const float4 *>(src)[q];
    d[4 * q] = v.x;
    d[4 * q + 1] = v.y;
    d[4 * q + 2] = v.z;
    d[4 * q + 3] = v.w;
  }
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

}  // namespace fused

// 3-D TMA map over a [tokens, heads, D] bf16 tensor with 64 (D) x 1 x 64
// (tokens) boxes in the 128-byte swizzle.  Returns GDR_OK or an error code.
int fused_make_map(CUtensorMap *m, const void *base, int64_t D, int64_t heads, int64_t tokens);

}  // namespace gdr
