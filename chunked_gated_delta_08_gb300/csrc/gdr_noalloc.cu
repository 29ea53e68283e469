// gdr_noalloc.cu -- the chunked forward with its scratch in a fixed device
// array, for callers that must not allocate device memory.
//
// Some callers cannot call cudaMalloc or take memory from an allocator: code
// that runs under a framework whose allocator owns every byte of the device
// (and would be bypassed), code that runs where allocation calls are not
// allowed or would synchronize the device, and embedded or real-time callers
// that must not allocate after start-up.  gdr_fwd_noalloc serves them: it
// runs the same chunked kernels as gdr_fwd with GDR_ALGO_CHUNKED, but its
// scratch (chunk map, gate cumsum, w, u, v_new, per-chunk states) lives in
// the array below, which every GPU that loads the library holds until the
// process exits.
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "gdr.h"
#include "gdr_internal.h"

namespace gdr {
namespace {

constexpr size_t kScratchBytes = size_t(64) << 20;  // GDR_NOALLOC_SCRATCH_BYTES in gdr.h
static_assert(kScratchBytes == GDR_NOALLOC_SCRATCH_BYTES, "scratch size and header disagree");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of the array on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device, with that device current, and cached.
int scratch_address(void **out) {
  int dev;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_error(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return set_error(GDR_ERR_CUDA, "device ordinal out of range");
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_addr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_error(e, "cudaGetSymbolAddress(no-allocation scratch)");
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return GDR_OK;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace
}  // namespace gdr

using namespace gdr;

extern "C" int gdr_fwd_noalloc(const gdr_desc *desc, const void *q, const void *k, const void *v, const float *g,
                               const void *beta, const float *h0, const int64_t *cu_seqlens, int chunk_size,
                               int use_qk_l2norm, void *o, float *ht, void *stream) {
  int rc = validate_request(desc, chunk_size, cu_seqlens);
  if (rc != GDR_OK) return rc;
  const gdr_desc &d = *desc;
  if (d.B * d.T > 0 && (!q || !k || !v || !g || !beta || !o))
    return set_error(GDR_ERR_NULLPTR, "q, k, v, g, beta and o must be non-NULL");
  gdr_chunked_sizes s;
  chunked_scratch_sizes(d, chunk_size, cu_seqlens, &s);
  const size_t parts[7] = {cu_seqlens ? align256(s.chunk_indices_bytes) : 0,
                           cu_seqlens ? align256(s.chunk_offsets_bytes) : 0,
                           align256(s.gcum_bytes),
                           align256(s.w_bytes),
                           align256(s.u_bytes),
                           align256(s.v_new_bytes),
                           align256(s.h_bytes)};
  size_t total = 0;
  for (size_t x : parts) total += x;
  if (total > kScratchBytes)
    return set_error(GDR_ERR_SHAPE, "gdr_fwd_noalloc: this problem needs " + std::to_string(total) +
                                        " bytes of scratch; the fixed array holds " +
                                        std::to_string(kScratchBytes));
  void *base = nullptr;
  if ((rc = scratch_address(&base)) != GDR_OK) return rc;
  char *p = static_cast<char *>(base);
  ChunkedArgs a{};
  a.d = d;
  a.C = chunk_size;
  a.l2 = use_qk_l2norm ? 1 : 0;
  a.q = q;
  a.k = k;
  a.v = v;
  a.beta = beta;
  a.g = g;
  a.h0 = h0;
  a.cu = cu_seqlens;
  a.chunk_indices = cu_seqlens ? (int64_t *)p : nullptr;
  p += parts[0];
  a.chunk_offsets = cu_seqlens ? (int64_t *)p : nullptr;
  p += parts[1];
  a.gcum = (float *)p;
  p += parts[2];
  a.w = (float *)p;
  p += parts[3];
  a.u = (float *)p;
  p += parts[4];
  a.v_new = (float *)p;
  p += parts[5];
  a.h = (float *)p;
  a.ht = ht;
  a.o = o;
  a.nt_max = s.nt_max;
  a.status = nullptr;  // nothing is allocated, not even a status word
  a.stream = (cudaStream_t)stream;
  if (cu_seqlens) rc = launch_chunk_index(a);
  if (rc == GDR_OK) rc = launch_chunk_prepare(a);
  if (rc == GDR_OK) rc = launch_chunk_fwd_h(a);
  if (rc == GDR_OK) rc = launch_chunk_fwd_o(a);
  return rc;
}
