// gdr_api.cu -- the C ABI of libgdr.so: argument validation, scratch
// management, dispatch between the fused and the chunked forms, and the
// error / status reporting.  See include/gdr.h for the contract.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdio>
#include <mutex>
#include <string>

#include "gdr.h"
#include "gdr_internal.h"

namespace gdr {

static thread_local std::string g_last_error;
static std::atomic<int64_t> g_launches{0};

void count_launch(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

int set_error(int code, const std::string &msg) {
  g_last_error = msg;
  return code;
}

int cuda_error(cudaError_t e, const char *what) {
  return set_error(GDR_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int *g_status[kMaxDevices] = {};
cudaMemPool_t g_pool[kMaxDevices] = {};

int current_device(int *dev) {
  cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return cuda_error(e, "cudaGetDevice");
  if (*dev < 0 || *dev >= kMaxDevices) return set_error(GDR_ERR_CUDA, "device ordinal out of range");
  return GDR_OK;
}

// A library-owned stream-ordered pool that keeps its memory between calls.
int scratch_pool(int dev, cudaMemPool_t *out) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_pool[dev]) {
    cudaMemPoolProps props = {};
    props.allocType = cudaMemAllocationTypePinned;
    props.handleTypes = cudaMemHandleTypeNone;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t pool;
    cudaError_t e = cudaMemPoolCreate(&pool, &props);
    if (e != cudaSuccess) return cuda_error(e, "cudaMemPoolCreate");
    uint64_t keep = UINT64_MAX;
    e = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
    if (e != cudaSuccess) return cuda_error(e, "cudaMemPoolSetAttribute");
    g_pool[dev] = pool;
  }
  *out = g_pool[dev];
  return GDR_OK;
}

int validate(const gdr_desc *d, int chunk_size, const int64_t *cu) {
  if (!d) return set_error(GDR_ERR_NULLPTR, "desc is NULL");
  if (chunk_size != 32 && chunk_size != 64)
    return set_error(GDR_ERR_CHUNK_SIZE, "chunk_size must be either 32 or 64");
  if (d->dtype != GDR_F32 && d->dtype != GDR_BF16) return set_error(GDR_ERR_DTYPE, "dtype must be GDR_F32 or GDR_BF16");
  if (d->gate != GDR_GATE_SCALAR && d->gate != GDR_GATE_PER_K)
    return set_error(GDR_ERR_DTYPE, "gate must be GDR_GATE_SCALAR or GDR_GATE_PER_K");
  if (d->algo < GDR_ALGO_AUTO || d->algo > GDR_ALGO_SPLIT) return set_error(GDR_ERR_DTYPE, "unknown algo");
  if (d->flags & ~GDR_FLAG_BETA_LOGITS) return set_error(GDR_ERR_DTYPE, "unknown bits in flags");
  if (d->B < 0 || d->T < 0) return set_error(GDR_ERR_SHAPE, "B and T must be >= 0");
  if (d->H <= 0 || d->HV <= 0) return set_error(GDR_ERR_SHAPE, "H and HV must be >= 1");
  if (d->HV % d->H != 0) return set_error(GDR_ERR_SHAPE, "HV must be a multiple of H");
  if (d->K < 1 || d->K > 256 || d->V < 1 || d->V > 256) return set_error(GDR_ERR_SHAPE, "K and V must be in [1, 256]");
  if (d->HV > 65535) return set_error(GDR_ERR_SHAPE, "HV must be <= 65535");
  if (cu) {
    if (d->B != 1) return set_error(GDR_ERR_SHAPE, "cu_seqlens requires B == 1");
    if (d->N < 0) return set_error(GDR_ERR_SHAPE, "N must be >= 0");
  } else if (d->N != d->B) {
    return set_error(GDR_ERR_SHAPE, "N must equal B when cu_seqlens is NULL");
  }
  return GDR_OK;
}

int64_t nt_max_of(const gdr_desc &d, int C, const int64_t *cu) {
  return cu ? nt_upper_bound(d, C) : d.B * cdiv(d.T, C);
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

void sizes_of(const gdr_desc &d, int C, const int64_t *cu, gdr_chunked_sizes *s) {
  const int64_t tok = d.B * d.T;
  s->nt_max = nt_max_of(d, C, cu);
  s->chunk_indices_bytes = sizeof(int64_t) * 2 * (size_t)s->nt_max;
  s->chunk_offsets_bytes = sizeof(int64_t) * (size_t)(d.N + 1);
  s->gcum_bytes = sizeof(float) * (size_t)(tok * d.HV * (d.gate == GDR_GATE_PER_K ? d.K : 1));
  s->w_bytes = sizeof(float) * (size_t)(tok * d.HV * d.K);
  s->u_bytes = sizeof(float) * (size_t)(tok * d.HV * d.V);
  s->v_new_bytes = s->u_bytes;
  s->h_bytes = sizeof(float) * (size_t)(s->nt_max * d.HV * d.K * d.V);
}

// Whether prepare may form k e^{G_L - G} for the state scan: only where prepare's q/k row loader and
// the scan's row loader both take their vector forms (K % 4 == 0, K <= 128, k 16-byte aligned), so
// the formed rows equal the ones the scan would form, bit for bit.
bool kb_formable(const gdr_desc &d, const void *k) {
  return d.K % 4 == 0 && d.K <= 128 && (reinterpret_cast<uintptr_t>(k) & 15u) == 0;
}

int run_chunked(const gdr_desc &d, const void *q, const void *k, const void *v, const float *g, const void *beta,
                const float *h0, const int64_t *cu, int C, int l2, void *o, float *ht, cudaStream_t stream) {
  int dev, rc;
  if ((rc = current_device(&dev)) != GDR_OK) return rc;
  int *status = device_status_word(dev, &rc);
  if (!status) return rc;
  cudaMemPool_t pool;
  if ((rc = scratch_pool(dev, &pool)) != GDR_OK) return rc;
  gdr_chunked_sizes s;
  sizes_of(d, C, cu, &s);
  const size_t offs[7] = {0,
                          align256(s.chunk_indices_bytes),
                          align256(s.chunk_offsets_bytes),
                          align256(s.gcum_bytes),
                          align256(s.w_bytes),
                          align256(s.u_bytes),
                          align256(s.v_new_bytes)};
  // k e^{G_L - G} formed once by prepare for the state scan, where both take their vector row loaders
  const bool formed_kb = kb_formable(d, k);
  size_t total = align256(s.h_bytes) + (formed_kb ? align256(s.w_bytes) : 0);
  for (size_t x : offs) total += x;
  char *base = nullptr;
  cudaError_t e = cudaMallocFromPoolAsync((void **)&base, total > 0 ? total : 256, pool, stream);
  if (e != cudaSuccess) return cuda_error(e, "cudaMallocFromPoolAsync (chunked scratch)");
  char *p = base;
  ChunkedArgs a{};
  a.d = d;
  a.C = C;
  a.l2 = l2;
  a.q = q; a.k = k; a.v = v; a.beta = beta; a.g = g; a.h0 = h0; a.cu = cu;
  a.chunk_indices = cu ? (int64_t *)p : nullptr; p += offs[1];
  a.chunk_offsets = cu ? (int64_t *)p : nullptr; p += offs[2];
  a.gcum = (float *)p; p += offs[3];
  a.w = (float *)p; p += offs[4];
  a.u = (float *)p; p += offs[5];
  a.v_new = (float *)p; p += offs[6];
  a.h = (float *)p; p += align256(s.h_bytes);
  a.kb = formed_kb ? (float *)p : nullptr;
  a.ht = ht;
  a.o = o;
  a.nt_max = s.nt_max;
  a.status = status;
  a.stream = stream;
  if (cu) rc = launch_chunk_index(a);
  if (rc == GDR_OK) rc = launch_chunk_prepare(a);
  if (rc == GDR_OK) rc = launch_chunk_fwd_h(a);
  if (rc == GDR_OK) rc = launch_chunk_fwd_o(a);
  e = cudaFreeAsync(base, stream);
  if (rc == GDR_OK && e != cudaSuccess) rc = cuda_error(e, "cudaFreeAsync (chunked scratch)");
  return rc;
}

// The chunked form with the state scan split into segments of kSplitTokens
// tokens: prepare, segment transitions, merge, segment rescans, fwd_o.
constexpr int kSplitTokens = 1024;

int run_split(const gdr_desc &d, const void *q, const void *k, const void *v, const float *g, const void *beta,
              const float *h0, const int64_t *cu, int C, int l2, void *o, float *ht, cudaStream_t stream) {
  int dev, rc;
  if ((rc = current_device(&dev)) != GDR_OK) return rc;
  int *status = device_status_word(dev, &rc);
  if (!status) return rc;
  cudaMemPool_t pool;
  if ((rc = scratch_pool(dev, &pool)) != GDR_OK) return rc;
  gdr_chunked_sizes s;
  sizes_of(d, C, cu, &s);
  const int S = kSplitTokens / C;
  const int64_t nseg_max = nt_max_of(d, S * C, cu);
  const size_t sz[10] = {s.chunk_indices_bytes, s.chunk_offsets_bytes, s.gcum_bytes, s.w_bytes, s.u_bytes,
                         s.v_new_bytes, s.h_bytes, sizeof(int64_t) * 2 * (size_t)nseg_max,
                         sizeof(int64_t) * (size_t)(d.N + 1), 0};
  const size_t x_bytes = sizeof(float) * (size_t)(nseg_max * d.HV * d.K * (d.V + d.K));
  const size_t sin_bytes = sizeof(float) * (size_t)(nseg_max * d.HV * d.K * d.V);
  size_t total = align256(x_bytes) + align256(sin_bytes);
  for (size_t x : sz) total += align256(x);
  char *base = nullptr;
  cudaError_t e = cudaMallocFromPoolAsync((void **)&base, total > 0 ? total : 256, pool, stream);
  if (e != cudaSuccess) return cuda_error(e, "cudaMallocFromPoolAsync (split scratch)");
  char *ptr[9];
  char *p = base;
  for (int i = 0; i < 9; ++i) {
    ptr[i] = p;
    p += align256(sz[i]);
  }
  ChunkedArgs a{};
  a.d = d;
  a.C = C;
  a.l2 = l2;
  a.q = q; a.k = k; a.v = v; a.beta = beta; a.g = g; a.h0 = h0; a.cu = cu;
  a.chunk_indices = cu ? (int64_t *)ptr[0] : nullptr;
  a.chunk_offsets = cu ? (int64_t *)ptr[1] : nullptr;
  a.gcum = (float *)ptr[2];
  a.w = (float *)ptr[3];
  a.u = (float *)ptr[4];
  a.v_new = (float *)ptr[5];
  a.h = (float *)ptr[6];
  a.ht = ht;
  a.o = o;
  a.nt_max = s.nt_max;
  a.status = status;
  a.stream = stream;
  SplitArgs sp{};
  sp.S = S;
  sp.nseg_max = nseg_max;
  sp.seg_indices = cu ? (int64_t *)ptr[7] : nullptr;
  sp.seg_offsets = cu ? (int64_t *)ptr[8] : nullptr;
  sp.X = (float *)p;
  sp.s_in = (float *)(p + align256(x_bytes));
  if (cu) {
    rc = launch_chunk_index(a);
    if (rc == GDR_OK) {  // the same index over segments (chunks of S*C tokens)
      ChunkedArgs sa = a;
      sa.C = S * C;
      sa.nt_max = nseg_max;
      sa.chunk_indices = sp.seg_indices;
      sa.chunk_offsets = sp.seg_offsets;
      rc = launch_chunk_index(sa);
    }
  }
  if (rc == GDR_OK) rc = launch_chunk_prepare(a);
  if (rc == GDR_OK) rc = launch_split_transitions(a, sp);
  if (rc == GDR_OK) rc = launch_split_merge(a, sp);
  if (rc == GDR_OK) rc = launch_split_final(a, sp);
  if (rc == GDR_OK) rc = launch_chunk_fwd_o(a);
  e = cudaFreeAsync(base, stream);
  if (rc == GDR_OK && e != cudaSuccess) rc = cuda_error(e, "cudaFreeAsync (split scratch)");
  return rc;
}

// The per-token form; the varlen layout first runs the chunk index to
// validate cu_seqlens (its offsets are the only scratch).
int run_recurrent(const gdr_desc &d, const void *q, const void *k, const void *v, const float *g, const void *beta,
                  const float *h0, const int64_t *cu, int C, int l2, void *o, float *ht, cudaStream_t stream) {
  int dev, rc;
  if ((rc = current_device(&dev)) != GDR_OK) return rc;
  int *status = device_status_word(dev, &rc);
  if (!status) return rc;
  ChunkedArgs a{};
  a.d = d;
  a.C = C;
  a.l2 = l2;
  a.q = q; a.k = k; a.v = v; a.beta = beta; a.g = g; a.h0 = h0; a.cu = cu;
  a.o = o;
  a.ht = ht;
  a.status = status;
  a.stream = stream;
  char *base = nullptr;
  if (cu) {
    cudaMemPool_t pool;
    if ((rc = scratch_pool(dev, &pool)) != GDR_OK) return rc;
    cudaError_t e = cudaMallocFromPoolAsync((void **)&base, sizeof(int64_t) * (size_t)(d.N + 1), pool, stream);
    if (e != cudaSuccess) return cuda_error(e, "cudaMallocFromPoolAsync (recurrent scratch)");
    a.chunk_offsets = (int64_t *)base;
    a.nt_max = 0;
    rc = launch_chunk_index(a);
  }
  if (rc == GDR_OK) rc = launch_recurrent_fwd(a);
  if (base) {
    cudaError_t e = cudaFreeAsync(base, stream);
    if (rc == GDR_OK && e != cudaSuccess) rc = cuda_error(e, "cudaFreeAsync (recurrent scratch)");
  }
  return rc;
}

// The backward: the forward recompute (chunk index, prepare, fwd_h) into
// pool scratch, then the five backward kernels.
int run_bwd(const gdr_desc &d, const void *q, const void *k, const void *v, const float *g, const void *beta,
            const float *h0, const int64_t *cu, int C, int l2, const void *d_o, const float *dht, void *dq,
            void *dk, void *dv, float *dg, void *dbeta, float *dh0, cudaStream_t stream) {
  int dev, rc;
  if ((rc = current_device(&dev)) != GDR_OK) return rc;
  int *status = device_status_word(dev, &rc);
  if (!status) return rc;
  cudaMemPool_t pool;
  if ((rc = scratch_pool(dev, &pool)) != GDR_OK) return rc;
  gdr_chunked_sizes s;
  sizes_of(d, C, cu, &s);
  // forward: chunk maps, gcum, w, u, v_new, h; backward: dvn, dhc, dqa, dka, dga, dW
  const size_t sz[13] = {s.chunk_indices_bytes, s.chunk_offsets_bytes, s.gcum_bytes, s.w_bytes, s.u_bytes,
                         s.v_new_bytes, s.h_bytes, s.u_bytes, s.h_bytes, s.w_bytes, s.w_bytes, s.gcum_bytes,
                         s.w_bytes};
  size_t total = 0;
  for (size_t x : sz) total += align256(x);
  char *base = nullptr;
  cudaError_t e = cudaMallocFromPoolAsync((void **)&base, total > 0 ? total : 256, pool, stream);
  if (e != cudaSuccess) return cuda_error(e, "cudaMallocFromPoolAsync (backward scratch)");
  char *ptr[13];
  char *p = base;
  for (int i = 0; i < 13; ++i) {
    ptr[i] = p;
    p += align256(sz[i]);
  }
  BwdArgs b{};
  ChunkedArgs &a = b.f;
  a.d = d;
  a.C = C;
  a.l2 = l2;
  a.q = q; a.k = k; a.v = v; a.beta = beta; a.g = g; a.h0 = h0; a.cu = cu;
  a.chunk_indices = cu ? (int64_t *)ptr[0] : nullptr;
  a.chunk_offsets = cu ? (int64_t *)ptr[1] : nullptr;
  a.gcum = (float *)ptr[2];
  a.w = (float *)ptr[3];
  a.u = (float *)ptr[4];
  a.v_new = (float *)ptr[5];
  a.h = (float *)ptr[6];
  a.ht = nullptr;
  a.o = nullptr;
  a.nt_max = s.nt_max;
  a.status = status;
  a.stream = stream;
  b.d_o = d_o;
  b.dht = dht;
  b.dvn = (float *)ptr[7];
  b.dhc = (float *)ptr[8];
  b.dqa = (float *)ptr[9];
  b.dka = (float *)ptr[10];
  b.dga = (float *)ptr[11];
  b.dW = (float *)ptr[12];
  b.dq = dq; b.dk = dk; b.dv = dv; b.dbeta = dbeta; b.dg = dg; b.dh0 = dh0;
  a.kb = kb_formable(d, k) ? b.dka : nullptr;  // free until dqkg; the reverse scan reads these rows too
  if (cu) rc = launch_chunk_index(a);
  if (rc == GDR_OK) rc = launch_chunk_prepare(a);
  if (rc == GDR_OK) rc = launch_chunk_fwd_h(a);
  if (rc == GDR_OK) rc = launch_bwd_dv_local(b);
  if (rc == GDR_OK) rc = launch_bwd_dh(b);
  if (rc == GDR_OK) rc = launch_bwd_dqkg(b);
  if (rc == GDR_OK) rc = launch_bwd_wy(b);
  if (rc == GDR_OK) rc = launch_bwd_finalize(b);
  e = cudaFreeAsync(base, stream);
  if (rc == GDR_OK && e != cudaSuccess) rc = cuda_error(e, "cudaFreeAsync (backward scratch)");
  return rc;
}

}  // namespace

int validate_request(const gdr_desc *d, int chunk_size, const int64_t *cu) { return validate(d, chunk_size, cu); }

void chunked_scratch_sizes(const gdr_desc &d, int C, const int64_t *cu, gdr_chunked_sizes *s) {
  sizes_of(d, C, cu, s);
}

int *device_status_word(int dev, int *err) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_status[dev]) {
    int *p = nullptr;
    cudaError_t e = cudaMalloc((void **)&p, sizeof(int));
    if (e == cudaSuccess) e = cudaMemset(p, 0, sizeof(int));
    if (e != cudaSuccess) {
      *err = cuda_error(e, "status word allocation");
      return nullptr;
    }
    g_status[dev] = p;
  }
  *err = GDR_OK;
  return g_status[dev];
}

// Implemented in gdr_fused.cu: returns GDR_ERR_UNSUPPORTED (without setting the
// message) when the fused form does not cover the request.
int run_fused(const gdr_desc &d, const void *q, const void *k, const void *v, const float *g, const void *beta,
              const float *h0, const int64_t *cu, int C, int l2, void *o, float *ht, int *status,
              cudaStream_t stream);

}  // namespace gdr

using namespace gdr;

extern "C" {

int gdr_fwd(const gdr_desc *desc, const void *q, const void *k, const void *v, const float *g, const void *beta,
            const float *h0, const int64_t *cu_seqlens, int chunk_size, int use_qk_l2norm, void *o, float *ht,
            void *stream) {
  int rc = validate(desc, chunk_size, cu_seqlens);
  if (rc != GDR_OK) return rc;
  const gdr_desc &d = *desc;
  const int64_t tok = d.B * d.T;
  if (tok > 0 && (!q || !k || !v || !g || !beta || !o))
    return set_error(GDR_ERR_NULLPTR, "q, k, v, g, beta and o must be non-NULL");
  const int l2 = use_qk_l2norm ? 1 : 0;
  cudaStream_t s = (cudaStream_t)stream;
  if (d.algo == GDR_ALGO_RECURRENT || (d.algo == GDR_ALGO_AUTO && !cu_seqlens && d.T <= 16))
    return run_recurrent(d, q, k, v, g, beta, h0, cu_seqlens, chunk_size, l2, o, ht, s);
  if (d.algo == GDR_ALGO_SPLIT) return run_split(d, q, k, v, g, beta, h0, cu_seqlens, chunk_size, l2, o, ht, s);
  if (d.algo != GDR_ALGO_CHUNKED) {
    int dev;
    if ((rc = current_device(&dev)) != GDR_OK) return rc;
    int *status = device_status_word(dev, &rc);
    if (!status) return rc;
    rc = run_fused(d, q, k, v, g, beta, h0, cu_seqlens, chunk_size, l2, o, ht, status, s);
    if (rc != GDR_ERR_UNSUPPORTED || d.algo == GDR_ALGO_FUSED) {
      if (rc == GDR_ERR_UNSUPPORTED) set_error(rc, "the fused form does not support this request");
      return rc;
    }
    // dense, long, and too few state-scan blocks to fill the GPU: split the scan
    if (!cu_seqlens && d.T >= 4 * kSplitTokens && d.N * d.HV * cdiv(d.V, 32) < 152)
      return run_split(d, q, k, v, g, beta, h0, cu_seqlens, chunk_size, l2, o, ht, s);
  }
  return run_chunked(d, q, k, v, g, beta, h0, cu_seqlens, chunk_size, l2, o, ht, s);
}

int gdr_bwd(const gdr_desc *desc, const void *q, const void *k, const void *v, const float *g, const void *beta,
            const float *h0, const int64_t *cu_seqlens, int chunk_size, int use_qk_l2norm, const void *d_o,
            const float *dht, void *dq, void *dk, void *dv, float *dg, void *dbeta, float *dh0, void *stream) {
  int rc = validate(desc, chunk_size, cu_seqlens);
  if (rc != GDR_OK) return rc;
  const gdr_desc &d = *desc;
  if (d.K > 128) return set_error(GDR_ERR_SHAPE, "gdr_bwd supports K <= 128");
  const int64_t tok = d.B * d.T;
  if (tok > 0 && (!q || !k || !v || !g || !beta || !d_o || !dq || !dk || !dv || !dg || !dbeta))
    return set_error(GDR_ERR_NULLPTR, "q, k, v, g, beta, d_o, dq, dk, dv, dg and dbeta must be non-NULL");
  return run_bwd(d, q, k, v, g, beta, h0, cu_seqlens, chunk_size, use_qk_l2norm ? 1 : 0, d_o, dht, dq, dk, dv, dg,
                 dbeta, dh0, (cudaStream_t)stream);
}

int gdr_chunked_sizes_get(const gdr_desc *desc, int chunk_size, int varlen, gdr_chunked_sizes *out) {
  if (!out) return set_error(GDR_ERR_NULLPTR, "out is NULL");
  // any non-NULL pointer selects the varlen checks and bound; it is never read
  static const int64_t marker = 0;
  const int64_t *cu = varlen ? &marker : nullptr;
  int rc = validate(desc, chunk_size, cu);
  if (rc != GDR_OK) return rc;
  sizes_of(*desc, chunk_size, cu, out);
  return GDR_OK;
}

static int stage_prologue(const gdr_desc *desc, int chunk_size, const int64_t *cu, ChunkedArgs *a, void *stream) {
  int rc = validate(desc, chunk_size, cu);
  if (rc != GDR_OK) return rc;
  int dev;
  if ((rc = current_device(&dev)) != GDR_OK) return rc;
  a->status = device_status_word(dev, &rc);
  if (!a->status) return rc;
  a->d = *desc;
  a->C = chunk_size;
  a->cu = cu;
  a->nt_max = nt_max_of(*desc, chunk_size, cu);
  a->stream = (cudaStream_t)stream;
  return GDR_OK;
}

int gdr_chunk_index(const gdr_desc *desc, const int64_t *cu_seqlens, int chunk_size, int64_t *chunk_indices,
                    int64_t *chunk_offsets, void *stream) {
  ChunkedArgs a{};
  int rc = stage_prologue(desc, chunk_size, cu_seqlens, &a, stream);
  if (rc != GDR_OK) return rc;
  if (!chunk_indices || !chunk_offsets) return set_error(GDR_ERR_NULLPTR, "chunk_indices and chunk_offsets required");
  a.chunk_indices = chunk_indices;
  a.chunk_offsets = chunk_offsets;
  return launch_chunk_index(a);
}

int gdr_chunk_prepare(const gdr_desc *desc, const void *k, const void *v, const float *g, const void *beta,
                      const int64_t *cu_seqlens, const int64_t *chunk_indices, int chunk_size, int use_qk_l2norm,
                      float *gcum, float *w, float *u, void *stream) {
  ChunkedArgs a{};
  int rc = stage_prologue(desc, chunk_size, cu_seqlens, &a, stream);
  if (rc != GDR_OK) return rc;
  if (a.d.B * a.d.T > 0 && (!k || !v || !g || !beta || !gcum || !w || !u))
    return set_error(GDR_ERR_NULLPTR, "k, v, g, beta, gcum, w, u required");
  if (cu_seqlens && !chunk_indices) return set_error(GDR_ERR_NULLPTR, "varlen layout needs chunk_indices");
  a.k = k; a.v = v; a.g = g; a.beta = beta;
  a.chunk_indices = cu_seqlens ? (int64_t *)chunk_indices : nullptr;
  a.l2 = use_qk_l2norm ? 1 : 0;
  a.gcum = gcum; a.w = w; a.u = u;
  return launch_chunk_prepare(a);
}

int gdr_chunk_fwd_h(const gdr_desc *desc, const void *k, const float *w, const float *u, const float *gcum,
                    const float *h0, const int64_t *cu_seqlens, const int64_t *chunk_offsets, int chunk_size,
                    int use_qk_l2norm, float *h, float *v_new, float *ht, void *stream) {
  ChunkedArgs a{};
  int rc = stage_prologue(desc, chunk_size, cu_seqlens, &a, stream);
  if (rc != GDR_OK) return rc;
  if (a.d.B * a.d.T > 0 && (!k || !w || !u || !gcum)) return set_error(GDR_ERR_NULLPTR, "k, w, u, gcum required");
  if (cu_seqlens && !chunk_offsets) return set_error(GDR_ERR_NULLPTR, "varlen layout needs chunk_offsets");
  a.k = k; a.w = (float *)w; a.u = (float *)u; a.gcum = (float *)gcum; a.h0 = h0;
  a.chunk_offsets = cu_seqlens ? (int64_t *)chunk_offsets : nullptr;
  a.l2 = use_qk_l2norm ? 1 : 0;
  a.h = h; a.v_new = v_new; a.ht = ht;
  return launch_chunk_fwd_h(a);
}

int gdr_chunk_fwd_o(const gdr_desc *desc, const void *q, const void *k, const float *v_new, const float *h,
                    const float *gcum, const int64_t *cu_seqlens, const int64_t *chunk_indices, int chunk_size,
                    int use_qk_l2norm, void *o, void *stream) {
  ChunkedArgs a{};
  int rc = stage_prologue(desc, chunk_size, cu_seqlens, &a, stream);
  if (rc != GDR_OK) return rc;
  if (a.d.B * a.d.T > 0 && (!q || !k || !v_new || !h || !gcum || !o))
    return set_error(GDR_ERR_NULLPTR, "q, k, v_new, h, gcum, o required");
  if (cu_seqlens && !chunk_indices) return set_error(GDR_ERR_NULLPTR, "varlen layout needs chunk_indices");
  a.q = q; a.k = k; a.v_new = (float *)v_new; a.h = (float *)h; a.gcum = (float *)gcum;
  a.chunk_indices = cu_seqlens ? (int64_t *)chunk_indices : nullptr;
  a.l2 = use_qk_l2norm ? 1 : 0;
  a.o = o;
  return launch_chunk_fwd_o(a);
}

int gdr_device_status(void *stream, int clear) {
  int dev, rc;
  if ((rc = current_device(&dev)) != GDR_OK) return rc;
  int *word = device_status_word(dev, &rc);
  if (!word) return rc;
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_error(e, "cudaStreamSynchronize");
  int host = 0;
  e = cudaMemcpy(&host, word, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_error(e, "reading the status word");
  if (clear && host != 0) {
    e = cudaMemset(word, 0, sizeof(int));
    if (e != cudaSuccess) return cuda_error(e, "clearing the status word");
  }
  if (host == GDR_ERR_SEQLENS) set_error(host, "cu_seqlens is not non-decreasing from 0 to T");
  if (host == GDR_ERR_TIMEOUT) set_error(host, "a bounded device-side wait expired");
  return host;
}

const char *gdr_last_error(void) { return g_last_error.c_str(); }

int64_t gdr_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int gdr_version(void) { return 100; }

}  // extern "C"
