// gdr_internal.h -- declarations shared by the translation units of libgdr.so.
// Host-side only; device helpers live in gdr_device.cuh.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <string>

#include "gdr.h"

namespace gdr {

// Records a message for gdr_last_error() on this thread and returns `code`.
int set_error(int code, const std::string &msg);
int cuda_error(cudaError_t e, const char *what);

// Counts kernel launches (gdr_launch_count).
void count_launch(int n = 1);

// Per-device 4-byte status word that kernels set on a detected problem
// (bad cu_seqlens, an expired bounded wait).  Zero means OK.
int *device_status_word(int device, int *err);

// Geometry shared by the launchers: number of chunks in the dense layout,
// and an upper bound on NT for the varlen layout.
inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int64_t nt_upper_bound(const gdr_desc &d, int C) {
  // sum_n ceil(len_n / C) <= (T + N (C - 1)) / C when the lengths sum to T
  return d.N > 0 ? (d.B * d.T + d.N * (int64_t)(C - 1)) / C : 0;
}

struct ChunkedArgs {
  gdr_desc d;
  int C;
  int l2;
  const void *q, *k, *v, *beta;
  const float *g, *h0;
  const int64_t *cu;
  int64_t *chunk_indices, *chunk_offsets;  // may be null in the dense layout
  float *gcum, *w, *u, *h, *v_new, *ht;
  float *kb;  // nullable: k e^{G_L - G} rows [B*T, HV, K] fp32, formed by prepare, read by fwd_h
  void *o;
  int64_t nt_max;
  int *status;
  cudaStream_t stream;
};

// The backward: the forward recompute (prepare, fwd_h) runs through `f`;
// the rest are the backward's own scratch and outputs.
struct BwdArgs {
  ChunkedArgs f;
  const void *d_o;           // upstream gradient of o [B,T,HV,V], input dtype
  const float *dht;          // upstream gradient of ht [N,HV,K,V], nullable
  float *dvn;                // [B*T,HV,V]: dL/dv_new (local part, then complete)
  float *dhc;                // [NT,HV,K,V]: dL/d(state leaving chunk c)
  float *dqa, *dka;          // [B*T,HV,K]: dL/dq^, dL/dk^ per value head
  float *dga;                // [B*T,HV,gw]: dL/dGamma from the output and state terms
  float *dW;                 // [B*T,HV,K]: dL/dw
  void *dq, *dk, *dv, *dbeta;  // outputs in the input dtype
  float *dg, *dh0;           // outputs, fp32 (dh0 nullable)
};

int launch_bwd_dv_local(const BwdArgs &a);
int launch_bwd_dh(const BwdArgs &a);
int launch_bwd_dqkg(const BwdArgs &a);
int launch_bwd_wy(const BwdArgs &a);
int launch_bwd_finalize(const BwdArgs &a);

// Argument checks shared by the entry points, and the chunked form's scratch
// sizes (gdr_api.cu).
int validate_request(const gdr_desc *d, int chunk_size, const int64_t *cu);
void chunked_scratch_sizes(const gdr_desc &d, int C, const int64_t *cu, gdr_chunked_sizes *s);

// Launchers of the chunked (three-kernel) form; return GDR_OK or an error.
int launch_chunk_index(const ChunkedArgs &a);
int launch_chunk_prepare(const ChunkedArgs &a);
int launch_chunk_fwd_h(const ChunkedArgs &a);
int launch_chunk_fwd_o(const ChunkedArgs &a);

// The intra-sequence split of the state scan (gdr_split.cu).  Segments are
// S chunks long; seg_indices / seg_offsets are the chunk index built with a
// chunk length of S*C tokens (varlen only).
struct SplitArgs {
  int S;
  int64_t nseg_max;
  int64_t *seg_indices, *seg_offsets;
  float *X;     // [nseg_max, HV, K, V + K]: [S_ext | M] per segment
  float *s_in;  // [nseg_max, HV, K, V]: state entering each segment
};
int launch_split_transitions(const ChunkedArgs &a, const SplitArgs &sp);
int launch_split_merge(const ChunkedArgs &a, const SplitArgs &sp);
int launch_split_final(const ChunkedArgs &a, const SplitArgs &sp);

// The per-token form (gdr_recurrent.cu): reads q, k, v, g, beta, h0, cu,
// chunk_offsets (varlen only, from launch_chunk_index), writes o and ht.
int launch_recurrent_fwd(const ChunkedArgs &a);

}  // namespace gdr
