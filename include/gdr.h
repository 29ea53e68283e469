/*
 * gdr.h -- C ABI of the GB300 (sm_103a) chunked gated delta rule forward.
 *
 * The operation (the gated delta rule, GDN with a scalar gate, KDA with a
 * per-key-channel gate), per sequence and value head, with S a K x V state:
 *
 *   S_t = (I - beta_t k_t k_t^T) Diag(exp g_t) S_{t-1} + beta_t k_t v_t^T
 *   o_t = S_t^T q_t
 *
 * evaluated chunk by chunk through the WY / UT-transform form
 * S^r = P^r S^0 + H^r, P^r = I - sum_i k^i w^i^T ("FLA 算子内核正确性测试与覆盖矩阵",
 * section 二), with the per-chunk state h stored at each chunk's START
 * ("flash-linear-attention KCP 精度失效根因排查手册", section on h/dh semantics).
 * The kernel order is the pages' forward order: chunk index -> prepare
 * (L2 norm, gate cumsum, A, triangular solve, w, u) -> state scan (fwd_h)
 * -> output (fwd_o) (KCP handbook, section on the debug-script layout).
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers to contiguous row-major memory,
 *    owned by the caller; the library never frees or retains them.
 *  - Shapes travel in a gdr_desc.  Token index t runs over B*T flat tokens.
 *      q, k        [B, T, H, K]      dtype (fp32 or bf16)
 *      v, o        [B, T, HV, V]     dtype
 *      g           [B, T, HV] (GDN) or [B, T, HV, K] (KDA), fp32, natural-log decay
 *      beta        [B, T, HV]        dtype (already in (0, 1); no sigmoid is applied)
 *      h0, ht      [N, HV, K, V]     fp32, nullable
 *      cu_seqlens  [N + 1]           int64, nullable; requires B == 1
 *    Value head hv reads q/k head hv / (HV / H) (grouped value heads, GVA).
 *  - q is not scaled (scale 1).  o has the dtype of q, k, v.
 *  - Calls are asynchronous on `stream` (a cudaStream_t passed as void*; NULL
 *    is the legacy default stream) and never synchronize the host, except
 *    gdr_device_status.
 *  - Every entry point returns GDR_OK (0) or a negative gdr_status.  On error
 *    nothing has been launched and gdr_last_error() holds a message for the
 *    calling thread.
 *  - The current CUDA device must be the one that owns the pointers.
 */
#ifndef GDR_H
#define GDR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gdr_status {
  GDR_OK = 0,
  GDR_ERR_CHUNK_SIZE = -1,  /* chunk_size not in {32, 64}: "chunk_size must be either 32 or 64" */
  GDR_ERR_SHAPE = -2,       /* bad sizes: HV % H != 0, K or V outside [1, 256], B != 1 with cu_seqlens, ... */
  GDR_ERR_DTYPE = -3,       /* unknown dtype / gate / algorithm code */
  GDR_ERR_NULLPTR = -4,     /* a required pointer is NULL */
  GDR_ERR_ALIGN = -5,       /* a pointer the fused path stages with TMA is not 16-byte aligned */
  GDR_ERR_CUDA = -6,        /* a CUDA runtime call failed (message has the CUDA error string) */
  GDR_ERR_TIMEOUT = -7,     /* a bounded device-side wait expired (reported by gdr_device_status) */
  GDR_ERR_SEQLENS = -8,     /* cu_seqlens not monotone or not spanning [0, T] (gdr_device_status) */
  GDR_ERR_UNSUPPORTED = -9  /* valid request that the chosen algorithm does not implement */
} gdr_status;

typedef enum gdr_dtype { GDR_F32 = 0, GDR_BF16 = 1 } gdr_dtype;
typedef enum gdr_gate { GDR_GATE_SCALAR = 0, GDR_GATE_PER_K = 1 } gdr_gate;
typedef enum gdr_algo {
  GDR_ALGO_AUTO = 0,     /* fused single pass where supported, else the chunked three-kernel form */
  GDR_ALGO_CHUNKED = 1,  /* chunk index -> prepare -> fwd_h -> fwd_o; warp-level tensor-core products in
                            3 x TF32 for fp32 inputs; for bf16 inputs the Gram matrices and the solve in
                            3 x TF32, the other products in one bf16 pass (fp32 accumulation) */
  GDR_ALGO_FUSED = 2,    /* one persistent pass per (sequence, value head), tcgen05 tensor cores */
  GDR_ALGO_RECURRENT = 3, /* token by token, state in registers (decode and other short inputs) */
  GDR_ALGO_SPLIT = 4      /* chunked, state scan split into 1024-token segments merged by transitions */
} gdr_algo;

typedef struct gdr_desc {
  int64_t B, T, H, HV, K, V;
  int64_t N;       /* number of sequences: B when cu_seqlens is NULL, else len(cu_seqlens) - 1 */
  int32_t dtype;   /* gdr_dtype of q, k, v, beta, o */
  int32_t gate;    /* gdr_gate */
  int32_t algo;    /* gdr_algo */
  int32_t flags;   /* GDR_FLAG_* bits; other bits must be 0 */
} gdr_desc;

/*
 * GDR_FLAG_BETA_LOGITS: beta holds logits x and every kernel uses
 * sigmoid(x) = 1 / (1 + exp(-x)) in its place (the coverage guide, section 三,
 * tests "raw beta" beside "beta after sigmoid").  gdr_bwd then returns
 * dL/dx = dL/dbeta * beta (1 - beta) in dbeta.
 */
#define GDR_FLAG_BETA_LOGITS 1

/*
 * gdr_fwd -- the chunked forward of the gated delta rule.
 *   chunk_size     32 or 64; anything else returns GDR_ERR_CHUNK_SIZE (the
 *                  coverage guide, section 三, rejects chunk_size = 16 this way).
 *   use_qk_l2norm  nonzero: q and k are L2-normalized per token and head inside
 *                  the kernels, x / sqrt(sum x^2 + 1e-6); zero: used as given.
 *   h0             initial state, NULL means zero.
 *   ht             final state output, NULL means not wanted.
 *   cu_seqlens     NULL for dense batches; else the varlen layout.  Its values
 *                  are read on the device: they must be non-decreasing with
 *                  cu[0] = 0 and cu[N] = T; a violation makes every output
 *                  untouched and is reported by gdr_device_status.
 * Scratch (the chunked form's w, u, h, v_new) is taken stream-ordered from a
 * library-owned memory pool on `stream` and returned to it before the call's
 * work completes; the fused form needs none.
 * GDR_ALGO_AUTO picks the recurrent form for dense inputs with T <= 16, then
 * the fused form where it applies, else the chunked form.  The recurrent form
 * (the coverage guide's fused_recurrent path, section 三) follows the
 * per-token recurrence directly; with it, ht may alias h0 for in-place
 * decode.  GDR_ALGO_SPLIT is the chunked form with the state scan split
 * inside each sequence (the KCP handbook's segment transition M and end
 * state S_ext, merged on one GPU): segments of 1024 tokens run in parallel,
 * for inputs with few (sequence, value head) pairs and long sequences.
 * AUTO takes it when the fused form does not apply, the input is dense with
 * T >= 4096, and N * HV * ceil(V / 32) < 152 (fewer state-scan blocks than
 * the GPU has SMs).
 */
int gdr_fwd(const gdr_desc *desc, const void *q, const void *k, const void *v, const float *g,
            const void *beta, const float *h0, const int64_t *cu_seqlens, int chunk_size,
            int use_qk_l2norm, void *o, float *ht, void *stream);

/*
 * gdr_bwd -- the backward of gdr_fwd: gradients of L = sum(o * do) +
 * sum(ht * dht) with respect to q, k, v, g, beta and h0 (the optional
 * backward of the problem statement; the coverage guide, section 三, grades
 * dq, dk, dv, dg, dbeta and dh0, and the KCP handbook's debug-script layout
 * names its chunk stages bwd_dAu -> bwd_dhu -> bwd_dv -> bwd_o -> bwd_wy ->
 * bwd_dqk_intra).  The forward's intermediates are recomputed, not taken from
 * a previous call.
 *   Inputs as gdr_fwd (desc->algo is ignored), plus
 *   d_o    upstream gradient of o, [B,T,HV,V] in the input dtype;
 *   dht    upstream gradient of ht, [N,HV,K,V] fp32; NULL means zero.
 *   Outputs (caller-owned device memory, every element written):
 *   dq, dk [B,T,H,K], dv [B,T,HV,V], dbeta [B,T,HV] in the input dtype;
 *   dg shaped like g, fp32; dh0 [N,HV,K,V] fp32, NULL means not wanted
 *   (it is the gradient with respect to the initial state, zero or not).
 * With grouped value heads, dq and dk sum over the HV/H value heads that
 * share a q/k head.  K must be <= 128 (GDR_ERR_SHAPE otherwise).  Scratch
 * (about 4 K + 5 V floats per token and value head, plus two fp32 states per
 * chunk and value head) comes from the same library-owned pool as gdr_fwd's.
 * Invalid cu_seqlens leave the outputs untouched and set GDR_ERR_SEQLENS in
 * the status word.
 */
int gdr_bwd(const gdr_desc *desc, const void *q, const void *k, const void *v, const float *g,
            const void *beta, const float *h0, const int64_t *cu_seqlens, int chunk_size,
            int use_qk_l2norm, const void *d_o, const float *dht, void *dq, void *dk, void *dv,
            float *dg, void *dbeta, float *dh0, void *stream);

/*
 * Stage entry points of the chunked form, with caller-provided scratch, so the
 * per-chunk intermediates can be inspected.  Sizes come from gdr_chunked_sizes.
 *
 *   gdr_chunk_index    cu_seqlens [N+1] -> chunk_indices [nt_max, 2] (sequence,
 *                      chunk-in-sequence), chunk_offsets [N+1] (first chunk of
 *                      each sequence; chunk_offsets[N] = NT).  Rows >= NT of
 *                      chunk_indices are set to -1.  int64 throughout
 *                      (coverage guide, section 四: address arithmetic in int64).
 *                      With cu_seqlens NULL it describes the dense layout.
 *   gdr_chunk_prepare  per (chunk, value head): gate cumsum Gamma (fp32, [B*T, HV]
 *                      or [B*T, HV, K]), A = tril(beta K K^T * decay, -1),
 *                      T = (I + A)^-1, w = T diag(beta) (K * exp Gamma)
 *                      ([B*T, HV, K] fp32) and u = T diag(beta) V ([B*T, HV, V] fp32).
 *   gdr_chunk_fwd_h    per (sequence, value head, V-tile), sequential over
 *                      chunks: h [NT, HV, K, V] fp32 (state entering each chunk),
 *                      v_new = u - w h ([B*T, HV, V] fp32), and ht.
 *   gdr_chunk_fwd_o    per (chunk, value head): o = (q * exp Gamma) h +
 *                      tril(q k^T * decay) v_new.
 */
typedef struct gdr_chunked_sizes {
  int64_t nt_max;              /* upper bound on the number of chunks NT */
  size_t chunk_indices_bytes;  /* int64 [nt_max, 2] */
  size_t chunk_offsets_bytes;  /* int64 [N + 1] */
  size_t gcum_bytes;           /* fp32 gate cumsum */
  size_t w_bytes, u_bytes, v_new_bytes, h_bytes;
} gdr_chunked_sizes;

/* varlen nonzero: sizes for the cu_seqlens layout (nt_max is then an upper bound). */
int gdr_chunked_sizes_get(const gdr_desc *desc, int chunk_size, int varlen, gdr_chunked_sizes *out);
int gdr_chunk_index(const gdr_desc *desc, const int64_t *cu_seqlens, int chunk_size,
                    int64_t *chunk_indices, int64_t *chunk_offsets, void *stream);
int gdr_chunk_prepare(const gdr_desc *desc, const void *k, const void *v, const float *g,
                      const void *beta, const int64_t *cu_seqlens, const int64_t *chunk_indices,
                      int chunk_size, int use_qk_l2norm, float *gcum, float *w, float *u, void *stream);
int gdr_chunk_fwd_h(const gdr_desc *desc, const void *k, const float *w, const float *u,
                    const float *gcum, const float *h0, const int64_t *cu_seqlens,
                    const int64_t *chunk_offsets, int chunk_size, int use_qk_l2norm, float *h,
                    float *v_new, float *ht, void *stream);
int gdr_chunk_fwd_o(const gdr_desc *desc, const void *q, const void *k, const float *v_new,
                    const float *h, const float *gcum, const int64_t *cu_seqlens,
                    const int64_t *chunk_indices, int chunk_size, int use_qk_l2norm, void *o,
                    void *stream);

/*
 * gdr_fwd_noalloc -- the chunked forward without any device allocation.
 * The pages have no counterpart to this entry point; it exists for callers
 * that cannot allocate device memory: code whose framework allocator owns all
 * device memory, code running where allocation calls are forbidden or would
 * synchronize, and callers that must not allocate after start-up.  It takes
 * the same arguments as gdr_fwd and computes the same results as gdr_fwd with
 * GDR_ALGO_CHUNKED (desc->algo is ignored).  Its scratch is one fixed device
 * array of GDR_NOALLOC_SCRATCH_BYTES that every GPU loading the library holds
 * until the process exits; requests needing more return GDR_ERR_SHAPE with a
 * message giving both sizes (about 2.6 KB per token and value head at
 * K = V = 128, so e.g. 1024 tokens x 16 heads fit).
 *   - The first call on a device looks up the array's device address (once
 *     per device, with that device current); make that first call before any
 *     stream capture.  The address is kept for the life of the process: it
 *     does not survive cudaDeviceReset (or any other teardown of the device's
 *     primary context), after which this entry point must not be called
 *     again in the same process.
 *   - Every call shares the one array: calls whose work overlaps on the GPU
 *     (concurrent streams, or several host threads) race and corrupt each
 *     other's results; serialize them.  Every scratch byte a call reads it
 *     first writes, so nothing carries over from one call to the next.
 *   - No status word exists for this path: with invalid cu_seqlens the
 *     outputs are left untouched and nothing is recorded.
 */
#define GDR_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
int gdr_fwd_noalloc(const gdr_desc *desc, const void *q, const void *k, const void *v, const float *g,
                    const void *beta, const float *h0, const int64_t *cu_seqlens, int chunk_size,
                    int use_qk_l2norm, void *o, float *ht, void *stream);

/*
 * gdr_device_status -- synchronizes `stream`, then returns (and, if `clear`,
 * resets) the library's device-side status word for the current device:
 * GDR_OK, GDR_ERR_SEQLENS or GDR_ERR_TIMEOUT.  Also returns GDR_ERR_CUDA if
 * the stream itself reports an error.
 */
int gdr_device_status(void *stream, int clear);

/* Message for the last error on the calling thread ("" if none). */
const char *gdr_last_error(void);

/* Number of kernels this library has launched in this process (all devices). */
int64_t gdr_launch_count(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int gdr_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GDR_H */
