/*
 * sdpa.h — C ABI of the GB300 (sm_103a) fused scaled-dot-product attention library.
 *
 * What it computes.  For every batch b and query head hq (KV head hk = hq / (h_q / h_kv)):
 *
 *     S   = attn_scale * Q K^T                  (scores, then the scale)
 *     S  += bias                                 (optional: ALiBi, or a bias tensor)
 *     S  += mask   (causal: -inf where key j > query i, top-left or bottom-right aligned;
 *                   variable lengths: -inf on padded keys; otherwise no mask)
 *     P   = softmax(S) over each row
 *     O   = (P * keep / (1 - p)) V               (optional dropout; O has Q's shape)
 *     LSE = log(sum_j exp(S_ij))                 (natural log, per query row)
 *
 * [attention codelab "Speeding up attention on GPU with cuDNN and TransformerEngine",
 *  §1 "How attention works" (the four steps) and §7 "Adding a causal mask";
 *  cuDNN 9 blog "Accelerating Transformers with NVIDIA cuDNN 9", "SDPA as a cuDNN
 *  graph", Fig. 4 (BMM1 -> scale -> causal mask -> softmax -> BMM2); the SDPA node's
 *  second output "stats" is the per-row statistic kept for training, read here as the
 *  log-sum-exp; the walkthrough's options bias, use_alibi_mask, use_padding_mask with
 *  seq_len_q / seq_len_kv, and dropout; the codelab's §10 FP8 recipe.]  The backward pass
 *  returns dQ, dK, dV (and, on request, the bias gradient) for an incoming dO, using the LSE
 *  kept by the forward pass (the blog's "fprop + bprop" figure; the pages give no formula,
 *  the derivative is the analytic one).
 *
 * Conventions shared by every entry point
 *  - All tensors are *logical* BHSD [b][h][s][d] views over caller memory described by
 *    four element strides (sdpa_strides_t).  The innermost stride must be 1.  A BSHD
 *    buffer is passed with strides (s*h*d, d, h*d, 1) — no copy is made [cuDNN-in-Python
 *    post: the GPT-2-like example views a BSHD buffer as BHSD with as_strided].
 *  - Pointers are DEVICE pointers on the current CUDA device; bases must be 16-byte
 *    aligned and every non-unit stride, in bytes, a multiple of 16 (they are handed to
 *    the tensor-memory-accelerator (TMA) unit as is).
 *  - Ownership: the caller owns every buffer.  The library allocates no device memory,
 *    frees nothing, does not synchronise the stream and keeps no pointer after return.
 *  - Work is enqueued asynchronously on `stream` (0 = legacy default stream).
 *  - Errors: arguments are validated on the host before anything is launched; a non-OK
 *    status comes with a message from sdpa_last_error_string().  Unsupported inputs are an
 *    error, never a silent fallback.  Launch failures return SDPA_ERR_CUDA.
 *  - Thread safety: re-entrant.  Concurrent calls must not share a workspace.
 */
#ifndef SDPA_GB300_H
#define SDPA_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SDPA_API __attribute__((visibility("default")))
#else
#define SDPA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SDPA_OK = 0,
  SDPA_ERR_INVALID_ARG = 1,   /* null pointer, non-positive size, h_q % h_kv != 0, ... */
  SDPA_ERR_UNSUPPORTED = 2,   /* valid request this library does not implement (e.g. d=96) */
  SDPA_ERR_LAYOUT = 3,        /* stride / alignment not expressible to the TMA unit */
  SDPA_ERR_WORKSPACE = 4,     /* workspace missing or smaller than sdpa_workspace_size() */
  SDPA_ERR_CUDA = 5,          /* a CUDA runtime/driver call failed (message has the code) */
  SDPA_ERR_TIMEOUT = 6        /* a bounded device wait gave up (see sdpa_device_error) */
} sdpa_status_t;

typedef enum {
  SDPA_DTYPE_F16 = 0,         /* IEEE binary16 */
  SDPA_DTYPE_BF16 = 1,        /* bfloat16 */
  SDPA_DTYPE_E4M3 = 2,        /* OCP FP8 E4M3 (finite max 448): Q, K, V (forward and backward) */
  SDPA_DTYPE_E5M2 = 3         /* OCP FP8 E5M2 (max 57344): dO of an FP8 backward pass only */
} sdpa_dtype_t;

/* Element strides of a logical [b][h][s][d] view.  d must be 1. */
typedef struct {
  int64_t b, h, s, d;
} sdpa_strides_t;

/* One attention problem.  Fields not used by a call are ignored. */
typedef struct {
  int32_t b;           /* batch, >= 1 */
  int32_t h_q;         /* query heads, >= 1 */
  int32_t h_kv;        /* key/value heads, >= 1, h_q % h_kv == 0 (MHA: ==, GQA: <, MQA: 1);
                          query head hq reads KV head hq / (h_q / h_kv) [codelab §9] */
  int32_t s_q;         /* query rows, >= 1 */
  int32_t s_kv;        /* key/value rows, >= 1 */
  int32_t d;           /* head dim of Q, K and V: 64, 128 or 256 */
  int32_t in_dtype;    /* sdpa_dtype_t of Q, K, V (and of dO for the backward pass) */
  int32_t out_dtype;   /* sdpa_dtype_t of O (and dQ/dK/dV): == in_dtype for F16/BF16;
                          BF16 or F16 for E4M3 inputs */
  float attn_scale;    /* multiplies Q K^T before the mask and softmax; any finite value
                          (usually 1/sqrt(d)) [cuDNN 9 blog, Fig. 4: scale node after BMM1] */
  int32_t causal;      /* 0: no mask.  1: top-left causal, key j visible to query i iff j <= i
                          (row 0 sees only key 0) [codelab §7].  2: bottom-right causal, key j
                          visible to query i iff j <= i + len_kv - len_q (the last query sees
                          every key, as when decoding against a KV cache) */
  sdpa_strides_t q, k, v, o;         /* forward and backward */
  sdpa_strides_t dout, dq, dk, dv;   /* backward only (dout = incoming gradient dO) */
  const float* descale_q;  /* E4M3 only: DEVICE pointers to one fp32 each; the real value of */
  const float* descale_k;  /* a stored code x is decode(x) * descale (per-tensor scaling of    */
  const float* descale_v;  /* the delayed-scaling FP8 recipe, codelab §10).  NULL otherwise.   */
  /* Variable lengths (the SDPA node's padding mask with per-batch sequence lengths, cuDNN 9
   * blog walkthrough).  Optional DEVICE pointers to b int32 values; NULL = every row valid.
   * For batch b only query rows i < len_q[b] and keys j < len_kv[b] take part (values are
   * clamped to [0, s_q] and [0, s_kv]).  Rows with no visible key — padded rows, or early rows
   * of a bottom-right mask with len_kv < len_q — give O = 0 and LSE = -inf, and padded rows of
   * dQ, dK and dV are 0. */
  const int32_t* seq_lens_q;
  const int32_t* seq_lens_kv;
  /* ALiBi (the SDPA node's ALiBi-mask option, cuDNN 9 blog walkthrough; the pages name it but
   * do not define it, and this is the linear-bias reading).  0 = off.  1 = the scaled score of
   * (i, j) gains m_hq * (j - i - off) before the mask and softmax, off = len_kv - len_q under
   * bottom-right causal alignment and 0 otherwise: zero on the aligned diagonal, a penalty
   * growing linearly with the distance to earlier keys.  ALiBi needs a causal mask (causal 1
   * or 2: every visible key is then at or before the aligned diagonal); with causal = 0 it is
   * refused with SDPA_ERR_UNSUPPORTED.  m_hq = alibi_slopes[hq] (a DEVICE
   * pointer to h_q finite fp32 values >= 0; a negative slope counts as 0), or, when
   * alibi_slopes is NULL, the geometric slopes 2^(-8 (hq + 1) / h_q).  F16 and BF16 inputs
   * only; the bias has no gradient. */
  int32_t alibi;
  const float* alibi_slopes;
  /* Dropout (the SDPA node's dropout option, cuDNN 9 blog walkthrough; named, not defined by
   * the pages).  dropout_p in [0, 1); 0 = off.  With p > 0 each softmax probability P_ij is
   * kept where its keep bit is set and scaled by 1/(1 - p), so O = (P * keep) V / (1 - p); the
   * LSE is that of the undropped softmax.  The keep bits come from sdpa_dropout_mask: the
   * forward pass reads `dropout_mask` (row-major), the backward pass `dropout_mask_t` (the
   * same bits transposed); both DEVICE pointers, 16-byte aligned.  F16/BF16 inputs only. */
  float dropout_p;
  const uint32_t* dropout_mask;
  const uint32_t* dropout_mask_t;
  /* FP8 backward (the HYBRID recipe of the codelab's TransformerEngine section: E4M3 in the
   * forward pass, E5M2 for gradients).  Read only when in_dtype is E4M3 and the call is
   * sdpa_bwd: dO has dout_dtype (E5M2 or E4M3) with the per-tensor descale *descale_do
   * (DEVICE pointer); Q, K, V are E4M3 with descale_q/k/v; O and dQ, dK, dV have out_dtype
   * (BF16 or F16).  The codes are widened exactly to out_dtype in the workspace and the
   * descales folded into the kernels' scale factors; the MMAs run at 16-bit precision. */
  int32_t dout_dtype;
  const float* descale_do;
  /* Additive bias (the SDPA node's bias input, cuDNN 9 blog walkthrough).  NULL = none; else
   * a DEVICE pointer to a logical [b][h_q][s_q][s_kv] tensor of in_dtype (F16/BF16) whose
   * element strides are bias_strides (b, h, s, and d = the key stride, which must be 1); a
   * zero b or h stride broadcasts one slice over the batch or the heads.  The bias is added
   * to the scaled scores before the mask and softmax and is treated as a constant (no
   * gradient is produced).  Base 16-byte aligned; non-zero b/h/s strides multiples of 8.
   * Not combined with alibi (fold ALiBi into the tensor instead).  A backward pass with a
   * bias needs workspace for a transposed copy (sdpa_workspace_size accounts for it); its
   * gradient is available through dbias. */
  const void* bias;
  sdpa_strides_t bias_strides;
  /* Bias gradient (sdpa_bwd only; needs `bias`): NULL = not wanted; else a DEVICE pointer to
   * a tensor of the bias's shape and dtype, strides dbias_strides (zero b/h strides exactly
   * where bias_strides has them), overwritten with dL/dbias = dS — the gradient of the
   * scaled scores — summed over the broadcast dimensions.  Same alignment rules as bias.
   * The workspace then also holds an fp32 accumulator (sdpa_workspace_size accounts for it). */
  void* dbias;
  sdpa_strides_t dbias_strides;
} sdpa_problem_t;

/*
 * Workspace bytes that sdpa_fwd (is_backward = 0) or sdpa_bwd (is_backward = 1) needs for
 * `p`.  Writes *bytes; never launches anything.  The forward pass needs 0 bytes; the
 * backward pass needs fp32 scratch for dQ accumulation and the per-row Delta term
 * (4*b*h_q*round_up(s_q,128)*(d+1) bytes plus alignment).
 * [cuDNN-in-Python post: the workspace size is queried, then allocated by the caller.]
 */
SDPA_API sdpa_status_t sdpa_workspace_size(const sdpa_problem_t* p, int is_backward, size_t* bytes);

/*
 * Forward pass: O (and, when lse != NULL, the per-row log-sum-exp) from Q, K, V.
 *   q:   [b][h_q][s_q][d]   in_dtype, strides p->q
 *   k,v: [b][h_kv][s_kv][d] in_dtype, strides p->k, p->v
 *   o:   [b][h_q][s_q][d]   out_dtype, strides p->o; overwritten
 *   lse: NULL (inference: no statistics written) or fp32 [b][h_q][s_q] dense row-major;
 *        lse[(b*h_q + hq)*s_q + i] = ln sum_j exp(S_ij) over the visible keys; overwritten.
 *        The SDPA node's "stats" output, kept for training [cuDNN 9 blog, SDPA walkthrough;
 *        cuDNN-in-Python post].
 *   workspace / workspace_bytes: may be NULL / 0 (the forward pass needs none).
 * E4M3 inputs require descale_q/k/v and give a BF16 or F16 O.
 */
SDPA_API sdpa_status_t sdpa_fwd(const sdpa_problem_t* p, const void* q, const void* k, const void* v,
                       void* o, float* lse, void* workspace, size_t workspace_bytes,
                       void* stream /* cudaStream_t */);

/*
 * Backward pass: dQ, dK, dV of O for the incoming gradient dO, recomputing P from the LSE
 * written by sdpa_fwd on the same inputs.
 *   q, k, v, o: as in sdpa_fwd (o is the forward output); dout: [b][h_q][s_q][d], in_dtype
 *   lse: fp32 [b][h_q][s_q] from sdpa_fwd (required)
 *   dq: Q's shape, dk/dv: K's/V's shape, all out_dtype (== in_dtype); overwritten.  dK and
 *       dV hold the sum over the query heads of each KV group (GQA/MQA).
 *   workspace: >= sdpa_workspace_size(p, 1) bytes, 256-byte aligned; its contents on entry
 *       do not matter and are clobbered.
 * F16/BF16, or E4M3 Q/K/V with E5M2 or E4M3 dO (see dout_dtype).
 */
SDPA_API sdpa_status_t sdpa_bwd(const sdpa_problem_t* p, const void* q, const void* k, const void* v,
                       const void* o, const void* dout, const float* lse, void* dq, void* dk,
                       void* dv, void* workspace, size_t workspace_bytes,
                       void* stream /* cudaStream_t */);

/*
 * Size of the built-in scratch that sdpa_bwd_noalloc uses: 32 MiB of device memory, held by
 * every GPU on which the library's kernels are loaded, until the process exits.
 */
#define SDPA_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)

/*
 * sdpa_bwd_noalloc: the backward pass of sdpa_bwd for callers that cannot allocate device
 * memory — for example a plugin running inside a host framework that owns all device
 * memory and offers no allocator, or a latency-critical loop that must not call cudaMalloc
 * (which can synchronise the device).  Arguments and results are those of sdpa_bwd minus
 * the workspace: the scratch comes from a fixed array inside the library
 * (SDPA_NOALLOC_SCRATCH_BYTES), so nothing is allocated or freed.  The pages have no
 * counterpart of this entry point.
 *   - Problems whose workspace (sdpa_workspace_size(p, 1)) exceeds the array are rejected
 *     with SDPA_ERR_UNSUPPORTED and a message giving both sizes; use sdpa_bwd then.
 *   - The first call on a device looks up the array's device address (with that device
 *     current); make that first call before any stream capture.  The address is kept for
 *     the life of the process, so do not call this entry point again on a device after
 *     cudaDeviceReset() there (the reset unloads the module that holds the array).
 *   - Every call shares the one array (whatever it held is overwritten; each call clears
 *     what must start at zero), so calls whose executions overlap on the GPU — on different
 *     streams, or from different threads — race and give wrong results.  Serialise them.
 */
SDPA_API sdpa_status_t sdpa_bwd_noalloc(const sdpa_problem_t* p, const void* q, const void* k,
                                        const void* v, const void* o, const void* dout,
                                        const float* lse, void* dq, void* dk, void* dv,
                                        void* stream /* cudaStream_t */);

/*
 * Byte sizes of the two dropout keep-mask arrays of `p` (b, h_q, s_q, s_kv are read):
 *   mask:   uint32 [b*h_q][s_q][ceil(s_kv/128)*4]   (key j of row i at bit 16*(j%2) + (j%32)/2
 *           of word j/32: the two keys of an even/odd pair sit 16 bits apart)
 *   mask_t: uint32 [b*h_q][s_kv][ceil(s_q/128)*4]   (row i of key j at bit 16*(i%2) + (i%32)/2
 *           of word i/32: the two rows of an even/odd pair sit 16 bits apart)
 */
SDPA_API sdpa_status_t sdpa_dropout_mask_size(const sdpa_problem_t* p, size_t* bytes, size_t* bytes_t);

/*
 * Draws the dropout keep bits for p->dropout_p (in [0, 1)) with the counter-based generator
 * Philox4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3",
 * SC'11).  Element n of the row-major grid [b*h_q][s_q][ceil(s_kv/128)*128] takes the 16-bit
 * half n%2 (0 = low) of 32-bit word (n%8)/2 of the block for the 128-bit counter (n/8, offset)
 * and the 64-bit key seed (each as 32-bit words, low word first), and is kept iff that value
 * is >= round(dropout_p * 65536).  The same (seed, offset) gives the same bits on every run
 * and device; advance `offset` between steps for fresh draws.
 *   mask, mask_t: DEVICE arrays of sdpa_dropout_mask_size bytes, 16-byte aligned; either may
 *   be NULL (not written).  Bits of padded positions (keys >= s_kv in `mask`, rows >= s_q in
 *   `mask_t`) are written too and are not used.  When p->causal is 1 or 2 and no seq_lens
 *   are given, 128x128 tiles that lie wholly above the causal diagonal are not written (the
 *   attention kernels never use them); pass causal = 0 for the full grid.
 */
SDPA_API sdpa_status_t sdpa_dropout_mask(const sdpa_problem_t* p, uint64_t seed, uint64_t offset,
                                         uint32_t* mask, uint32_t* mask_t, void* stream /* cudaStream_t */);

/* Message for the last non-OK status returned on the calling thread ("" if none).  The
 * pointer stays valid until the next library call on this thread [cuDNN 9 blog: errors
 * come with a retrievable last-error string]. */
SDPA_API const char* sdpa_last_error_string(void);

/*
 * Device-side error word of the current device: bit 0 = a bounded wait inside a kernel
 * gave up (the kernel then skipped its remaining work and returned without faulting);
 * bit 1 = shared memory was not 1024-byte aligned (the kernel did nothing).
 * Synchronises the device, writes the word to *flags and clears it.  Returns SDPA_OK, or
 * SDPA_ERR_CUDA if the synchronisation or copy failed.
 */
SDPA_API sdpa_status_t sdpa_device_error(uint32_t* flags);

/* Library version as major*10000 + minor*100 + patch. */
SDPA_API int sdpa_version(void);

/* sizeof(sdpa_problem_t) as compiled into the library, so that bindings built from this
 * header can check their copy of the struct layout. */
SDPA_API size_t sdpa_problem_struct_size(void);

#ifdef __cplusplus
}
#endif

#endif /* SDPA_GB300_H */
