/*
 * mla.h -- C ABI of libmla.so: absorbed Multi-head Latent Attention (MLA)
 * decode over a paged latent cache, hand-written for NVIDIA B300 (sm_103a).
 *
 * The operation (page "02 · DeepSeek-V2 analysis", sections 1.2-1.3, 6.1 and
 * the closing walk of one token through a layer): every token of a layer
 * caches one row of d_c + d_r elements, the RMSNorm'd latent c^KV (d_c = 512)
 * followed by one RoPE key k^R (d_r = 64) that all heads share.  With W^UK
 * absorbed into the query, head h of a query token attends directly over the
 * cached rows:
 *
 *     x_s   = softmax_scale * ( q_nope[h] . c_s  +  q_rope[h] . k^R_s )
 *     a_s   = softmax_s(x_s)          over the visible history s
 *     out[h]= sum_s a_s c_s           (in R^{d_c}; W^UV / W^O applied later)
 *     lse[h]= ln sum_s exp(x_s)
 *
 * with softmax_scale = 1/sqrt(d_h + d_h^R) (eq 18: the per-head width of the
 * concatenated content and RoPE key, not d_c + d_r).
 *
 * Conventions shared by all calls
 *  - Every pointer argument is a DEVICE pointer owned by the caller, except
 *    the mla_cache_t descriptor itself and `status_out`, which are host
 *    pointers read/written during the call only.  The library never
 *    allocates, frees or synchronises device memory in these calls (except
 *    mla_decode_read_status, which synchronises the stream it is given).
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Every call only enqueues work on it and returns.
 *  - Errors are returned, never thrown.  Argument checks that can be done on
 *    the host return MLA_ERR_INVALID_ARG / MLA_ERR_UNSUPPORTED before
 *    anything is launched.  A launch failure returns MLA_ERR_CUDA.  Checks
 *    that need device data (sequence lengths, page ids) are done in the
 *    kernels, which skip the offending work and record MLA_ERR_INVALID_ARG
 *    in the workspace status word; mla_decode_read_status returns it.
 *  - Calls are thread-safe.  The only library state is a per-device cache of
 *    the SM count and kernel attributes.
 *
 * Cache layout: data[num_pages][page_size][d_c + d_r], row = [c_kv || k_R].
 * Token `pos` of sequence `b` lives in page page_table[b][pos / page_size],
 * slot pos % page_size.  A contiguous cache is the identity page table.
 */
#ifndef MLA_H_
#define MLA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MLA_API __attribute__((visibility("default")))
#else
#define MLA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum mla_status {
    MLA_OK = 0,
    MLA_ERR_INVALID_ARG = 1,  /* bad pointer, size, stride or alignment   */
    MLA_ERR_UNSUPPORTED = 2,  /* valid but not implemented (shape, dtype) */
    MLA_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed        */
    MLA_ERR_TIMEOUT = 4,      /* a bounded in-kernel wait ran out         */
    MLA_ERR_WORKSPACE = 5     /* workspace missing or too small           */
} mla_status_t;

typedef enum mla_dtype {
    MLA_BF16 = 0,             /* bfloat16 */
    MLA_FP32 = 1,             /* IEEE float32 */
    MLA_FP8 = 2               /* low-precision cache rows (cache only, see below) */
} mla_dtype_t;

/*
 * Low-precision cache (dtype MLA_FP8): "02 · DeepSeek-V2 analysis",
 * sections 1.3 and 6.2, say the deployed cache is quantised further (to
 * about 6 bits per element) and warn that the quantisation scales must not
 * mix the axis the absorbed product contracts; the page gives no format.
 * This library's format: each token's row is 656 bytes,
 *     bytes [0, 512)    the 512 latent values as FP8 E4M3 codes
 *                       (OCP "E4M3FN": bias 7, max 448, no infinities),
 *     bytes [512, 528)  4 fp32 scales, one per 128 consecutive latent values,
 *     bytes [528, 656)  the 64 RoPE-key values in bf16,
 * value = E4M3(code) * scale.  The scale runs along one token's latent,
 * so it commutes with both contractions over tokens.  `data` is then
 * uint8 [num_pages][page_size][656] (d_c = 512, d_r = 64 only), 16-byte
 * aligned.  mla_cache_append forms the bf16 row (exactly as for a bf16
 * cache) and quantises it: s = amax/448 (fp32 division; 1 for an all-zero
 * group), code = nearest E4M3 (ties to even, saturating) of the
 * fp32-rounded quotient x/s.
 */

/* Describes a paged latent cache.  Plain data; the caller owns both arrays. */
typedef struct mla_cache {
    void* data;                /* device [num_pages][page_size][d_c + d_r] (MLA_FP8: [..][656] bytes) */
    const int32_t* page_table; /* device int32 [B][max_pages_per_seq], page ids     */
    int32_t dtype;             /* mla_dtype_t of `data`                             */
    int32_t num_seqs;          /* rows of page_table (sequences addressable)        */
    int32_t num_pages;         /* pages in the pool (>= 1)                          */
    int32_t page_size;         /* tokens per page: must be 64                       */
    int32_t d_c;               /* latent width: 512 for bf16; 4..512, mult. of 4, fp32 */
    int32_t d_r;               /* RoPE key width: 64 for bf16, 2..64 (even) fp32    */
    int32_t max_pages_per_seq; /* row stride of page_table (>= 1)                   */
} mla_cache_t;

/* flags for mla_cache_append */
#define MLA_APPEND_RMSNORM 1u  /* c_kv row := RMSNorm(c_kv_raw) * gamma          */
#define MLA_APPEND_ROPE    2u  /* k_R row  := RoPE(k_R_raw, position)            */

/*
 * mla_cache_append -- write T new tokens into the cache.
 * Follows the DeepSeek-V2 analysis page: an RMSNorm after the compressed
 * latent (section 1.2), the shared key k^R rotated by RoPE at the token's
 * position and cached (section 1.3, eq 14-15), "the token's 576 elements
 * join the cache" (walk of one token); RoPE rotates the pairs (2i, 2i+1)
 * (page "DeepSeek-V3 model structure", section 2(3)).
 *
 *  ckv_raw  [T][d_c], kr_raw [T][d_r]: in_dtype (bf16 or fp32), row-major.
 *  gamma    [d_c] fp32 or NULL (= all ones).  Used with MLA_APPEND_RMSNORM.
 *  eps      RMSNorm epsilon: y = x / sqrt(mean(x^2) + eps) * gamma.
 *  rope_base  theta_i = rope_base^(-2i/d_r); angle = position * theta_i;
 *           (y_2i, y_2i+1) = (x_2i cos - x_2i+1 sin, x_2i sin + x_2i+1 cos).
 *  seq_ids, positions [T] int32: destination sequence and position.
 *  Without a flag the corresponding part is copied (converted to the cache
 *  dtype).  Arithmetic in fp32 (angles in fp64), one rounding to the cache
 *  dtype (round to nearest even).  Out-of-range seq_id / position / page id
 *  skip the row (nothing is written); that is not reported.
 *  Returns MLA_OK, MLA_ERR_INVALID_ARG (NULL pointers, T < 0, bad cache
 *  descriptor), MLA_ERR_UNSUPPORTED, MLA_ERR_CUDA.  T = 0 is a no-op.
 */
MLA_API mla_status_t mla_cache_append(const mla_cache_t* cache,
                              const void* ckv_raw, const void* kr_raw, int32_t in_dtype,
                              const float* gamma, float eps, float rope_base,
                              const int32_t* seq_ids, const int32_t* positions, int32_t T,
                              uint32_t flags, void* stream);

/*
 * RoPE with YaRN context extension (DeepSeek-V2 analysis page, section 3.2
 * "YaRN extends 4K to 128K").  In MLA only the decoupled RoPE key k^R and the
 * RoPE queries carry positions, so YaRN acts on those d_r dims alone; the
 * page gives the extension factor s = 40, alpha = 1, beta = 32 (4K x 40 =
 * 160K).  Frequency of pair i (the page refers to the published YaRN rule
 * for the interpolation; that rule is what is implemented):
 *     theta_i   = base^(-2i/d_r),   r_i = original_max_position * theta_i / (2 pi)
 *     gamma_i   = clamp((r_i - alpha) / (beta - alpha), 0, 1)
 *     theta'_i  = theta_i * (gamma_i + (1 - gamma_i) / s)
 * i.e. pairs that turn more than beta times over the original window keep
 * their frequency, pairs that turn less than alpha times are interpolated by
 * 1/s, and a linear ramp joins the two.  yarn_factor = 1 is plain RoPE.
 */
typedef struct mla_rope {
    float base;                     /* RoPE base, e.g. 10000                        */
    float yarn_factor;              /* s >= 1; 1 = no extension                     */
    float yarn_alpha;               /* ramp start (turns over the window), 1        */
    float yarn_beta;                /* ramp end, > yarn_alpha, 32                   */
    int32_t original_max_position;  /* window before extension, e.g. 4096 (>= 1)   */
} mla_rope_t;

/*
 * mla_cache_append_rope -- mla_cache_append with the RoPE frequencies of
 * `rope` (host pointer, read during the call).  Arguments and errors as
 * mla_cache_append; MLA_ERR_INVALID_ARG also for base <= 0, yarn_factor < 1,
 * yarn_beta <= yarn_alpha or original_max_position < 1 when
 * MLA_APPEND_ROPE is set.  mla_cache_append(..., rope_base, ...) equals this
 * call with yarn_factor = 1.
 */
MLA_API mla_status_t mla_cache_append_rope(const mla_cache_t* cache,
                              const void* ckv_raw, const void* kr_raw, int32_t in_dtype,
                              const float* gamma, float eps, const mla_rope_t* rope,
                              const int32_t* seq_ids, const int32_t* positions, int32_t T,
                              uint32_t flags, void* stream);

/*
 * mla_yarn_softmax_scale -- softmax scale of a YaRN-extended model.  YaRN's
 * attention temperature sqrt(1/t) = coef * ln(s) + 1 (coef = 0.0707 in
 * DeepSeek-V2, 0.1 in the original YaRN; the page's "sqrt(t)" is a typo for
 * sqrt(1/t)) scales q and k each in the original, i.e. the logits by 1/t.
 * Because only d_r of the dims carry RoPE in MLA, the temperature is moved
 * onto the softmax scale: returns softmax_scale * (coef * ln(s) + 1)^2
 * (s = 40: factor 1.2608^2 = 1.590).  s <= 1 returns softmax_scale.
 * Host-only arithmetic; no device work.
 */
MLA_API float mla_yarn_softmax_scale(float softmax_scale, float yarn_factor, float coef);

/*
 * mla_decode -- absorbed MLA attention of Q query tokens per sequence.
 *
 *  seq_lens [B] int32 (device): cached tokens of each sequence, INCLUDING
 *           its Q query tokens (already appended).  Query j (0 <= j < Q) of
 *           sequence b sits at position seq_lens[b]-Q+j and sees positions
 *           0..seq_lens[b]-Q+j (causal).  A query that sees no position gets
 *           out = 0 and lse = -inf.  0 <= seq_lens[b] <= max_pages_per_seq*64.
 *  q_nope   [B][Q][H][d_c] absorbed content queries, cache dtype.
 *  q_rope   [B][Q][H][d_r] RoPE queries, already rotated at their position.
 *  softmax_scale  usually 1/sqrt(d_h + d_h^R).
 *  out      [B][Q][H][d_c], cache dtype.   lse [B][Q][H] fp32 or NULL.
 *  workspace / workspace_bytes: device scratch of at least
 *           mla_decode_workspace_size(B, Q, H, d_c, 0, 0) bytes, 256-byte
 *           aligned, owned by the caller; its contents are not needed
 *           between calls.  Calls sharing a workspace must not overlap.
 *  Shapes: bf16 cache needs d_c = 512, d_r = 64, page_size = 64, Q*H <= 4096,
 *  16-byte aligned cache/q/out; fp32 cache needs d_c <= 512 (multiple of 4)
 *  and d_r <= 64 (even).  B <= cache->num_seqs.  The work is split across the
 *  SMs by a balanced partition of all key tiles (flash-decoding), then
 *  partial results are merged by log-sum-exp.
 *  Equivalent to mla_decode_plan(n_split = 0) + mla_decode_attend +
 *  mla_decode_combine.
 */
MLA_API mla_status_t mla_decode(const mla_cache_t* cache, const int32_t* seq_lens, int32_t B,
                        const void* q_nope, const void* q_rope, int32_t Q, int32_t H,
                        float softmax_scale, void* out, float* lse,
                        void* workspace, size_t workspace_bytes, void* stream);

/*
 * mla_decode_split_combine -- same result as mla_decode, but every sequence's
 * visible keys are cut into n_split (1..1024) equal chunks of whole 64-token
 * tiles; each chunk yields a partial (fp32 out, lse) and the chunks are merged
 * by log-sum-exp: lse = ln sum_j exp(lse_j), out = sum_j exp(lse_j - lse) out_j.
 * Chunks past the end of a short sequence are empty and contribute nothing.
 * Workspace: mla_decode_workspace_size(B, Q, H, d_c, n_split, 0).
 */
MLA_API mla_status_t mla_decode_split_combine(const mla_cache_t* cache, const int32_t* seq_lens, int32_t B,
                                      const void* q_nope, const void* q_rope, int32_t Q, int32_t H,
                                      float softmax_scale, int32_t n_split, void* out, float* lse,
                                      void* workspace, size_t workspace_bytes, void* stream);

/*
 * Bytes of workspace needed by a decode of this shape.  n_split = 0 selects
 * the balanced partition of mla_decode, n_split >= 1 the uniform split of
 * mla_decode_split_combine.  num_sms = 0 queries the current device.
 * Returns 0 for invalid arguments.
 */
MLA_API size_t mla_decode_workspace_size(int32_t B, int32_t Q, int32_t H, int32_t d_c,
                                 int32_t n_split, int32_t num_sms);

/*
 * The three phases of a decode, callable one by one.  The plan depends only
 * on seq_lens, B, Q, H, n_split and the device, so a caller that decodes
 * several layers with the same lengths may plan once and attend/combine per
 * layer.  mla_decode_plan writes the partition of work into `workspace`;
 * mla_decode_attend runs the attention kernel and writes final rows into
 * out/lse and partial rows into the workspace; mla_decode_combine merges the
 * partial rows.  All three take the same workspace and the same n_split
 * (0 = balanced); the cache dtype and the unit size select the kernel:
 * bf16 or low-precision (E4M3) rows with more than 16 query rows per unit
 * (Q * H > 16) take the two-SM tcgen05 kernel, bf16 rows with Q * H <= 16
 * the single-SM warp-MMA kernel, fp32 rows the CUDA-core kernel.  Plan,
 * attend and combine must see the same cache, Q, H and n_split.
 */
MLA_API mla_status_t mla_decode_plan(const mla_cache_t* cache, const int32_t* seq_lens, int32_t B,
                             int32_t Q, int32_t H, int32_t n_split,
                             void* workspace, size_t workspace_bytes, void* stream);
MLA_API mla_status_t mla_decode_attend(const mla_cache_t* cache, const int32_t* seq_lens, int32_t B,
                               const void* q_nope, const void* q_rope, int32_t Q, int32_t H,
                               float softmax_scale, int32_t n_split, void* out, float* lse,
                               void* workspace, size_t workspace_bytes, void* stream);
MLA_API mla_status_t mla_decode_combine(const mla_cache_t* cache, int32_t B, int32_t Q, int32_t H,
                                int32_t n_split, void* out, float* lse,
                                void* workspace, size_t workspace_bytes, void* stream);

/*
 * Synchronises `stream`, then returns (and clears) the status word the
 * kernels of the last decode on `workspace` recorded: MLA_OK,
 * MLA_ERR_INVALID_ARG (bad sequence length or page id met on the device) or
 * MLA_ERR_TIMEOUT (a bounded wait ran out; the kernel stopped cleanly).
 * The code is also stored in *status_out when status_out is not NULL.
 */
MLA_API mla_status_t mla_decode_read_status(void* workspace, size_t workspace_bytes, void* stream,
                                    int32_t* status_out);

/*
 * Self-test of the bounded wait used by every in-kernel wait: launches one
 * block that waits on a barrier nothing ever completes, gives up after
 * `timeout_us` microseconds, records MLA_ERR_TIMEOUT in the workspace status
 * word and exits.  Lets a test exercise the timeout path without a hang.
 */
MLA_API mla_status_t mla_selftest_bounded_wait(void* workspace, size_t workspace_bytes,
                                       uint32_t timeout_us, void* stream);

/*
 * mla_decode_noalloc -- mla_decode for callers that cannot give the library
 * any device memory of its own (no workspace argument).  The pages have no
 * counterpart to this entry point; it exists for integration only.
 *
 * Callers such as a plugin that only receives its input and output buffers
 * from a host framework, or a serving loop that forbids device allocation
 * after start-up, cannot call cudaMalloc.  This entry point runs exactly the
 * decode of mla_decode (same arguments minus the workspace, same results)
 * using a fixed scratch array of MLA_NOALLOC_SCRATCH_BYTES compiled into the
 * library: it calls no allocator.  Every GPU that loads the library holds the
 * array until the process exits.
 *  - Returns MLA_ERR_WORKSPACE, launching nothing, when the decode needs more
 *    scratch than MLA_NOALLOC_SCRATCH_BYTES, i.e. more than
 *    mla_decode_workspace_size(B, Q, H, d_c, 0, clusters) bytes.  On a
 *    148-SM B300 that allows up to 117 units on the bf16 path and 43 on the
 *    fp32 path (a unit is one sequence x up to 128 query rows j*H+h, so
 *    B = 117 sequences at H = 128, Q = 1).
 *  - All calls on a device share the array; each call rewrites what it reads,
 *    but calls that overlap on the GPU race and must be serialised.
 *  - The first call on each device looks up the array's device address (with
 *    that device current); make that first call before any stream capture.
 *  - Device-side problems (bad lengths, page ids) give zero rows as in
 *    mla_decode; their status word is internal and not reported here.
 */
#define MLA_NOALLOC_SCRATCH_BYTES (48u << 20)
MLA_API mla_status_t mla_decode_noalloc(const mla_cache_t* cache, const int32_t* seq_lens, int32_t B,
                                        const void* q_nope, const void* q_rope, int32_t Q, int32_t H,
                                        float softmax_scale, void* out, float* lse, void* stream);

/* Static description of a status code. */
/*
 * Absorption GEMMs either side of the attention ("02 · DeepSeek-V2
 * analysis", section 1.2, the paragraph on absorbing W^UK into the query, and
 * section 6.1, where each head aggregates the latents with its own weights
 * and W^UV is applied afterwards).  bf16 in and out, fp32 accumulation on
 * the tensor cores.
 *
 *  mla_absorb_query:  q_nope[n][h][:] = W^UK[h]^T q_c[n][h][:]
 *      w_uk   [H][d_h][d_c]   (the up-projection of keys, per head)
 *      q_c    [n_rows][H][d_h] content queries
 *      q_nope [n_rows][H][d_c] absorbed queries, the input of mla_decode
 *  mla_absorb_output: o[n][h][:] = W^UV[h] u[n][h][:]
 *      w_uv   [H][d_h][d_c]   (the up-projection of values, per head)
 *      u      [n_rows][H][d_c] aggregated latents, the output of mla_decode
 *      o      [n_rows][H][d_h] per-head attention outputs (W^O is applied
 *             by the caller)
 *
 *  All arrays are dense row-major device memory owned by the caller; w and
 *  the activation input must be 16-byte aligned.  d_h and d_c must be
 *  multiples of 128 (MLA_ERR_UNSUPPORTED otherwise); n_rows = 0 is a no-op.
 *  status: NULL or a device int32 that receives MLA_ERR_TIMEOUT if an
 *  in-kernel wait ran out (the kernel then stops cleanly; the output is
 *  undefined).  Asynchronous on `stream`.
 */
MLA_API mla_status_t mla_absorb_query(const void* w_uk, const void* q_c, void* q_nope, int32_t n_rows,
                                      int32_t H, int32_t d_h, int32_t d_c, int32_t* status, void* stream);
MLA_API mla_status_t mla_absorb_output(const void* w_uv, const void* u, void* o, int32_t n_rows,
                                       int32_t H, int32_t d_h, int32_t d_c, int32_t* status, void* stream);

/* ------------------------------------------------------------------------
 * Expanded (prefill) attention
 *
 * "02 · DeepSeek-V2 analysis", sections 1.2-1.3 (eq 10-11 up-projections,
 * eq 14-18 decoupled RoPE and the scaled two-part score) and section 6
 * (prefill may materialise K and V; decode absorbs them; the two forms are
 * one function in exact arithmetic).  For the first T tokens of sequence
 * `seq` of the cache (already appended, positions 0..T-1):
 *
 *   K^C[t][h] = W^UK[h] c_t,  V[t][h] = W^UV[h] c_t        (materialised)
 *   o[t][h]   = sum_{s<=t} softmax_s(scale ([q_c[t][h] || q_r[t][h]] .
 *                                           [K^C[s][h] || k^R_s])) V[s][h]
 *   lse[t][h] = ln sum_{s<=t} exp(scale * score)
 *
 * with c_t the cached latent row (d_c = 512) and k^R_s the cached, rotated
 * RoPE key (d_r = 64, shared by every head).  Causal: query t sees keys
 * 0..t.  bf16 cache only; d_h = 128 and H even (MLA_ERR_UNSUPPORTED
 * otherwise).
 *
 *   w_uk, w_uv  bf16 [H][128][512]   per-head key / value up-projections
 *   q_c         bf16 [T][H][128]     content queries
 *   q_r         bf16 [T][H][64]      RoPE queries, already rotated at t
 *   out         bf16 [T][H][128]     per-head outputs (W^O applied by the caller)
 *   lse         fp32 [T][H] or NULL
 *   workspace   caller-owned device memory of mla_prefill_workspace_size(T, H)
 *               bytes, 256-byte aligned: a status word (read it with
 *               mla_decode_read_status) and the materialised K^C and V.
 *
 * All pointers are device memory owned by the caller, 16-byte aligned.
 * Asynchronous on `stream`; host-side checks return before any launch,
 * device-side checks (page ids) and in-kernel timeouts are recorded in the
 * workspace status word.
 * ---------------------------------------------------------------------- */
MLA_API size_t mla_prefill_workspace_size(int32_t T, int32_t H);
MLA_API mla_status_t mla_prefill_expanded(const mla_cache_t* cache, int32_t seq, int32_t T, const void* w_uk,
                                          const void* w_uv, const void* q_c, const void* q_r, int32_t H,
                                          float softmax_scale, void* out, float* lse, void* workspace,
                                          size_t workspace_bytes, void* stream);
/* The two phases of mla_prefill_expanded, same arguments and workspace:
 * mla_prefill_project materialises K^C and V in the workspace (and clears
 * its status word); mla_prefill_attend then runs the causal attention over
 * them.  A caller that wants the materialised K / V for several query sets
 * projects once. */
MLA_API mla_status_t mla_prefill_project(const mla_cache_t* cache, int32_t seq, int32_t T, const void* w_uk,
                                         const void* w_uv, int32_t H, void* workspace, size_t workspace_bytes,
                                         void* stream);
MLA_API mla_status_t mla_prefill_attend(const mla_cache_t* cache, int32_t seq, int32_t T, const void* q_c,
                                        const void* q_r, int32_t H, float softmax_scale, void* out, float* lse,
                                        void* workspace, size_t workspace_bytes, void* stream);

MLA_API const char* mla_status_string(mla_status_t status);

/* Library version as major*10000 + minor*100 + patch. */
MLA_API int32_t mla_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MLA_H_ */
