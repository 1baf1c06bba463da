/*
 * decode_step.h — C ABI of the GB300 (sm_103a) single-token decode step.
 *
 * Every call takes plain pointers and sizes.  Unless stated otherwise:
 *  - Buffers are DEVICE pointers owned by the caller; the library allocates
 *    no device memory in any call (a decode step "runs with zero heap
 *    allocations", "Inside the engine", section 1, "CausalLM: the forward
 *    path").  Scratch space is a caller-supplied workspace whose size a
 *    *_workspace_bytes call reports; a workspace must be zero-filled before
 *    its first use and is left ready for the next call by every call.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *    default stream) and return before the GPU work finishes.
 *  - Every length argument is an element count.  Each buffer's real length
 *    is passed next to it and checked against the length the operation
 *    needs, as the "LLM inference kernels" page's contract checks do
 *    ("Status vocabulary and the shape checks (contract)", "Guarantees").
 *    On any refusal the call returns before launching anything and leaves
 *    every output untouched.
 *  - Only what the host can see is checked on the host.  Values that live in
 *    device memory (token ids, positions, sequence lengths) are checked by the
 *    kernels: an out-of-range value is clamped or skipped and a bit is set in
 *    the workspace's error word (see ds_workspace_error).
 *  - Identical inputs give bit-identical outputs run to run: no reduction
 *    depends on the order in which thread blocks finish.
 *  - fp32 activations; weights fp32 or bf16; KV cache fp32 or bf16; fp32
 *    accumulation.
 */
#ifndef DECODE_STEP_H
#define DECODE_STEP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(_WIN32)
#define DS_API
#else
#define DS_API __attribute__((visibility("default")))
#endif

/* A cudaStream_t, declared without the CUDA headers. */
typedef struct CUstream_st *ds_stream_t;

/* ---------------------------------------------------------------------
 * Status vocabulary.  560-571 keep the numbers and meanings of the
 * "LLM inference kernels" page ("Status vocabulary and the shape checks
 * (contract)"); 572-577 are this library's additions in the unused part of
 * the same 560-579 range.
 * ------------------------------------------------------------------- */
enum {
    DS_OK = 560,                      /* ran; every output element is defined */
    DS_EMPTY_DIMENSION = 561,         /* a required dimension was < 1 */
    DS_A_LENGTH_MISMATCH = 562,       /* first operand's length != n */
    DS_B_LENGTH_MISMATCH = 563,       /* second operand's length != n */
    DS_DIMENSION_TOO_LARGE = 564,     /* a dimension exceeds DS_MAX_DIM */
    DS_CODE_OUT_OF_RANGE = 565,       /* ds_status_name's answer for an unknown code */
    DS_CACHE_LENGTH_MISMATCH = 566,   /* cache length / position out of range */
    DS_NEW_LENGTH_MISMATCH = 567,     /* appended values' length != n_new */
    DS_LOGITS_LENGTH_MISMATCH = 568,  /* logits length != n_rows * n */
    DS_GEMV_A_LENGTH_MISMATCH = 569,  /* matrix length != rows * cols */
    DS_GEMV_X_LENGTH_MISMATCH = 570,  /* vector length != the reduced dimension */
    DS_CACHE_CAPACITY_EXCEEDED = 571, /* an append would overrun the reserved cache */
    DS_BAD_DTYPE = 572,               /* dtype or layout code not supported here */
    DS_CUDA_ERROR = 573,              /* a CUDA runtime call failed */
    DS_WORKSPACE_TOO_SMALL = 574,     /* workspace NULL or smaller than required */
    DS_BAD_SAMPLING_PARAM = 575,      /* temperature/top_k/top_p outside their domain */
    DS_TOKEN_OUT_OF_RANGE = 576,      /* a host-visible token id outside [0, vocab) */
    DS_BAD_ARGUMENT = 577             /* NULL pointer, misaligned pointer or bad count */
};

/* Largest accepted dimension (per dimension), 1 << 24, as on the
 * "LLM inference kernels" page ("Status vocabulary and the shape checks"). */
#define DS_MAX_DIM (1LL << 24)

/* Storage dtypes. */
enum { DS_F32 = 0, DS_BF16 = 1 };

/* RoPE layouts: pairs (p, p + head_dim/2) — the GPT-NeoX split-half
 * convention ("LLM inference kernels", "Two gaps, not three") — or pairs
 * (2p, 2p + 1) ("The forward pass end to end", "The code"). */
enum { DS_ROPE_HALF_SPLIT = 0, DS_ROPE_INTERLEAVED = 1 };

/* Bits of a workspace's error word (set by kernels, never by the host). */
enum {
    DS_ERR_TOKEN_RANGE = 1,   /* a device-side token id was outside [0, vocab); clamped */
    DS_ERR_POSITION = 2,      /* a device-side position or length exceeded the cache */
    DS_ERR_WAIT_TIMEOUT = 4,  /* a bounded wait inside a kernel gave up */
    DS_ERR_SAMPLING = 8       /* a sampler row had no finite logits */
};

/* Name of a status code ("ds_ok", "ds_a_length_mismatch", ...);
 * "ds_code_out_of_range" for anything else.  Static storage. */
DS_API const char *ds_status_name(int code);

/* The residual-add shape check of the "LLM inference kernels" contract:
 * 561 if n < 1, 564 if n > DS_MAX_DIM, 562 if a_len != n, 563 if b_len != n,
 * else 560.  Host only. */
DS_API int ds_residual_dims_check(int64_t n, int64_t a_len, int64_t b_len);

/* Copy a workspace's error word (int32 at byte 0 of every workspace) to
 * *host_word and clear it.  Synchronises `stream`. */
DS_API int ds_workspace_error(void *workspace, int32_t *host_word, ds_stream_t stream);

/* Number of streaming multiprocessors the library sizes its grids for on the
 * current device (0 when no device is usable). */
DS_API int ds_device_sm_count(void);

/* ---------------------------------------------------------------------
 * Projections
 * ------------------------------------------------------------------- */

/* Workspace bytes ds_gemv_transposed needs for a rows x cols matrix. */
DS_API size_t ds_gemv_workspace_bytes(int64_t rows, int64_t cols, int a_dtype);

/* y = A^T x: y[j] = sum_i A[i * cols + j] * x[i] for j < cols.
 * The transposed mat-vec of "LLM inference kernels" ("A parallel path for
 * one frozen kernel's known-slow shape"): A is row-major with `rows` input
 * rows and `cols` output columns, the layout of every decode-step projection.
 *   A: rows*cols elements of a_dtype (a_len must equal rows*cols, else 569)
 *   x: rows fp32 (x_len must equal rows, else 570); y: cols fp32 (y_len must
 *   equal cols, else 562); 561 / 564 for an empty / oversized dimension.
 *   workspace: ds_gemv_workspace_bytes(rows, cols, a_dtype) bytes, zeroed
 *   before first use.
 * Weight rows stream through shared memory with bulk asynchronous copies when
 * A is 16-byte aligned and cols * element size is a multiple of 16 bytes;
 * other shapes run a plain-load kernel with the same result definition. */
DS_API int ds_gemv_transposed(const void *A, int64_t a_len, int a_dtype, const float *x,
                              int64_t x_len, int64_t rows, int64_t cols, float *y,
                              int64_t y_len, void *workspace, size_t workspace_bytes,
                              ds_stream_t stream);

/* ds_gemv_transposed for callers that cannot allocate device memory (for
 * example a host whose device memory is all owned by its own allocator, or a
 * plug-in handed nothing but one operation's inputs and outputs).  The pages
 * have no counterpart of this call.  Same arguments, result and checks as
 * ds_gemv_transposed, minus the workspace: the split-reduction scratch comes
 * from a fixed area compiled into the library, which every GPU that loads the
 * library keeps (ds_gemv_transposed_noalloc_max_bytes() bytes, 1 MiB) until
 * the process exits.  A matrix on the streamed path (A 16-byte aligned and
 * cols * element size a multiple of 16 bytes) whose scratch
 * (ds_gemv_workspace_bytes) does not fit in the area is refused with
 * DS_DIMENSION_TOO_LARGE; any other matrix runs the plain-load kernel, which
 * uses no scratch.  The call allocates nothing: on the streamed path it clears
 * the band counters with one asynchronous memset, then launches the kernel on
 * `stream`.
 *  - The first call on a device (that device current) looks up the area's
 *    device address, which is kept for the life of the process; make that
 *    first call before any stream capture.  After cudaDeviceReset the kept
 *    address is stale: the call must not be used again in that process.
 *  - All calls share the one area and it keeps the last call's contents:
 *    calls whose GPU work overlaps (other streams, other threads) race on it
 *    and must be ordered by the caller.
 *  - A kernel's error bits (DS_ERR_*) collect in the area's error word across
 *    calls until ds_gemv_transposed_noalloc_error reads and clears it. */
DS_API int ds_gemv_transposed_noalloc(const void *A, int64_t a_len, int a_dtype, const float *x,
                                      int64_t x_len, int64_t rows, int64_t cols, float *y,
                                      int64_t y_len, ds_stream_t stream);
DS_API size_t ds_gemv_transposed_noalloc_max_bytes(void);
/* Copy the no-allocation area's error word (of the current device) to
 * *host_word and clear it, as ds_workspace_error does for a workspace.
 * Synchronises `stream`. */
DS_API int ds_gemv_transposed_noalloc_error(int32_t *host_word, ds_stream_t stream);

/* y = W x: y[r] = sum_c W[r * cols + c] * x[c] for r < rows — the
 * untransposed form the "LLM inference kernels" page uses for lm_head.
 *   W: rows*cols of w_dtype (569), x: cols fp32 (570), y: rows fp32 (562). */
DS_API int ds_gemv(const void *W, int64_t w_len, int w_dtype, const float *x, int64_t x_len,
                   int64_t rows, int64_t cols, float *y, int64_t y_len, ds_stream_t stream);

/* ---------------------------------------------------------------------
 * Batched projections (tensor cores)
 *
 * When one step decodes n sequences ("Inside the engine", section 4:
 * batched decode, one token per sequence per step) each projection applies
 * the same matrix to n activation vectors: a skinny GEMM, run on the tcgen05
 * tensor cores with bf16 operands and fp32 accumulation.  n is 1..256.
 * ------------------------------------------------------------------- */

/* Workspace bytes ds_gemm_transposed / ds_gemm need for n vectors and a
 * rows x cols matrix (either orientation); 0 for an unsupported shape. */
DS_API size_t ds_gemm_workspace_bytes(int64_t n, int64_t rows, int64_t cols);

/* Y[s][j] = sum_i A[i * cols + j] * X[s * rows + i] for s < n, j < cols:
 * ds_gemv_transposed's y = A^T x ("LLM inference kernels", "A parallel path
 * for one frozen kernel's known-slow shape") for the n rows of X at once.
 *   A: bf16 rows*cols (a_len, else 569); X: bf16 n*rows (x_len, else 570);
 *   Y: fp32 n*cols (y_len, else 562).  rows and cols multiples of 8, A and X
 *   16-byte aligned (577).  561 / 564 for an empty / oversized dimension
 *   (n > 256 included).  workspace: ds_gemm_workspace_bytes(n, rows, cols)
 *   bytes, zeroed before first use. */
DS_API int ds_gemm_transposed(const void *A, int64_t a_len, const void *X, int64_t x_len, int64_t n,
                              int64_t rows, int64_t cols, float *Y, int64_t y_len, void *workspace,
                              size_t workspace_bytes, ds_stream_t stream);

/* Y[s][r] = sum_c W[r * cols + c] * X[s * cols + c] for s < n, r < rows: the
 * untransposed form of the output head (ds_gemv) for n vectors.
 *   W: bf16 rows*cols (569); X: bf16 n*cols (570); Y: fp32 n*rows (562);
 *   cols a multiple of 8; other checks as ds_gemm_transposed. */
DS_API int ds_gemm(const void *W, int64_t w_len, const void *X, int64_t x_len, int64_t n, int64_t rows,
                   int64_t cols, float *Y, int64_t y_len, void *workspace, size_t workspace_bytes,
                   ds_stream_t stream);

/* ---------------------------------------------------------------------
 * Decode glue
 * ------------------------------------------------------------------- */

/* out[i] = a[i] + b[i] in fp32 for i < n ("LLM inference kernels",
 * "Residual add").  a_len/b_len must equal n (562/563); out has n elements and
 * may alias a or b. */
DS_API int ds_residual_add(const float *a, int64_t a_len, const float *b, int64_t b_len,
                           float *out, int64_t n, ds_stream_t stream);

/* residual += x (fp32, in place), then h = residual * (mean(residual^2) + eps)^(-1/2) * w,
 * the square sum accumulated in fp32 ("decode-ops", "Usage" and
 * "API — Method"; "The forward pass end to end", "The code", rmsnorm).
 * x may be NULL (plain RMSNorm; x_len ignored).  residual_len (562), x_len
 * (563), w_len and h_len (562) must equal n; w is fp32 or bf16. */
DS_API int ds_add_rmsnorm(float *residual, int64_t residual_len, const float *x, int64_t x_len,
                          const void *w, int64_t w_len, int w_dtype, float eps, float *h,
                          int64_t h_len, int64_t n, ds_stream_t stream);

/* Rotate q (n_qh heads) and k (n_kh heads, may be NULL with n_kh = 0) of
 * head_dim values each, in place, to position `pos`: pair p turns by
 * pos * base^(-2p/head_dim), the head_dim/2 angles formed once per call in fp64
 * on the host and rounded to fp32 ("decode-ops", "API — Method"), the rotation
 * applied in fp32 on the device.  layout: DS_ROPE_*.
 * q_len must be n_qh*head_dim (562), k_len n_kh*head_dim (563); head_dim
 * even and <= 1024 (577); pos >= 0 (566). */
DS_API int ds_rope(float *q, int64_t q_len, float *k, int64_t k_len, int64_t pos, int n_qh,
                   int n_kh, int head_dim, double base, int layout, ds_stream_t stream);

/* Reserved-capacity KV append: write the n_new fp32 values into
 * cache[cache_len, cache_len + n_new) in place, converted to cache_dtype
 * (bf16: round to nearest even) ("LLM inference kernels", "The hot loop
 * doesn't call kv_cache_append_flat").  `capacity` is the cache's reserved
 * element count.  561 for n_new < 1, 567 if new_len != n_new, 566 if
 * cache_len < 0, 571 if cache_len + n_new > capacity. */
DS_API int ds_kv_cache_append(void *cache, int cache_dtype, int64_t capacity, int64_t cache_len,
                              const float *new_vals, int64_t new_len, int64_t n_new,
                              ds_stream_t stream);

/* out[i] = silu(gate[i]) * up[i], silu(z) = z / (1 + e^-z), fp32
 * ("decode-ops", "Usage": silu_mul).  gate_len (562), up_len (563) equal n. */
DS_API int ds_silu_mul(const float *gate, int64_t gate_len, const float *up, int64_t up_len,
                       float *out, int64_t n, ds_stream_t stream);

/* ---------------------------------------------------------------------
 * Attention
 * ------------------------------------------------------------------- */

/* Workspace bytes for ds_gqa_decode_attn. */
DS_API size_t ds_attention_workspace_bytes(int n_seqs, int n_qh, int n_kvh, int head_dim,
                                           int64_t max_ctx);

/* Grouped-query attention of one new query token per sequence over its
 * cached positions ("The forward pass end to end", "The code":
 * forward_token's attention; split across the context and reduced, "Inside
 * the engine", section 1).  For sequence s and query head h, the KV head is
 * g = h / (n_qh / n_kvh); scores q_h . k_t * scale over t < seq_lens[s],
 * softmax, and out[s][h][:] = sum_t w_t v_t.
 *   q: [n_seqs][n_qh][head_dim] fp32.  out: same shape fp32.
 *   k_cache / v_cache: rows of n_kvh*head_dim elements of kv_dtype,
 *   `cache_rows` rows each; position t of sequence s is row
 *   blk * block_tokens + t % block_tokens with blk = block_table[s *
 *   max_blocks_per_seq + t / block_tokens], or, with block_table NULL,
 *   blk = s * max_blocks_per_seq + t / block_tokens (a contiguous slot per
 *   sequence, "Inside the engine", section 3).
 *   seq_lens: device int32 [n_seqs]; a length outside
 *   [1, max_blocks_per_seq*block_tokens] is clamped and flags DS_ERR_POSITION.
 *   n_qh must be a multiple of n_kvh; head_dim a multiple of 4 up to 128, or of 8 up to 256.
 *   workspace: ds_attention_workspace_bytes(...) with max_ctx >= every length. */
DS_API int ds_gqa_decode_attn(const float *q, const void *k_cache, const void *v_cache,
                              int kv_dtype, int64_t cache_rows, const int32_t *block_table,
                              int max_blocks_per_seq, int block_tokens, const int32_t *seq_lens,
                              int n_seqs, int n_qh, int n_kvh, int head_dim, float scale,
                              float *out, void *workspace, size_t workspace_bytes,
                              ds_stream_t stream);

/* ---------------------------------------------------------------------
 * Picking the next token
 * ------------------------------------------------------------------- */

DS_API size_t ds_argmax_workspace_bytes(int n_rows, int64_t n);

/* ids[r] = first index of the maximum of row r of logits [n_rows][n]
 * ("LLM inference kernels", "KV-cache growth and greedy argmax": ties go to
 * the first id; "decode-ops", "Correctness": exact against torch.argmax, NaN
 * ranking above every number).  max_logit (optional) gets the row maxima.
 * logits_len must be n_rows*n (568). */
DS_API int ds_greedy_argmax(const float *logits, int64_t logits_len, int n_rows, int64_t n,
                            int32_t *ids, float *max_logit, void *workspace,
                            size_t workspace_bytes, ds_stream_t stream);

DS_API size_t ds_sample_workspace_bytes(int n_rows, int64_t n);

/* Per row r of logits [n_rows][n], with the explicit uniform draw u[r] in
 * [0,1): temperature -> top-k -> softmax over the survivors -> top-p ->
 * renormalise -> inverse CDF at u ("decode-ops", "API — Method", the
 * HuggingFace warper order).  In this order: l' = l / T (fp32); survivors =
 * the top_k largest l', ties to the lower index, in descending order;
 * e_i = exp(l'_i - l'_max) (fp32); p_i = e_i / (sum of e over the
 * survivors); keep the prefix whose exclusive running sum of p is < top_p (at
 * least one; top_p >= 1 keeps all); token = first kept survivor whose
 * inclusive running sum exceeds u * (sum of kept p), else the last kept.
 * The running sums are exact sums of the e_i, each rounded to a multiple of
 * 2^-F of the largest (F = min(46, 63 - ceil(log2 n)): 2^-46 at a 128,256
 * vocabulary), so the token does not depend on summation order.
 *   temperature <= 0: greedy (first index of the maximum).
 *   top_k: any value; <= 0 or >= n means no top-k cut.
 *   top_p in (0, 1].  575 for a parameter outside its domain.
 *   u: device fp32 [n_rows]; ids: device int32 [n_rows].
 * A row whose largest scaled logit is NaN or infinite gets the first index of
 * that value and sets DS_ERR_SAMPLING in the workspace's error word.
 * Each row runs as one cluster of up to 8 thread blocks; no allocation, no
 * workspace beyond the error word. */
DS_API int ds_sample(const float *logits, int64_t logits_len, int n_rows, int64_t n,
                     float temperature, int top_k, float top_p, const float *u, int32_t *ids,
                     void *workspace, size_t workspace_bytes, ds_stream_t stream);

/* ---------------------------------------------------------------------
 * The decode step
 * ------------------------------------------------------------------- */

/* Model shape ("The forward pass end to end", "The code": Config, with the
 * head dimension explicit). */
typedef struct {
    int32_t vocab, d, n_layer, n_qh, n_kvh, head_dim, ff;
    int32_t rope_layout; /* DS_ROPE_* */
    double rope_base;
    float eps;           /* RMSNorm epsilon */
    int32_t tied;        /* 1: the output head is the embedding table */
    int32_t w_dtype;     /* DS_F32 or DS_BF16, for emb, out and projections */
    int32_t kv_dtype;    /* DS_F32 or DS_BF16 */
    int32_t max_seqs;    /* largest n_seqs a step will be given, 1..256.  Above 1 every step
                          * runs the batched path: the projections as GEMMs over the batch on
                          * the tcgen05 tensor cores ("Inside the engine", section 4: batched
                          * decode), which needs bf16 weights (else 572) and a head_dim that
                          * divides 128 (else 577). */
    int32_t max_ctx;     /* largest position + 1 a step will see */
    /* Long-context RoPE scaling as Llama 3.1 checkpoints define it (not on the
     * pages): pair p's frequency f = rope_base^(-2p/head_dim), wavelength
     * w = 2 pi / f, becomes f where w < rope_orig_max_pos / rope_high_freq_factor,
     * f / rope_factor where w > rope_orig_max_pos / rope_low_freq_factor, and
     * (1 - s) f / rope_factor + s f in between, with
     * s = (rope_orig_max_pos / w - rope_low_freq_factor) /
     *     (rope_high_freq_factor - rope_low_freq_factor).
     * rope_factor 0 (a zeroed struct): no scaling.  Otherwise rope_factor >= 1,
     * 0 < rope_low_freq_factor < rope_high_freq_factor and rope_orig_max_pos > 0
     * (else 577).  Applies to every position of the model's RoPE table. */
    double rope_factor;
    double rope_low_freq_factor, rope_high_freq_factor;
    double rope_orig_max_pos;
} ds_model_config;

/* Device pointers to the weights, in this storage layout:
 *   emb [vocab][d]; out [vocab][d] (ignored when tied); final_norm [d] fp32;
 *   per layer (host arrays of n_layer device pointers):
 *   n1, n2 [d] fp32;  wqkv [d][(n_qh + 2 n_kvh) head_dim] with the q columns,
 *   then k, then v;  wo [n_qh head_dim][d];  wgu [d][2 ff] with the gate
 *   columns, then up;  wd [ff][d].  Projections are [in][out] row-major and
 *   applied as y = W^T x.  The library keeps the pointers, not copies: the
 *   weights must outlive the model. */
typedef struct {
    const void *emb;
    const void *out;
    const float *final_norm;
    const float *const *n1;
    const void *const *wqkv;
    const void *const *wo;
    const float *const *n2;
    const void *const *wgu;
    const void *const *wd;
    /* Optional QK-norm, as Qwen3 checkpoints define it (not on the pages):
     * host arrays of n_layer device pointers to fp32 [head_dim] weights, or
     * both NULL (no QK-norm; a zeroed struct has none).  Every q head is
     * scaled by 1 / sqrt(mean of its head_dim squares + eps) and by q_norm,
     * every k head likewise with k_norm, after the projection and before
     * RoPE; v is untouched.  One set without the other: 577. */
    const float *const *q_norm;
    const float *const *k_norm;
} ds_model_weights;

/* The KV cache: per layer one K and one V buffer of rows of n_kvh*head_dim
 * elements (kv_dtype), addressed as in ds_gqa_decode_attn ("Inside the
 * engine", section 3: KvPool holds one K and one V buffer per layer). */
typedef struct {
    void *const *k;             /* host array of n_layer device pointers */
    void *const *v;             /* host array of n_layer device pointers */
    int64_t rows;               /* rows each per-layer buffer holds */
    int32_t block_tokens;       /* positions per block */
    int32_t max_blocks;         /* blocks per sequence */
    const int32_t *block_table; /* device int32 [max_seqs][max_blocks], or NULL */
} ds_kv_cache;

/* Sampling parameters for a whole step (see ds_sample); NULL means greedy. */
typedef struct {
    float temperature;
    int32_t top_k;
    float top_p;
} ds_sampling;

typedef struct ds_model ds_model;

/* Bytes of the model workspace (activations, split reductions, RoPE table,
 * error word) for a configuration. */
DS_API size_t ds_model_workspace_bytes(const ds_model_config *cfg);

/* Validate the configuration and weights, carve the caller's workspace
 * (zeroed here) and build the RoPE table (angles in fp64 on the device).
 * Synchronises the device.  The model object lives in host memory. */
DS_API int ds_model_create(const ds_model_config *cfg, const ds_model_weights *weights,
                           void *workspace, size_t workspace_bytes, ds_model **out);
DS_API void ds_model_destroy(ds_model *model);

/* Workspace pointer of a model (its error word is at byte 0). */
DS_API void *ds_model_workspace(ds_model *model);

/* Flags of ds_decode_step. */
#define DS_STEP_ADVANCE 1u     /* after picking: tokens[s] = next_ids[s], pos[s] += 1 (on device) */
#define DS_STEP_PHASE_TIMES 2u /* record a device timestamp at every phase boundary of the step */
#define DS_STEP_TRACE 4u       /* also record per-CTA timestamps inside every phase (see ds_model_trace) */

/* One decode step for n_seqs sequences: for each sequence s, token
 * tokens[s] at position pos[s] ("The forward pass end to end", "What a
 * forward step does"; "LLM inference kernels", "How this composes into a
 * decode step").  A model with max_seqs 1 runs the step as one persistent
 * kernel; a model with max_seqs > 1 runs the batched path (one launch per
 * operation, projections on the tensor cores, each fp32 activation handed to
 * them as a bf16 pair hi + lo, 16 significant bits), every sequence at its own
 * position in its own blocks of the K/V cache.  The step: embed; per layer
 * RMSNorm -> fused q|k|v projection -> RoPE on
 * q and k with the K/V write at pos ("Inside the engine", section 1: qkPrep)
 * -> attention over positions 0..pos -> output projection + residual ->
 * RMSNorm -> fused gate|up projection with SiLU-gate -> down projection +
 * residual; final RMSNorm -> output head -> greedy argmax (sampling NULL) or
 * the sampler with draws u[s].
 *   tokens, pos: device int32 [n_seqs]; next_ids: device int32 [n_seqs];
 *   u: device fp32 [n_seqs] (sampling only); logits_out: optional device fp32
 *   [n_seqs][vocab].  n_seqs in [1, max_seqs].
 * Bad device-side tokens/positions are clamped/skipped and flag the model's
 * error word. */
DS_API int ds_decode_step(ds_model *model, const ds_kv_cache *kv, int32_t *tokens, int32_t *pos,
                          int n_seqs, const ds_sampling *sampling, const float *u,
                          int32_t *next_ids, float *logits_out, unsigned flags,
                          ds_stream_t stream);

/* n_steps greedy decode steps of one sequence in ONE kernel launch: step i
 * decodes tokens[0] at pos[0] + i and feeds its pick to step i + 1 on the
 * device, so the weight stream runs on from one step's output head into the
 * next step's first layer without a launch in between ("Inside the engine",
 * section 4: the decode loop's steps issued back to back on the device).
 * Each step is a whole ds_decode_step (same result, same K/V writes).
 *   ids_out: optional device int32 [n_steps], the pick of every step;
 *   next_ids: device int32 [1], the last pick.  With DS_STEP_ADVANCE,
 *   tokens[0] and pos[0] end at the last pick and pos[0] + n_steps.
 * Batch-1 models (max_seqs 1) on the persistent step kernel only (577
 * otherwise); n_steps >= 1 (561); logits are not written. */
DS_API int ds_decode_steps(ds_model *model, const ds_kv_cache *kv, int32_t *tokens, int32_t *pos, int n_steps,
                           int32_t *ids_out, int32_t *next_ids, unsigned flags, ds_stream_t stream);

/* stepSeq(sequence, tokens, offset, count): `count` prompt tokens of one
 * sequence at positions offset .. offset + count - 1, run as chunks of at
 * most max_seqs rows, each chunk one batch of rows through the batched path
 * ("Inside the engine", section 1: prefill runs a chunk of prompt tokens as a
 * batch of rows through the batched projections; decode is the one-token
 * chunk of the same step).  Row j of a chunk is the token at position
 * offset + c0 + j: its K and V are written to sequence `seq`'s blocks and it
 * attends positions 0 .. offset + c0 + j of that sequence (earlier chunks'
 * rows and its own chunk's earlier rows included), so the cache ends as
 * `count` decode steps would leave it.  Only the last token goes through the
 * final norm, the head and the greedy argmax.
 *   tokens: device int32 [count] (tokens_len must equal count, else 562);
 *   seq in [0, max_seqs) (577; with a block table, its row seq, else the
 *   contiguous slot seq); next_id: device int32 [1], the greedy pick after
 *   the last token; logits_out: optional device fp32 [vocab], that token's
 *   logits (the model's own buffer is used when NULL).
 * Models with max_seqs > 1 only (577 otherwise); count >= 1 (561);
 * offset >= 0 and offset + count within the cache and max_ctx (571).
 * Uses the model's workspace: calls on one model are serialised on a stream. */
DS_API int ds_step_seq(ds_model *model, const ds_kv_cache *kv, const int32_t *tokens, int64_t tokens_len,
                       int32_t seq, int32_t offset, int32_t count, int32_t *next_id, float *logits_out,
                       ds_stream_t stream);

/* Device timestamps (ns, globaltimer) of the last step run with
 * DS_STEP_PHASE_TIMES: [0] start, then the start of every phase in order
 * (per layer: q|k|v, attention, o, gate|up, down), then the head, then the
 * end — 5*n_layer + 3 values for a batch-1 step.  Copies at most cap values
 * to ns_out (host), the count to *n_out; synchronises `stream`. */
DS_API int ds_model_phase_times(ds_model *model, uint64_t *ns_out, int cap, int *n_out,
                                ds_stream_t stream);

/* Per-CTA timestamps (ns) of the last step run with DS_STEP_TRACE, laid out
 * [phase][cta][5]: phase start, prologue done, last weight stage consumed,
 * epilogue done, and the producer warp's last weight request of the phase
 * (zero where a point does not apply).  Phases as in ds_model_phase_times.
 * Copies at most cap_words values; *n_ctas gets the CTA count. */
DS_API int ds_model_trace(ds_model *model, uint64_t *out, size_t cap_words, size_t *n_words,
                          int *n_ctas, ds_stream_t stream);

/* A decode step captured once as a CUDA graph and replayed ("Inside the
 * engine", section 4: the launch sequence of a step replayed as a captured
 * graph).  Arguments as ds_decode_step; the pointed-to device buffers are
 * read at every launch, so with DS_STEP_ADVANCE each launch decodes the next
 * token.  Capture uses `stream`, which must not be capturing already. */
typedef struct ds_step_graph ds_step_graph;
DS_API int ds_step_graph_create(ds_model *model, const ds_kv_cache *kv, int32_t *tokens,
                                int32_t *pos, int n_seqs, const ds_sampling *sampling,
                                const float *u, int32_t *next_ids, float *logits_out,
                                unsigned flags, ds_stream_t stream, ds_step_graph **out);
DS_API int ds_step_graph_launch(ds_step_graph *graph, ds_stream_t stream);
DS_API void ds_step_graph_destroy(ds_step_graph *graph);

/* Per-kernel timing of one decode step: the step's kernels are launched one
 * at a time on `stream` with CUDA events around each, `reps` times, and the
 * mean duration of each launch slot is written to ms_out[i] with its kernel
 * kind in kinds_out[i] (DS_KIND_*).  *n_out gets the number of slots (at most
 * cap).  Runs the step `reps` times: with DS_STEP_ADVANCE the state advances. */
enum {
    DS_KIND_EMBED = 0,
    DS_KIND_QKV = 1,
    DS_KIND_ATTENTION = 2,
    DS_KIND_O_PROJ = 3,
    DS_KIND_GATE_UP = 4,
    DS_KIND_DOWN = 5,
    DS_KIND_HEAD = 6,
    DS_KIND_SAMPLE = 7,
    DS_KIND_COUNT = 8
};
/* Mean duration, in microseconds, of one launch of the step's kernels of one
 * kind (DS_KIND_*, not DS_KIND_SAMPLE), measured with CUDA events around
 * `reps` passes over all of that kind's launches of a step (every layer's),
 * launched back to back on `stream` as in a step.  The kernels read and write
 * the model's buffers and the cache row at pos[0] as a step would (the
 * residual stream is left changed), but tokens and pos are not advanced.
 * Synchronises `stream`. */
DS_API int ds_decode_kernel_time(ds_model *model, const ds_kv_cache *kv, int32_t *tokens,
                                 int32_t *pos, int kind, int reps, float *us_per_launch,
                                 ds_stream_t stream);

DS_API int ds_decode_step_profile(ds_model *model, const ds_kv_cache *kv, int32_t *tokens,
                                  int32_t *pos, int n_seqs, const ds_sampling *sampling,
                                  const float *u, int32_t *next_ids, float *logits_out,
                                  unsigned flags, int reps, float *ms_out, int32_t *kinds_out,
                                  int cap, int *n_out, ds_stream_t stream);

/* ---------------------------------------------------------------------
 * Continuous-batching scheduler slice over the paged K/V pool (host only)
 * ("Inside the engine", section 2: admission, chunks, preemption, resume).
 * It decides, step by step, which requests run, as prompt chunks or decode
 * rows, and which pool blocks each one's block-table row maps; the caller
 * runs the rows (ds_step_seq for a chunk, ds_decode_step for decode rows)
 * and reports back.  Policy (the page's, read for a pool whose blocks hold
 * every layer's K/V of block_tokens positions):
 *   - a request's tokens are its prompt plus what it has generated; its
 *     cached prefix is the positions whose K/V sit in its blocks;
 *   - admission, strictly first come first served over the waiting list
 *     (preempted requests first, by preemption order, then new ones by
 *     submission): the head is admitted when a block-table row is free and
 *     the free blocks cover all its tokens plus headroom_blocks; those
 *     blocks are taken (lowest block numbers first); otherwise admission
 *     stops for this step;
 *   - chunks: a request with uncached tokens runs them in chunks of at most
 *     `chunk`; the chunk that reaches the last token also yields the next
 *     token; a request whose tokens are all cached but the last runs one
 *     decode row (the last token), which yields the next token;
 *   - preemption: a decode row whose position needs a new block takes the
 *     lowest free one; with none free, the youngest running request (last
 *     submitted) is preempted — its blocks and row freed, its cache
 *     forgotten — until one is free or the request itself was the youngest;
 *     older requests claim blocks first;
 *   - resume: a preempted request waits ahead of new ones, first preempted
 *     first, and recomputes its whole prefix (prompt and generated tokens)
 *     through the chunked path;
 *   - completion: a request that has generated max_new tokens, or that the
 *     caller reports finished, frees its blocks and row at ds_sched_commit;
 *     the next plan admits into them.
 * ------------------------------------------------------------------- */
typedef struct {
    int32_t n_blocks;        /* blocks in the pool */
    int32_t block_tokens;    /* positions per block */
    int32_t max_blocks;      /* block-table width: blocks per request at most */
    int32_t max_running;     /* block-table rows: requests running at once (a model's max_seqs) */
    int32_t chunk;           /* prompt tokens a request runs per step at most */
    int32_t headroom_blocks; /* free blocks demanded beyond a request's tokens at admission */
} ds_sched_config;

/* One row of a planned step. */
typedef struct {
    int64_t request; /* the caller's id */
    int32_t slot;    /* block-table row (the sequence index the kernels address) */
    int32_t offset;  /* position of the row's first token */
    int32_t count;   /* tokens: a chunk of the prompt (or of a resumed prefix), or 1 */
    int32_t decode;  /* 1: the decode row of a request whose tokens are all cached but the last */
    int32_t yields;  /* 1: the row ends at the request's last token and yields its next one */
} ds_sched_row;

typedef struct ds_sched ds_sched;

/* 561 for a count < 1 (headroom_blocks may be 0), 564 beyond DS_MAX_DIM,
 * 577 for NULL.  The scheduler lives in host memory. */
DS_API int ds_sched_create(const ds_sched_config *cfg, ds_sched **out);
DS_API void ds_sched_destroy(ds_sched *sched);

/* Queue a request (ids unique among live requests, else 577): prompt_len >= 1
 * and max_new >= 1 (561); prompt_len + max_new - 1 positions must fit one
 * block-table row (571). */
DS_API int ds_sched_submit(ds_sched *sched, int64_t request, int32_t prompt_len, int32_t max_new);

/* Plan the next step: admit, grow, preempt, and list one row per running
 * request, oldest first, in rows[0 .. *n_rows) (cap >= max_running, else
 * 574).  block_table (host int32 [max_running][max_blocks]) receives every
 * row's blocks, -1 past a request's blocks and in free rows.  preempted
 * (optional, capacity max_running) receives the ids preempted by this plan,
 * *n_preempted their count.  A plan must be committed before the next one
 * (577 otherwise). */
DS_API int ds_sched_plan(ds_sched *sched, ds_sched_row *rows, int32_t cap, int32_t *n_rows,
                         int32_t *block_table, int64_t *preempted, int32_t *n_preempted);

/* The planned step ran: every row's tokens are cached, the rows that yield
 * add a generated token, and requests that reached max_new or appear in
 * finished[0 .. n_finished) free their blocks and rows.  577 without a plan
 * to commit. */
DS_API int ds_sched_commit(ds_sched *sched, const int64_t *finished, int32_t n_finished);

/* Counts: [0] free blocks, [1] running, [2] waiting, [3] finished,
 * [4] preemptions so far. */
DS_API int ds_sched_stats(const ds_sched *sched, int64_t *out5);

/* Generated tokens of a live or finished request (-1: unknown id). */
DS_API int64_t ds_sched_generated(const ds_sched *sched, int64_t request);

#ifdef __cplusplus
}
#endif

#endif /* DECODE_STEP_H */
