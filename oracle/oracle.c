/*
 * Decode-step oracle — TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously correct CPU statement of what one single-token
 * decode step of a Llama/Qwen-style decoder computes.  Only the tests, the
 * smoke check and bench.py's CPU-baseline leg load this library; the product
 * (the CUDA library and its Python binding) never does.  It shares no code,
 * header, table or helper with the CUDA path.
 *
 * Conventions
 *  - Stored operands are fp32 or bf16 (dtype code 0 = fp32, 1 = bf16).  They
 *    are widened to fp64 exactly; sums and products are carried in fp64.
 *  - Projection weights use the transposed convention of "LLM inference
 *    kernels", section "A parallel path for one frozen kernel's known-slow
 *    shape": A is row-major with m = input rows and n = output columns, and
 *    y = A^T x.  The output head / embedding is [vocab, d] row-major and is
 *    applied untransposed (y = W x), as that section says of lm_head.
 *  - The residual stream is stored in fp32 after every update, and K/V rows
 *    are stored in the cache dtype after passing through fp32, because the
 *    model's activations are fp32 ("decode-ops", "Requirements and limits").
 *    Everything the model does not store is kept in fp64.
 *  - The sampler's scaled logits and exponentials are fp32; its sums and
 *    decisions are fp64 (see or_sample).
 *
 * Parity pins for every function live in tests/ (worked examples printed on
 * the pages, closed forms, invariants, brute force).  Nothing here is tuned;
 * the only concession to size is an OpenMP pragma over independent output
 * elements (each output is still summed by one thread in index order).
 */
#include <math.h>
#include <stdint.h>
#ifdef _OPENMP
#include <omp.h>
#endif
#include <stdlib.h>
#include <string.h>

#define OR_F32 0
#define OR_BF16 1

/* Status vocabulary of "LLM inference kernels", section "Status vocabulary
 * and the shape checks (contract)"; codes 572+ are this library's additions in
 * the unused part of the same 560-579 range. */
#define OR_OK 560
#define OR_EMPTY_DIMENSION 561
#define OR_A_LENGTH_MISMATCH 562
#define OR_B_LENGTH_MISMATCH 563
#define OR_DIMENSION_TOO_LARGE 564
#define OR_CACHE_LENGTH_MISMATCH 566
#define OR_NEW_LENGTH_MISMATCH 567
#define OR_LOGITS_LENGTH_MISMATCH 568
#define OR_GEMV_A_LENGTH_MISMATCH 569
#define OR_GEMV_X_LENGTH_MISMATCH 570
#define OR_CACHE_CAPACITY_EXCEEDED 571
#define OR_BAD_SAMPLING_PARAM 575
#define OR_MAX_DIM (1LL << 24)

/* Threads the OpenMP loops use (1 without OpenMP). */
int or_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Set the threads later OpenMP loops use (ignored without OpenMP). */
void or_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ------------------------------------------------------------------ */
/* element access                                                      */
/* ------------------------------------------------------------------ */

/* bf16 is the upper 16 bits of an IEEE binary32; widening is exact. */
static double load_elem(const void *p, int64_t i, int dtype) {
    if (dtype == OR_F32) return (double)((const float *)p)[i];
    uint32_t bits = (uint32_t)((const uint16_t *)p)[i] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* Round a binary32 to bf16, round-to-nearest, ties to even, NaN kept NaN. */
uint16_t or_f32_to_bf16(float f) {
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    if ((bits & 0x7f800000u) == 0x7f800000u && (bits & 0x007fffffu) != 0)
        return (uint16_t)((bits >> 16) | 0x0040u); /* quiet NaN */
    uint32_t lower = bits & 0xffffu;
    uint32_t upper = bits >> 16;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;
    return (uint16_t)upper;
}

/* Store an fp64 value as an fp32 activation, then in the buffer's dtype. */
static void store_elem(void *p, int64_t i, int dtype, double v) {
    float f = (float)v;
    if (dtype == OR_F32)
        ((float *)p)[i] = f;
    else
        ((uint16_t *)p)[i] = or_f32_to_bf16(f);
}

/* ------------------------------------------------------------------ */
/* contract: the exact-length shape checks                             */
/* ------------------------------------------------------------------ */

/* "LLM inference kernels", "Status vocabulary and the shape checks":
 * a dimension < 1 is refused (561), a dimension above 1<<24 is refused (564),
 * then each operand's real length must equal its claimed length. */
int or_residual_dims_check(int64_t n, int64_t a_len, int64_t b_len) {
    if (n < 1) return OR_EMPTY_DIMENSION;
    if (n > OR_MAX_DIM) return OR_DIMENSION_TOO_LARGE;
    if (a_len != n) return OR_A_LENGTH_MISMATCH;
    if (b_len != n) return OR_B_LENGTH_MISMATCH;
    return OR_OK;
}

/* ------------------------------------------------------------------ */
/* projections                                                         */
/* ------------------------------------------------------------------ */

/* y[j] = sum_i A[i, j] * x[i], A row-major with `rows` input rows and `cols`
 * output columns ("LLM inference kernels", "A parallel path for one frozen
 * kernel's known-slow shape": the transposed mat-vec summed down each
 * column). */
void or_gemv_transposed(const void *A, int a_dtype, const double *x,
                        int64_t rows, int64_t cols, double *y) {
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < cols; ++j) {
        double acc = 0.0;
        for (int64_t i = 0; i < rows; ++i) acc += load_elem(A, i * cols + j, a_dtype) * x[i];
        y[j] = acc;
    }
}

/* y[r] = sum_c W[r, c] * x[c] — the untransposed form used for the output
 * head ("The forward pass end to end", "The code": logits are the output
 * matrix times the normalised state). */
void or_gemv(const void *W, int w_dtype, const double *x, int64_t rows, int64_t cols,
             double *y) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        double acc = 0.0;
        for (int64_t c = 0; c < cols; ++c) acc += load_elem(W, r * cols + c, w_dtype) * x[c];
        y[r] = acc;
    }
}

/* ------------------------------------------------------------------ */
/* residual add, RMSNorm, SiLU-gate                                    */
/* ------------------------------------------------------------------ */

/* out[i] = a[i] + b[i] in fp32 ("LLM inference kernels", "Residual add"). */
void or_residual_add(const float *a, const float *b, float *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = a[i] + b[i];
}

/* y = x * (mean(x^2) + eps)^(-1/2) * g ("The forward pass end to end",
 * "The code", rmsnorm; "Root Mean Square Layer Normalization"). */
void or_rmsnorm(const double *x, const void *g, int g_dtype, int64_t n, double eps,
                double *y) {
    double ss = 0.0;
    for (int64_t i = 0; i < n; ++i) ss += x[i] * x[i];
    double s = 1.0 / sqrt(ss / (double)n + eps);
    for (int64_t i = 0; i < n; ++i) y[i] = x[i] * s * load_elem(g, i, g_dtype);
}

/* residual += x (stored fp32), then h = RMSNorm(residual) * w ("decode-ops",
 * "Usage": add_rmsnorm adds into the residual, then normalises).  x may be
 * NULL, which leaves the residual unchanged (plain RMSNorm). */
void or_add_rmsnorm(float *residual, const float *x, const void *w, int w_dtype,
                    int64_t n, double eps, double *h) {
    double *r = (double *)malloc((size_t)n * sizeof(double));
    for (int64_t i = 0; i < n; ++i) {
        if (x) residual[i] = residual[i] + x[i];
        r[i] = (double)residual[i];
    }
    or_rmsnorm(r, w, w_dtype, n, eps, h);
    free(r);
}

/* silu(z) = z / (1 + e^-z) ("The forward pass end to end", "The code"). */
static double silu(double z) { return z / (1.0 + exp(-z)); }

/* out[i] = silu(gate[i]) * up[i] ("decode-ops", "Usage": silu_mul). */
void or_silu_mul(const double *gate, const double *up, double *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = silu(gate[i]) * up[i];
}

/* ------------------------------------------------------------------ */
/* rotary position embedding                                           */
/* ------------------------------------------------------------------ */

#define OR_ROPE_HALF_SPLIT 0
#define OR_ROPE_INTERLEAVED 1

/* Rotation frequency of pair p (0 <= p < hd/2): base^(-2p/hd).  With
 * long-context scaling (sc != NULL and sc[0] != 0; sc = {factor, low_factor,
 * high_factor, orig_max_pos}) the frequency is remapped by its wavelength
 * w = 2 pi / f, as Llama 3.1 checkpoints define it (not on the pages): a pair
 * that turns more than high_factor times within orig_max_pos positions keeps
 * f, one that turns fewer than low_factor times turns factor times slower,
 * and in between f / factor and f are blended with the weight
 * s = (orig_max_pos / w - low_factor) / (high_factor - low_factor) on f. */
double or_rope_freq(int64_t p, int64_t hd, double base, const double *sc) {
    const double f = pow(base, -(double)(2 * p) / (double)hd);
    if (!sc || sc[0] == 0.0) return f;
    const double factor = sc[0], lo = sc[1], hi = sc[2], orig = sc[3];
    const double two_pi = 6.283185307179586476925286766559;
    const double w = two_pi / f;
    if (w < orig / hi) return f;
    if (w > orig / lo) return f / factor;
    const double s = (orig / w - lo) / (hi - lo);
    return (1.0 - s) * (f / factor) + s * f;
}

/* Rotate every head of `vec` (n_heads * hd values) to position `pos`.
 * Pair p turns by theta_p = pos * f_p (f_p from or_rope_freq; unscaled,
 * f_p = base^(-2p/hd)):
 *   a' = a cos(theta) - b sin(theta),  b' = a sin(theta) + b cos(theta).
 * Interleaved layout pairs (2p, 2p+1) ("The forward pass end to end", "The
 * code", rope); half-split layout pairs (p, p + hd/2), the GPT-NeoX split-half
 * convention ("LLM inference kernels", "Two gaps, not three").  Angles are
 * formed in fp64 ("decode-ops", "API — Method"). */
void or_rope(double *vec, int64_t n_heads, int64_t hd, int64_t pos, double base, int layout, const double *sc) {
    for (int64_t h = 0; h < n_heads; ++h) {
        double *v = vec + h * hd;
        for (int64_t p = 0; p < hd / 2; ++p) {
            double theta = (double)pos * or_rope_freq(p, hd, base, sc);
            double c = cos(theta), s = sin(theta);
            int64_t ia = layout == OR_ROPE_INTERLEAVED ? 2 * p : p;
            int64_t ib = layout == OR_ROPE_INTERLEAVED ? 2 * p + 1 : p + hd / 2;
            double a = v[ia], b = v[ib];
            v[ia] = a * c - b * s;
            v[ib] = a * s + b * c;
        }
    }
}

/* ------------------------------------------------------------------ */
/* KV cache                                                            */
/* ------------------------------------------------------------------ */

/* Reserved-capacity append: write n_new values at [cache_len, cache_len+n_new)
 * of a buffer reserved once at `capacity` elements; refuse an overrun with
 * 571 ("LLM inference kernels", "The hot loop doesn't call
 * kv_cache_append_flat"; an empty append is refused, "Guarantees"). */
int or_kv_cache_append(void *cache, int dtype, int64_t capacity, int64_t cache_len,
                       const double *new_vals, int64_t new_len, int64_t n_new) {
    if (n_new < 1 || capacity < 1) return OR_EMPTY_DIMENSION;
    if (n_new > OR_MAX_DIM || cache_len > OR_MAX_DIM || capacity > OR_MAX_DIM)
        return OR_DIMENSION_TOO_LARGE;
    if (cache_len < 0) return OR_CACHE_LENGTH_MISMATCH;
    if (new_len != n_new) return OR_NEW_LENGTH_MISMATCH;
    if (cache_len + n_new > capacity) return OR_CACHE_CAPACITY_EXCEEDED;
    for (int64_t i = 0; i < n_new; ++i) store_elem(cache, cache_len + i, dtype, new_vals[i]);
    return OR_OK;
}

/* Address of the row holding position t of sequence `seq` in a cache laid out
 * as blocks of `block_tokens` positions, each position a row of row_elems.
 * With a block table, logical block b of the sequence lives in physical block
 * table[seq * max_blocks + b]; without one, a sequence owns `max_blocks`
 * consecutive blocks starting at block seq * max_blocks ("Inside the engine",
 * "3. The K/V cache and the block store": slot s at element s x plane). */
static int64_t cache_row(int64_t seq, int64_t t, const int32_t *block_table,
                         int64_t max_blocks, int64_t block_tokens) {
    int64_t b = t / block_tokens;
    int64_t phys = block_table ? (int64_t)block_table[seq * max_blocks + b] : seq * max_blocks + b;
    return phys * block_tokens + t % block_tokens;
}

/* ------------------------------------------------------------------ */
/* grouped-query attention for one new token                           */
/* ------------------------------------------------------------------ */

/* For query head h, its KV head is g = h / (n_qh / n_kvh).  Scores
 * s_t = (q_h . k_{t,g}) * scale over every cached position t in [0, n_ctx)
 * (the current one included), w = softmax(s) with the maximum subtracted,
 * out_h = sum_t w_t v_{t,g} ("The forward pass end to end", "The code":
 * forward_token's attention loop and softmax). */
void or_gqa_attention(const double *q, const void *k_cache, const void *v_cache, int kv_dtype,
                      const int32_t *block_table, int64_t max_blocks, int64_t block_tokens,
                      int64_t seq, int64_t n_ctx, int64_t n_qh, int64_t n_kvh, int64_t hd,
                      double scale, double *out) {
    int64_t group = n_qh / n_kvh;
    int64_t row_elems = n_kvh * hd;
    double *s = (double *)malloc((size_t)n_ctx * sizeof(double));
    for (int64_t h = 0; h < n_qh; ++h) {
        int64_t g = h / group;
        const double *qh = q + h * hd;
        double m = -INFINITY;
        for (int64_t t = 0; t < n_ctx; ++t) {
            int64_t base = cache_row(seq, t, block_table, max_blocks, block_tokens) * row_elems + g * hd;
            double acc = 0.0;
            for (int64_t i = 0; i < hd; ++i) acc += qh[i] * load_elem(k_cache, base + i, kv_dtype);
            s[t] = acc * scale;
            if (s[t] > m) m = s[t];
        }
        double z = 0.0;
        for (int64_t t = 0; t < n_ctx; ++t) {
            s[t] = exp(s[t] - m);
            z += s[t];
        }
        for (int64_t i = 0; i < hd; ++i) out[h * hd + i] = 0.0;
        for (int64_t t = 0; t < n_ctx; ++t) {
            int64_t base = cache_row(seq, t, block_table, max_blocks, block_tokens) * row_elems + g * hd;
            double w = s[t] / z;
            for (int64_t i = 0; i < hd; ++i) out[h * hd + i] += w * load_elem(v_cache, base + i, kv_dtype);
        }
    }
    free(s);
}

/* ------------------------------------------------------------------ */
/* picking the next token                                              */
/* ------------------------------------------------------------------ */

/* Is a "greater" than b under torch.argmax's ordering, where NaN ranks above
 * every number?  Ties are not greater, so the first index wins. */
static int ranks_above(float a, float b) {
    if (isnan(a)) return !isnan(b);
    if (isnan(b)) return 0;
    return a > b;
}

/* First index of the maximum ("LLM inference kernels", "KV-cache growth and
 * greedy argmax": ties resolve to the first matching id; "decode-ops",
 * "Correctness": exact against torch.argmax, ties included). */
int64_t or_argmax(const float *logits, int64_t n, float *max_logit) {
    int64_t best = 0;
    for (int64_t i = 1; i < n; ++i)
        if (ranks_above(logits[i], logits[best])) best = i;
    if (max_logit) *max_logit = logits[best];
    return best;
}

typedef struct {
    float key;
    int64_t idx;
} keyed;

/* Descending key, then ascending index: the survivor order of "decode-ops",
 * "API — Method" (heap pops in descending logit order, ties to the lower
 * index). */
static int by_key_desc(const void *pa, const void *pb) {
    const keyed *a = (const keyed *)pa, *b = (const keyed *)pb;
    if (a->key > b->key) return -1;
    if (a->key < b->key) return 1;
    return (a->idx > b->idx) - (a->idx < b->idx);
}

/* Temperature -> top-k -> softmax over survivors -> top-p -> renormalise ->
 * inverse CDF at the caller's uniform draw u in [0,1) ("decode-ops",
 * "API — Method", the HuggingFace warper order).  The pages give the sampler
 * f32 logits and exp (exp(0) == 1), and leave the precision of its running
 * sums open; here the scaled logits and the exponentials are fp32 and every
 * sum, ratio and comparison after them is fp64, so that the token depends on
 * the method's values, not on the order in which a long sum is taken:
 *   l'_i = l_i / T (fp32);  survivors = first top_k of (l' desc, index asc),
 *   all if top_k <= 0 or top_k >= n;  e_i = expf(l'_i - l'_max) (fp32);
 *   S = sum e_i;  p_i = e_i / S;  keep the prefix whose exclusive running sum
 *   of p is < top_p (at least one; top_p >= 1 keeps all);  S2 = sum of the
 *   kept p;  token = first kept with inclusive running sum > u * S2, else the
 *   last kept.
 * T <= 0 means greedy.  `margin` (optional) receives the smallest distance,
 * as a fraction of the mass, between a running sum and the threshold it was
 * compared with (top_p for the exclusive sums the top-p cut tests, u * S2 / S2
 * for the inclusive sums of the draw), so that a caller can tell a draw or a
 * cut that sits on a boundary.  Returns the token id, or -1 for a parameter
 * outside its domain (top_p <= 0, u outside [0,1)). */
int64_t or_sample(const float *logits, int64_t n, float temperature, int64_t top_k,
                  float top_p, float u, double *margin) {
    if (margin) *margin = INFINITY;
    if (temperature <= 0.0f) return or_argmax(logits, n, NULL);
    if (!(top_p > 0.0f) || !(u >= 0.0f && u < 1.0f)) return -1;
    keyed *c = (keyed *)malloc((size_t)n * sizeof(keyed));
    for (int64_t i = 0; i < n; ++i) {
        c[i].key = logits[i] / temperature;
        c[i].idx = i;
    }
    qsort(c, (size_t)n, sizeof(keyed), by_key_desc);
    int64_t k = (top_k <= 0 || top_k >= n) ? n : top_k;
    double *p = (double *)malloc((size_t)k * sizeof(double));
    double S = 0.0;
    for (int64_t i = 0; i < k; ++i) {
        const float e = expf(c[i].key - c[0].key);
        p[i] = (double)e;
        S += p[i];
    }
    for (int64_t i = 0; i < k; ++i) p[i] = p[i] / S;
    int64_t kept = k;
    if (top_p < 1.0f) {
        double excl = 0.0;
        kept = 0;
        while (kept < k && (kept == 0 || excl < (double)top_p)) {
            if (kept > 0 && margin) {
                const double d = fabs(excl - (double)top_p);
                if (d < *margin) *margin = d;
            }
            excl += p[kept];
            ++kept;
        }
        if (kept < k && margin) {  /* the comparison that stopped the cut */
            const double d = fabs(excl - (double)top_p);
            if (d < *margin) *margin = d;
        }
    }
    double S2 = 0.0;
    for (int64_t i = 0; i < kept; ++i) S2 += p[i];
    const double target = (double)u * S2;
    double incl = 0.0;
    int64_t chosen = -1;
    for (int64_t i = 0; i < kept; ++i) {
        incl += p[i];
        if (margin) {
            const double d = fabs(incl - target) / S2;
            if (d < *margin) *margin = d;
        }
        if (chosen < 0 && incl > target) chosen = i;
    }
    if (chosen < 0) chosen = kept - 1;
    int64_t token = c[chosen].idx;
    free(p);
    free(c);
    return token;
}

/* ------------------------------------------------------------------ */
/* the decode step                                                     */
/* ------------------------------------------------------------------ */

/* Model description, passed as plain integers so that no struct layout is
 * shared with any other component. */
typedef struct {
    int64_t vocab, d, n_layer, n_qh, n_kvh, hd, ff;
    int64_t rope_layout; /* OR_ROPE_* */
    int64_t tied;        /* 1: the output head is the embedding table */
    int64_t w_dtype;     /* dtype of emb / out / projections */
    int64_t kv_dtype;
    int64_t block_tokens, max_blocks; /* cache geometry, see cache_row */
    int64_t qk_norm;     /* 1: every q and k head is RMS-normalised before RoPE */
    double rope_base, eps;
    double rope_scaling[4]; /* factor (0: none), low_factor, high_factor, orig_max_pos */
} or_model;

static void unpack(or_model *m, const int64_t *iv, const double *dv) {
    m->vocab = iv[0];
    m->d = iv[1];
    m->n_layer = iv[2];
    m->n_qh = iv[3];
    m->n_kvh = iv[4];
    m->hd = iv[5];
    m->ff = iv[6];
    m->rope_layout = iv[7];
    m->tied = iv[8];
    m->w_dtype = iv[9];
    m->kv_dtype = iv[10];
    m->block_tokens = iv[11];
    m->max_blocks = iv[12];
    m->qk_norm = iv[13];
    m->rope_base = dv[0];
    m->eps = dv[1];
    for (int i = 0; i < 4; ++i) m->rope_scaling[i] = dv[2 + i];
}

/* Weight pointers, in this order:
 *   [0] emb [vocab, d]   [1] out [vocab, d] (unused when tied)
 *   [2] final norm weight [d] fp32
 *   then per layer l, at 3 + 6l:
 *   n1 [d] fp32 | wqkv [d, (n_qh + 2 n_kvh) hd] (q columns, then k, then v)
 *   | wo [n_qh hd, d] | n2 [d] fp32 | wgu [d, 2 ff] (gate columns, then up)
 *   | wd [ff, d]
 *   and, with qk_norm, after the layers, per layer l at 3 + 6 n_layer + 2l:
 *   q_norm [hd] fp32 | k_norm [hd] fp32
 * Caches: k_caches[l], v_caches[l], rows of n_kvh * hd in cache_row layout. */

/* One token through the model at position `pos` of sequence `seq`, with the
 * cache holding positions [0, pos) already; appends this position's K and V
 * and writes `vocab` logits ("The forward pass end to end", "What a forward
 * step does" and "The code": forward_token; "LLM inference kernels", "How
 * this composes into a decode step").  `residual_out` (optional, [d]) gets the
 * final residual stream. */
int or_decode_step(const int64_t *iv, const double *dv, const void *const *weights,
                   void *const *k_caches, void *const *v_caches, const int32_t *block_table,
                   int64_t seq, int64_t token, int64_t pos, double *logits) {
    or_model m;
    unpack(&m, iv, dv);
    if (token < 0 || token >= m.vocab || pos < 0 || pos >= m.block_tokens * m.max_blocks) return -1;
    const int64_t d = m.d, hd = m.hd, nq = m.n_qh * hd, nkv = m.n_kvh * hd, ff = m.ff;
    const int64_t nqkv = nq + 2 * nkv;
    float *x = (float *)malloc((size_t)d * sizeof(float));
    double *xd = (double *)malloc((size_t)d * sizeof(double));
    double *h = (double *)malloc((size_t)d * sizeof(double));
    double *qkv = (double *)malloc((size_t)nqkv * sizeof(double));
    double *att = (double *)malloc((size_t)nq * sizeof(double));
    double *o = (double *)malloc((size_t)d * sizeof(double));
    double *gu = (double *)malloc((size_t)2 * ff * sizeof(double));
    double *f = (double *)malloc((size_t)ff * sizeof(double));
    double *gate = (double *)malloc((size_t)ff * sizeof(double));
    double *up = (double *)malloc((size_t)ff * sizeof(double));
    double *hbuf = (double *)malloc((size_t)hd * sizeof(double));

    /* x = E[token] */
    for (int64_t i = 0; i < d; ++i) x[i] = (float)load_elem(weights[0], token * d + i, (int)m.w_dtype);

    for (int64_t l = 0; l < m.n_layer; ++l) {
        const void *const *L = weights + 3 + 6 * l;
        /* h = RMSNorm(x, n1) */
        for (int64_t i = 0; i < d; ++i) xd[i] = x[i];
        or_rmsnorm(xd, L[0], OR_F32, d, m.eps, h);
        /* q | k | v = Wqkv^T h */
        or_gemv_transposed(L[1], (int)m.w_dtype, h, d, nqkv, qkv);
        double *q = qkv, *k = qkv + nq, *v = qkv + nq + nkv;
        /* QK-norm as Qwen3 checkpoints define it (not on the pages): every q
         * head and every k head RMS-normalised over its head_dim values with
         * the layer's q_norm or k_norm weight, before the rotation */
        if (m.qk_norm) {
            const void *qn = weights[3 + 6 * m.n_layer + 2 * l], *kn = weights[3 + 6 * m.n_layer + 2 * l + 1];
            for (int64_t hh = 0; hh < m.n_qh + m.n_kvh; ++hh) {
                double *head = hh < m.n_qh ? q + hh * hd : k + (hh - m.n_qh) * hd;
                or_rmsnorm(head, hh < m.n_qh ? qn : kn, OR_F32, hd, m.eps, hbuf);
                for (int64_t i = 0; i < hd; ++i) head[i] = hbuf[i];
            }
        }
        /* rotate q and k (never v) to this position */
        or_rope(q, m.n_qh, hd, pos, m.rope_base, (int)m.rope_layout, m.rope_scaling);
        or_rope(k, m.n_kvh, hd, pos, m.rope_base, (int)m.rope_layout, m.rope_scaling);
        /* append this position's K and V before attending */
        int64_t row = cache_row(seq, pos, block_table, m.max_blocks, m.block_tokens);
        for (int64_t i = 0; i < nkv; ++i) {
            store_elem(k_caches[l], row * nkv + i, (int)m.kv_dtype, k[i]);
            store_elem(v_caches[l], row * nkv + i, (int)m.kv_dtype, v[i]);
        }
        /* attend over positions 0..pos */
        or_gqa_attention(q, k_caches[l], v_caches[l], (int)m.kv_dtype, block_table, m.max_blocks,
                         m.block_tokens, seq, pos + 1, m.n_qh, m.n_kvh, hd, 1.0 / sqrt((double)hd),
                         att);
        /* x += Wo^T att */
        or_gemv_transposed(L[2], (int)m.w_dtype, att, nq, d, o);
        for (int64_t i = 0; i < d; ++i) x[i] = (float)((double)x[i] + o[i]);
        /* h = RMSNorm(x, n2); f = silu(gate . h) * (up . h) */
        for (int64_t i = 0; i < d; ++i) xd[i] = x[i];
        or_rmsnorm(xd, L[3], OR_F32, d, m.eps, h);
        or_gemv_transposed(L[4], (int)m.w_dtype, h, d, 2 * ff, gu);
        for (int64_t i = 0; i < ff; ++i) {
            gate[i] = gu[i];
            up[i] = gu[ff + i];
        }
        or_silu_mul(gate, up, f, ff);
        /* x += Wd^T f */
        or_gemv_transposed(L[5], (int)m.w_dtype, f, ff, d, o);
        for (int64_t i = 0; i < d; ++i) x[i] = (float)((double)x[i] + o[i]);
    }
    /* logits = Out . RMSNorm(x, final) */
    for (int64_t i = 0; i < d; ++i) xd[i] = x[i];
    or_rmsnorm(xd, weights[2], OR_F32, d, m.eps, h);
    or_gemv(m.tied ? weights[0] : weights[1], (int)m.w_dtype, h, m.vocab, d, logits);

    free(x);
    free(xd);
    free(h);
    free(qkv);
    free(att);
    free(o);
    free(gu);
    free(f);
    free(gate);
    free(up);
    free(hbuf);
    return 0;
}

/* Full recompute without cache reuse: run tokens[0..n) through fresh caches
 * (the caller passes zeroed scratch caches) and return the logits of the last
 * position ("The forward pass end to end", "The correctness test"). */
int or_recompute_logits(const int64_t *iv, const double *dv, const void *const *weights,
                        void *const *k_scratch, void *const *v_scratch, const int32_t *tokens,
                        int64_t n, double *logits) {
    for (int64_t t = 0; t < n; ++t) {
        int rc = or_decode_step(iv, dv, weights, k_scratch, v_scratch, NULL, 0, tokens[t], t, logits);
        if (rc) return rc;
    }
    return 0;
}
