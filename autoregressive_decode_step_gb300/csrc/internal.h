// Internal interfaces between the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

#include "../../include/decode_step.h"

namespace ds {

// Every workspace starts with this header; the error word is at byte 0.
constexpr size_t kWsHeader = 256;

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// SM count of the current device (cached per device).
int sm_count();

// Launch `kernel` with cudaLaunchKernelEx; `pdl` adds the programmatic
// stream-serialisation attribute so the kernel may begin while its
// predecessor on the stream finishes.
template <typename... KArgs, typename... Args>
cudaError_t launch_ex(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                      cudaStream_t stream, bool pdl, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ------------------------------------------------------------------ GEMV
enum Pro { PRO_PLAIN = 0, PRO_RMSNORM = 1 };
enum Epi { EPI_STORE = 0, EPI_ADD = 1, EPI_SILU = 2, EPI_QKV = 3 };

// Bytes of one band's row segment in shared memory, rows per pipeline stage
// and stages of the transposed GEMV's ring.
#ifndef DS_GT_ROWS
#define DS_GT_ROWS 64
#endif
#ifndef DS_GT_STAGES
#define DS_GT_STAGES 4
#endif
#ifndef DS_ST_BOX_ROWS
#define DS_ST_BOX_ROWS 16
#endif
constexpr int kGtBoxRows = DS_ST_BOX_ROWS;  // rows of one tensor-map box (the unit of work)
constexpr int kGtBandBytes = 512;
constexpr int kGtRows = DS_GT_ROWS;
constexpr int kGtStages = DS_GT_STAGES;
constexpr int kGtConsumerWarps = 8;

struct GemvTArgs {
    CUtensorMap tm0;      // 2-D map of sub-tile 0: {sub_cols, K}, box {band columns, kGtBoxRows}
    CUtensorMap tm1;      // same for sub-tile 1 (EPI_SILU's up columns)
    const char *a0;       // element (k, c) of sub-tile 0 at a0 + k*row_stride + c*es
    const char *a1;       // sub-tile 1 (the up columns for EPI_SILU) or nullptr
    long long row_stride; // bytes between consecutive rows
    int K;                // reduced dimension (rows)
    int sub_cols;         // columns of each sub-tile source
    int n_bands;
    const float *x;       // PRO_PLAIN: x[K]; PRO_RMSNORM: the residual [K]
    const float *norm_w;  // PRO_RMSNORM weight [K] (fp32)
    float eps;
    int xs_cap;           // floats of shared memory for this CTA's slice of x
    float *partials;      // (grid + n_bands) * band_cols floats
    int *counters;        // n_bands ints, zero between launches
    int *err;
    float *y;             // STORE/ADD: y[sub_cols]; SILU: f[sub_cols]; QKV: q out
    // EPI_QKV: RoPE on the q and k columns, K/V written at position pos[0]
    // of sequence 0.
    void *k_cache;
    void *v_cache;
    int kv_dtype;
    const int *pos;
    int nq_cols, nkv_cols, head_dim, rope_layout;
    const float *rope_cos, *rope_sin;  // [rope_rows][head_dim / 2]
    int rope_rows;
    const int *block_table;
    int block_tokens, max_blocks;
    // QK-norm before RoPE (null: none): every q / k head scaled by
    // 1/sqrt(mean of its squares + eps) and by these [head_dim] weights
    const float *q_norm, *k_norm;
};

// Columns of one band (partial sums per band) for an element size.
inline int gemv_t_band_cols(int es) { return kGtBandBytes / es; }
int gemv_t_grid(int K, int n_bands);
size_t gemv_t_partial_floats(int grid, int n_bands, int es);
// Can the tensor-map kernel stream this matrix?
bool gemv_t_streamable(const void *a0, const void *a1, long long row_stride, int sub_cols, int es);
// Encode a.tm0 (and a.tm1 when a.a1 is set) from a0/a1, row_stride, sub_cols
// and K for a matrix of the given dtype; false if the driver refuses.
bool gemv_t_make_maps(GemvTArgs &a, int dtype);
cudaError_t launch_gemv_t(const GemvTArgs &a, int dtype, int pro, int epi, int grid,
                          cudaStream_t stream, bool pdl);
// ds_gemv_transposed after its host checks: y = A^T x with the split
// reduction's scratch at `ws` (ds_gemv_workspace_bytes bytes, unused when
// gemv_t_uses_workspace is false: the plain-load kernel then runs).
int gemv_transposed_run(const void *A, int a_dtype, const float *x, int64_t rows, int64_t cols, float *y,
                        char *ws, cudaStream_t s);
bool gemv_t_uses_workspace(const void *A, int64_t cols, int a_dtype);
// Bytes at the start of ds_gemv_transposed's workspace that the streamed
// path needs at zero when it starts: the header (error word) and the band
// counters; the partial sums after them need no clearing.
size_t gemv_t_zeroed_bytes(int64_t cols, int a_dtype);

struct GemvNArgs {
    const char *W;        // [rows][cols]
    int rows, cols;
    const float *x;       // PRO_PLAIN: x[cols]; PRO_RMSNORM: the residual [cols]
    const float *norm_w;
    float eps;
    float *y;             // [rows]
    // fused greedy argmax over the rows (do_argmax != 0)
    int do_argmax;
    float *part_val;      // [grid]
    int *part_idx;        // [grid]
    int *counter;         // 1 int, zero between launches
    int *ids_out;         // 1 int
    float *max_out;       // 1 float or nullptr
    int *tokens_adv;      // DS_STEP_ADVANCE targets or nullptr
    int *pos_adv;
    int *err;
};
int gemv_n_grid(int rows, int cols, int es);
bool gemv_n_streamable(const void *W, int rows, int cols, int es);
cudaError_t launch_gemv_n(const GemvNArgs &a, int dtype, int pro, int grid, cudaStream_t stream,
                          bool pdl);

// ------------------------------------------------------------------ attention
struct AttnArgs {
    const float *q;       // [n_seqs][n_qh * hd]
    const void *k_cache;
    const void *v_cache;
    int kv_dtype;
    long long cache_rows;
    const int *block_table;
    int max_blocks, block_tokens;
    const int *seq_lens;  // [n_seqs] or nullptr (then n_ctx = pos[s] + 1)
    const int *pos;
    const int *row_seq;   // [n_seqs]: the sequence whose blocks row s reads, or nullptr (s itself)
    int n_qh, n_kvh, hd;
    float scale;
    float *out;           // [n_seqs][n_qh * hd]
    void *out_bf16;       // optional bf16 pair of out (the batched o projection's input): hi here,
    long long out_bf16_lo; // lo this many elements further (0: hi only)
    float *partials;
    int *counters;        // n_seqs * n_kvh ints, zero between launches
    int *err;
    int n_splits;
};
// Paged flash-decoding over whole cache blocks (head_dim 128, 16-position
// blocks, 2 or 4 query heads per KV head, at most 8 KV heads).
struct PagedAttnArgs {
    CUtensorMap tk, tv;    // bf16 caches, 128-byte swizzle: 3-D maps {64, cache_rows, 2 n_kvh} with one box per
                           // block (box3d), else 2-D maps {n_kvh * 128, cache_rows} with boxes {64, 16}
    int box3d;
    const float *q;        // [n_seqs][n_qh * 128]
    const void *k_cache;   // rows of n_kvh * 128 elements of kv_dtype
    const void *v_cache;
    int kv_dtype;
    long long cache_rows;
    const int *block_table;  // [n_seqs][max_blocks] or nullptr (contiguous slots)
    int max_blocks;
    const int *seq_lens;   // [n_seqs] or nullptr (then n_ctx = pos[s] + 1)
    const int *pos;
    const int *row_seq;    // [n_seqs]: the sequence whose blocks row s reads, or nullptr (s itself)
    int n_seqs, n_qh, n_kvh;
    float scale;
    float *out;            // [n_seqs][n_qh * 128]
    void *out_bf16;        // optional bf16 pair of out: hi here, lo out_bf16_lo elements further
    long long out_bf16_lo;
    float *partials;       // paged_attention_partial_floats(n_seqs, n_qh)
    int *counters;         // n_seqs * n_kvh ints, zero between launches
    int *err;
    int stages;            // set by the launcher
};
bool paged_attention_supported(int n_qh, int n_kvh, int hd, int block_tokens, int n_seqs, int kv_dtype);
// Encode a.tk / a.tv for bf16 caches (the tensor-core variant); false if the driver refuses.
bool paged_attention_maps(PagedAttnArgs &a);
size_t paged_attention_partial_floats(int n_seqs, int n_qh);
cudaError_t launch_paged_attention(const PagedAttnArgs &a, cudaStream_t stream, bool pdl);
cudaError_t prepare_paged_attention();

int attention_splits(int n_seqs, int n_kvh, long long max_ctx);
size_t attention_partial_floats(int n_seqs, int n_qh, int n_kvh, int hd, int n_splits);
cudaError_t launch_attention(const AttnArgs &a, int n_seqs, cudaStream_t stream, bool pdl);

// ------------------------------------------------------------------ small ops
cudaError_t launch_embed(const void *emb, int w_dtype, int vocab, int d, const int *tokens,
                         float *x, int *err, int n_seqs, cudaStream_t stream, bool pdl);
// Long-context frequency scaling of the RoPE table (factor 0: none).
struct RopeScaling {
    double factor, low_freq_factor, high_freq_factor, orig_max_pos;
};
cudaError_t launch_rope_table(float *cos_t, float *sin_t, int rows, int head_dim, double base, RopeScaling sc,
                              cudaStream_t stream);
cudaError_t launch_rmsnorm_rows_bf16(const float *x, const float *w, float eps, void *h, long long lo_off,
                                     int n_rows, int d, cudaStream_t stream, bool pdl);
// pos[j] = pos0 + j and row_seq[j] = seq for j < n (no programmatic overlap
// with the launch before it)
cudaError_t launch_chunk_rows(int *pos, int *row_seq, int pos0, int seq, int n, cudaStream_t stream);

// ------------------------------------------------------------------ picking
struct ArgmaxArgs {
    const float *logits;
    int n_rows;
    long long n;
    int *ids;
    float *max_logit;
    float *part_val;
    int *part_idx;
    int *counters;        // n_rows ints
    int *tokens_adv, *pos_adv;
    int *err;
    int blocks_per_row;
};
int argmax_blocks_per_row(long long n);
cudaError_t launch_argmax(const ArgmaxArgs &a, cudaStream_t stream, bool pdl);

struct SampleArgs {
    const float *logits;
    int n_rows;
    long long n;
    float temperature;
    int top_k;
    float top_p;
    const float *u;
    int *ids;
    int *tokens_adv, *pos_adv;
    int *err;
};
cudaError_t launch_sample(const SampleArgs &a, cudaStream_t stream, bool pdl);

// ------------------------------------------------------------------ the step kernel
constexpr int kStMaxLayers = 128;
constexpr int kStMaxSplits = 64;

struct StepLayer {  // aligned as CUtensorMap requires
    CUtensorMap maps[5];  // q|k|v, o, gate, up, down
    const float *n1, *n2;
    const float *qn, *kn;  // QK-norm weights [head_dim] or null
};

struct StepParams {
    const StepLayer *layers;
    int n_layer;
    const char *emb, *head;
    const float *final_norm;
    int vocab, d, nq_cols, nkv_cols, hd, ff, rope_layout, kv_dtype, n_kvh, n_qh;
    float eps;
    const float *rope_cos, *rope_sin;
    int rope_rows;
    const int *block_table;
    int block_tokens, max_blocks;
    int *tokens, *pos, *next_ids;
    float *logits;
    int advance, greedy;
    // activations handed between CTAs, as tagged 64-bit words (value, phase tag)
    unsigned long long *xt;   // residual [d]
    unsigned long long *qt;   // rotated q [n_qh * hd]
    unsigned long long *kvt;  // this position's k then v [2 * n_kvh * hd], as the cache holds them
    unsigned long long *ft;   // SiLU(gate) * up [ff]
    unsigned long long *sst;  // per-band square sums of the residual [n_ss]
    int n_ss;
    unsigned long long *pt;   // projection partials: 4 buffers (one per kind) of pt_stride words
    size_t pt_stride;
    unsigned long long *at;   // attention split records [n_kvh][attn_splits][GQ * (hd + 2)]
    float *am_val;
    int *am_idx;
    int *am_counter;
    unsigned long long *epoch;  // steps completed (tags derive from it)
    int n_steps;                // greedy steps this launch decodes (tokens hand over on the device)
    int *ids_out;               // optional: the id picked at every step [n_steps]
    unsigned long long *tokt;   // tagged word: a step's pick, read by the next step's embed
    int *err;
    int *abort_flag;
    unsigned long long *phase_times;  // optional: globaltimer at every phase start, then at the end
    unsigned long long *trace;        // optional: [phase][cta][5] per-CTA timestamps
    int nb_qkv, nb_o, nb_gu, nb_d;
    int attn_splits;
    int stages;             // ring stages in use
    // the cached K/V of each CTA's attention item streamed through the ring
    // (between the q|k|v and o stages of a layer) when kv_tma is set:
    const CUtensorMap *kv_maps;  // per layer: K map, V map; 2-D {n_kvh * hd, rows}, boxes {hd, block_tokens}
    int kv_tma;
    int kv_align;           // attention split boundaries are multiples of this (whole blocks)
    int kv_stage_pos;       // positions per K/V stage
    int scratch_floats;     // shared scratch after the ring
    int max_inflight;       // weight stages requested and not yet landed at most (0: no cap)
    int chain_inflight;     // the same while the attention chain runs (o and K/V stages; 0: max_inflight)
    int chain_gu_stages;    // first gate|up stages issued under chain_inflight
    void *kc[kStMaxLayers];
    void *vc[kStMaxLayers];
};

size_t step_layer_bytes();
void step_layer_fill(void *dst, const CUtensorMap *maps5, const float *n1, const float *n2, const float *qn,
                     const float *kn);
int step_scratch_floats(const ds_model_config *c, int grid, int nb_qkv, int nb_o, int nb_gu, int nb_d);
bool step_supported(const ds_model_config *c);
int step_stages(int scratch_floats);
int step_inflight_setting();
void step_chain_setting(int *cap, int *gu_stages);
int step_stage_bytes();  // bytes of one ring stage of the step kernel
size_t step_smem_bytes(int stages, int scratch_floats);
cudaError_t launch_step(const void *params, int w_dtype, int kv_dtype, int gq, int grid, cudaStream_t stream);

}  // namespace ds
