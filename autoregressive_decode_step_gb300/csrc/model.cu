// The decode step: model object, workspace layout, the per-step launch
// sequence, CUDA-graph capture and per-kernel timing.
//
// Per layer the step launches five kernels ("The forward pass end to end",
// "What a forward step does"; "Inside the engine", section 1):
//   1. fused q|k|v projection with RMSNorm in its prologue and RoPE + the K/V
//      cache write in its epilogue (qkPrep);
//   2. split-context grouped-query attention with its cross-split reduce;
//   3. output projection with the residual add in its epilogue;
//   4. fused gate|up projection with RMSNorm in its prologue and SiLU-gate in
//      its epilogue;
//   5. down projection with the residual add in its epilogue;
// then the output head with the final RMSNorm in its prologue and the greedy
// argmax fused in (or the sampler after it).  Every kernel is launched with
// programmatic dependent launch, so each one's weight stream starts while its
// predecessor drains.
#include <cstring>
#include <new>
#include <vector>

#include "common.cuh"
#include "internal.h"
#include "tc.h"

namespace ds {
cudaError_t prepare_kernels();
}

struct ds_model {
    ds_model_config cfg;
    const void *emb, *out;
    const float *final_norm;
    std::vector<const float *> n1, n2;
    std::vector<const float *> qn, kn;  // QK-norm weights per layer (empty: none)
    std::vector<const void *> wqkv, wo, wgu, wd;
    char *ws;
    size_t ws_bytes;
    int *err;
    float *x, *q, *att, *f, *logits, *rope_cos, *rope_sin;
    int *g_counters;
    float *g_partials;
    int *a_counters;
    float *a_partials;
    float *am_val;
    int *am_idx;
    int *am_counter;
    int grid_qkv, grid_o, grid_gu, grid_d, grid_head;
    int nb_qkv, nb_o, nb_gu, nb_d;
    int attn_splits;
    int es;
    // tensor maps of every projection, per layer: qkv, o, gate, up, down
    std::vector<CUtensorMap> maps;
    // the persistent step kernel
    bool step_ok;
    int step_grid, step_splits, step_stages, step_scratch;
    int step_inflight;  // weight stages in flight at most (0: no cap)
    int step_chain_inflight, step_chain_gu;  // the cap during the attention chain
    ds::StepLayer *step_layers;
    unsigned *step_bar;
    int *step_abort;
    unsigned long long *phase_times;
    int n_phase_times;
    unsigned long long *trace;
    size_t trace_words;
    // tagged activation words and partials of the step kernel
    unsigned long long *st_x, *st_q, *st_kv, *st_f, *st_ss, *st_part, *st_att;
    size_t st_part_stride;
    // the batched step (max_seqs > 1): projections on the tensor cores
    bool batched;
    int b_splits;
    void *h_bf, *att_bf, *f_bf;  // projection inputs as bf16 pairs: [2][max_seqs][d | nq | ff], hi then lo
    int *b_am_counters;          // argmax arrival counters, one per sequence
    int *seq_rows;               // [2][max_seqs]: a prompt chunk's positions, then each row's sequence
    std::vector<ds::TcArgs> tc;  // per layer: q|k|v, o, gate|up, down; then the head
    // tensor maps of the K/V buffers for the paged attention, per layer, and
    // the cache they were encoded for (re-encoded when a step passes another)
    // K/V tensor maps of the persistent step kernel (device copy in the
    // workspace), and the cache they were encoded for
    CUtensorMap *kv_maps_dev;
    const void *kv_k0 = nullptr;
    long long kv_rows_enc = -1;
    int kv_bt_enc = -1;
    int kv_tma_cur = 0;
    std::vector<CUtensorMap> pa_maps;
    std::vector<int> pa_box3d;
    std::vector<const void *> pa_k, pa_v;
    std::vector<long long> pa_rows;
};

struct ds_step_graph {
    cudaGraph_t graph;
    cudaGraphExec_t exec;
};

namespace {

using namespace ds;

struct Layout {
    size_t x, q, att, f, logits, rope_cos, rope_sin, g_counters, g_partials, a_counters, a_partials, am_val,
        am_idx, am_counter, step_layers, step_bar, phase_times, trace, st_x, st_q, st_kv, st_f, st_ss, st_part,
        st_att, h_bf, att_bf, f_bf, tc_counters, tc_partials, tc_ssq, b_am_counters, seq_rows, kv_maps, total;
    int b_splits, tc_tiles;
    size_t st_part_stride;
    int grid_qkv, grid_o, grid_gu, grid_d, grid_head, nb_qkv, nb_o, nb_gu, nb_d, attn_splits;
    bool step_ok;
    int step_grid, step_splits, step_stages, step_scratch, n_phase_times;
};

int validate(const ds_model_config *c) {
    if (!c) return DS_BAD_ARGUMENT;
    if (c->vocab < 1 || c->d < 1 || c->n_layer < 0 || c->n_qh < 1 || c->n_kvh < 1 || c->head_dim < 2 || c->ff < 1 ||
        c->max_seqs < 1 || c->max_ctx < 1)
        return DS_EMPTY_DIMENSION;
    if (c->vocab > DS_MAX_DIM || c->d > DS_MAX_DIM || c->ff > DS_MAX_DIM || c->max_ctx > DS_MAX_DIM ||
        (int64_t)c->n_qh * c->head_dim > DS_MAX_DIM)
        return DS_DIMENSION_TOO_LARGE;
    if ((c->w_dtype != DS_F32 && c->w_dtype != DS_BF16) || (c->kv_dtype != DS_F32 && c->kv_dtype != DS_BF16) ||
        (c->rope_layout != DS_ROPE_HALF_SPLIT && c->rope_layout != DS_ROPE_INTERLEAVED))
        return DS_BAD_DTYPE;
    const int gq = c->n_qh / c->n_kvh;
    if (c->n_qh % c->n_kvh || (gq != 1 && gq != 2 && gq != 4 && gq != 8)) return DS_BAD_ARGUMENT;
    if (c->head_dim % 4 || c->head_dim > 256 || (c->head_dim > 128 && c->head_dim % 8)) return DS_BAD_ARGUMENT;
    const int es = c->w_dtype == DS_BF16 ? 2 : 4;
    // every projection streams whole 16-byte chunks; a band holds whole heads
    if (((int64_t)c->d * es) % 16 || ((int64_t)c->ff * es) % 16 || ((int64_t)c->n_qh * c->head_dim * es) % 16 ||
        ((int64_t)c->n_kvh * c->head_dim * es) % 16)
        return DS_BAD_ARGUMENT;
    if (gemv_t_band_cols(es) % c->head_dim) return DS_BAD_ARGUMENT;
    if (!gemv_n_streamable(nullptr, c->vocab, c->d, es)) return DS_BAD_ARGUMENT;
    if (!(c->eps >= 0.0f) || !(c->rope_base > 0.0)) return DS_BAD_ARGUMENT;
    if (c->rope_factor != 0.0 &&
        !(c->rope_factor >= 1.0 && c->rope_low_freq_factor > 0.0 &&
          c->rope_high_freq_factor > c->rope_low_freq_factor && c->rope_orig_max_pos > 0.0 &&
          c->rope_factor < 1e300 && c->rope_high_freq_factor < 1e300 && c->rope_orig_max_pos < 1e300))
        return DS_BAD_ARGUMENT;
    if (c->max_seqs > 256) return DS_DIMENSION_TOO_LARGE;
    if (c->max_seqs > 1) {
        // the batched step runs its projections on bf16 tensor cores, with
        // whole heads in every 128-feature tile
        if (c->w_dtype != DS_BF16) return DS_BAD_DTYPE;
        if (128 % c->head_dim) return DS_BAD_ARGUMENT;
    }
    return DS_OK;
}

size_t carve(size_t &off, size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes, 256);
    return at;
}

Layout make_layout(const ds_model_config *c) {
    Layout L = {};
    const int es = c->w_dtype == DS_BF16 ? 2 : 4;
    const int bc = gemv_t_band_cols(es);
    const int nq = c->n_qh * c->head_dim, nkv = c->n_kvh * c->head_dim;
    const int S = c->max_seqs;
    L.nb_qkv = (nq + 2 * nkv + bc - 1) / bc;
    L.nb_o = (c->d + bc - 1) / bc;
    L.nb_gu = (c->ff + bc / 2 - 1) / (bc / 2);
    L.nb_d = (c->d + bc - 1) / bc;
    L.grid_qkv = gemv_t_grid(c->d, L.nb_qkv);
    L.grid_o = gemv_t_grid(nq, L.nb_o);
    L.grid_gu = gemv_t_grid(c->d, L.nb_gu);
    L.grid_d = gemv_t_grid(c->ff, L.nb_d);
    L.grid_head = gemv_n_grid(c->vocab, c->d, es);
    L.attn_splits = attention_splits(S, c->n_kvh, c->max_ctx);
    // the persistent step kernel: one CTA per SM
    L.step_grid = sm_count();
    L.step_ok = step_supported(c) && c->n_kvh <= L.step_grid;
    if (L.step_ok) {
        L.step_splits = std::max(1, std::min(L.step_grid / c->n_kvh, kStMaxSplits));
        L.step_scratch = step_scratch_floats(c, L.step_grid, L.nb_qkv, L.nb_o, L.nb_gu, L.nb_d);
        L.step_stages = step_stages(L.step_scratch);
        L.step_ok = L.step_stages >= 2;
    }
    L.n_phase_times = 5 * c->n_layer + 4;
    // the batched step: attention splits of about 256 positions at the
    // largest context; tensor-core tiles of the largest projection
    const bool batched = S > 1;
    L.b_splits = batched ? (int)std::min<long long>(kStMaxSplits, std::max<long long>(1, (c->max_ctx + 255) / 256)) : 0;
    if (batched) {
        const int nqkv = nq + 2 * nkv;
        L.tc_tiles = std::max(std::max(tc_m_tiles(nqkv, TC_QKV), tc_m_tiles(c->d, TC_ADD)),
                              std::max(tc_m_tiles(c->ff, TC_SILU), tc_m_tiles(c->vocab, TC_STORE)));
        // counted in 128-feature sub-tiles: a pairing never needs more partial
        // space than (SMs + sub-tiles) single sub-tiles
    }
    size_t partial = 0;
    partial = std::max(partial, gemv_t_partial_floats(L.grid_qkv, L.nb_qkv, es));
    partial = std::max(partial, gemv_t_partial_floats(L.grid_o, L.nb_o, es));
    partial = std::max(partial, gemv_t_partial_floats(L.grid_gu, L.nb_gu, es));
    partial = std::max(partial, gemv_t_partial_floats(L.grid_d, L.nb_d, es));
    const int max_nb = std::max(std::max(L.nb_qkv, L.nb_o), std::max(L.nb_gu, L.nb_d));
    partial = std::max(partial, gemv_t_partial_floats(L.step_grid, max_nb, es));
    const int max_bands = std::max(std::max(L.nb_qkv, L.nb_o), std::max(L.nb_gu, L.nb_d));
    size_t off = kWsHeader;
    L.x = carve(off, (size_t)S * c->d * 4);
    L.q = carve(off, (size_t)S * nq * 4);
    L.att = carve(off, (size_t)S * nq * 4);
    L.f = carve(off, (size_t)S * c->ff * 4);
    L.logits = carve(off, (size_t)S * c->vocab * 4);
    L.rope_cos = carve(off, (size_t)c->max_ctx * (c->head_dim / 2) * 4);
    L.rope_sin = carve(off, (size_t)c->max_ctx * (c->head_dim / 2) * 4);
    L.g_counters = carve(off, (size_t)max_bands * 4);
    L.g_partials = carve(off, partial * 4);
    L.a_counters = carve(off, (size_t)S * c->n_kvh * 4);
    size_t a_part = attention_partial_floats(S, c->n_qh, c->n_kvh, c->head_dim,
                                             std::max(std::max(L.attn_splits, L.step_splits), L.b_splits));
    if (batched) a_part = std::max(a_part, paged_attention_partial_floats(S, c->n_qh));
    L.a_partials = carve(off, a_part * 4);
    const size_t am_slots = std::max((size_t)std::max(L.grid_head, L.step_grid),
                                     (size_t)S * argmax_blocks_per_row(c->vocab));
    L.am_val = carve(off, am_slots * 4);
    L.am_idx = carve(off, am_slots * 4);
    L.am_counter = carve(off, 4);
    L.step_layers = carve(off, (size_t)std::max(c->n_layer, 1) * step_layer_bytes());
    L.kv_maps = carve(off, (size_t)2 * std::max(c->n_layer, 1) * sizeof(CUtensorMap));
    L.step_bar = carve(off, 32);  // arrival count (u64), epoch (u64), abort flag (int, + pad), handed-over token (u64)
    L.phase_times = carve(off, (size_t)L.n_phase_times * 8);
    L.trace = carve(off, (size_t)L.n_phase_times * L.step_grid * 5 * 8);
    if (L.step_ok) {
        const int gq = c->n_qh / c->n_kvh;
        L.st_x = carve(off, (size_t)c->d * 8);
        L.st_q = carve(off, (size_t)nq * 8);
        L.st_kv = carve(off, (size_t)2 * nkv * 8);
        L.st_f = carve(off, (size_t)c->ff * 8);
        L.st_ss = carve(off, (size_t)L.nb_o * 8);
        // partial slot = CTA + band, one buffer per projection kind
        L.st_part_stride = (size_t)(L.step_grid + max_bands) * bc;
        L.st_part = carve(off, 4 * L.st_part_stride * 8);
        L.st_att = carve(off, (size_t)c->n_kvh * L.step_splits * gq * (c->head_dim + 2) * 8);
    }
    if (batched) {
        L.h_bf = carve(off, (size_t)2 * S * c->d * 2);
        L.att_bf = carve(off, (size_t)2 * S * nq * 2);
        L.f_bf = carve(off, (size_t)2 * S * c->ff * 2);
        L.tc_counters = carve(off, (size_t)L.tc_tiles * 4);
        L.tc_partials = carve(off, tc_partial_floats(L.tc_tiles, tc_n_pad(S), 2) * 4);
        // per 128-feature tile of the residual, each sequence's square sum (the folded RMSNorms)
        L.tc_ssq = carve(off, (size_t)tc_m_tiles(c->d, TC_ADD) * S * 4);
        L.b_am_counters = carve(off, (size_t)S * 4);
        L.seq_rows = carve(off, (size_t)2 * S * 4);  // a prompt chunk's positions, then its rows' sequence
    }
    L.total = off;
    return L;
}

int check_kv(const ds_model *m, const ds_kv_cache *kv) {
    if (!kv || !kv->k || !kv->v) return DS_BAD_ARGUMENT;
    if (kv->block_tokens < 1 || kv->max_blocks < 1 || kv->rows < 1) return DS_EMPTY_DIMENSION;
    const int64_t cap = (int64_t)kv->block_tokens * kv->max_blocks;
    if (cap > DS_MAX_DIM) return DS_DIMENSION_TOO_LARGE;
    if (!kv->block_table && cap * m->cfg.max_seqs > kv->rows) return DS_CACHE_CAPACITY_EXCEEDED;
    const int es = m->cfg.kv_dtype == DS_BF16 ? 2 : 4;
    for (int l = 0; l < m->cfg.n_layer; ++l) {
        if (!kv->k[l] || !kv->v[l]) return DS_BAD_ARGUMENT;
        if (((uintptr_t)kv->k[l] | (uintptr_t)kv->v[l]) & 15) return DS_BAD_ARGUMENT;
    }
    (void)es;
    return DS_OK;
}

// Optional per-launch event recorder used by the profiler.
struct Recorder {
    std::vector<cudaEvent_t> ev;
    std::vector<int> kind;
    size_t used = 0;
    cudaStream_t stream;
    bool record(int k) {
        if (used >= ev.size()) {
            cudaEvent_t e;
            if (cudaEventCreate(&e) != cudaSuccess) return false;
            ev.push_back(e);
            kind.push_back(k);
        }
        kind[used] = k;
        return cudaEventRecord(ev[used++], stream) == cudaSuccess;
    }
    ~Recorder() {
        for (auto e : ev) cudaEventDestroy(e);
    }
};

// Launch one decode step; with only_kind >= 0 launch just the kernels of
// that kind (DS_KIND_*), in step order, for timing.
int run_step(ds_model *m, const ds_kv_cache *kv, int32_t *tokens, int32_t *pos, int n_seqs,
             const ds_sampling *sampling, const float *u, int32_t *next_ids, float *logits_out, unsigned flags,
             cudaStream_t s, Recorder *rec, int only_kind = -1) {
    const ds_model_config &c = m->cfg;
    const int es = m->es;
    const int nq = c.n_qh * c.head_dim, nkv = c.n_kvh * c.head_dim;
    const bool pdl = rec == nullptr;
    const bool greedy = sampling == nullptr || !(sampling->temperature > 0.0f);
    const bool advance = (flags & DS_STEP_ADVANCE) != 0;
    float *logits = logits_out ? logits_out : m->logits;
    cudaError_t e;
#define DS_TRY(expr, kind)                                   \
    do {                                                     \
        if (only_kind < 0 || only_kind == (kind)) {          \
            e = (expr);                                      \
            if (e != cudaSuccess) return DS_CUDA_ERROR;      \
            if (rec && !rec->record(kind)) return DS_CUDA_ERROR; \
        }                                                    \
    } while (0)

    if (rec && !rec->record(-1)) return DS_CUDA_ERROR;
    DS_TRY(launch_embed(m->emb, c.w_dtype, c.vocab, c.d, tokens, m->x, m->err, n_seqs, s, pdl), DS_KIND_EMBED);

    GemvTArgs g = {};
    g.err = m->err;
    g.counters = m->g_counters;
    g.partials = m->g_partials;
    g.eps = c.eps;
    for (int l = 0; l < c.n_layer; ++l) {
        // 1. q|k|v = Wqkv^T RMSNorm(x, n1); RoPE; K/V written at pos
        GemvTArgs a = g;
        a.a0 = static_cast<const char *>(m->wqkv[l]);
        a.row_stride = (long long)(nq + 2 * nkv) * es;
        a.K = c.d;
        a.sub_cols = nq + 2 * nkv;
        a.n_bands = m->nb_qkv;
        a.x = m->x;
        a.norm_w = m->n1[l];
        a.y = m->q;
        a.k_cache = kv->k[l];
        a.v_cache = kv->v[l];
        a.kv_dtype = c.kv_dtype;
        a.pos = pos;
        a.nq_cols = nq;
        a.nkv_cols = nkv;
        a.head_dim = c.head_dim;
        a.rope_layout = c.rope_layout;
        a.rope_cos = m->rope_cos;
        a.rope_sin = m->rope_sin;
        a.rope_rows = c.max_ctx;
        a.block_table = kv->block_table;
        a.block_tokens = kv->block_tokens;
        a.max_blocks = kv->max_blocks;
        a.q_norm = m->qn.empty() ? nullptr : m->qn[l];
        a.k_norm = m->kn.empty() ? nullptr : m->kn[l];
        a.tm0 = m->maps[5 * l + 0];
        DS_TRY(launch_gemv_t(a, c.w_dtype, PRO_RMSNORM, EPI_QKV, m->grid_qkv, s, pdl), DS_KIND_QKV);

        // 2. attention over positions 0..pos
        AttnArgs at = {};
        at.q = m->q;
        at.k_cache = kv->k[l];
        at.v_cache = kv->v[l];
        at.kv_dtype = c.kv_dtype;
        at.cache_rows = kv->rows;
        at.block_table = kv->block_table;
        at.max_blocks = kv->max_blocks;
        at.block_tokens = kv->block_tokens;
        at.seq_lens = nullptr;
        at.pos = pos;
        at.n_qh = c.n_qh;
        at.n_kvh = c.n_kvh;
        at.hd = c.head_dim;
        at.scale = 1.0f / sqrtf((float)c.head_dim);
        at.out = m->att;
        at.partials = m->a_partials;
        at.counters = m->a_counters;
        at.err = m->err;
        at.n_splits = m->attn_splits;
        DS_TRY(launch_attention(at, n_seqs, s, pdl), DS_KIND_ATTENTION);

        // 3. x += Wo^T att
        a = g;
        a.a0 = static_cast<const char *>(m->wo[l]);
        a.row_stride = (long long)c.d * es;
        a.K = nq;
        a.sub_cols = c.d;
        a.n_bands = m->nb_o;
        a.x = m->att;
        a.y = m->x;
        a.tm0 = m->maps[5 * l + 1];
        DS_TRY(launch_gemv_t(a, c.w_dtype, PRO_PLAIN, EPI_ADD, m->grid_o, s, pdl), DS_KIND_O_PROJ);

        // 4. f = silu(Wg^T h) * (Wu^T h), h = RMSNorm(x, n2)
        a = g;
        a.a0 = static_cast<const char *>(m->wgu[l]);
        a.a1 = static_cast<const char *>(m->wgu[l]) + (size_t)c.ff * es;
        a.row_stride = (long long)2 * c.ff * es;
        a.K = c.d;
        a.sub_cols = c.ff;
        a.n_bands = m->nb_gu;
        a.x = m->x;
        a.norm_w = m->n2[l];
        a.y = m->f;
        a.tm0 = m->maps[5 * l + 2];
        a.tm1 = m->maps[5 * l + 3];
        DS_TRY(launch_gemv_t(a, c.w_dtype, PRO_RMSNORM, EPI_SILU, m->grid_gu, s, pdl), DS_KIND_GATE_UP);

        // 5. x += Wd^T f
        a = g;
        a.a0 = static_cast<const char *>(m->wd[l]);
        a.row_stride = (long long)c.d * es;
        a.K = c.ff;
        a.sub_cols = c.d;
        a.n_bands = m->nb_d;
        a.x = m->f;
        a.y = m->x;
        a.tm0 = m->maps[5 * l + 4];
        DS_TRY(launch_gemv_t(a, c.w_dtype, PRO_PLAIN, EPI_ADD, m->grid_d, s, pdl), DS_KIND_DOWN);
    }

    // logits = Out . RMSNorm(x, final); greedy argmax fused
    GemvNArgs h = {};
    h.W = static_cast<const char *>(c.tied ? m->emb : m->out);
    h.rows = c.vocab;
    h.cols = c.d;
    h.x = m->x;
    h.norm_w = m->final_norm;
    h.eps = c.eps;
    h.y = logits;
    h.do_argmax = greedy ? 1 : 0;
    h.part_val = m->am_val;
    h.part_idx = m->am_idx;
    h.counter = m->am_counter;
    h.ids_out = next_ids;
    h.max_out = nullptr;
    h.tokens_adv = advance ? tokens : nullptr;
    h.pos_adv = advance ? pos : nullptr;
    h.err = m->err;
    DS_TRY(launch_gemv_n(h, c.w_dtype, PRO_RMSNORM, m->grid_head, s, pdl), DS_KIND_HEAD);

    if (!greedy) {
        SampleArgs sa = {};
        sa.logits = logits;
        sa.n_rows = n_seqs;
        sa.n = c.vocab;
        sa.temperature = sampling->temperature;
        sa.top_k = sampling->top_k;
        sa.top_p = sampling->top_p;
        sa.u = u;
        sa.ids = next_ids;
        sa.tokens_adv = advance ? tokens : nullptr;
        sa.pos_adv = advance ? pos : nullptr;
        sa.err = m->err;
        DS_TRY(launch_sample(sa, s, pdl), DS_KIND_SAMPLE);
    }
#undef DS_TRY
    return DS_OK;
}

int check_step(ds_model *m, const ds_kv_cache *kv, int32_t *tokens, int32_t *pos, int n_seqs,
               const ds_sampling *sampling, const float *u, int32_t *next_ids) {
    if (!m) return DS_BAD_ARGUMENT;
    if (n_seqs < 1) return DS_EMPTY_DIMENSION;
    if (n_seqs > m->cfg.max_seqs) return DS_DIMENSION_TOO_LARGE;
    if (!tokens || !pos || !next_ids) return DS_BAD_ARGUMENT;
    int st = check_kv(m, kv);
    if (st != DS_OK) return st;
    if (sampling && sampling->temperature > 0.0f) {
        if (!(sampling->top_p > 0.0f) || sampling->top_p > 1.0f) return DS_BAD_SAMPLING_PARAM;
        if (!u) return DS_BAD_ARGUMENT;
    } else if (sampling && sampling->temperature != sampling->temperature) {
        return DS_BAD_SAMPLING_PARAM;
    }
    return DS_OK;
}

}  // namespace

extern "C" DS_API size_t ds_model_workspace_bytes(const ds_model_config *cfg) {
    if (validate(cfg) != DS_OK) return 0;
    return make_layout(cfg).total;
}

extern "C" DS_API int ds_model_create(const ds_model_config *cfg, const ds_model_weights *w, void *workspace,
                                      size_t workspace_bytes, ds_model **out) {
    if (!out) return DS_BAD_ARGUMENT;
    *out = nullptr;
    int st = validate(cfg);
    if (st != DS_OK) return st;
    if (!w || !w->emb || (!cfg->tied && !w->out) || !w->final_norm) return DS_BAD_ARGUMENT;
    if (cfg->n_layer > 0 && (!w->n1 || !w->wqkv || !w->wo || !w->n2 || !w->wgu || !w->wd)) return DS_BAD_ARGUMENT;
    const Layout L = make_layout(cfg);
    if (!workspace || workspace_bytes < L.total) return DS_WORKSPACE_TOO_SMALL;
    if ((uintptr_t)workspace & 255) return DS_BAD_ARGUMENT;
    auto aligned = [](const void *p) { return p && ((uintptr_t)p & 15) == 0; };
    if (!aligned(w->emb) || (!cfg->tied && !aligned(w->out))) return DS_BAD_ARGUMENT;
    if (!aligned(w->final_norm)) return DS_BAD_ARGUMENT;
    for (int l = 0; l < cfg->n_layer; ++l)
        if (!aligned(w->wqkv[l]) || !aligned(w->wo[l]) || !aligned(w->wgu[l]) || !aligned(w->wd[l]) ||
            !aligned(w->n1[l]) || !aligned(w->n2[l]))
            return DS_BAD_ARGUMENT;
    // QK-norm: both weight sets or neither
    const bool qk_norm = w->q_norm || w->k_norm;
    if (qk_norm) {
        if (!w->q_norm || !w->k_norm) return DS_BAD_ARGUMENT;
        for (int l = 0; l < cfg->n_layer; ++l)
            if (!w->q_norm[l] || !w->k_norm[l] || ((uintptr_t)w->q_norm[l] & 3) || ((uintptr_t)w->k_norm[l] & 3))
                return DS_BAD_ARGUMENT;
    }

    ds_model *m = new (std::nothrow) ds_model();
    if (!m) return DS_BAD_ARGUMENT;
    m->cfg = *cfg;
    m->es = cfg->w_dtype == DS_BF16 ? 2 : 4;
    m->emb = w->emb;
    m->out = cfg->tied ? w->emb : w->out;
    m->final_norm = w->final_norm;
    for (int l = 0; l < cfg->n_layer; ++l) {
        m->n1.push_back(w->n1[l]);
        m->n2.push_back(w->n2[l]);
        m->wqkv.push_back(w->wqkv[l]);
        m->wo.push_back(w->wo[l]);
        m->wgu.push_back(w->wgu[l]);
        m->wd.push_back(w->wd[l]);
        if (qk_norm) {
            m->qn.push_back(w->q_norm[l]);
            m->kn.push_back(w->k_norm[l]);
        }
    }
    char *ws = static_cast<char *>(workspace);
    m->ws = ws;
    m->ws_bytes = workspace_bytes;
    m->err = reinterpret_cast<int *>(ws);
    m->x = reinterpret_cast<float *>(ws + L.x);
    m->q = reinterpret_cast<float *>(ws + L.q);
    m->att = reinterpret_cast<float *>(ws + L.att);
    m->f = reinterpret_cast<float *>(ws + L.f);
    m->logits = reinterpret_cast<float *>(ws + L.logits);
    m->rope_cos = reinterpret_cast<float *>(ws + L.rope_cos);
    m->rope_sin = reinterpret_cast<float *>(ws + L.rope_sin);
    m->g_counters = reinterpret_cast<int *>(ws + L.g_counters);
    m->g_partials = reinterpret_cast<float *>(ws + L.g_partials);
    m->a_counters = reinterpret_cast<int *>(ws + L.a_counters);
    m->a_partials = reinterpret_cast<float *>(ws + L.a_partials);
    m->am_val = reinterpret_cast<float *>(ws + L.am_val);
    m->am_idx = reinterpret_cast<int *>(ws + L.am_idx);
    m->am_counter = reinterpret_cast<int *>(ws + L.am_counter);
    m->grid_qkv = L.grid_qkv;
    m->grid_o = L.grid_o;
    m->grid_gu = L.grid_gu;
    m->grid_d = L.grid_d;
    m->grid_head = L.grid_head;
    m->nb_qkv = L.nb_qkv;
    m->nb_o = L.nb_o;
    m->nb_gu = L.nb_gu;
    m->nb_d = L.nb_d;
    m->attn_splits = L.attn_splits;

    // tensor maps of every projection
    {
        const int es = m->es;
        const int nq = cfg->n_qh * cfg->head_dim, nkv = cfg->n_kvh * cfg->head_dim;
        m->maps.resize((size_t)5 * cfg->n_layer);
        for (int l = 0; l < cfg->n_layer; ++l) {
            GemvTArgs a = {};
            a.a0 = static_cast<const char *>(m->wqkv[l]);
            a.row_stride = (long long)(nq + 2 * nkv) * es;
            a.K = cfg->d;
            a.sub_cols = nq + 2 * nkv;
            bool ok = gemv_t_make_maps(a, cfg->w_dtype);
            m->maps[5 * l + 0] = a.tm0;
            a = GemvTArgs{};
            a.a0 = static_cast<const char *>(m->wo[l]);
            a.row_stride = (long long)cfg->d * es;
            a.K = nq;
            a.sub_cols = cfg->d;
            ok = ok && gemv_t_make_maps(a, cfg->w_dtype);
            m->maps[5 * l + 1] = a.tm0;
            a = GemvTArgs{};
            a.a0 = static_cast<const char *>(m->wgu[l]);
            a.a1 = static_cast<const char *>(m->wgu[l]) + (size_t)cfg->ff * es;
            a.row_stride = (long long)2 * cfg->ff * es;
            a.K = cfg->d;
            a.sub_cols = cfg->ff;
            ok = ok && gemv_t_make_maps(a, cfg->w_dtype);
            m->maps[5 * l + 2] = a.tm0;
            m->maps[5 * l + 3] = a.tm1;
            a = GemvTArgs{};
            a.a0 = static_cast<const char *>(m->wd[l]);
            a.row_stride = (long long)cfg->d * es;
            a.K = cfg->ff;
            a.sub_cols = cfg->d;
            ok = ok && gemv_t_make_maps(a, cfg->w_dtype);
            m->maps[5 * l + 4] = a.tm0;
            if (!ok) {
                delete m;
                return DS_CUDA_ERROR;
            }
        }
    }
    m->step_ok = L.step_ok;
    m->step_grid = L.step_grid;
    m->step_splits = L.step_splits;
    m->step_stages = L.step_stages;
    m->step_scratch = L.step_scratch;
    m->step_inflight = step_inflight_setting();
    step_chain_setting(&m->step_chain_inflight, &m->step_chain_gu);
    m->step_layers = reinterpret_cast<StepLayer *>(ws + L.step_layers);
    m->kv_maps_dev = reinterpret_cast<CUtensorMap *>(ws + L.kv_maps);
    m->step_bar = reinterpret_cast<unsigned *>(ws + L.step_bar);
    m->step_abort = reinterpret_cast<int *>(ws + L.step_bar + 16);
    m->phase_times = reinterpret_cast<unsigned long long *>(ws + L.phase_times);
    m->n_phase_times = L.n_phase_times;
    m->trace = reinterpret_cast<unsigned long long *>(ws + L.trace);
    m->trace_words = (size_t)L.n_phase_times * L.step_grid * 5;
    m->st_x = reinterpret_cast<unsigned long long *>(ws + L.st_x);
    m->st_q = reinterpret_cast<unsigned long long *>(ws + L.st_q);
    m->st_kv = reinterpret_cast<unsigned long long *>(ws + L.st_kv);
    m->st_f = reinterpret_cast<unsigned long long *>(ws + L.st_f);
    m->st_ss = reinterpret_cast<unsigned long long *>(ws + L.st_ss);
    m->st_part = reinterpret_cast<unsigned long long *>(ws + L.st_part);
    m->st_att = reinterpret_cast<unsigned long long *>(ws + L.st_att);
    m->st_part_stride = L.st_part_stride;

    m->batched = cfg->max_seqs > 1;
    m->b_splits = L.b_splits;
    if (m->batched) {
        m->h_bf = ws + L.h_bf;
        m->att_bf = ws + L.att_bf;
        m->f_bf = ws + L.f_bf;
        m->b_am_counters = reinterpret_cast<int *>(ws + L.b_am_counters);
        m->seq_rows = reinterpret_cast<int *>(ws + L.seq_rows);
        const int S = cfg->max_seqs, es = 2;
        const int nq = cfg->n_qh * cfg->head_dim, nkv = cfg->n_kvh * cfg->head_dim, nqkv = nq + 2 * nkv;
        // pair = 2: two 128-feature sub-tiles per stage share one activation tile
        // (the large gate|up and head matrices always; q|k|v, o and down up to
        // 128 vectors, where both accumulators still fit in tensor memory):
        // an SM's intake per weight byte then carries half the activation bytes
        auto mk = [&](int epi, int a_mn, const void *A0, const void *A1, long long stride, int M, int K, void *X,
                      TcArgs &a, int pair) {
            a = TcArgs{};
            a.a_mn = a_mn;
            a.M = M;
            a.K = K;
            a.n = S;
            a.n_pad = tc_n_pad(S);
            a.split = 1;  // fp32 activations as bf16 hi + lo rows, S rows apart
            a.b_lo_row = S;
            a.epi = epi;
            a.msub = pair == 2 ? 2 : 1;
            // two accumulators (one tile's epilogue overlapping the next
            // tile's MMAs) where TMEM holds them; above 128 vectors a paired
            // tile keeps one, which still halves the activation tiles
            // streamed per weight byte
            a.acc_bufs = 2 * a.msub * a.n_pad <= 512 ? 2 : 1;
            a.m_tiles = (tc_m_tiles(M, epi) + a.msub - 1) / a.msub;
            a.stages = tc_stages(a.n_pad, 1, a.msub);
            a.tmem_cols = tc_tmem_cols(a.acc_bufs, a.msub, a.n_pad);
            a.partials = reinterpret_cast<float *>(ws + L.tc_partials);
            a.counters = reinterpret_cast<int *>(ws + L.tc_counters);
            a.err = m->err;
            return tc_make_maps(a, A0, A1, stride, X);
        };
        m->tc.resize((size_t)4 * cfg->n_layer + 1);
        bool ok = true;
        for (int l = 0; l < cfg->n_layer && ok; ++l) {
            TcArgs &q = m->tc[4 * l + 0];
            const int pair_small = tc_n_pad(S) <= 128 ? 2 : 1;
            ok = ok && mk(TC_QKV, 1, m->wqkv[l], nullptr, (long long)nqkv * es, nqkv, cfg->d, m->h_bf, q, pair_small);
            q.y = m->q;
            q.ldy = nq;
            q.rope_cos = m->rope_cos;
            q.rope_sin = m->rope_sin;
            q.rope_rows = cfg->max_ctx;
            q.nq_cols = nq;
            q.nkv_cols = nkv;
            q.head_dim = cfg->head_dim;
            q.rope_layout = cfg->rope_layout;
            q.kv_dtype = cfg->kv_dtype;
            q.q_norm = qk_norm ? w->q_norm[l] : nullptr;
            q.k_norm = qk_norm ? w->k_norm[l] : nullptr;
            q.qk_eps = cfg->eps;
            TcArgs &o = m->tc[4 * l + 1];
            ok = ok && mk(TC_ADD, 1, m->wo[l], nullptr, (long long)cfg->d * es, cfg->d, nq, m->att_bf, o, pair_small);
            o.y = m->x;
            o.ldy = cfg->d;
            TcArgs &gu = m->tc[4 * l + 2];
            ok = ok && mk(TC_SILU, 1, m->wgu[l], static_cast<const char *>(m->wgu[l]) + (size_t)cfg->ff * es,
                          (long long)2 * cfg->ff * es, cfg->ff, cfg->d, m->h_bf, gu, 2);
            gu.yb = static_cast<__nv_bfloat16 *>(m->f_bf);
            gu.yb_lo = (long long)S * cfg->ff;
            gu.ldy = cfg->ff;
            TcArgs &dn = m->tc[4 * l + 3];
            ok = ok && mk(TC_ADD, 1, m->wd[l], nullptr, (long long)cfg->d * es, cfg->d, cfg->ff, m->f_bf, dn, pair_small);
            dn.y = m->x;
            dn.ldy = cfg->d;
            // RMSNorms folded into the projections: o and down also write the
            // next norm's input (x * weight, hi/lo) and per-tile square sums;
            // gate|up and the next layer's q|k|v apply the 1/rms scale
            float *ssq = reinterpret_cast<float *>(ws + L.tc_ssq);
            auto fold_out = [&](TcArgs &a, const float *nw) {
                a.nw = nw;
                a.hb = static_cast<__nv_bfloat16 *>(m->h_bf);
                a.hb_lo = (long long)S * cfg->d;
                a.ssq = ssq;
                a.ss_ld = S;
            };
            auto fold_in = [&](TcArgs &a) {
                a.ssq_in = ssq;
                a.ss_tiles = tc_m_tiles(cfg->d, TC_ADD);
                a.ss_ld = S;
                a.ss_d = cfg->d;
                a.eps = cfg->eps;
            };
            fold_out(o, w->n2[l]);
            fold_in(gu);
            if (l + 1 < cfg->n_layer) fold_out(dn, w->n1[l + 1]);
            if (l > 0) fold_in(q);
        }
        TcArgs &hd = m->tc[(size_t)4 * cfg->n_layer];
        ok = ok && mk(TC_STORE, 0, m->out, nullptr, (long long)cfg->d * es, cfg->vocab, cfg->d, m->h_bf, hd, 2);
        hd.ldy = cfg->vocab;
        if (!ok || prepare_tc_kernels() != cudaSuccess || prepare_paged_attention() != cudaSuccess) {
            delete m;
            return DS_CUDA_ERROR;
        }
    }

    std::vector<unsigned char> layer_img((size_t)std::max(cfg->n_layer, 1) * step_layer_bytes(), 0);
    for (int l = 0; l < cfg->n_layer; ++l)
        step_layer_fill(layer_img.data() + (size_t)l * step_layer_bytes(), &m->maps[5 * l], w->n1[l], w->n2[l],
                        qk_norm ? w->q_norm[l] : nullptr, qk_norm ? w->k_norm[l] : nullptr);
    if (prepare_kernels() != cudaSuccess || cudaMemset(workspace, 0, L.total) != cudaSuccess ||
        cudaMemcpy(m->step_layers, layer_img.data(), layer_img.size(), cudaMemcpyHostToDevice) != cudaSuccess ||
        launch_rope_table(m->rope_cos, m->rope_sin, cfg->max_ctx, cfg->head_dim, cfg->rope_base,
                          RopeScaling{cfg->rope_factor, cfg->rope_low_freq_factor, cfg->rope_high_freq_factor,
                                      cfg->rope_orig_max_pos},
                          nullptr) !=
            cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess) {
        delete m;
        return DS_CUDA_ERROR;
    }
    *out = m;
    return DS_OK;
}

extern "C" DS_API void ds_model_destroy(ds_model *m) { delete m; }

extern "C" DS_API void *ds_model_workspace(ds_model *m) { return m ? m->ws : nullptr; }

// Positions per K/V stage of the step kernel's ring (K rows then V rows of
// one head in a 64 KB stage, a multiple of 64 and of the block size, at most
// 256), or 0 when the cache geometry cannot stream through the ring.
int kv_stage_positions(const ds_model_config &c, int block_tokens) {
    const int es = c.kv_dtype == DS_BF16 ? 2 : 4;
    const int row = c.head_dim * es;
    if (row % 16 || c.head_dim > 128 || ((long long)c.n_kvh * row) % 16) return 0;
    int P = std::min(256, step_stage_bytes() / (2 * row)) / 64 * 64;
    if (P < 64 || block_tokens < 1 || block_tokens > 256 || P % block_tokens) return 0;
    // every box of a block lands block_tokens * row bytes after the previous
    // one: tensor copies need 128-byte-aligned shared-memory destinations
    if (((long long)block_tokens * row) % 128 || ((long long)P * row) % 128) return 0;
    return P;
}

// Encode the step kernel's per-layer K/V maps for this cache and upload them,
// when the cache differs from the one they were made for.  Runs before any
// capture (a synchronous copy of a few KB).
int ensure_kv_maps(ds_model *m, const ds_kv_cache *kv, cudaStream_t s) {
    const ds_model_config &c = m->cfg;
    if (!m->step_ok || m->batched) return DS_OK;
    if (m->kv_k0 == kv->k[0] && m->kv_rows_enc == kv->rows && m->kv_bt_enc == kv->block_tokens) return DS_OK;
    m->kv_tma_cur = 0;
    if (kv_stage_positions(c, kv->block_tokens) > 0) {
        std::vector<CUtensorMap> maps((size_t)2 * c.n_layer);
        const int es = c.kv_dtype == DS_BF16 ? 2 : 4;
        const long long cols = (long long)c.n_kvh * c.head_dim;
        bool ok = true;
        for (int l = 0; l < c.n_layer && ok; ++l)
            ok = encode_tiled_2d(&maps[2 * l], kv->k[l], c.kv_dtype, cols, kv->rows, cols * es, c.head_dim,
                                 kv->block_tokens, false) &&
                 encode_tiled_2d(&maps[2 * l + 1], kv->v[l], c.kv_dtype, cols, kv->rows, cols * es, c.head_dim,
                                 kv->block_tokens, false);
        if (ok) {
            if (cudaMemcpyAsync(m->kv_maps_dev, maps.data(), maps.size() * sizeof(CUtensorMap), cudaMemcpyHostToDevice,
                                s) != cudaSuccess ||
                cudaStreamSynchronize(s) != cudaSuccess)
                return DS_CUDA_ERROR;
            m->kv_tma_cur = 1;
        }
    }
    m->kv_k0 = kv->k[0];
    m->kv_rows_enc = kv->rows;
    m->kv_bt_enc = kv->block_tokens;
    return DS_OK;
}

// One step through the persistent step kernel (and the sampler after it).
int run_step_fused(ds_model *m, const ds_kv_cache *kv, int32_t *tokens, int32_t *pos, int n_seqs,
                   const ds_sampling *sampling, const float *u, int32_t *next_ids, float *logits_out, unsigned flags,
                   cudaStream_t s, int n_steps = 1, int32_t *ids_out = nullptr) {
    const ds_model_config &c = m->cfg;
    const bool greedy = sampling == nullptr || !(sampling->temperature > 0.0f);
    const bool advance = (flags & DS_STEP_ADVANCE) != 0;
    float *logits = logits_out ? logits_out : m->logits;
    StepParams p;
    std::memset(&p, 0, sizeof p);
    p.layers = m->step_layers;
    p.n_layer = c.n_layer;
    p.emb = static_cast<const char *>(m->emb);
    p.head = static_cast<const char *>(c.tied ? m->emb : m->out);
    p.final_norm = m->final_norm;
    p.vocab = c.vocab;
    p.d = c.d;
    p.nq_cols = c.n_qh * c.head_dim;
    p.nkv_cols = c.n_kvh * c.head_dim;
    p.hd = c.head_dim;
    p.ff = c.ff;
    p.rope_layout = c.rope_layout;
    p.kv_dtype = c.kv_dtype;
    p.n_kvh = c.n_kvh;
    p.n_qh = c.n_qh;
    p.eps = c.eps;
    p.rope_cos = m->rope_cos;
    p.rope_sin = m->rope_sin;
    p.rope_rows = c.max_ctx;
    p.block_table = kv->block_table;
    p.block_tokens = kv->block_tokens;
    p.max_blocks = kv->max_blocks;
    p.tokens = tokens;
    p.pos = pos;
    p.next_ids = next_ids;
    p.logits = logits;
    p.advance = advance && greedy;
    p.greedy = greedy;
    p.xt = m->st_x;
    p.qt = m->st_q;
    p.kvt = m->st_kv;
    p.ft = m->st_f;
    p.sst = m->st_ss;
    p.n_ss = m->nb_o;
    p.pt = m->st_part;
    p.pt_stride = m->st_part_stride;
    p.at = m->st_att;
    p.am_val = m->am_val;
    p.am_idx = m->am_idx;
    p.am_counter = m->am_counter;
    p.epoch = reinterpret_cast<unsigned long long *>(m->step_bar) + 1;
    p.n_steps = n_steps;
    p.ids_out = ids_out;
    p.tokt = reinterpret_cast<unsigned long long *>(m->step_bar) + 3;
    p.err = m->err;
    p.abort_flag = m->step_abort;
    p.phase_times = (n_steps == 1 && (flags & (DS_STEP_PHASE_TIMES | DS_STEP_TRACE))) ? m->phase_times : nullptr;
    p.trace = (n_steps == 1 && (flags & DS_STEP_TRACE)) ? m->trace : nullptr;
    p.nb_qkv = m->nb_qkv;
    p.nb_o = m->nb_o;
    p.nb_gu = m->nb_gu;
    p.nb_d = m->nb_d;
    p.attn_splits = m->step_splits;
    p.stages = m->step_stages;
    p.kv_maps = m->kv_maps_dev;
    p.kv_tma = m->kv_tma_cur && m->kv_bt_enc == kv->block_tokens && m->kv_k0 == kv->k[0];
    p.kv_stage_pos = p.kv_tma ? kv_stage_positions(c, kv->block_tokens) : 0;
    p.kv_align = p.kv_tma ? std::max(8, kv->block_tokens) : 1;
    p.scratch_floats = m->step_scratch;
    p.max_inflight = m->step_inflight;
    p.chain_inflight = m->step_chain_inflight;
    p.chain_gu_stages = m->step_chain_gu;
    for (int l = 0; l < c.n_layer; ++l) {
        p.kc[l] = kv->k[l];
        p.vc[l] = kv->v[l];
    }
    if (launch_step(&p, c.w_dtype, c.kv_dtype, c.n_qh / c.n_kvh, m->step_grid, s) != cudaSuccess)
        return DS_CUDA_ERROR;
    if (!greedy) {
        SampleArgs sa = {};
        sa.logits = logits;
        sa.n_rows = n_seqs;
        sa.n = c.vocab;
        sa.temperature = sampling->temperature;
        sa.top_k = sampling->top_k;
        sa.top_p = sampling->top_p;
        sa.u = u;
        sa.ids = next_ids;
        sa.tokens_adv = advance ? tokens : nullptr;
        sa.pos_adv = advance ? pos : nullptr;
        sa.err = m->err;
        if (launch_sample(sa, s, false) != cudaSuccess) return DS_CUDA_ERROR;
    }
    return DS_OK;
}

// One batched step for n sequences ("Inside the engine", section 4: batched
// decode, one token per sequence per step).  Activations stay fp32; each
// projection input is handed to the tensor cores as a bf16 pair hi + lo.  Per
// layer RMSNorm rows ->
// q|k|v on the tensor cores (RoPE + K/V write at each sequence's position in
// the epilogue) -> split-context attention over each sequence's blocks (fp32
// and bf16 outputs) -> o on the tensor cores (+ residual) -> RMSNorm rows ->
// gate|up (SiLU-gate to bf16) -> down (+ residual); final RMSNorm rows ->
// head -> per-row greedy argmax or sampler.  Every launch may begin while its
// predecessor drains (programmatic dependent launch).
// Embed and every layer of a batched step over n rows: row r is token
// tokens[r] at position pos[r], its K/V written to and read from the blocks
// of sequence row_seq[r] (row r's own when row_seq is null).  Leaves the
// residual of every row in m->x.
int run_layers_batched(ds_model *m, const ds_kv_cache *kv, const int32_t *tokens, const int32_t *pos,
                       const int32_t *row_seq, int n, cudaStream_t s) {
    const ds_model_config &c = m->cfg;
    const bool pdl = true;
#define DS_TRYB(expr)                               \
    do {                                            \
        if ((expr) != cudaSuccess) return DS_CUDA_ERROR; \
    } while (0)
    auto gemm = [&](TcArgs a) { return launch_tc_gemm(a, tc_grid(a.m_tiles, a.K), s, pdl); };
    const long long h_lo = (long long)c.max_seqs * c.d;  // hi rows, then lo rows
    DS_TRYB(launch_embed(m->emb, c.w_dtype, c.vocab, c.d, tokens, m->x, m->err, n, s, pdl));
    for (int l = 0; l < c.n_layer; ++l) {
        // the first layer's norm runs alone; every later one is folded into
        // the projection writing the residual and the one reading it
        if (l == 0) DS_TRYB(launch_rmsnorm_rows_bf16(m->x, m->n1[l], c.eps, m->h_bf, h_lo, n, c.d, s, pdl));
        TcArgs a = m->tc[4 * l + 0];
        a.n = n;
        a.pos = pos;
        a.row_seq = row_seq;
        a.block_table = kv->block_table;
        a.max_blocks = kv->max_blocks;
        a.block_tokens = kv->block_tokens;
        a.cache_rows = kv->rows;
        a.k_cache = kv->k[l];
        a.v_cache = kv->v[l];
        DS_TRYB(gemm(a));
        if (paged_attention_supported(c.n_qh, c.n_kvh, c.head_dim, kv->block_tokens, n, c.kv_dtype)) {
            PagedAttnArgs pa = {};
            if (c.kv_dtype == DS_BF16) {
                if (m->pa_maps.empty()) {
                    m->pa_maps.resize((size_t)2 * c.n_layer);
                    m->pa_k.assign(c.n_layer, nullptr);
                    m->pa_v.assign(c.n_layer, nullptr);
                    m->pa_rows.assign(c.n_layer, -1);
                    m->pa_box3d.assign(c.n_layer, 0);
                }
                if (m->pa_k[l] != kv->k[l] || m->pa_v[l] != kv->v[l] || m->pa_rows[l] != kv->rows) {
                    PagedAttnArgs enc = {};
                    enc.k_cache = kv->k[l];
                    enc.v_cache = kv->v[l];
                    enc.n_kvh = c.n_kvh;
                    enc.cache_rows = kv->rows;
                    if (!paged_attention_maps(enc)) return DS_CUDA_ERROR;
                    m->pa_maps[2 * l] = enc.tk;
                    m->pa_maps[2 * l + 1] = enc.tv;
                    m->pa_box3d[l] = enc.box3d;
                    m->pa_k[l] = kv->k[l];
                    m->pa_v[l] = kv->v[l];
                    m->pa_rows[l] = kv->rows;
                }
                pa.tk = m->pa_maps[2 * l];
                pa.tv = m->pa_maps[2 * l + 1];
                pa.box3d = m->pa_box3d[l];
            }
            pa.q = m->q;
            pa.k_cache = kv->k[l];
            pa.v_cache = kv->v[l];
            pa.kv_dtype = c.kv_dtype;
            pa.cache_rows = kv->rows;
            pa.block_table = kv->block_table;
            pa.max_blocks = kv->max_blocks;
            pa.seq_lens = nullptr;
            pa.pos = pos;
            pa.row_seq = row_seq;
            pa.n_seqs = n;
            pa.n_qh = c.n_qh;
            pa.n_kvh = c.n_kvh;
            pa.scale = 1.0f / sqrtf((float)c.head_dim);
            pa.out = m->att;
            pa.out_bf16 = m->att_bf;
            pa.out_bf16_lo = (long long)c.max_seqs * c.n_qh * c.head_dim;
            pa.partials = m->a_partials;
            pa.counters = m->a_counters;
            pa.err = m->err;
            DS_TRYB(launch_paged_attention(pa, s, pdl));
        } else {
            AttnArgs at = {};
            at.q = m->q;
            at.k_cache = kv->k[l];
            at.v_cache = kv->v[l];
            at.kv_dtype = c.kv_dtype;
            at.cache_rows = kv->rows;
            at.block_table = kv->block_table;
            at.max_blocks = kv->max_blocks;
            at.block_tokens = kv->block_tokens;
            at.seq_lens = nullptr;
            at.pos = pos;
            at.row_seq = row_seq;
            at.n_qh = c.n_qh;
            at.n_kvh = c.n_kvh;
            at.hd = c.head_dim;
            at.scale = 1.0f / sqrtf((float)c.head_dim);
            at.out = m->att;
            at.out_bf16 = m->att_bf;
            at.out_bf16_lo = (long long)c.max_seqs * c.n_qh * c.head_dim;
            at.partials = m->a_partials;
            at.counters = m->a_counters;
            at.err = m->err;
            at.n_splits = m->b_splits;
            DS_TRYB(launch_attention(at, n, s, pdl));
        }
        a = m->tc[4 * l + 1];
        a.n = n;
        DS_TRYB(gemm(a));
        a = m->tc[4 * l + 2];
        a.n = n;
        DS_TRYB(gemm(a));
        a = m->tc[4 * l + 3];
        a.n = n;
        DS_TRYB(gemm(a));
    }
#undef DS_TRYB
    return DS_OK;
}

int run_step_batched(ds_model *m, const ds_kv_cache *kv, int32_t *tokens, int32_t *pos, int n,
                     const ds_sampling *sampling, const float *u, int32_t *next_ids, float *logits_out, unsigned flags,
                     cudaStream_t s) {
    const ds_model_config &c = m->cfg;
    const bool greedy = sampling == nullptr || !(sampling->temperature > 0.0f);
    const bool advance = (flags & DS_STEP_ADVANCE) != 0;
    float *logits = logits_out ? logits_out : m->logits;
    const bool pdl = true;
#define DS_TRYB(expr)                               \
    do {                                            \
        if ((expr) != cudaSuccess) return DS_CUDA_ERROR; \
    } while (0)
    {
        const int st = run_layers_batched(m, kv, tokens, pos, nullptr, n, s);
        if (st != DS_OK) return st;
    }
    const long long h_lo = (long long)c.max_seqs * c.d;  // hi rows, then lo rows
    auto gemm = [&](TcArgs a) { return launch_tc_gemm(a, tc_grid(a.m_tiles, a.K), s, pdl); };
    DS_TRYB(launch_rmsnorm_rows_bf16(m->x, m->final_norm, c.eps, m->h_bf, h_lo, n, c.d, s, pdl));
    TcArgs hd = m->tc[(size_t)4 * c.n_layer];
    hd.n = n;
    hd.y = logits;
    DS_TRYB(gemm(hd));
    if (greedy) {
        ArgmaxArgs am = {};
        am.logits = logits;
        am.n_rows = n;
        am.n = c.vocab;
        am.ids = next_ids;
        am.max_logit = nullptr;
        am.part_val = m->am_val;
        am.part_idx = m->am_idx;
        am.counters = m->b_am_counters;
        am.tokens_adv = advance ? tokens : nullptr;
        am.pos_adv = advance ? pos : nullptr;
        am.err = m->err;
        am.blocks_per_row = argmax_blocks_per_row(c.vocab);
        DS_TRYB(launch_argmax(am, s, pdl));
    } else {
        SampleArgs sa = {};
        sa.logits = logits;
        sa.n_rows = n;
        sa.n = c.vocab;
        sa.temperature = sampling->temperature;
        sa.top_k = sampling->top_k;
        sa.top_p = sampling->top_p;
        sa.u = u;
        sa.ids = next_ids;
        sa.tokens_adv = advance ? tokens : nullptr;
        sa.pos_adv = advance ? pos : nullptr;
        sa.err = m->err;
        DS_TRYB(launch_sample(sa, s, pdl));
    }
#undef DS_TRYB
    return DS_OK;
}

// The step for this model: the batched path, the persistent step kernel
// (batch 1) or the per-kernel launch sequence.
int dispatch_step(ds_model *m, const ds_kv_cache *kv, int32_t *tokens, int32_t *pos, int n_seqs,
                  const ds_sampling *sampling, const float *u, int32_t *next_ids, float *logits_out, unsigned flags,
                  cudaStream_t s) {
    if (m->batched) return run_step_batched(m, kv, tokens, pos, n_seqs, sampling, u, next_ids, logits_out, flags, s);
    if (m->step_ok && n_seqs == 1)
        return run_step_fused(m, kv, tokens, pos, n_seqs, sampling, u, next_ids, logits_out, flags, s);
    return run_step(m, kv, tokens, pos, n_seqs, sampling, u, next_ids, logits_out, flags, s, nullptr);
}

extern "C" DS_API int ds_decode_step(ds_model *m, const ds_kv_cache *kv, int32_t *tokens, int32_t *pos, int n_seqs,
                                     const ds_sampling *sampling, const float *u, int32_t *next_ids,
                                     float *logits_out, unsigned flags, ds_stream_t stream) {
    int st = check_step(m, kv, tokens, pos, n_seqs, sampling, u, next_ids);
    if (st != DS_OK) return st;
    st = ensure_kv_maps(m, kv, reinterpret_cast<cudaStream_t>(stream));
    if (st != DS_OK) return st;
    return dispatch_step(m, kv, tokens, pos, n_seqs, sampling, u, next_ids, logits_out, flags,
                         reinterpret_cast<cudaStream_t>(stream));
}

extern "C" DS_API int ds_decode_steps(ds_model *m, const ds_kv_cache *kv, int32_t *tokens, int32_t *pos,
                                      int n_steps, int32_t *ids_out, int32_t *next_ids, unsigned flags,
                                      ds_stream_t stream) {
    if (n_steps < 1) return DS_EMPTY_DIMENSION;
    int st = check_step(m, kv, tokens, pos, 1, nullptr, nullptr, next_ids);
    if (st != DS_OK) return st;
    if (!m->step_ok || m->batched) return DS_BAD_ARGUMENT;  // the persistent batch-1 kernel only
    st = ensure_kv_maps(m, kv, reinterpret_cast<cudaStream_t>(stream));
    if (st != DS_OK) return st;
    return run_step_fused(m, kv, tokens, pos, 1, nullptr, nullptr, next_ids, nullptr, flags & DS_STEP_ADVANCE,
                          reinterpret_cast<cudaStream_t>(stream), n_steps, ids_out);
}

extern "C" DS_API int ds_step_seq(ds_model *m, const ds_kv_cache *kv, const int32_t *tokens, int64_t tokens_len,
                                  int32_t seq, int32_t offset, int32_t count, int32_t *next_id, float *logits_out,
                                  ds_stream_t stream) {
    if (!m) return DS_BAD_ARGUMENT;
    if (count < 1) return DS_EMPTY_DIMENSION;
    if (tokens_len != count) return DS_A_LENGTH_MISMATCH;
    if (!tokens || !next_id) return DS_BAD_ARGUMENT;
    if (!m->batched) return DS_BAD_ARGUMENT;  // chunks are batches of rows: the tensor-core path
    int st = check_kv(m, kv);
    if (st != DS_OK) return st;
    const ds_model_config &c = m->cfg;
    if (seq < 0 || seq >= c.max_seqs) return DS_BAD_ARGUMENT;
    const int64_t cap = std::min<int64_t>((int64_t)kv->block_tokens * kv->max_blocks, c.max_ctx);
    if (offset < 0 || (int64_t)offset + count > cap) return DS_CACHE_CAPACITY_EXCEEDED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int S = c.max_seqs;
    int last = 0;  // rows of the last chunk
    for (int c0 = 0; c0 < count; c0 += S) {
        const int nc = std::min(S, count - c0);
        // the chunk's positions and sequence, written after everything
        // before it on the stream has finished reading the last chunk's
        if (launch_chunk_rows(m->seq_rows, m->seq_rows + S, offset + c0, seq, nc, s) != cudaSuccess)
            return DS_CUDA_ERROR;
        st = run_layers_batched(m, kv, tokens + c0, m->seq_rows, m->seq_rows + S, nc, s);
        if (st != DS_OK) return st;
        last = nc;
    }
    // the last token only: final norm, head, greedy pick
    float *logits = logits_out ? logits_out : m->logits;
    const long long h_lo = (long long)S * c.d;
    if (launch_rmsnorm_rows_bf16(m->x + (long long)(last - 1) * c.d, m->final_norm, c.eps, m->h_bf, h_lo, 1, c.d, s,
                                 true) != cudaSuccess)
        return DS_CUDA_ERROR;
    TcArgs hd = m->tc[(size_t)4 * c.n_layer];
    hd.n = 1;
    hd.y = logits;
    if (launch_tc_gemm(hd, tc_grid(hd.m_tiles, hd.K), s, true) != cudaSuccess) return DS_CUDA_ERROR;
    ArgmaxArgs am = {};
    am.logits = logits;
    am.n_rows = 1;
    am.n = c.vocab;
    am.ids = next_id;
    am.part_val = m->am_val;
    am.part_idx = m->am_idx;
    am.counters = m->b_am_counters;
    am.err = m->err;
    am.blocks_per_row = argmax_blocks_per_row(c.vocab);
    if (launch_argmax(am, s, true) != cudaSuccess) return DS_CUDA_ERROR;
    return DS_OK;
}

extern "C" DS_API int ds_model_phase_times(ds_model *m, uint64_t *ns_out, int cap, int *n_out, ds_stream_t stream) {
    if (!m || !ns_out || !n_out || cap < 1) return DS_BAD_ARGUMENT;
    const int n = std::min(cap, m->n_phase_times);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(ns_out, m->phase_times, (size_t)n * 8, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return DS_CUDA_ERROR;
    *n_out = n;
    return DS_OK;
}

extern "C" DS_API int ds_step_graph_create(ds_model *m, const ds_kv_cache *kv, int32_t *tokens, int32_t *pos,
                                           int n_seqs, const ds_sampling *sampling, const float *u,
                                           int32_t *next_ids, float *logits_out, unsigned flags, ds_stream_t stream,
                                           ds_step_graph **out) {
    if (!out) return DS_BAD_ARGUMENT;
    *out = nullptr;
    int st = check_step(m, kv, tokens, pos, n_seqs, sampling, u, next_ids);
    if (st != DS_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (!s) return DS_BAD_ARGUMENT;  // the legacy stream cannot be captured
    st = ensure_kv_maps(m, kv, s);  // uploads, if any, happen outside the capture
    if (st != DS_OK) return st;
    if (cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal) != cudaSuccess) return DS_CUDA_ERROR;
    st = dispatch_step(m, kv, tokens, pos, n_seqs, sampling, u, next_ids, logits_out, flags, s);
    cudaGraph_t graph = nullptr;
    cudaError_t e = cudaStreamEndCapture(s, &graph);
    if (st != DS_OK || e != cudaSuccess) {
        if (graph) cudaGraphDestroy(graph);
        cudaGetLastError();
        return st != DS_OK ? st : DS_CUDA_ERROR;
    }
    cudaGraphExec_t exec = nullptr;
    if (cudaGraphInstantiate(&exec, graph, 0) != cudaSuccess) {
        cudaGraphDestroy(graph);
        return DS_CUDA_ERROR;
    }
    ds_step_graph *g = new (std::nothrow) ds_step_graph();
    if (!g) {
        cudaGraphExecDestroy(exec);
        cudaGraphDestroy(graph);
        return DS_BAD_ARGUMENT;
    }
    g->graph = graph;
    g->exec = exec;
    *out = g;
    return DS_OK;
}

extern "C" DS_API int ds_step_graph_launch(ds_step_graph *g, ds_stream_t stream) {
    if (!g) return DS_BAD_ARGUMENT;
    return cudaGraphLaunch(g->exec, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? DS_OK : DS_CUDA_ERROR;
}

extern "C" DS_API void ds_step_graph_destroy(ds_step_graph *g) {
    if (!g) return;
    cudaGraphExecDestroy(g->exec);
    cudaGraphDestroy(g->graph);
    delete g;
}

extern "C" DS_API int ds_decode_step_profile(ds_model *m, const ds_kv_cache *kv, int32_t *tokens, int32_t *pos,
                                             int n_seqs, const ds_sampling *sampling, const float *u,
                                             int32_t *next_ids, float *logits_out, unsigned flags, int reps,
                                             float *ms_out, int32_t *kinds_out, int cap, int *n_out,
                                             ds_stream_t stream) {
    if (reps < 1 || !ms_out || !kinds_out || !n_out || cap < 1) return DS_BAD_ARGUMENT;
    if (m && m->batched) return DS_BAD_ARGUMENT;  // per-kernel timing covers the batch-1 launch sequence
    int st = check_step(m, kv, tokens, pos, n_seqs, sampling, u, next_ids);
    if (st != DS_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    Recorder rec;
    rec.stream = s;
    std::vector<double> sum;
    int slots = 0;
    for (int r = 0; r < reps; ++r) {
        rec.used = 0;
        st = run_step(m, kv, tokens, pos, n_seqs, sampling, u, next_ids, logits_out, flags, s, &rec);
        if (st != DS_OK) return st;
        if (cudaStreamSynchronize(s) != cudaSuccess) return DS_CUDA_ERROR;
        slots = (int)rec.used - 1;
        if (sum.empty()) sum.assign(slots, 0.0);
        for (int i = 0; i < slots; ++i) {
            float ms = 0.0f;
            if (cudaEventElapsedTime(&ms, rec.ev[i], rec.ev[i + 1]) != cudaSuccess) return DS_CUDA_ERROR;
            sum[i] += ms;
        }
    }
    const int n = std::min(cap, slots);
    for (int i = 0; i < n; ++i) {
        ms_out[i] = (float)(sum[i] / reps);
        kinds_out[i] = rec.kind[i + 1];
    }
    *n_out = n;
    return DS_OK;
}

extern "C" DS_API int ds_decode_kernel_time(ds_model *m, const ds_kv_cache *kv, int32_t *tokens, int32_t *pos,
                                            int kind, int reps, float *us_per_launch, ds_stream_t stream) {
    if (reps < 1 || !us_per_launch || kind < 0 || kind >= DS_KIND_COUNT || kind == DS_KIND_SAMPLE)
        return DS_BAD_ARGUMENT;
    if (m && m->batched) return DS_BAD_ARGUMENT;
    int st = check_step(m, kv, tokens, pos, 1, nullptr, nullptr, m ? m->am_idx : nullptr);
    if (st != DS_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // next ids go to a scratch word of the workspace, so the caller's state
    // is not advanced
    int32_t *scratch_ids = reinterpret_cast<int32_t *>(m->ws) + 1;
    cudaEvent_t e0, e1;
    if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) return DS_CUDA_ERROR;
    st = run_step(m, kv, tokens, pos, 1, nullptr, nullptr, scratch_ids, nullptr, 0, s, nullptr, kind);  // warm
    if (st == DS_OK && cudaEventRecord(e0, s) != cudaSuccess) st = DS_CUDA_ERROR;
    for (int r = 0; r < reps && st == DS_OK; ++r)
        st = run_step(m, kv, tokens, pos, 1, nullptr, nullptr, scratch_ids, nullptr, 0, s, nullptr, kind);
    float ms = 0.0f;
    if (st == DS_OK && (cudaEventRecord(e1, s) != cudaSuccess || cudaEventSynchronize(e1) != cudaSuccess ||
                        cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess))
        st = DS_CUDA_ERROR;
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    if (st != DS_OK) return st;
    const int per_step = (kind == DS_KIND_EMBED || kind == DS_KIND_HEAD) ? 1 : m->cfg.n_layer;
    *us_per_launch = 1000.0f * ms / (float)(reps * std::max(per_step, 1));
    return DS_OK;
}

extern "C" DS_API int ds_model_trace(ds_model *m, uint64_t *out, size_t cap_words, size_t *n_words, int *n_ctas,
                                     ds_stream_t stream) {
    if (!m || !out || !n_words || !n_ctas) return DS_BAD_ARGUMENT;
    const size_t n = std::min(cap_words, m->trace_words);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(out, m->trace, n * 8, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return DS_CUDA_ERROR;
    *n_words = n;
    *n_ctas = m->step_grid;
    return DS_OK;
}
