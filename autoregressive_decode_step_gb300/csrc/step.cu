// The whole batch-1 decode step as one persistent kernel.
//
// One CTA per SM (cooperative launch), eight consumer warps and one producer
// warp.  The step is a fixed sequence of phases ("The forward pass end to
// end", "What a forward step does"; "Inside the engine", section 1):
//   embed | per layer: q|k|v (RMSNorm prologue, RoPE + K/V write epilogue) |
//   attention | o (+ residual) | gate|up (RMSNorm prologue, SiLU epilogue) |
//   down (+ residual) | final RMSNorm + output head + greedy argmax.
// Activations pass between phases as tagged 64-bit words (value + the phase
// sequence number) that readers poll, so a CTA starts a phase as soon as the
// slice of the previous phase's output it needs has arrived; there is no grid
// barrier.  The producer warp never waits for activations: weights do not
// depend on them, so it streams the next phase's weight boxes into the
// shared-memory ring while consumers finish a phase, wait for their inputs
// or run attention.  The weight stream therefore runs across phase
// boundaries without the drain and refill a kernel launch per phase would
// cost.
//
// Arithmetic per phase is the same as the standalone kernels': stream-K
// ranges of 16-row x 512-byte tensor-map boxes for the transposed projections,
// fixed-order cross-CTA reductions by the CTA holding each band's last box,
// whole-row bulk copies for the head.  Activations written by other CTAs are
// read through L2 (ld.global.cg) so no stale L1 line is ever used.  Every wait is
// bounded: a tagged-word poll or mbarrier wait that times out sets the error
// word and an abort flag, after which the remaining phases run without
// waiting.
#include <algorithm>
#include <climits>
#include <cstdio>
#include <cstdlib>
#include <cstring>

#include "common.cuh"
#include "internal.h"

namespace ds {

constexpr int kStConsumerWarps = 8;
constexpr int kStConsumers = kStConsumerWarps * 32;
constexpr int kStThreads = kStConsumers + 32;
#ifndef DS_ST_STAGE_BYTES
#define DS_ST_STAGE_BYTES 65536
#endif
constexpr int kStStageBytes = DS_ST_STAGE_BYTES;
constexpr int kStMaxStages = 16;
#ifndef DS_ST_BOX_ROWS
#define DS_ST_BOX_ROWS 16
#endif
constexpr int kStBoxRows = DS_ST_BOX_ROWS;
constexpr int kStBandBytes = 512;
#ifndef DS_ST_ATTN_MIN_PER
#define DS_ST_ATTN_MIN_PER 64
#endif
constexpr int kStAttnMinPer = DS_ST_ATTN_MIN_PER;  // fewest positions per attention split
// split records an attention merge requests at once (all of a head's splits
// in one batch up to this count)
constexpr int kStMergeBatch = 20;
constexpr int kStBoxesPerStage = kStStageBytes / (kStBoxRows * kStBandBytes);  // 8 boxes of 16 rows at 64 KB
constexpr size_t kStSmemLimit = 227 * 1024;
#ifndef DS_ST_MAX_INFLIGHT
#define DS_ST_MAX_INFLIGHT 0
#endif
constexpr int kStMaxInflight = DS_ST_MAX_INFLIGHT;  // weight stages requested and not landed (0: no cap)
#ifndef DS_ST_CHAIN_INFLIGHT
#define DS_ST_CHAIN_INFLIGHT 1
#endif
#ifndef DS_ST_CHAIN_GU_STAGES
#define DS_ST_CHAIN_GU_STAGES 3
#endif
constexpr int kStChainInflight = DS_ST_CHAIN_INFLIGHT;  // the cap during the attention chain (0: the plain cap)
constexpr int kStChainGuStages = DS_ST_CHAIN_GU_STAGES;  // first gate|up stages counted as chain stages

__device__ __forceinline__ float ldcg(const float *p) { return __ldcg(p); }

__device__ __forceinline__ bool aborted(const StepParams &p) {
    return *reinterpret_cast<volatile int *>(p.abort_flag) != 0;
}

__device__ __forceinline__ void raise_abort(const StepParams &p, int bit) {
    flag_error(p.err, bit);
    atomicExch(p.abort_flag, 1);
}

// Bounded mbarrier wait that also gives up once the step is aborted.
__device__ __forceinline__ bool st_wait(uint64_t *bar, uint32_t parity, const StepParams &p) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 0) {
            if (aborted(p)) return false;
            if (global_timer_ns() - t0 > kWaitLimitNs) {
                raise_abort(p, DS_ERR_WAIT_TIMEOUT);
                return false;
            }
        }
    }
}

__device__ __forceinline__ void mark_phase(const StepParams &p, int &phase) {
    if (p.phase_times && blockIdx.x == 0 && threadIdx.x == 0) p.phase_times[phase] = global_timer_ns();
    ++phase;
}

// Per-CTA trace point k (0 phase start, 1 prologue done, 2 last stage
// consumed, 3 epilogue done; 4 is the producer's last issue of the phase).
__device__ __forceinline__ void trace_point(const StepParams &p, int phase, int k) {
    if (p.trace && (threadIdx.x == 0 || k == 4))
        p.trace[((size_t)phase * gridDim.x + blockIdx.x) * 5 + k] = global_timer_ns();
}

// ---------------------------------------------------------------- producer
struct Ring {
    unsigned char *base;
    uint64_t *full, *empty;
    int stages;
};

// Wait until ring slot `fill` is free, announce `bytes` on its full barrier;
// returns the slot's shared-memory address or nullptr once aborted.
__device__ __forceinline__ unsigned char *ring_acquire(const Ring &r, uint32_t fill, uint32_t bytes,
                                                       const StepParams &p) {
    const int s = fill % r.stages;
    const uint32_t use = fill / r.stages;
    if (use > 0 && !st_wait(&r.empty[s], (use - 1) & 1, p)) return nullptr;
    mbar_arrive_expect_tx(&r.full[s], bytes);
    return r.base + (size_t)s * kStStageBytes;
}

// Cursor over every weight stage this CTA streams in a step, in order: per
// layer the q|k|v, o, gate|up and down boxes of this CTA's range, then its
// rows of the head.
struct StageCursor {
    int l, ph;  // layer and phase (0 q|k|v, 4 cached K/V, 1 o, 2 gate|up, 3 down); l == n_layer: head
    const CUtensorMap *m0, *m1;
    int UB, sub_band_cols;
    uint32_t box_bytes;
    long long u, u1;
    int band, j, j1;
    int rr, r1, rps;
    long long row_bytes;
    bool done;
    int n_ctx;        // positions the step attends (its own included)
    int kv_t, kv_tc;  // K/V phase: the next cached position to stream, and the end
};

struct StageDesc {
    bool head, kv;
    const CUtensorMap *m0, *m1;
    int col, row0, nb;
    uint32_t box_bytes, bytes;
    const char *src;
    int kv_t, layer;
};

// Positions per attention split and the number of splits in use for a step
// attending n_ctx positions: at least kStAttnMinPer per split, rounded up to
// whole cache blocks when the cached K/V streams through the ring.
// Does this step stream its cached K/V through the ring?  Only when a split
// holds at least one full stage of positions: shorter splits are served
// sooner from L2 (prefetched during the q|k|v phase) than from a ring slot
// queued behind the q|k|v weights.  The producer and the consumers decide
// alike, from the same position.
__device__ __forceinline__ bool kv_streamed(int n_ctx, const StepParams &p) {
    return p.kv_tma && (n_ctx + p.attn_splits - 1) / p.attn_splits >= p.kv_stage_pos;
}

// Positions per attention split and the number of splits in use for a step
// attending n_ctx positions: at least kStAttnMinPer per split, rounded up to
// whole cache blocks when the cached K/V streams through the ring.
__device__ __forceinline__ void attention_split_n(int n_ctx, const StepParams &p, int &per, int &n_eff) {
    per = max(kStAttnMinPer, (n_ctx + p.attn_splits - 1) / p.attn_splits);
    if (kv_streamed(n_ctx, p)) per = (per + p.kv_align - 1) / p.kv_align * p.kv_align;
    n_eff = (n_ctx + per - 1) / per;
}

// The phase after `ph` in a layer's order q|k|v, [K/V], o, gate|up, down.
__device__ __forceinline__ int next_ph(int ph, int n_ctx, const StepParams &p) {
    if (ph == 0) return kv_streamed(n_ctx, p) ? 4 : 1;
    if (ph == 4) return 1;
    return ph + 1;  // 1 -> 2 -> 3 -> 4 means "next layer" (handled by the caller)
}

template <int ES>
__device__ void cursor_phase(StageCursor &c, const StepParams &p) {
    constexpr int BAND_COLS = kStBandBytes / ES;
    const int G0 = gridDim.x;
    for (;;) {
        if (c.l >= p.n_layer) {
            const long long rows = p.vocab;
            c.row_bytes = (long long)p.d * ES;
            c.rps = (int)max(1LL, (long long)kStStageBytes / c.row_bytes);
            c.rr = (int)(rows * blockIdx.x / G0);
            c.r1 = (int)(rows * (blockIdx.x + 1) / G0);
            c.done = c.rr >= c.r1;
            return;
        }
        if (c.ph == 4) {  // this CTA's cached K/V positions, if it has an attention item
            const int n_items = p.n_kvh * p.attn_splits;
            c.kv_t = c.kv_tc = 0;
            if ((int)blockIdx.x < n_items) {
                const int split = blockIdx.x % p.attn_splits;
                int per, n_eff;
                attention_split_n(c.n_ctx, p, per, n_eff);
                const int t0 = min(c.n_ctx, split * per), t1 = min(c.n_ctx, t0 + per);
                c.kv_t = t0;
                c.kv_tc = min(t1, c.n_ctx - 1);
            }
            if (c.kv_t < c.kv_tc) return;
            c.ph = 1;  // nothing cached to stream here
            continue;
        }
        const StepLayer &L = p.layers[c.l];
        int K, nb;
        c.m1 = nullptr;
        if (c.ph == 0) { c.m0 = &L.maps[0]; K = p.d; nb = p.nb_qkv; }
        else if (c.ph == 1) { c.m0 = &L.maps[1]; K = p.nq_cols; nb = p.nb_o; }
        else if (c.ph == 2) { c.m0 = &L.maps[2]; c.m1 = &L.maps[3]; K = p.d; nb = p.nb_gu; }
        else { c.m0 = &L.maps[4]; K = p.ff; nb = p.nb_d; }
        c.sub_band_cols = c.m1 ? BAND_COLS / 2 : BAND_COLS;
        c.box_bytes = kStBoxRows * c.sub_band_cols * ES;
        c.UB = (K + kStBoxRows - 1) / kStBoxRows;
        const long long W = (long long)nb * c.UB;
        const int G = (int)min((long long)G0, W);
        const bool in = (int)blockIdx.x < G;
        c.u = in ? W * blockIdx.x / G : 0;
        c.u1 = in ? W * (blockIdx.x + 1) / G : 0;
        if (c.u < c.u1) {
            c.band = (int)(c.u / c.UB);
            c.j = (int)(c.u - (long long)c.band * c.UB);
            c.j1 = (int)min((long long)c.UB, c.j + (c.u1 - c.u));
            return;
        }
        // nothing for this CTA here
        if (c.ph == 3) {
            c.ph = 0;
            ++c.l;
        } else {
            c.ph = next_ph(c.ph, c.n_ctx, p);
        }
    }
}

template <int ES>
__device__ void cursor_begin(StageCursor &c, const StepParams &p) {
    c.l = 0;
    c.ph = 0;
    c.done = false;
    cursor_phase<ES>(c, p);
}

template <int ES>
__device__ bool cursor_desc(const StageCursor &c, const StepParams &p, StageDesc &d) {
    if (c.done) return false;
    if (c.l >= p.n_layer) {
        const int nr = min(c.rps, c.r1 - c.rr);
        d.head = true;
        d.src = p.head + (long long)c.rr * c.row_bytes;
        d.bytes = (uint32_t)(nr * c.row_bytes);
        return true;
    }
    d.head = false;
    d.kv = c.ph == 4;
    if (d.kv) {
        const int P = p.kv_stage_pos, bt = p.block_tokens;
        const int t_end = min(c.kv_t + P, c.kv_tc);
        d.kv_t = c.kv_t;
        d.layer = c.l;
        d.nb = (t_end - c.kv_t + bt - 1) / bt;  // whole blocks (kv_t is block-aligned)
        d.box_bytes = (uint32_t)(bt * p.hd * (p.kv_dtype == DS_BF16 ? 2 : 4));
        d.bytes = 2u * (uint32_t)d.nb * d.box_bytes;
        return true;
    }
    d.m0 = c.m0;
    d.m1 = c.m1;
    d.col = c.band * c.sub_band_cols;
    d.row0 = c.j * kStBoxRows;
    d.nb = min(kStBoxesPerStage, c.j1 - c.j);
    d.box_bytes = c.box_bytes;
    d.bytes = (uint32_t)d.nb * c.box_bytes * (c.m1 ? 2 : 1);
    return true;
}

template <int ES>
__device__ void cursor_advance(StageCursor &c, const StepParams &p) {
    if (c.done) return;
    if (c.l >= p.n_layer) {
        c.rr += c.rps;
        c.done = c.rr >= c.r1;
        return;
    }
    if (c.ph == 4) {
        c.kv_t += p.kv_stage_pos;
        if (c.kv_t < c.kv_tc) return;
        c.ph = 1;
        cursor_phase<ES>(c, p);
        return;
    }
    const int nb = min(kStBoxesPerStage, c.j1 - c.j);
    c.j += nb;
    c.u += nb;
    if (c.j < c.j1) return;
    if (c.u < c.u1) {  // next segment (band) of this phase
        c.band = (int)(c.u / c.UB);
        c.j = (int)(c.u - (long long)c.band * c.UB);
        c.j1 = (int)min((long long)c.UB, c.j + (c.u1 - c.u));
        return;
    }
    if (c.ph == 3) {
        c.ph = 0;
        ++c.l;
    } else {
        c.ph = next_ph(c.ph, c.n_ctx, p);
    }
    cursor_phase<ES>(c, p);
}

// Issue the copies of one stage into ring slot `s`.
__device__ __forceinline__ void issue_stage(const StageDesc &d, unsigned char *dst, uint64_t *bar, uint64_t pol,
                                            const StepParams &p) {
    if (d.head) {
        bulk_g2s(dst, d.src, d.bytes, bar, pol);
        return;
    }
    if (d.kv) {  // whole blocks of this CTA's KV head: K rows, then (kv_stage_pos rows further) V rows
        const int bt = p.block_tokens;
        const int g = blockIdx.x / p.attn_splits;
        const CUtensorMap *mk = p.kv_maps + 2 * d.layer, *mv = mk + 1;
        const int x = g * p.hd;
        const int row_bytes = (int)d.box_bytes / bt;
        for (int i = 0; i < d.nb; ++i) {
            const int b = (d.kv_t + i * bt) / bt;
            const int blk = p.block_table ? __ldg(p.block_table + b) : b;
            tma_box_g2s(dst + i * d.box_bytes, mk, x, blk * bt, bar, pol);
            tma_box_g2s(dst + (size_t)p.kv_stage_pos * row_bytes + i * d.box_bytes, mv, x, blk * bt, bar, pol);
        }
        return;
    }
    for (int b = 0; b < d.nb; ++b) {
        tma_box_g2s(dst + b * d.box_bytes, d.m0, d.col, d.row0 + b * kStBoxRows, bar, pol);
        if (d.m1) tma_box_g2s(dst + kStStageBytes / 2 + b * d.box_bytes, d.m1, d.col, d.row0 + b * kStBoxRows, bar, pol);
    }
}

// The producer: every weight stage of the step, in order, through the ring.
// At most p.max_inflight stages are requested and not yet landed at any time
// (0: every free slot is requested at once): the ring still buffers
// p.stages landed stages for consumers that are busy elsewhere, but fewer
// bytes queue in the memory system ahead of the phase hand-offs' polls.
template <int ES>
__device__ void produce_all(const Ring &r, const StepParams &p) {
    const uint64_t pol = policy_evict_first();
    uint32_t fill = 0;
    bool ok = true;
    const int pos0 = __ldcg(p.pos);
    const int cap = p.max_blocks * p.block_tokens;
    const uint32_t inflight = p.max_inflight > 0 && p.max_inflight < r.stages ? (uint32_t)p.max_inflight : 0u;
    // stages requested while the consumers run the attention chain (the o
    // projection's and cached K/V stages, and the first p.chain_gu_stages of
    // gate|up): fewer bytes in flight there keep the hand-off polls fast, and
    // the ring fills before the chain ends either way
    const uint32_t inflight_chain =
        p.chain_inflight > 0 && p.chain_inflight < r.stages ? (uint32_t)p.chain_inflight : inflight;
    for (int step = 0; step < p.n_steps && ok; ++step) {  // weights do not depend on the token
        StageCursor fc;
        fc.n_ctx = min(max(pos0 + step + 1, 1), cap);
        cursor_begin<ES>(fc, p);
        StageDesc d;
        int cur_ph = -1, ph_stage = 0;
        while (cursor_desc<ES>(fc, p, d)) {
            const int s = fill % r.stages;
            const uint32_t use = fill / r.stages;
            if (use > 0 && !st_wait(&r.empty[s], (use - 1) & 1, p)) {
                ok = false;
                break;
            }
            const int ph_now = d.head ? 5 : fc.ph;
            ph_stage = ph_now == cur_ph ? ph_stage + 1 : 0;
            cur_ph = ph_now;
            const bool chain = ph_now == 1 || ph_now == 4 || (ph_now == 2 && ph_stage < p.chain_gu_stages);
            const uint32_t cap_now = chain ? inflight_chain : inflight;
            if (cap_now && fill >= cap_now) {  // stage fill - cap has landed (its slot is not yet reused)
                const uint32_t f = fill - cap_now;
                if (!st_wait(&r.full[f % r.stages], (f / r.stages) & 1, p)) {
                    ok = false;
                    break;
                }
            }
            mbar_arrive_expect_tx(&r.full[s], d.bytes);
            issue_stage(d, r.base + (size_t)s * kStStageBytes, &r.full[s], pol, p);
            cursor_advance<ES>(fc, p);
            ++fill;
        }
    }
    const uint32_t first = fill > (uint32_t)r.stages ? fill - r.stages : 0;
    for (uint32_t f = first; f < fill; ++f)
        if (!st_wait(&r.full[f % r.stages], (f / r.stages) & 1, p)) break;
}

// ---------------------------------------------------------------- tagged words
// Every activation one CTA hands to another within a step travels as one
// 64-bit word: the fp32 value in the low half and, in the high half, the
// sequence number of the phase that wrote it.  A reader polls the word until
// the tag it expects appears, so readiness arrives with the data: no flag, no
// fence, no counter and no grid barrier between phases.  Tags are
// seq(id) = (epoch mod 2^22) * 1024 + id + 1 for phase id `id` of the launch
// numbered `epoch`.  Every tagged word is rewritten in every launch, so a
// stale word carries an earlier phase's tag or the previous launch's, never
// the one its reader waits for.
using u64 = unsigned long long;

struct Seq {
    uint32_t base;
    __device__ __forceinline__ uint32_t operator()(int id) const { return base + (uint32_t)id + 1u; }
};
// phase ids: 0 embed; layer l: 1+5l q|k|v, 2+5l attention, 3+5l o, 4+5l gate|up,
// 5+5l down; 1+5L the head.  The residual layer l reads was written by phase 5l.
__device__ __forceinline__ int ph_qkv(int l) { return 1 + 5 * l; }

__device__ __forceinline__ u64 tag_pack(float v, uint32_t tag) {
    return ((u64)tag << 32) | (u64)__float_as_uint(v);
}
__device__ __forceinline__ void st_tag(u64 *a, float v, uint32_t tag) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(a), "l"(tag_pack(v, tag)) : "memory");
}
__device__ __forceinline__ u64 ld_tag(const u64 *a) {
    u64 v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(a) : "memory");
    return v;
}
// Poll `a` until it carries `tag` (bounded; gives up once the step is aborted).
__device__ __forceinline__ u64 tag_wait_slow(const u64 *a, uint32_t tag, const StepParams &p) {
    if (aborted(p)) return 0;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        const u64 v = ld_tag(a);
        if ((uint32_t)(v >> 32) == tag) return v;
        if ((it & 31u) == 0) {
            if (aborted(p)) return 0;
            if (global_timer_ns() - t0 > kWaitLimitNs) {
                raise_abort(p, DS_ERR_WAIT_TIMEOUT);
                return 0;
            }
        }
    }
}
// The value of word `v` already loaded from `a`, polling if it lacked `tag`.
__device__ __forceinline__ float tag_value(u64 v, const u64 *a, uint32_t tag, const StepParams &p) {
    if ((uint32_t)(v >> 32) != tag) v = tag_wait_slow(a, tag, p);
    return __uint_as_float((uint32_t)v);
}
__device__ __forceinline__ float ld_wait(const u64 *a, uint32_t tag, const StepParams &p) {
    return tag_value(ld_tag(a), a, tag, p);
}
// Words w[i] loaded from a[i] (a[i] == nullptr: unused slot): until every
// one carries `tag`, reload all the stale ones together, so a batch that
// arrived late costs one L2 round trip per poll, not one per word.  Gives up
// (stale words read as 0) once the step is aborted or the wait limit passes.
template <int N>
__device__ __forceinline__ void tag_fix_at(u64 (&w)[N], const u64 *const (&a)[N], uint32_t tag,
                                           const StepParams &p) {
    auto stale = [&]() {
        bool st = false;
#pragma unroll
        for (int i = 0; i < N; ++i) st = st || (a[i] && (uint32_t)(w[i] >> 32) != tag);
        return st;
    };
    if (!stale()) return;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
#pragma unroll
        for (int i = 0; i < N; ++i)
            if (a[i] && (uint32_t)(w[i] >> 32) != tag) w[i] = ld_tag(a[i]);
        if (!stale()) return;
        if ((it & 15u) == 0 && (aborted(p) || global_timer_ns() - t0 > kWaitLimitNs)) {
            if (!aborted(p)) raise_abort(p, DS_ERR_WAIT_TIMEOUT);
#pragma unroll
            for (int i = 0; i < N; ++i)
                if (a[i] && (uint32_t)(w[i] >> 32) != tag) w[i] = 0;
            return;
        }
    }
}
// The same for words w[0..n) loaded from base[i * stride].
template <int N>
__device__ __forceinline__ void tag_fix(u64 (&w)[N], const u64 *base, size_t stride, int n, uint32_t tag,
                                        const StepParams &p) {
    bool ok = true;
#pragma unroll
    for (int i = 0; i < N; ++i)
        if (i < n) ok = ok && (uint32_t)(w[i] >> 32) == tag;
    if (ok) return;
    const u64 *a[N];
#pragma unroll
    for (int i = 0; i < N; ++i) a[i] = i < n ? base + (size_t)i * stride : nullptr;
    tag_fix_at<N>(w, a, tag, p);
}
__device__ __forceinline__ float tag_f(u64 w) { return __uint_as_float((uint32_t)w); }

// Values of the launch every consumer thread keeps: the position and the tag base.
struct StepCtx {
    Seq seq;
    int pos;     // the position this step writes and attends up to
    bool pos_ok;
    int n_ctx;   // positions attended: pos + 1, clamped to the cache
};

// ---------------------------------------------------------------- consumers
__device__ __forceinline__ float silu_st(float z) { return z / (1.0f + expf(-z)); }

// The first square-sum word thread t < 32 adds in scale_from_sst, loaded
// ahead of time (0 for the other threads).
__device__ __forceinline__ u64 sst_first(const StepParams &p) {
    return threadIdx.x < 32 && (int)threadIdx.x < p.n_ss ? ld_tag(p.sst + threadIdx.x) : 0ull;
}

// RMS scale 1/sqrt(mean(r^2) + eps) of the residual whose per-band square sums
// (tagged `tag`) are p.sst[0..n_ss), summed in lane order then across lanes;
// `first` is thread t's word p.sst[t] as sst_first loaded it.
__device__ float scale_from_sst(const StepParams &p, int n, uint32_t tag, float *red, u64 first) {
    const int t = threadIdx.x;
    if (t < 32) {
        float v = 0.0f;
        if (t < p.n_ss) v += tag_value(first, p.sst + t, tag, p);
        for (int b = t + 32; b < p.n_ss; b += 32) v += ld_wait(p.sst + b, tag, p);
        v = warp_sum(v);
        if (t == 0) red[0] = v;
    }
    named_sync(1, kStConsumers);
    const float tot = red[0];
    named_sync(1, kStConsumers);
    return 1.0f / sqrtf(tot / (float)n + p.eps);
}

// Sum of squares of v over the 256 consumer threads (t >= count adds 0).
__device__ float block_sumsq(float v, float *red) {
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    float s2 = warp_sum(v * v);
    if (lane == 0) red[warp] = s2;
    named_sync(1, kStConsumers);
    float tot = 0.0f;
    for (int w = 0; w < kStConsumerWarps; ++w) tot += red[w];
    named_sync(1, kStConsumers);
    return tot;
}

// QK-norm of one band of the q|k|v output (Qwen3's per-head RMSNorm before
// RoPE): v[t] holds column col0 + t (t < band_cols, heads of hd columns
// aligned to the band); every q head is scaled by 1/sqrt(mean of its squares
// + eps) and by qn, every k head by its own scale and kn, v columns are left
// alone.  hsum: 8 floats of shared scratch.  All consumer threads call it.
__device__ void qk_norm_band(float *v, float *hsum, int col0, int band_cols, const float *qn, const float *kn,
                             int nq_cols, int nkv_cols, int hd, float eps) {
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int col = col0 + t;
    const bool normed = t < band_cols && col < nq_cols + nkv_cols;
    const float x = normed ? v[t] : 0.0f;
    float s2 = x * x;
    if (hd >= 32) {  // a head spans hd / 32 whole warps
        s2 = warp_sum(s2);
        if (lane == 0) hsum[warp] = s2;
        named_sync(1, kStConsumers);
        const int w0 = (t / hd) * (hd >> 5);
        s2 = 0.0f;
        for (int w = w0; w < w0 + (hd >> 5); ++w) s2 += hsum[w];
    } else {  // a head is an aligned group of hd lanes
        for (int o = hd >> 1; o > 0; o >>= 1) s2 += __shfl_xor_sync(0xffffffffu, s2, o);
    }
    if (normed) {
        const bool is_q = col < nq_cols;
        const int i = (is_q ? col : col - nq_cols) % hd;
        v[t] = x * (1.0f / sqrtf(s2 / (float)hd + eps)) * __ldg((is_q ? qn : kn) + i);
    }
    named_sync(1, kStConsumers);
}

enum { ST_STORE = 0, ST_ADD = 1, ST_SILU = 2, ST_QKV = 3 };
enum { SRC_PLAIN = 0, SRC_NORM = 1, SRC_ATTN = 2 };

template <int GQ>
__device__ void stage_attention_rows(int k0, int k1, float *xs, float *red, uint32_t tag, const StepCtx &cx,
                                     const StepParams &p);

// One transposed projection phase (id `pid`): this CTA's stream-K range of
// boxes from the ring, the cross-CTA reduction and the fused epilogue.
//  - The input slice this range needs is polled from the tagged input (or
//    merged from the attention splits) and kept in shared memory; an
//    RMSNorm's weight is applied there and its 1/rms scale, a scalar, in the
//    epilogue, so a phase never waits for the whole previous output.
//  - A band this CTA covers whole is finished as soon as it is streamed.  A
//    band shared by several CTAs is settled by the CTA holding its last box:
//    the others store their column sums as tagged partials and move on; the
//    settler, after its own range, polls those partials, adds them in CTA
//    order with its own, and runs the epilogue.
template <typename T, int EPI, int SRC, int GQ>
__device__ void consume_gt(const Ring &r, uint32_t &fill, int K, int sub_cols, int n_bands, const u64 *xin,
                           uint32_t in_tag, const float *norm_w, u64 *y, uint32_t yold_tag, int layer, int pid,
                           const StepCtx &cx, float *scratch, const StepParams &p, int phase) {
    constexpr bool NORM = SRC == SRC_NORM;
    constexpr int ES = sizeof(T);
    constexpr int LE = 16 / ES;
    constexpr int BAND_COLS = kStBandBytes / ES;
    constexpr bool PAIRED = EPI == ST_SILU;
    constexpr int SUB_BAND_COLS = PAIRED ? BAND_COLS / 2 : BAND_COLS;
    constexpr int SUB_ROW_BYTES = SUB_BAND_COLS * ES;
    float *red = scratch;                  // [8][256]
    float *vals = red + kStConsumerWarps * 256;
    float *xs = vals + 256 + 16;
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int UB = (K + kStBoxRows - 1) / kStBoxRows;
    const long long W = (long long)n_bands * UB;
    // only min(grid, W) CTAs take part, so that every one has a non-empty
    // range and the contributors to a band are consecutive CTAs
    const int G = (int)min((long long)gridDim.x, W);
    const bool in = (int)blockIdx.x < G;
    const long long u0 = in ? W * blockIdx.x / G : 0, u1 = in ? W * (blockIdx.x + 1) / G : 0;
    const uint32_t out_tag = cx.seq(pid);
    // one partial buffer per projection kind: the same kind of the next layer
    // cannot start writing before every settlement of this one has read it
    const int kind = (pid - 1) % 5;  // 0 q|k|v, 2 o, 3 gate|up, 4 down
    u64 *part = p.pt + (size_t)(kind == 0 ? 0 : kind - 1) * p.pt_stride;
    trace_point(p, phase, 0);
    if (!in) return;

    if (SRC == SRC_ATTN) {  // the slice of the attention output, merged here
        int off = 0;
        for (long long u = u0; u < u1;) {
            const int band = (int)(u / UB);
            const int j0 = (int)(u - (long long)band * UB);
            const int j1 = (int)min((long long)UB, j0 + (u1 - u));
            u += j1 - j0;
            const int k0 = j0 * kStBoxRows, k1 = j1 * kStBoxRows;
            stage_attention_rows<GQ>(k0, min(k1, K), xs + off, red, in_tag, cx, p);
            for (int k = K + t; k < k1; k += kStConsumers) xs[off + k - k0] = 0.0f;
            off += k1 - k0;
        }
        named_sync(1, kStConsumers);
    } else {  // this CTA's slice of the input (times the norm weight; zero past K)
        int off = 0;
        for (long long u = u0; u < u1;) {
            const int band = (int)(u / UB);
            const int j0 = (int)(u - (long long)band * UB);
            const int j1 = (int)min((long long)UB, j0 + (u1 - u));
            u += j1 - j0;
            const int k0 = j0 * kStBoxRows, k1 = j1 * kStBoxRows;
            for (int kb = k0; kb < k1; kb += 8 * kStConsumers) {
                u64 v[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int k = kb + q * kStConsumers + t;
                    v[q] = (k < k1 && k < K) ? ld_tag(xin + k) : 0ull;
                }
                const int nv = min(8, max(0, (min(k1, K) - kb - t + kStConsumers - 1) / kStConsumers));
                tag_fix<8>(v, xin + kb + t, kStConsumers, nv, in_tag, p);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int k = kb + q * kStConsumers + t;
                    if (k < k1) {
                        float o = 0.0f;
                        if (k < K) {
                            o = tag_f(v[q]);
                            if (NORM) o *= __ldg(norm_w + k);
                        }
                        xs[off + k - k0] = o;
                    }
                }
            }
            off += k1 - k0;
        }
        named_sync(1, kStConsumers);
    }
    trace_point(p, phase, 1);

    float scale = 1.0f;
    bool have_scale = !NORM;
    // the RMSNorm's square sums, requested now and summed at the first epilogue
    const u64 ss_w = NORM ? sst_first(p) : 0ull;
    // What an epilogue of `band` reads besides the column sums, requested
    // before those are waited for so that one L2 round trip covers all: for
    // q|k|v, RoPE's cos/sin of this thread's column and the cache row of pos.
    struct EpiIn {
        float c, sn;
        long long row;
    };
    auto epi_in = [&](int band) {
        EpiIn e{1.0f, 0.0f, 0};
        if (EPI == ST_QKV && cx.pos_ok) {
            const int col = band * BAND_COLS + t;
            if (t < BAND_COLS && col < p.nq_cols + p.nkv_cols) {
                const int hd = p.hd, half = hd >> 1;
                const int i = (col - (col < p.nq_cols ? 0 : p.nq_cols)) % hd;
                const int pair = p.rope_layout == DS_ROPE_HALF_SPLIT ? (i < half ? i : i - half) : i >> 1;
                e.c = __ldg(p.rope_cos + (size_t)cx.pos * half + pair);
                e.sn = __ldg(p.rope_sin + (size_t)cx.pos * half + pair);
            }
            const int blk = p.block_table ? __ldcg(p.block_table + cx.pos / p.block_tokens) : cx.pos / p.block_tokens;
            e.row = (long long)blk * p.block_tokens + cx.pos % p.block_tokens;
        }
        return e;
    };
    // the band this CTA settles (see below) is the first of its range when
    // that range starts inside a band and reaches the band's end
    const int b_first = (int)(u0 / UB);
    const bool settles = u0 % UB != 0 && u1 >= (long long)(b_first + 1) * UB;
    const EpiIn own_in = settles ? epi_in(b_first) : EpiIn{1.0f, 0.0f, 0};
    // the fused epilogue of one band whose column sums v (thread t < BAND_COLS)
    // are final; yw is the residual word already loaded (ST_ADD), ein what
    // epi_in(band) loaded
    auto epilogue = [&](int band, float v, u64 yw, const EpiIn &ein) {
        if (NORM && !have_scale) {
            scale = scale_from_sst(p, K, in_tag, red, ss_w);
            have_scale = true;
        }
        if (EPI == ST_STORE || EPI == ST_ADD) {
            const int col = band * BAND_COLS + t;
            const bool ok = t < BAND_COLS && col < sub_cols;
            float out = v * scale;
            if (EPI == ST_ADD && ok) out += tag_value(yw, y + col, yold_tag, p);
            if (ok) st_tag(y + col, out, out_tag);
            if (EPI == ST_ADD) {  // this band's share of the next RMSNorm
                const float ss = block_sumsq(ok ? out : 0.0f, red);
                if (t == 0) st_tag(p.sst + band, ss, out_tag);
            }
        } else if (EPI == ST_SILU) {
            vals[t] = v * scale;
            named_sync(1, kStConsumers);
            const int col = band * SUB_BAND_COLS + t;
            if (t < SUB_BAND_COLS && col < sub_cols) st_tag(y + col, silu_st(vals[t]) * vals[t + SUB_BAND_COLS], out_tag);
            named_sync(1, kStConsumers);
        } else {  // ST_QKV: RoPE on q and k; K/V written at pos and handed to attention
            vals[t] = v * scale;
            named_sync(1, kStConsumers);
            const StepLayer &QL = p.layers[layer];
            if (QL.qn) qk_norm_band(vals, vals + 256, band * BAND_COLS, BAND_COLS, QL.qn, QL.kn, p.nq_cols,
                                    p.nkv_cols, p.hd, p.eps);
            const int col = band * BAND_COLS + t;
            const int total = p.nq_cols + 2 * p.nkv_cols;
            if (t < BAND_COLS && col < total) {
                float out = vals[t];
                if (col < p.nq_cols + p.nkv_cols) {
                    const int hd = p.hd, half = hd >> 1;
                    const int region = col < p.nq_cols ? 0 : p.nq_cols;
                    const int i = (col - region) % hd;
                    float a, b;
                    bool first_of_pair;
                    if (p.rope_layout == DS_ROPE_HALF_SPLIT) {
                        first_of_pair = i < half;
                        a = first_of_pair ? vals[t] : vals[t - half];
                        b = first_of_pair ? vals[t + half] : vals[t];
                    } else {
                        first_of_pair = (i & 1) == 0;
                        a = first_of_pair ? vals[t] : vals[t - 1];
                        b = first_of_pair ? vals[t + 1] : vals[t];
                    }
                    const float c = ein.c, sn = ein.sn;  // 1 and 0 where pos is past the tables
                    out = first_of_pair ? a * c - b * sn : a * sn + b * c;
                }
                if (col < p.nq_cols) {
                    st_tag(y + col, out, out_tag);
                } else {
                    const int kv = col - p.nq_cols;  // k then v
                    if (cx.pos_ok) {
                        const long long row = ein.row;
                        if (kv < p.nkv_cols)
                            store_as(p.kc[layer], row * p.nkv_cols + kv, p.kv_dtype, out);
                        else
                            store_as(p.vc[layer], row * p.nkv_cols + kv - p.nkv_cols, p.kv_dtype, out);
                    }
                    // attention reads this position from here, as the cache holds it
                    const float held = p.kv_dtype == DS_BF16 ? __bfloat162float(__float2bfloat16_rn(out)) : out;
                    st_tag(p.kvt + kv, held, out_tag);
                }
            }
            named_sync(1, kStConsumers);
        }
    };

    int own_band = -1, own_first = 0;  // the shared band this CTA settles
    float own_v = 0.0f;
    int seg_off = 0;
    for (long long u = u0; u < u1;) {
        const int band = (int)(u / UB);
        const int j0 = (int)(u - (long long)band * UB);
        const int j1 = (int)min((long long)UB, j0 + (u1 - u));
        u += j1 - j0;
        const float *xseg = xs + seg_off - j0 * kStBoxRows;
        seg_off += (j1 - j0) * kStBoxRows;

        float acc[LE];
#pragma unroll
        for (int e = 0; e < LE; ++e) acc[e] = 0.0f;
        for (int j = j0; j < j1; j += kStBoxesPerStage) {
            const int nr = min(kStBoxesPerStage, j1 - j) * kStBoxRows;
            const int s = fill % r.stages;
            const uint32_t use = fill / r.stages;
            if (st_wait(&r.full[s], use & 1, p)) {
                const unsigned char *st = r.base + (size_t)s * kStStageBytes;
                const unsigned char *lane_base =
                    PAIRED ? st + (lane >> 4) * (kStStageBytes / 2) + (lane & 15) * 16 : st + lane * 16;
                const int kr = j * kStBoxRows;
#pragma unroll 4
                for (int rr = warp; rr < nr; rr += kStConsumerWarps) {
                    const float xk = xseg[kr + rr];
                    const uint4 w = *reinterpret_cast<const uint4 *>(lane_base + rr * SUB_ROW_BYTES);
                    float fv[LE];
                    widen16(w, fv);
#pragma unroll
                    for (int e = 0; e < LE; ++e) acc[e] = fmaf(fv[e], xk, acc[e]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&r.empty[s]);
            ++fill;
        }
        if (u >= u1) trace_point(p, phase, 2);

        // cross-warp reduction of the band's column sums, fixed order
#pragma unroll
        for (int e = 0; e < LE; ++e) red[warp * BAND_COLS + lane * LE + e] = acc[e];
        named_sync(1, kStConsumers);
        float v = 0.0f;
        if (t < BAND_COLS)
            for (int w = 0; w < kStConsumerWarps; ++w) v += red[w * BAND_COLS + t];
        named_sync(1, kStConsumers);

        if (j0 == 0 && j1 == UB) {  // whole band here: final now
            u64 yw = 0;
            if (EPI == ST_ADD && t < BAND_COLS && band * BAND_COLS + t < sub_cols) yw = ld_tag(y + band * BAND_COLS + t);
            epilogue(band, v, yw, epi_in(band));
        } else if (j1 == UB) {  // this CTA holds the band's last box: it settles
            own_band = band;
            own_v = v;
            own_first = (int)((((long long)band * UB + 1) * G - 1) / W);
        } else if (t < BAND_COLS) {
            st_tag(part + (size_t)(blockIdx.x + band) * BAND_COLS + t, v, out_tag);
        }
    }

    if (own_band >= 0) {
        // the other contributors are CTAs own_first .. this one - 1, partial
        // slot CTA + band; their loads go out together with the residual's
        u64 yw = 0;
        const int col = own_band * BAND_COLS + t;
        if (EPI == ST_ADD && t < BAND_COLS && col < sub_cols) yw = ld_tag(y + col);
        float tot = 0.0f;
        if (t < BAND_COLS) {
            const int n = (int)blockIdx.x - own_first;
            const u64 *base = part + (size_t)(own_first + own_band) * BAND_COLS + t;
            for (int c0 = 0; c0 < n; c0 += 8) {
                u64 w[8];
#pragma unroll
                for (int c = 0; c < 8; ++c) w[c] = c0 + c < n ? ld_tag(base + (size_t)(c0 + c) * BAND_COLS) : 0ull;
                tag_fix<8>(w, base + (size_t)c0 * BAND_COLS, BAND_COLS, n - c0, out_tag, p);
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    if (c0 + c < n) tot += tag_f(w[c]);
            }
            tot += own_v;
        }
        epilogue(own_band, tot, yw, own_in);
    }
    trace_point(p, phase, 3);
}

// K or V dims [d0, d0+4) of one cache row, through L2.
template <typename KT>
__device__ __forceinline__ void load4(const KT *base, long long off, bool ok, float (&f)[4]) {
    if (!ok) {
        f[0] = f[1] = f[2] = f[3] = 0.0f;
        return;
    }
    if (sizeof(KT) == 2) {
        uint2 w;
        asm volatile("ld.global.cg.v2.u32 {%0, %1}, [%2];" : "=r"(w.x), "=r"(w.y) : "l"(base + off));
        f[0] = __uint_as_float(w.x << 16);
        f[1] = __uint_as_float(w.x & 0xffff0000u);
        f[2] = __uint_as_float(w.y << 16);
        f[3] = __uint_as_float(w.y & 0xffff0000u);
    } else {
        const float4 w = __ldcg(reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(base) + off));
        f[0] = w.x;
        f[1] = w.y;
        f[2] = w.z;
        f[3] = w.w;
    }
}

// Positions per attention split and the number of splits in use.
__device__ __forceinline__ void attention_split(const StepCtx &cx, const StepParams &p, int &per, int &n_eff) {
    attention_split_n(cx.n_ctx, p, per, n_eff);
}

// Request into L2 the K/V rows of this CTA's attention item of `layer`:
// rows before the current position, written by earlier steps.
template <typename KT>
__device__ void prefetch_attention(int layer, const StepCtx &cx, const StepParams &p) {
    const int n_items = p.n_kvh * p.attn_splits;
    if (kv_streamed(cx.n_ctx, p) || (int)blockIdx.x >= n_items) return;  // streamed through the ring instead
    const int g = blockIdx.x / p.attn_splits, split = blockIdx.x % p.attn_splits;
    int per, n_eff;
    attention_split(cx, p, per, n_eff);
    const int n_old = cx.n_ctx - 1;
    const int t0 = min(n_old, split * per), t1 = min(n_old, t0 + per);
    const int row_bytes = p.hd * (int)sizeof(KT);  // one head's row
    const int lines = (row_bytes + 127) / 128;
    const int n = (t1 - t0) * lines * 2;
    for (int i = threadIdx.x; i < n; i += kStConsumers) {
        const int kv = i & 1, rest = i >> 1;
        const int tt = t0 + rest / lines, line = rest % lines;
        const int b = tt / p.block_tokens;
        const long long blk = p.block_table ? (long long)__ldcg(p.block_table + b) : (long long)b;
        const long long off = ((blk * p.block_tokens + tt % p.block_tokens) * p.n_kvh + g) * (long long)row_bytes + line * 128;
        const char *base = static_cast<const char *>(kv ? p.vc[layer] : p.kc[layer]);
        asm volatile("prefetch.global.L2 [%0];" ::"l"(base + off));
    }
}

// One CTA's share of the attention phase (id `pid`): item (kv head g, split)
// = this CTA (CTAs past the items have none).  Eight warps take runs of RUN
// cached positions with an online softmax; the current position comes from
// the tagged copy the q|k|v phase handed over.  Warps merge in shared memory
// and the CTA publishes its split's (max, sum, accumulator) as tagged words;
// splits past the context publish an empty record.  The splits of a head are
// merged, in split order, by whoever reads the attention output next (the o
// projection's prologue).
//
// Within a warp, lane L holds dims 4L..4L+3 of every row.  The RUN x GQ
// partial dot products of a run are summed across the warp by halving
// exchanges (at each round a lane keeps one half of its values and sends the
// other half to the lane `b` apart), V - 1 shuffles in all instead of five per
// product; afterwards lane L holds the whole score of pair L >> SH (head
// pair / RUN, position pair % RUN), the lanes of one head form an aligned
// group, and the softmax runs on one score per lane.  The weights reach every
// lane through a few words of shared memory for the P.V products.
template <typename KT, int GQ>
__device__ void consume_attention(const Ring &r, uint32_t &fill, int layer, int pid, const StepCtx &cx,
                                  float *scratch, const StepParams &p, int phase) {
    constexpr int RUN = GQ >= 8 ? 4 : 8;              // positions per run
    constexpr int V = RUN * GQ;                       // scores per run (<= 32)
    constexpr int LV = V >= 32 ? 5 : V >= 16 ? 4 : V >= 8 ? 3 : V >= 4 ? 2 : 1;
    constexpr int SH = 5 - LV;                        // lane bits below a pair's index
    constexpr int WS = V + 8;                         // per-warp words: weights, then corrections
    static_assert(V <= 32 && (1 << LV) == V, "RUN * GQ must be a power of two up to 32");
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int hd = p.hd;
    const int n_items = p.n_kvh * p.attn_splits;
    trace_point(p, phase, 0);
    if ((int)blockIdx.x >= n_items) return;
    const int g = blockIdx.x / p.attn_splits, split = blockIdx.x % p.attn_splits;
    const uint32_t q_tag = cx.seq(pid - 1), out_tag = cx.seq(pid);
    const int rec = GQ * (hd + 2);
    u64 *out = p.at + (size_t)(g * p.attn_splits + split) * rec;
    float *s_acc = scratch;                                   // [8][GQ][hd]
    float *s_m = s_acc + kStConsumerWarps * GQ * hd;          // [8][GQ]
    float *s_l = s_m + kStConsumerWarps * GQ;                 // [8][GQ]
    float *s_q = s_l + kStConsumerWarps * GQ;                 // [GQ][hd]
    float *s_w = s_q + GQ * hd + warp * WS;                   // this warp's [V] weights, [GQ] corrections
    float *s_M = s_q + GQ * hd + kStConsumerWarps * WS;       // [GQ] merged max
    float *s_L = s_M + GQ;                                    // [GQ] merged sum

    int per, n_eff;
    attention_split(cx, p, per, n_eff);
    if (split >= n_eff) {  // no positions: an empty record
        for (int idx = t; idx < rec; idx += kStConsumers)
            st_tag(out + idx, idx < GQ ? -INFINITY : 0.0f, out_tag);
        trace_point(p, phase, 3);
        return;
    }
    const int t0 = min(cx.n_ctx, split * per), t1 = min(cx.n_ctx, t0 + per);
    const int tc = min(t1, cx.n_ctx - 1);  // cached positions [t0, tc)
    const bool has_cur = t1 == cx.n_ctx;
    const bool active = lane * 4 < hd;
    const int d0 = lane * 4;
    const long long row_elems = (long long)p.n_kvh * hd;
    const KT *kc = static_cast<const KT *>(p.kc[layer]);
    const KT *vc = static_cast<const KT *>(p.vc[layer]);

    float kf[RUN][4], vf[RUN][4];
    // bf16 caches: a run's rows are fetched packed (two registers per row) one
    // run ahead; K is unpacked for the scores and V for the products, each
    // just before its own next-run loads go out
    constexpr bool PACKED = sizeof(KT) == 2;
    uint2 rk[PACKED ? RUN : 1], rv[PACKED ? RUN : 1];
    auto row_off = [&](int tt) {
        const int b = tt / p.block_tokens;
        const long long blk = p.block_table ? (long long)__ldcg(p.block_table + b) : (long long)b;
        return (blk * p.block_tokens + tt % p.block_tokens) * row_elems + (long long)g * hd + d0;
    };
    auto load_packed = [&](uint2 (&rw)[PACKED ? RUN : 1], const KT *base, int tb) {
        if constexpr (PACKED) {
            const int nt = min(RUN, tc - tb);
#pragma unroll
            for (int i = 0; i < RUN; ++i) {
                rw[i] = make_uint2(0u, 0u);
                if (active && i < nt)
                    asm volatile("ld.global.cg.v2.u32 {%0, %1}, [%2];"
                                 : "=r"(rw[i].x), "=r"(rw[i].y) : "l"(base + row_off(tb + i)));
            }
        }
    };
    auto load_run = [&](int tb) {
        if constexpr (PACKED) {
            load_packed(rk, kc, tb);
            load_packed(rv, vc, tb);
        } else {
            const int nt = min(RUN, tc - tb);
#pragma unroll
            for (int i = 0; i < RUN; ++i) {
                const bool ok = active && i < nt;
                const long long off = ok ? row_off(tb + i) : 0;
                load4<KT>(kc, off, ok, kf[i]);
                load4<KT>(vc, off, ok, vf[i]);
            }
        }
    };
    auto unpack = [&](const uint2 (&rw)[PACKED ? RUN : 1], float (&f)[RUN][4]) {
        if constexpr (PACKED) {
#pragma unroll
            for (int i = 0; i < RUN; ++i) {
                f[i][0] = __uint_as_float(rw[i].x << 16);
                f[i][1] = __uint_as_float(rw[i].x & 0xffff0000u);
                f[i][2] = __uint_as_float(rw[i].y << 16);
                f[i][3] = __uint_as_float(rw[i].y & 0xffff0000u);
            }
        }
    };
    int tb = t0 + warp * RUN;
    const bool streamed = kv_streamed(cx.n_ctx, p);
    if (!streamed && tb < tc) load_run(tb);  // K/V requests go out before q is polled
    // the current position's k and v (handed over by the q|k|v phase), read by
    // the last warp: requested now, their arrival checked after the cached run
    const bool cur_warp = has_cur && warp == kStConsumerWarps - 1;
    u64 cw[8];
    const u64 *ca[8];
    {
        const u64 *kt = p.kvt + (size_t)g * hd + d0, *vt = p.kvt + p.nkv_cols + (size_t)g * hd + d0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            ca[e] = cur_warp && active ? kt + e : nullptr;
            ca[4 + e] = cur_warp && active ? vt + e : nullptr;
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) cw[e] = ca[e] ? ld_tag(ca[e]) : 0ull;
    }
    {   // the group's q rows, polled once by the whole CTA into shared memory
        const u64 *qg = p.qt + (size_t)g * GQ * hd;
        for (int i0 = 0; i0 < GQ * hd; i0 += 2 * kStConsumers) {
            u64 w[2];
#pragma unroll
            for (int k = 0; k < 2; ++k) w[k] = i0 + k * kStConsumers + t < GQ * hd ? ld_tag(qg + i0 + k * kStConsumers + t) : 0ull;
            const int nv = min(2, max(0, (GQ * hd - i0 - t + kStConsumers - 1) / kStConsumers));
            tag_fix<2>(w, qg + i0 + t, kStConsumers, nv, q_tag, p);
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int i = i0 + k * kStConsumers + t;
                if (i < GQ * hd) s_q[i] = tag_f(w[k]);
            }
        }
        named_sync(1, kStConsumers);
    }
    trace_point(p, phase, 1);
    const float scale = 1.0f / sqrtf((float)hd);
    const int pair = lane >> SH, pos_i = pair % RUN;
    const bool pair_lead = (lane & ((1 << SH) - 1)) == 0;
    float mh = -INFINITY, lh = 0.0f;  // this lane's head (pair / RUN): running max and sum
    float acc[GQ][4];
#pragma unroll
    for (int j = 0; j < GQ; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[j][e] = 0.0f;
    // the scores of the `nt` positions whose K rows are in kf: online-softmax
    // state updated, their weights and the heads' corrections left in s_w
    auto scores = [&](int nt) {
        float v[V];
#pragma unroll
        for (int j = 0; j < GQ; ++j) {
            const float4 qj = active ? *reinterpret_cast<const float4 *>(s_q + j * hd + d0) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int i = 0; i < RUN; ++i) {
                float dd = qj.x * kf[i][0];
                dd = fmaf(qj.y, kf[i][1], dd);
                dd = fmaf(qj.z, kf[i][2], dd);
                dd = fmaf(qj.w, kf[i][3], dd);
                v[j * RUN + i] = dd;
            }
        }
#pragma unroll
        for (int c = V, b = 16; c > 1; c >>= 1, b >>= 1) {
            const bool up = (lane & b) != 0;
#pragma unroll
            for (int k = 0; k < c / 2; ++k) {
                const float send = up ? v[k] : v[k + c / 2];
                const float keep = up ? v[k + c / 2] : v[k];
                v[k] = keep + __shfl_xor_sync(0xffffffffu, send, b);
            }
        }
        float s = v[0];
#pragma unroll
        for (int b = 1; b < (1 << SH); b <<= 1) s += __shfl_xor_sync(0xffffffffu, s, b);
        s = pos_i < nt ? s * scale : -INFINITY;
        float mx = s;
#pragma unroll
        for (int b = 1 << SH; b < (RUN << SH); b <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, b));
        const float mn = fmaxf(mh, mx);  // finite: nt >= 1
        const float corr = expf(mh - mn);
        const float w = pos_i < nt ? expf(s - mn) : 0.0f;
        float ws = w;
#pragma unroll
        for (int b = 1 << SH; b < (RUN << SH); b <<= 1) ws += __shfl_xor_sync(0xffffffffu, ws, b);
        lh = fmaf(lh, corr, ws);
        mh = mn;
        if (pair_lead) {
            s_w[pair] = w;
            if (pos_i == 0) s_w[V + pair / RUN] = corr;
        }
        __syncwarp();
    };
    // acc = acc * correction + weights . V rows (in vf); s_w free afterwards
    auto accumulate = [&]() {
#pragma unroll
        for (int j = 0; j < GQ; ++j) {
            const float cj = s_w[V + j];
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[j][e] *= cj;
#pragma unroll
            for (int i4 = 0; i4 < RUN; i4 += 4) {
                const float4 w4 = *reinterpret_cast<const float4 *>(s_w + j * RUN + i4);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    acc[j][e] = fmaf(w4.x, vf[i4][e], acc[j][e]);
                    acc[j][e] = fmaf(w4.y, vf[i4 + 1][e], acc[j][e]);
                    acc[j][e] = fmaf(w4.z, vf[i4 + 2][e], acc[j][e]);
                    acc[j][e] = fmaf(w4.w, vf[i4 + 3][e], acc[j][e]);
                }
            }
        }
        __syncwarp();
    };
    if (streamed) {
        // the cached positions arrive through the ring, kv_stage_pos per stage
        // (K rows, then V rows); warp w takes a stage's w-th eighth in runs
        const int P = p.kv_stage_pos, per_warp = P / kStConsumerWarps;
        const int row_bytes = hd * (int)sizeof(KT);
        auto read_rows = [&](const unsigned char *base, int rb, int nt, float (&f)[RUN][4]) {
#pragma unroll
            for (int i = 0; i < RUN; ++i) {
                const bool ok = active && i < nt;
                const size_t off = (size_t)(rb + i) * row_bytes + (size_t)d0 * sizeof(KT);
                if (sizeof(KT) == 2) {
                    uint2 w = make_uint2(0u, 0u);
                    if (ok) w = *reinterpret_cast<const uint2 *>(base + off);
                    f[i][0] = __uint_as_float(w.x << 16);
                    f[i][1] = __uint_as_float(w.x & 0xffff0000u);
                    f[i][2] = __uint_as_float(w.y << 16);
                    f[i][3] = __uint_as_float(w.y & 0xffff0000u);
                } else {
                    float4 w = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (ok) w = *reinterpret_cast<const float4 *>(base + off);
                    f[i][0] = w.x; f[i][1] = w.y; f[i][2] = w.z; f[i][3] = w.w;
                }
            }
        };
        for (int ts = t0; ts < tc; ts += P) {
            const int s = fill % r.stages;
            const uint32_t use = fill / r.stages;
            if (st_wait(&r.full[s], use & 1, p)) {
                const unsigned char *kb = r.base + (size_t)s * kStStageBytes;
                const unsigned char *vb = kb + (size_t)P * row_bytes;
                for (int rb = warp * per_warp; rb < (warp + 1) * per_warp; rb += RUN) {
                    const int nt = min(RUN, tc - (ts + rb));
                    if (nt <= 0) break;
                    read_rows(kb, rb, nt, kf);
                    scores(nt);
                    read_rows(vb, rb, nt, vf);
                    accumulate();
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&r.empty[s]);
            ++fill;
        }
        tb = tc;
    }
    while (tb < tc) {
        const int nt = min(RUN, tc - tb), tn = tb + kStConsumerWarps * RUN;
        if constexpr (PACKED) {
            // the next run's loads go out before this run's arithmetic
            unpack(rk, kf);
            if (tn < tc) load_packed(rk, kc, tn);
            scores(nt);
            unpack(rv, vf);
            if (tn < tc) load_packed(rv, vc, tn);
            accumulate();
        } else {
            scores(nt);
            accumulate();
            if (tn < tc) load_run(tn);
        }
        tb = tn;
    }
    if (cur_warp) {  // the current position
        tag_fix_at<8>(cw, ca, q_tag, p);
#pragma unroll
        for (int i = 0; i < RUN; ++i)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                kf[i][e] = i == 0 && active ? tag_f(cw[e]) : 0.0f;
                vf[i][e] = i == 0 && active ? tag_f(cw[4 + e]) : 0.0f;
            }
        scores(1);
        accumulate();
    }
    if (pair_lead && pos_i == 0) {
        s_m[warp * GQ + pair / RUN] = mh;
        s_l[warp * GQ + pair / RUN] = lh;
    }
#pragma unroll
    for (int j = 0; j < GQ; ++j)
        if (active)
#pragma unroll
            for (int e = 0; e < 4; ++e) s_acc[(warp * GQ + j) * hd + d0 + e] = acc[j][e];
    named_sync(1, kStConsumers);
    trace_point(p, phase, 2);

    // the warps' weights exp(m_w - M) per head, and the merged max and sum:
    // warp 0, one (head, warp) pair per lane, eight lanes per head
    if (warp == 0)
        for (int p0 = 0; p0 < GQ * kStConsumerWarps; p0 += 32) {
            const int pr = p0 + lane, j = pr / kStConsumerWarps, w = pr % kStConsumerWarps;
            const bool ok = pr < GQ * kStConsumerWarps;
            const float mw = ok ? s_m[w * GQ + j] : -INFINITY;
            float M = mw;
#pragma unroll
            for (int b = 1; b < kStConsumerWarps; b <<= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, b));
            const float c = mw == -INFINITY ? 0.0f : expf(mw - M);
            float L = ok ? s_l[w * GQ + j] * c : 0.0f;
#pragma unroll
            for (int b = 1; b < kStConsumerWarps; b <<= 1) L += __shfl_xor_sync(0xffffffffu, L, b);
            if (ok) {
                s_m[w * GQ + j] = c;  // each lane rewrites only the entry it read
                if (w == 0) {
                    s_M[j] = M;
                    s_L[j] = L;
                }
            }
        }
    named_sync(1, kStConsumers);
    for (int idx = t; idx < GQ * hd; idx += kStConsumers) {
        const int j = idx / hd;
        float A = 0.0f;
#pragma unroll
        for (int w = 0; w < kStConsumerWarps; ++w) A = fmaf(s_acc[(w * GQ + j) * hd + idx % hd], s_m[w * GQ + j], A);
        st_tag(out + 2 * GQ + idx, A, out_tag);
        if (idx % hd == 0) {
            st_tag(out + j, s_M[j], out_tag);
            st_tag(out + GQ + j, s_L[j], out_tag);
        }
    }
    trace_point(p, phase, 3);
}

// Attention output rows [k0, k1) (k indexes query head h = k / hd, dim
// k % hd), merged from the tagged split records of their KV heads in split
// order: out = sum_s w_s acc_s / sum_s w_s l_s with w_s = exp(m_s - max m),
// written to xs.  `red` holds the per-head weights.
template <int GQ>
__device__ void stage_attention_rows(int k0, int k1, float *xs, float *red, uint32_t tag, const StepCtx &cx,
                                     const StepParams &p) {
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int hd = p.hd;
    int per, n_eff;
    attention_split(cx, p, per, n_eff);
    const int rec = GQ * (hd + 2);
    const int h_lo = k0 / hd, h_hi = (k1 - 1) / hd;
    const int nh = h_hi - h_lo + 1;
    float *wt = red;                      // [nh][kStMaxSplits]
    float *Lh = red + nh * kStMaxSplits;  // [nh]
    for (int hl = warp; hl < nh; hl += kStConsumerWarps) {
        const int h = h_lo + hl, g = h / GQ, j = h % GQ;
        const u64 *base = p.at + (size_t)g * p.attn_splits * rec;
        const u64 *a[4];
        a[0] = lane < n_eff ? base + (size_t)lane * rec + j : nullptr;
        a[1] = lane < n_eff ? base + (size_t)lane * rec + GQ + j : nullptr;
        a[2] = lane + 32 < n_eff ? base + (size_t)(lane + 32) * rec + j : nullptr;
        a[3] = lane + 32 < n_eff ? base + (size_t)(lane + 32) * rec + GQ + j : nullptr;
        u64 w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) w[i] = a[i] ? ld_tag(a[i]) : 0ull;
        tag_fix_at<4>(w, a, tag, p);
        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;
        if (lane < n_eff) {
            m0 = tag_f(w[0]);
            l0 = tag_f(w[1]);
        }
        if (lane + 32 < n_eff) {
            m1 = tag_f(w[2]);
            l1 = tag_f(w[3]);
        }
        const float M = warp_max(fmaxf(m0, m1));
        const float w0 = (lane < n_eff && m0 != -INFINITY) ? expf(m0 - M) : 0.0f;
        const float w1 = (lane + 32 < n_eff && m1 != -INFINITY) ? expf(m1 - M) : 0.0f;
        wt[hl * kStMaxSplits + lane] = w0;
        wt[hl * kStMaxSplits + lane + 32] = w1;
        const float L = warp_sum(fmaf(w1, l1, w0 * l0));
        if (lane == 0) Lh[hl] = L;
    }
    named_sync(1, kStConsumers);
    for (int k = k0 + t; k < k1; k += kStConsumers) {
        const int h = k / hd, g = h / GQ, j = h % GQ, hl = h - h_lo;
        const u64 *rp = p.at + (size_t)g * p.attn_splits * rec + 2 * GQ + j * hd + k % hd;
        float A = 0.0f;
        for (int s0 = 0; s0 < n_eff; s0 += kStMergeBatch) {
            u64 w[kStMergeBatch];
#pragma unroll
            for (int i = 0; i < kStMergeBatch; ++i) w[i] = s0 + i < n_eff ? ld_tag(rp + (size_t)(s0 + i) * rec) : 0ull;
            tag_fix<kStMergeBatch>(w, rp + (size_t)s0 * rec, rec, n_eff - s0, tag, p);
#pragma unroll
            for (int i = 0; i < kStMergeBatch; ++i)
                if (s0 + i < n_eff) A = fmaf(tag_f(w[i]), wt[hl * kStMaxSplits + s0 + i], A);
        }
        xs[k - k0] = A / Lh[hl];
    }
    named_sync(1, kStConsumers);
}

// The best (value, index) of the 256 consumer threads' candidates under
// ranks_above, left in every thread: a shuffle tree per warp, then over the
// eight warps' winners (sv/si: 8 entries of shared scratch).
__device__ void block_best(float &bv, int &bi, float *sv, int *si) {
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ranks_above(ov, oi, bv, bi)) {
            bv = ov;
            bi = oi;
        }
    }
    if (lane == 0) {
        sv[warp] = bv;
        si[warp] = bi;
    }
    named_sync(1, kStConsumers);
    bv = sv[0];
    bi = si[0];
    for (int w = 1; w < kStConsumerWarps; ++w)
        if (ranks_above(sv[w], si[w], bv, bi)) {
            bv = sv[w];
            bi = si[w];
        }
    named_sync(1, kStConsumers);
}

// The head phase: logits of this CTA's rows, then (once every CTA has
// finished) the greedy pick and the launch's epoch advance.
template <typename T>
__device__ void consume_gn(const Ring &r, uint32_t &fill, uint32_t in_tag, float *scratch, const StepParams &p,
                           int step, int phase) {
    constexpr int LE = 16 / sizeof(T);
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int G = gridDim.x;
    const int cols = p.d, rows = p.vocab;
    const long long row_bytes = (long long)cols * sizeof(T);
    const int rps = (int)max(1LL, (long long)kStStageBytes / row_bytes);
    const int parts = rps >= kStConsumerWarps ? 1 : kStConsumerWarps / rps;
    const int r0 = (int)((long long)rows * blockIdx.x / G), r1 = (int)((long long)rows * (blockIdx.x + 1) / G);
    float *bestv = scratch;                              // [256]
    int *besti = reinterpret_cast<int *>(bestv + 256);   // [256]
    float *xs = bestv + 512;                             // [cols]
    float *rowpart = xs + cols;                          // [rows of this CTA][parts]
    trace_point(p, phase, 0);

    for (int i0 = 0; i0 < cols; i0 += 8 * kStConsumers) {
        u64 v[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int i = i0 + q * kStConsumers + t;
            v[q] = i < cols ? ld_tag(p.xt + i) : 0ull;
        }
        const int nv = min(8, max(0, (cols - i0 - t + kStConsumers - 1) / kStConsumers));
        tag_fix<8>(v, p.xt + i0 + t, kStConsumers, nv, in_tag, p);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int i = i0 + q * kStConsumers + t;
            if (i < cols) xs[i] = tag_f(v[q]) * __ldg(p.final_norm + i);
        }
    }
    named_sync(1, kStConsumers);
    const float scale = scale_from_sst(p, cols, in_tag, bestv, sst_first(p));
    trace_point(p, phase, 1);

    const int chunks = (int)(row_bytes / 16);
    for (int rr = r0; rr < r1; rr += rps) {
        const int nr = min(rps, r1 - rr);
        const int s = fill % r.stages;
        const uint32_t use = fill / r.stages;
        if (st_wait(&r.full[s], use & 1, p)) {
            const unsigned char *st = r.base + (size_t)s * kStStageBytes;
            if (parts == 1) {
                for (int q = warp; q < nr; q += kStConsumerWarps) {
                    const unsigned char *row = st + (size_t)q * row_bytes;
                    float a = 0.0f;
                    for (int c = lane; c < chunks; c += 32) {
                        const uint4 w = *reinterpret_cast<const uint4 *>(row + c * 16);
                        float fv[LE];
                        widen16(w, fv);
#pragma unroll
                        for (int e = 0; e < LE; ++e) a = fmaf(fv[e], xs[c * LE + e], a);
                    }
                    a = warp_sum(a);
                    if (lane == 0) rowpart[rr - r0 + q] = a;
                }
            } else {
                const int q = warp / parts, part = warp % parts;
                if (q < nr) {
                    const unsigned char *row = st + (size_t)q * row_bytes;
                    const int c0 = chunks * part / parts, c1 = chunks * (part + 1) / parts;
                    float a = 0.0f;
#pragma unroll 4
                    for (int c = c0 + lane; c < c1; c += 32) {
                        const uint4 w = *reinterpret_cast<const uint4 *>(row + c * 16);
                        float fv[LE];
                        widen16(w, fv);
#pragma unroll
                        for (int e = 0; e < LE; ++e) a = fmaf(fv[e], xs[c * LE + e], a);
                    }
                    a = warp_sum(a);
                    if (lane == 0) rowpart[(rr - r0 + q) * parts + part] = a;
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&r.empty[s]);
        ++fill;
    }
    named_sync(1, kStConsumers);
    trace_point(p, phase, 2);

    float bv = -INFINITY;
    int bi = INT_MAX;
    for (int q = t; q < r1 - r0; q += kStConsumers) {
        float logit = 0.0f;
        for (int k = 0; k < parts; ++k) logit += rowpart[q * parts + k];
        logit *= scale;
        p.logits[r0 + q] = logit;
        if (ranks_above(logit, r0 + q, bv, bi)) {
            bv = logit;
            bi = r0 + q;
        }
    }
    // this CTA's best row: a tree over the 256 consumer threads (ranks_above is
    // a total order, so any tree gives the first index of the maximum)
    block_best(bv, bi, bestv, besti);
    __shared__ int s_last;
    if (t == 0) {
        p.am_val[blockIdx.x] = bv;
        p.am_idx[blockIdx.x] = bi;
        trace_point(p, phase, 3);
        __threadfence();
        const int last = atomicAdd(p.am_counter, 1) == G - 1;  // every CTA is done with the step
        if (last) *p.am_counter = 0;
        s_last = last;
    }
    named_sync(1, kStConsumers);
    const bool last = s_last != 0;
    named_sync(1, kStConsumers);
    if (!last) return;
    __threadfence();
    // the step's pick: every CTA's best, read in parallel
    bv = -INFINITY;
    bi = INT_MAX;
    if (p.greedy) {
        for (int j = t; j < G; j += kStConsumers) {
            const float v = ldcg(&p.am_val[j]);
            const int ix = __ldcg(&p.am_idx[j]);
            if (ranks_above(v, ix, bv, bi)) {
                bv = v;
                bi = ix;
            }
        }
        block_best(bv, bi, bestv, besti);
    }
    if (t == 0) {
        if (p.greedy) {
            p.next_ids[0] = bi;
            if (p.ids_out) p.ids_out[step] = bi;
            if (p.advance) {
                p.tokens[0] = bi;
                p.pos[0] += 1;
            }
        }
        if (step + 1 < p.n_steps) {
            // the next step's embed waits for this word; the counter reset above
            // is visible before it is
            __threadfence();
            st_tag(p.tokt, __int_as_float(bi), in_tag);
        } else {
            // every CTA read the epoch at its start: advance it past this launch's steps
            asm volatile("red.relaxed.gpu.global.add.u64 [%0], %1;" ::"l"(p.epoch), "l"((u64)p.n_steps) : "memory");
        }
    }
}

template <typename T, typename KT, int GQ>
__global__ void __launch_bounds__(kStThreads, 1) step_kernel(const __grid_constant__ StepParams p) {
    extern __shared__ __align__(1024) unsigned char smem[];
    Ring r;
    r.base = smem;
    r.stages = p.stages;
    r.full = reinterpret_cast<uint64_t *>(smem + (size_t)p.stages * kStStageBytes);
    r.empty = r.full + kStMaxStages;  // 16 + 16 barriers: 256 bytes
    float *scratch = reinterpret_cast<float *>(smem + (size_t)p.stages * kStStageBytes + 256);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x;
    constexpr int ES = sizeof(T);

    if (threadIdx.x == 0) {
        for (int s = 0; s < r.stages; ++s) {
            mbar_init(&r.full[s], 1);
            mbar_init(&r.empty[s], kStConsumerWarps);
        }
        fence_mbarrier_init();
    }
    __syncthreads();

    if (warp == kStConsumerWarps) {
        // ---------------- producer: every weight byte of the step, in phase order
        if (lane == 0) produce_all<ES>(r, p);
        return;
    }

    // ---------------- consumers
    StepCtx cx;
    int tok;
    {
        __shared__ unsigned long long s_epoch;
        __shared__ int s_pos, s_tok;
        if (threadIdx.x == 0) {
            unsigned long long e;
            asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(e) : "l"(p.epoch) : "memory");
            s_epoch = e;
            s_pos = __ldcg(p.pos);
            s_tok = __ldcg(p.tokens);
        }
        named_sync(1, kStConsumers);
        cx.seq.base = (uint32_t)(s_epoch & 0x3FFFFFull) << 10;
        cx.pos = s_pos;
        tok = s_tok;
        named_sync(1, kStConsumers);
    }
    const int cap = p.max_blocks * p.block_tokens;
    const int pos0 = cx.pos;
    const uint32_t epoch0 = cx.seq.base >> 10;
    uint32_t fill = 0;
    for (int step = 0; step < p.n_steps; ++step) {
    cx.seq.base = ((epoch0 + (uint32_t)step) & 0x3FFFFFu) << 10;
    cx.pos = pos0 + step;
    cx.pos_ok = cx.pos >= 0 && cx.pos < p.rope_rows && cx.pos < cap;
    if (!cx.pos_ok && threadIdx.x == 0 && blockIdx.x == 0) flag_error(p.err, DS_ERR_POSITION);
    cx.n_ctx = min(max(cx.pos + 1, 1), cap);
    if (step > 0) {  // the previous step's pick, handed over as a tagged word
        __shared__ int s_next;
        if (threadIdx.x == 0) {
            const Seq prev{((epoch0 + (uint32_t)step - 1u) & 0x3FFFFFu) << 10};
            s_next = __float_as_int(ld_wait(p.tokt, prev(5 * p.n_layer), p));
        }
        named_sync(1, kStConsumers);
        tok = s_next;
        named_sync(1, kStConsumers);
    }

    int phase = 0;
    mark_phase(p, phase);
    trace_point(p, 0, 0);
    {   // embed (phase id 0): x = E[token]; every CTA writes a slice
        if (tok < 0 || tok >= p.vocab) {
            if (threadIdx.x == 0 && blockIdx.x == 0) flag_error(p.err, DS_ERR_TOKEN_RANGE);
            tok = min(max(tok, 0), p.vocab - 1);
        }
        const uint32_t tag = cx.seq(0);
        const T *row = reinterpret_cast<const T *>(p.emb) + (long long)tok * p.d;
        const int i0 = (int)((long long)p.d * blockIdx.x / G), i1 = (int)((long long)p.d * (blockIdx.x + 1) / G);
        for (int i = i0 + threadIdx.x; i < i1; i += kStConsumers) st_tag(p.xt + i, to_f32(row[i]), tag);
        // the square sum of band b of the row (the bands the residual
        // projections use), for the first RMSNorm
        for (int b = blockIdx.x; b < p.n_ss; b += G) {
            const int bc = kStBandBytes / (int)sizeof(T);
            const int col = b * bc + threadIdx.x;
            const float v = (threadIdx.x < bc && col < p.d) ? to_f32(row[col]) : 0.0f;
            const float ss = block_sumsq(v, scratch);
            if (threadIdx.x == 0) st_tag(p.sst + b, ss, tag);
        }
    }
    trace_point(p, 0, 3);
    for (int l = 0; l < p.n_layer; ++l) {
        const StepLayer &L = p.layers[l];
        const int ph = ph_qkv(l);
        const uint32_t x_in = cx.seq(5 * l);  // the residual as the previous layer left it
        prefetch_attention<KT>(l, cx, p);
        mark_phase(p, phase);
        consume_gt<T, ST_QKV, SRC_NORM, GQ>(r, fill, p.d, p.nq_cols + 2 * p.nkv_cols, p.nb_qkv, p.xt, x_in, L.n1,
                                            p.qt, 0, l, ph, cx, scratch, p, phase - 1);
        mark_phase(p, phase);
        consume_attention<KT, GQ>(r, fill, l, ph + 1, cx, scratch, p, phase - 1);
        mark_phase(p, phase);
        consume_gt<T, ST_ADD, SRC_ATTN, GQ>(r, fill, p.nq_cols, p.d, p.nb_o, nullptr, cx.seq(ph + 1), nullptr, p.xt,
                                            x_in, l, ph + 2, cx, scratch, p, phase - 1);
        mark_phase(p, phase);
        consume_gt<T, ST_SILU, SRC_NORM, GQ>(r, fill, p.d, p.ff, p.nb_gu, p.xt, cx.seq(ph + 2), L.n2, p.ft, 0, l,
                                             ph + 3, cx, scratch, p, phase - 1);
        mark_phase(p, phase);
        consume_gt<T, ST_ADD, SRC_PLAIN, GQ>(r, fill, p.ff, p.d, p.nb_d, p.ft, cx.seq(ph + 3), nullptr, p.xt,
                                             cx.seq(ph + 2), l, ph + 4, cx, scratch, p, phase - 1);
    }
    mark_phase(p, phase);
    consume_gn<T>(r, fill, cx.seq(5 * p.n_layer), scratch, p, step, phase - 1);
    mark_phase(p, phase);
    }
}

// ---------------------------------------------------------------- host
size_t step_layer_bytes() { return sizeof(StepLayer); }

// Host image of one layer's step descriptor: its five tensor maps and norms.
void step_layer_fill(void *dst, const CUtensorMap *maps5, const float *n1, const float *n2, const float *qn,
                     const float *kn) {
    StepLayer L;
    std::memset(&L, 0, sizeof L);
    for (int i = 0; i < 5; ++i) L.maps[i] = maps5[i];
    L.n1 = n1;
    L.n2 = n2;
    L.qn = qn;
    L.kn = kn;
    std::memcpy(dst, &L, sizeof L);
}

int step_max_layers() { return kStMaxLayers; }
int step_stage_bytes() { return kStStageBytes; }
int step_max_splits() { return kStMaxSplits; }

// Shared-memory floats the consumers need after the ring, for a config.
int step_scratch_floats(const ds_model_config *c, int grid, int nb_qkv, int nb_o, int nb_gu, int nb_d) {
    const int es = c->w_dtype == DS_BF16 ? 2 : 4;
    auto slice = [&](int K, int nb) {
        const long long UB = (K + kStBoxRows - 1) / kStBoxRows;
        return (long long)(((UB * nb + grid - 1) / grid + 1) * kStBoxRows);
    };
    const int nq = c->n_qh * c->head_dim;
    long long gt = std::max(std::max(slice(c->d, nb_qkv), slice(nq, nb_o)), std::max(slice(c->d, nb_gu), slice(c->ff, nb_d)));
    gt += kStConsumerWarps * 256 + 256 + 16;
    const int gq = c->n_qh / c->n_kvh;
    const long long at = std::max((long long)kStConsumerWarps * gq * c->head_dim, 2LL * kStMaxSplits * gq + 2 * gq) +
                         2LL * kStConsumerWarps * gq + (long long)gq * c->head_dim +
                         kStConsumerWarps * 40LL + 2LL * gq + 16;  // + per-warp run weights, merged max/sum
    const long long row_bytes = (long long)c->d * es;
    const long long rps = std::max(1LL, (long long)kStStageBytes / row_bytes);
    const long long parts = rps >= kStConsumerWarps ? 1 : kStConsumerWarps / rps;
    const long long rows_cap = (c->vocab + grid - 1) / grid + 1;
    const long long gn = 512 + c->d + rows_cap * parts;
    return (int)std::max(std::max(gt, at), gn);
}

bool step_supported(const ds_model_config *c) {
    const int es = c->w_dtype == DS_BF16 ? 2 : 4;
    if (c->n_layer > kStMaxLayers || c->max_seqs != 1) return false;
    if ((long long)c->d * es > kStStageBytes) return false;
    const int gq = c->n_qh / c->n_kvh;
    if (gq != 1 && gq != 2 && gq != 4 && gq != 8) return false;
    if (c->head_dim > 128) return false;
    return true;
}

// Shared memory of the step kernel with `stages` ring stages.
size_t step_smem_bytes(int stages, int scratch_floats) {
    return (size_t)stages * kStStageBytes + 256 + (size_t)scratch_floats * 4 + 64;
}

// Ring stages that fit beside `scratch_floats` of scratch (0 if none).
int step_stages(int scratch_floats) {
    for (int s = kStMaxStages; s >= 2; --s)
        if (step_smem_bytes(s, scratch_floats) <= kStSmemLimit) return s;
    return 0;
}

// Stages in flight at most (see produce_all); DS_STEP_INFLIGHT overrides the
// default, 0 meaning every free ring slot.
int step_inflight_setting() {
    int v = kStMaxInflight;
    const char *e = std::getenv("DS_STEP_INFLIGHT");
    if (e && *e) v = std::max(0, std::atoi(e));
    return v;
}

// The cap while the attention chain runs, and the gate|up stages it covers;
// DS_STEP_CHAIN_INFLIGHT="cap,gate_up_stages" overrides (cap 0: the plain cap).
void step_chain_setting(int *cap, int *gu_stages) {
    *cap = kStChainInflight;
    *gu_stages = kStChainGuStages;
    const char *e = std::getenv("DS_STEP_CHAIN_INFLIGHT");
    if (e && *e) {
        int c = 0, g = kStChainGuStages;
        const int n = std::sscanf(e, "%d,%d", &c, &g);
        if (n >= 1) *cap = std::max(0, c);
        if (n >= 2) *gu_stages = std::max(0, g);
    }
}

template <typename T, typename KT, int GQ>
static cudaError_t launch_step_t(const StepParams &p, int grid, cudaStream_t stream) {
    const size_t smem = step_smem_bytes(p.stages, p.scratch_floats);
    if (smem > kStSmemLimit) return cudaErrorInvalidValue;
    cudaError_t e =
        cudaFuncSetAttribute(step_kernel<T, KT, GQ>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kStThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, step_kernel<T, KT, GQ>, p);
}

template <typename T, typename KT>
static cudaError_t launch_step_g(const StepParams &p, int gq, int grid, cudaStream_t stream) {
    switch (gq) {
        case 1: return launch_step_t<T, KT, 1>(p, grid, stream);
        case 2: return launch_step_t<T, KT, 2>(p, grid, stream);
        case 4: return launch_step_t<T, KT, 4>(p, grid, stream);
        case 8: return launch_step_t<T, KT, 8>(p, grid, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_step(const void *params, int w_dtype, int kv_dtype, int gq, int grid, cudaStream_t stream) {
    const StepParams &p = *static_cast<const StepParams *>(params);
    if (w_dtype == DS_BF16)
        return kv_dtype == DS_BF16 ? launch_step_g<__nv_bfloat16, __nv_bfloat16>(p, gq, grid, stream)
                                   : launch_step_g<__nv_bfloat16, float>(p, gq, grid, stream);
    return kv_dtype == DS_BF16 ? launch_step_g<float, __nv_bfloat16>(p, gq, grid, stream)
                               : launch_step_g<float, float>(p, gq, grid, stream);
}

}  // namespace ds
