// Continuous-batching scheduler slice over the paged K/V pool ("Inside the
// engine", section 2: admission, chunks, preemption, resume).  Host code
// only: it decides which requests run in a step, as prompt chunks or decode
// rows, and which pool blocks each request's block-table row maps.  The
// policy, as the header states it, in the terms of a pool whose blocks hold
// every layer's K/V of block_tokens positions:
//   admission  strictly first come first served over the waiting requests
//              (the preempted ones first, by preemption order); the head is
//              admitted when a row is free and the free blocks cover all of
//              its tokens plus the headroom, which it takes then;
//   chunks     uncached tokens run in chunks of at most `chunk`; the row that
//              reaches a request's last token yields its next token;
//   preemption a decode row whose position needs a block takes the lowest
//              free one; with none free the youngest running request gives
//              up its blocks and row (and its cache) until one is free or
//              the request itself was the youngest; older requests go first;
//   resume     a preempted request recomputes its prompt and generated
//              tokens through the chunked path once re-admitted.
#include <algorithm>
#include <cstdint>
#include <map>
#include <set>
#include <vector>

#include "decode_step.h"

namespace {

enum { kWaiting = 0, kRunning = 1, kFinished = 2 };

struct Request {
    int64_t arrival = 0;  // submission order: smaller is older
    int32_t prompt = 0, max_new = 0, generated = 0, cached = 0;
    int32_t slot = -1;
    int state = kWaiting;
    std::vector<int32_t> blocks;
    int32_t tokens() const { return prompt + generated; }
};

int32_t blocks_for(int64_t positions, int32_t bt) { return (int32_t)((positions + bt - 1) / bt); }

}  // namespace

struct ds_sched {
    ds_sched_config cfg;
    std::set<int32_t> free_blocks, free_slots;
    std::map<int64_t, Request> reqs;
    std::vector<int64_t> running;      // oldest first
    std::vector<int64_t> waiting_pre;  // first preempted first
    std::vector<int64_t> waiting_new;  // first submitted first
    int64_t n_submitted = 0, n_preemptions = 0, n_finished = 0;
    bool planned = false;
    std::vector<ds_sched_row> rows;  // the plan awaiting its commit

    bool admit(int64_t id) {
        Request &r = reqs[id];
        const int32_t need = blocks_for(r.tokens(), cfg.block_tokens);
        if (free_slots.empty() || (int64_t)free_blocks.size() < (int64_t)need + cfg.headroom_blocks) return false;
        r.slot = *free_slots.begin();
        free_slots.erase(free_slots.begin());
        r.blocks.clear();
        for (int32_t i = 0; i < need; ++i) {
            r.blocks.push_back(*free_blocks.begin());
            free_blocks.erase(free_blocks.begin());
        }
        r.cached = 0;
        r.state = kRunning;
        auto at = std::upper_bound(running.begin(), running.end(), id,
                                   [&](int64_t a, int64_t b) { return reqs[a].arrival < reqs[b].arrival; });
        running.insert(at, id);
        return true;
    }

    void release(Request &r) {
        for (int32_t b : r.blocks) free_blocks.insert(b);
        r.blocks.clear();
        if (r.slot >= 0) free_slots.insert(r.slot);
        r.slot = -1;
    }

    void preempt_youngest(std::vector<int64_t> &out) {
        const int64_t id = running.back();
        running.pop_back();
        Request &r = reqs[id];
        release(r);
        r.cached = 0;
        r.state = kWaiting;
        waiting_pre.push_back(id);
        ++n_preemptions;
        out.push_back(id);
    }
};

extern "C" DS_API int ds_sched_create(const ds_sched_config *cfg, ds_sched **out) {
    if (!cfg || !out) return DS_BAD_ARGUMENT;
    *out = nullptr;
    if (cfg->n_blocks < 1 || cfg->block_tokens < 1 || cfg->max_blocks < 1 || cfg->max_running < 1 ||
        cfg->chunk < 1 || cfg->headroom_blocks < 0)
        return DS_EMPTY_DIMENSION;
    if (cfg->n_blocks > DS_MAX_DIM || cfg->block_tokens > DS_MAX_DIM || cfg->max_blocks > DS_MAX_DIM ||
        cfg->max_running > DS_MAX_DIM || cfg->chunk > DS_MAX_DIM || cfg->headroom_blocks > DS_MAX_DIM ||
        (int64_t)cfg->block_tokens * cfg->max_blocks > DS_MAX_DIM)
        return DS_DIMENSION_TOO_LARGE;
    ds_sched *s = new ds_sched();
    s->cfg = *cfg;
    for (int32_t b = 0; b < cfg->n_blocks; ++b) s->free_blocks.insert(b);
    for (int32_t i = 0; i < cfg->max_running; ++i) s->free_slots.insert(i);
    *out = s;
    return DS_OK;
}

extern "C" DS_API void ds_sched_destroy(ds_sched *s) { delete s; }

extern "C" DS_API int ds_sched_submit(ds_sched *s, int64_t request, int32_t prompt_len, int32_t max_new) {
    if (!s) return DS_BAD_ARGUMENT;
    if (prompt_len < 1 || max_new < 1) return DS_EMPTY_DIMENSION;
    auto it = s->reqs.find(request);
    if (it != s->reqs.end() && it->second.state != kFinished) return DS_BAD_ARGUMENT;
    // every position the request will feed, in one row and in the pool
    const int64_t positions = (int64_t)prompt_len + max_new - 1;
    if (positions > (int64_t)s->cfg.max_blocks * s->cfg.block_tokens ||
        (int64_t)blocks_for(positions, s->cfg.block_tokens) + s->cfg.headroom_blocks > s->cfg.n_blocks)
        return DS_CACHE_CAPACITY_EXCEEDED;
    Request r;
    r.arrival = s->n_submitted++;
    r.prompt = prompt_len;
    r.max_new = max_new;
    s->reqs[request] = r;
    s->waiting_new.push_back(request);
    return DS_OK;
}

extern "C" DS_API int ds_sched_plan(ds_sched *s, ds_sched_row *rows, int32_t cap, int32_t *n_rows,
                                    int32_t *block_table, int64_t *preempted, int32_t *n_preempted) {
    if (!s || !rows || !n_rows || !block_table) return DS_BAD_ARGUMENT;
    if (s->planned) return DS_BAD_ARGUMENT;
    if (cap < s->cfg.max_running) return DS_WORKSPACE_TOO_SMALL;
    const int32_t bt = s->cfg.block_tokens;
    // admission: preempted requests first; new ones only once none waits
    while (!s->waiting_pre.empty() && s->admit(s->waiting_pre.front())) s->waiting_pre.erase(s->waiting_pre.begin());
    if (s->waiting_pre.empty())
        while (!s->waiting_new.empty() && s->admit(s->waiting_new.front()))
            s->waiting_new.erase(s->waiting_new.begin());
    // decode rows claim the block of their position, oldest first
    std::vector<int64_t> gone;
    for (size_t i = 0; i < s->running.size(); ++i) {
        const int64_t id = s->running[i];
        Request &r = s->reqs[id];
        if (r.cached != r.tokens() - 1) continue;  // prefill: its blocks cover all its tokens
        if ((int64_t)r.blocks.size() * bt > r.cached) continue;
        bool self = false;
        while (s->free_blocks.empty()) {
            self = s->running.back() == id;
            s->preempt_youngest(gone);
            if (self) break;
        }
        if (self) break;  // it was the youngest: nothing younger is left to plan
        r.blocks.push_back(*s->free_blocks.begin());
        s->free_blocks.erase(s->free_blocks.begin());
    }
    // one row per running request, oldest first
    s->rows.clear();
    for (int64_t id : s->running) {
        const Request &r = s->reqs[id];
        ds_sched_row row;
        row.request = id;
        row.slot = r.slot;
        row.offset = r.cached;
        row.count = std::min(s->cfg.chunk, r.tokens() - r.cached);
        row.yields = r.cached + row.count == r.tokens() ? 1 : 0;
        row.decode = (r.cached == r.tokens() - 1 && r.generated >= 1) ? 1 : 0;
        s->rows.push_back(row);
    }
    const int64_t width = s->cfg.max_blocks;
    std::fill(block_table, block_table + (int64_t)s->cfg.max_running * width, -1);
    for (int64_t id : s->running) {
        const Request &r = s->reqs[id];
        std::copy(r.blocks.begin(), r.blocks.end(), block_table + (int64_t)r.slot * width);
    }
    std::copy(s->rows.begin(), s->rows.end(), rows);
    *n_rows = (int32_t)s->rows.size();
    if (preempted) std::copy(gone.begin(), gone.end(), preempted);
    if (n_preempted) *n_preempted = (int32_t)gone.size();
    s->planned = true;
    return DS_OK;
}

extern "C" DS_API int ds_sched_commit(ds_sched *s, const int64_t *finished, int32_t n_finished) {
    if (!s || (n_finished > 0 && !finished) || n_finished < 0) return DS_BAD_ARGUMENT;
    if (!s->planned) return DS_BAD_ARGUMENT;
    for (const ds_sched_row &row : s->rows) {
        Request &r = s->reqs[row.request];
        r.cached += row.count;
        if (row.yields) r.generated += 1;
    }
    std::set<int64_t> stop(finished, finished + std::max(n_finished, 0));
    auto done = [&](int64_t id) {
        Request &r = s->reqs[id];
        if (r.generated < r.max_new && !stop.count(id)) return false;
        s->release(r);
        r.state = kFinished;
        ++s->n_finished;
        return true;
    };
    s->running.erase(std::remove_if(s->running.begin(), s->running.end(), done), s->running.end());
    // a request reported finished while it waits leaves the queue too
    s->waiting_pre.erase(std::remove_if(s->waiting_pre.begin(), s->waiting_pre.end(),
                                        [&](int64_t id) { return stop.count(id) && done(id); }),
                         s->waiting_pre.end());
    s->waiting_new.erase(std::remove_if(s->waiting_new.begin(), s->waiting_new.end(),
                                        [&](int64_t id) { return stop.count(id) && done(id); }),
                         s->waiting_new.end());
    s->planned = false;
    return DS_OK;
}

extern "C" DS_API int ds_sched_stats(const ds_sched *s, int64_t *out5) {
    if (!s || !out5) return DS_BAD_ARGUMENT;
    out5[0] = (int64_t)s->free_blocks.size();
    out5[1] = (int64_t)s->running.size();
    out5[2] = (int64_t)(s->waiting_pre.size() + s->waiting_new.size());
    out5[3] = s->n_finished;
    out5[4] = s->n_preemptions;
    return DS_OK;
}

extern "C" DS_API int64_t ds_sched_generated(const ds_sched *s, int64_t request) {
    if (!s) return -1;
    auto it = s->reqs.find(request);
    return it == s->reqs.end() ? -1 : it->second.generated;
}
