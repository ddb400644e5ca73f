// scheduler.cpp -- the host continuous-batching scheduler of include/pa_sched.h.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <deque>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/pa.h"
#include "../../include/pa_alloc.h"
#include "../../include/pa_sched.h"

namespace {

struct Req {
    int64_t id;
    int n;          // prompt rows
    int m;          // tokens to produce
    int prefilled;  // prompt rows in the cache
    int generated;  // tokens produced (the last one not yet in the cache)
};

struct Planned {
    int64_t id;
    int rows;      // rows this step
    int len_after; // context after the step's append
    bool decode;
};

}  // namespace

struct pa_scheduler {
    pa_sched_params p{};
    int block_size = 0, num_blocks = 0;
    pa_block_allocator *alloc = nullptr;
    std::deque<Req> queue;
    std::vector<Req> running;               // admission order
    std::unordered_map<int64_t, int> known;  // 1 queued, 2 running
    int waiting = 0;                         // steps since the last admission
    std::vector<Planned> plan;
    bool planned = false;

    long long reserve(const Req &r) const {  // block-aligned prompt + max_new_tokens
        const long long t = (long long)r.n + r.m;
        return (t + block_size - 1) / block_size * block_size;
    }
};

extern "C" {

pa_scheduler *pa_sched_create(const pa_sched_params *params, int num_blocks, int block_size) {
    if (!params || num_blocks <= 0 || block_size <= 0) return nullptr;
    const pa_sched_params &p = *params;
    if (p.max_batch_prefill_tokens <= 0 || p.max_batch_total_tokens < 0 || p.max_waiting_tokens < 0 ||
        !(p.waiting_served_ratio >= 0.f) || p.max_batch_size < 0 || p.max_input_tokens <= 0 ||
        p.max_total_tokens <= 0)
        return nullptr;
    pa_scheduler *s = new (std::nothrow) pa_scheduler;
    if (!s) return nullptr;
    s->p = p;
    if (s->p.max_batch_total_tokens == 0 || (long long)s->p.max_batch_total_tokens > (long long)num_blocks * block_size)
        s->p.max_batch_total_tokens = num_blocks * block_size;
    s->block_size = block_size;
    s->num_blocks = num_blocks;
    s->alloc = pa_alloc_create(num_blocks, block_size, nullptr);
    if (!s->alloc) {
        delete s;
        return nullptr;
    }
    return s;
}

void pa_sched_destroy(pa_scheduler *s) {
    if (!s) return;
    pa_alloc_destroy(s->alloc);
    delete s;
}

int pa_sched_submit(pa_scheduler *s, int64_t request_id, int input_tokens, int max_new_tokens) {
    if (!s || s->known.count(request_id) || input_tokens < 1 || max_new_tokens < 1 ||
        input_tokens > s->p.max_input_tokens || (long long)input_tokens + max_new_tokens > s->p.max_total_tokens)
        return PA_ERR_INVALID_ARG;
    // without chunking a prompt is prefilled whole: it must fit one prefill
    if (!s->p.chunking && input_tokens > s->p.max_batch_prefill_tokens) return PA_ERR_INVALID_ARG;
    Req r{request_id, input_tokens, max_new_tokens, 0, 0};
    if (s->reserve(r) > s->p.max_batch_total_tokens) return PA_ERR_INVALID_ARG;  // could never run
    s->queue.push_back(r);
    s->known[request_id] = 1;
    return PA_OK;
}

int pa_sched_cancel(pa_scheduler *s, int64_t request_id) {
    if (!s) return PA_ERR_INVALID_ARG;
    auto it = s->known.find(request_id);
    if (it == s->known.end() || s->planned) return PA_ERR_INVALID_ARG;
    if (it->second == 1) {
        for (auto q = s->queue.begin(); q != s->queue.end(); ++q)
            if (q->id == request_id) {
                s->queue.erase(q);
                break;
            }
    } else {
        for (auto r = s->running.begin(); r != s->running.end(); ++r)
            if (r->id == request_id) {
                s->running.erase(r);
                break;
            }
        if (pa_alloc_num_blocks_of(s->alloc, request_id) > 0) pa_alloc_release(s->alloc, request_id);
    }
    s->known.erase(it);
    return PA_OK;
}

int pa_sched_plan(pa_scheduler *s, int max_seqs, int max_tokens, int width, int64_t *seq_ids,
                  int32_t *q_start_loc, int32_t *seq_lens, int32_t *block_table, int32_t *slot_mapping,
                  int *num_seqs, int *num_decode, int *num_tokens) {
    if (!s || s->planned || max_seqs < 0 || max_tokens < 0 || width <= 0 || !num_seqs || !num_decode ||
        !num_tokens)
        return PA_ERR_INVALID_ARG;
    const pa_sched_params &p = s->p;
    std::vector<Planned> plan;
    // every running request whose prompt is done decodes one token
    int decode_rows = 0;
    for (const Req &r : s->running)
        if (r.prefilled == r.n) {
            plan.push_back({r.id, 1, r.n + r.generated, true});
            ++decode_rows;
        }
    long long reserved = 0;
    for (const Req &r : s->running) reserved += s->reserve(r);
    const long long token_budget = (long long)p.max_batch_total_tokens - reserved;
    const int max_size = p.max_batch_size > 0 ? p.max_batch_size - (int)s->running.size() : 1 << 30;
    size_t take = 0;
    if (p.chunking) {
        long long budget = (long long)p.max_batch_prefill_tokens - decode_rows;
        for (const Req &r : s->running)  // prompts already under way go first
            if (r.prefilled < r.n && budget > 0) {
                const int c = (int)std::min<long long>(r.n - r.prefilled, budget);
                plan.push_back({r.id, c, r.prefilled + c, false});
                budget -= c;
            }
        long long res = 0;
        while (take < s->queue.size() && budget > 0 && (int)take < max_size) {
            const Req &e = s->queue[take];
            if (res + s->reserve(e) > token_budget) break;
            const int c = (int)std::min<long long>(e.n, budget);
            plan.push_back({e.id, c, c, false});
            budget -= c;
            res += s->reserve(e);
            ++take;
        }
    } else {
        // min_size: none when nothing runs or the wait is exceeded
        const bool forced = s->running.empty() || s->waiting >= p.max_waiting_tokens;
        const long long min_size =
            forced ? 0 : (long long)std::floor((double)s->running.size() * (double)p.waiting_served_ratio);
        if ((long long)s->queue.size() >= min_size) {
            long long pre = 0, res = 0;
            while (take < s->queue.size() && (int)take < max_size) {
                const Req &e = s->queue[take];
                if (pre + e.n > p.max_batch_prefill_tokens || res + s->reserve(e) > token_budget) break;
                pre += e.n;
                res += s->reserve(e);
                ++take;
            }
            if ((long long)take < min_size) take = 0;
        }
        for (size_t i = 0; i < take; ++i) plan.push_back({s->queue[i].id, s->queue[i].n, s->queue[i].n, false});
    }
    const int S = (int)plan.size();
    long long T = 0;
    for (const Planned &x : plan) T += x.rows;
    if (S > max_seqs || T > max_tokens) return PA_ERR_INVALID_ARG;
    for (const Planned &x : plan)
        if ((x.len_after + s->block_size - 1) / s->block_size > width) return PA_ERR_INVALID_ARG;
    // blocks for the step's new tokens (the reservations keep this within the pool)
    for (const Planned &x : plan) {
        const int rc = pa_alloc_ensure(s->alloc, x.id, x.len_after);
        if (rc) {  // not expected (reservations fit the pool): undo the admissions' blocks
            for (size_t i = 0; i < take; ++i)
                if (pa_alloc_num_blocks_of(s->alloc, s->queue[i].id) > 0) pa_alloc_release(s->alloc, s->queue[i].id);
            return rc;
        }
    }
    std::vector<int32_t> n_new(S), total(S);
    q_start_loc[0] = 0;
    for (int i = 0; i < S; ++i) {
        seq_ids[i] = plan[i].id;
        n_new[i] = plan[i].rows;
        total[i] = plan[i].len_after;
        seq_lens[i] = plan[i].len_after;
        q_start_loc[i + 1] = q_start_loc[i] + plan[i].rows;
    }
    int rc = S ? pa_alloc_block_table(s->alloc, seq_ids, S, width, -1, block_table) : PA_OK;
    if (!rc && S) rc = pa_alloc_slot_mapping(s->alloc, seq_ids, n_new.data(), total.data(), S, slot_mapping);
    if (rc) return rc;
    // admitted requests join the running batch now (their blocks exist)
    for (size_t i = 0; i < take; ++i) {
        s->running.push_back(s->queue.front());
        s->known[s->queue.front().id] = 2;
        s->queue.pop_front();
    }
    if (take > 0) s->waiting = 0;
    else if (!s->running.empty()) ++s->waiting;
    *num_seqs = S;
    *num_decode = decode_rows;
    *num_tokens = (int)T;
    s->plan = plan;
    s->planned = S > 0;
    return PA_OK;
}

int pa_sched_commit(pa_scheduler *s, int64_t *finished_out, int max_finished, int *num_finished) {
    if (!s || !num_finished) return PA_ERR_INVALID_ARG;
    int nf = 0;
    if (s->planned) {
        std::unordered_map<int64_t, const Planned *> by_id;
        for (const Planned &x : s->plan) by_id[x.id] = &x;
        std::vector<Req> keep;
        keep.reserve(s->running.size());
        for (Req &r : s->running) {
            auto it = by_id.find(r.id);
            if (it != by_id.end()) {
                const Planned &x = *it->second;
                if (x.decode) {
                    ++r.generated;
                } else {
                    r.prefilled += x.rows;
                    if (r.prefilled == r.n) r.generated = 1;
                }
            }
            if (r.generated >= r.m) {
                pa_alloc_release(s->alloc, r.id);
                s->known.erase(r.id);
                if (finished_out && nf < max_finished) finished_out[nf] = r.id;
                ++nf;
            } else {
                keep.push_back(r);
            }
        }
        s->running.swap(keep);
    }
    s->plan.clear();
    s->planned = false;
    *num_finished = nf;
    return PA_OK;
}

int pa_sched_stats(const pa_scheduler *s, int *queued, int *running, int *free_blocks, int *waiting_steps) {
    if (!s) return PA_ERR_INVALID_ARG;
    if (queued) *queued = (int)s->queue.size();
    if (running) *running = (int)s->running.size();
    if (free_blocks) *free_blocks = pa_alloc_num_free(s->alloc);
    if (waiting_steps) *waiting_steps = s->waiting;
    return PA_OK;
}

}  // extern "C"
