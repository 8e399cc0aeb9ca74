// Iteration-level scheduler (host, C++).
//
// garden.houmin.site Orca notes, 3.1.1 (workflow steps 1-5): the scheduler
// picks the requests to run, asks the engine for ONE iteration, appends each
// returned token to its request, removes the requests that are done and
// frees their memory, and may admit newly arrived requests at the very next
// iteration.  "論文解説: Orca", scheduler algorithm, and the arcsin2 ORCA
// notes, 4.2: FCFS order, a maximum batch size, and a K/V reservation of the
// request's maximum length taken at admission; admission stops at the first
// request that cannot be placed.  The "Continuous Batching" glossary page
// (limits): a cap on the tokens processed in one step.
//
// Readings where the pages are silent: candidates are ordered by
// (arrival, id) and the batch is the longest prefix of that order that fits
// (running requests always come first under FCFS-with-break); a request with
// output length T is done after its T-th token, the initiation iteration
// producing the first; the clock counts iterations and a tick with nothing to
// run does not call the engine.  Request-level mode (the baseline): a batch is
// formed only when the previous batch has completely finished.
//
// Cancellation (houmin 3.1.1: a request that leaves the pool has its memory
// freed at once): between iterations a waiting or running request can be
// dropped; its reservation is freed immediately, it never runs again, and a
// request-level batch whose other members are all done completes then.
// Chunked prefill (optional, iteration-level only): in the FCFS scan a request
// still in its prompt whose remaining prompt exceeds the budget left takes the
// budget left as a chunk (>= 1 token) and the scan stops; only the iteration
// that processes its last prompt token yields a token.
// Pipelining (houmin 3.1.3, n_workers): up to n_workers batches may be open
// (selected, not yet completed); a request in an open batch is not selectable,
// so open batches are disjoint, and completions come oldest first.  The clock
// advances when a batch is selected or an idle tick passes.
#include <algorithm>
#include <cstring>
#include <memory>
#include <new>
#include <numeric>
#include <unordered_map>
#include <vector>

#include "../../include/orca.h"
#include "kvpool.h"

namespace {

enum { W_WAITING = 0, W_RUNNING = 1, W_FINISHED = 2, W_CANCELLED = 3 };

struct Request {
    int64_t id = 0;
    double arrival = 0;
    std::vector<int32_t> prompt;
    int32_t out_len = 0;
    int32_t ctx0 = 0;
    int32_t ctx = 0;
    std::vector<int32_t> generated;
    int32_t pending = 0;
    int64_t kv_off = -1;
    int32_t state = W_WAITING;
    int64_t admitted_at = -1, finished_at = -1;
    int64_t last_iter = -1;  // engine iteration this request last ran in
    int32_t last_index = -1; // its index in that iteration's batch
    int32_t chunk = 0;       // its input rows in the batch being formed
    bool in_flight = false;  // member of an open batch

    // prompt tokens remain to be processed (never for requests entered with ctx0 > 0)
    bool in_prompt() const { return ctx0 == 0 && ctx < (int32_t)prompt.size(); }
    // rows needed to finish the current phase in one iteration
    int32_t n_input() const { return in_prompt() ? (int32_t)prompt.size() - ctx : 1; }
    bool done() const { return (int32_t)generated.size() >= out_len; }
};

bool fcfs_less(const Request *a, const Request *b) {
    if (a->arrival != b->arrival) return a->arrival < b->arrival;
    return a->id < b->id;
}

}  // namespace

struct OpenBatch {
    int64_t clock;  // the clock at its selection
    std::vector<Request *> reqs;
    std::vector<int32_t> chunk;  // each member's input rows in it
};

struct orca_sched {
    orca_sched_config cfg{};
    orca_engine *eng = nullptr;
    std::unique_ptr<orca::KVPool> own_pool;
    std::unordered_map<int64_t, std::unique_ptr<Request>> by_id;
    std::vector<Request *> live;  // unfinished requests, sorted by (arrival, id)
    std::vector<Request *> current_batch;  // request-level mode only
    std::vector<Request *> batch;          // batch being formed by orca_sched_next
    std::vector<OpenBatch> open;           // selected, not yet completed; oldest first
    int64_t clock = 0, iterations = 0, generated = 0, finished = 0, cancelled = 0;
    int64_t feedback_since = 0;  // first iteration run with token feedback on
    // descriptor arrays handed out by orca_sched_next
    std::vector<int64_t> d_id, d_kv;
    std::vector<int32_t> d_phase, d_n, d_ctx, d_tok;

    int32_t reserve_size(const Request &r) const {
        if (cfg.kv_reserve > 0) return cfg.kv_reserve;
        return (r.ctx0 ? r.ctx0 : (int32_t)r.prompt.size()) + r.out_len;
    }

    int kv_alloc(int64_t id, int32_t n, int64_t *off) {
        if (eng) return orca_kv_alloc(eng, id, n, off);
        int64_t o = own_pool->alloc(id, n);
        if (o == -1) return ORCA_ERR_KV_FULL;
        if (o < 0) return ORCA_ERR_INVALID;
        *off = o;
        return ORCA_OK;
    }
    void kv_free(int64_t id) {
        if (eng)
            orca_kv_free(eng, id);
        else
            own_pool->release(id);
    }
    int64_t kv_reserved() const;

    // The longest FCFS prefix of `cands` that fits; admits waiting ones.
    void admit_prefix(const std::vector<Request *> &cands, std::vector<Request *> &out) {
        out.clear();
        int64_t rows = 0;
        for (Request *r : cands) {
            int32_t n = r->n_input();
            if ((int32_t)out.size() >= cfg.max_batch) break;
            if (rows + n > cfg.max_tokens) {
                const int64_t left = cfg.max_tokens - rows;
                if (!(cfg.chunked_prefill && r->in_prompt() && left >= 1)) break;
                n = (int32_t)left;  // a chunk of the prompt; the budget is now used up
            }
            if (r->state == W_WAITING) {
                int64_t off = -1;
                if (kv_alloc(r->id, reserve_size(*r), &off) != ORCA_OK) break;
                r->kv_off = off;
                r->state = W_RUNNING;
                r->admitted_at = clock;
            }
            r->chunk = n;
            out.push_back(r);
            rows += n;
        }
    }

    // Request-level: the batch completes when every member is done or
    // cancelled; the reservations still held are released then.
    void close_request_batch() {
        if (cfg.mode != 1 || current_batch.empty()) return;
        for (Request *r : current_batch)
            if (!r->done() && r->state != W_CANCELLED) return;
        for (Request *r : current_batch)
            if (r->state != W_CANCELLED) kv_free(r->id);
        current_batch.clear();
    }
};

int64_t orca_sched::kv_reserved() const {
    int64_t t = 0;
    for (const Request *r : live)
        if (r->state == W_RUNNING) t += reserve_size(*r);
    if (cfg.mode == 1)
        for (const Request *r : current_batch)
            if (r->state == W_FINISHED) t += reserve_size(*r);
    return t;
}

extern "C" {

int orca_sched_create(const orca_sched_config *cfg, orca_engine *eng, orca_sched **out) {
    if (!cfg || !out) return ORCA_ERR_INVALID;
    if (cfg->max_batch <= 0 || cfg->max_tokens <= 0 || cfg->kv_reserve < 0 || (cfg->mode != 0 && cfg->mode != 1) ||
        (cfg->chunked_prefill != 0 && cfg->chunked_prefill != 1) || (cfg->chunked_prefill && cfg->mode != 0))
        return ORCA_ERR_INVALID;
    // pipelining: iteration-level only, and increment inputs must be literal tokens
    const int32_t nw = cfg->n_workers ? cfg->n_workers : 1;
    if (nw < 1 || nw > 64 || (nw > 1 && (cfg->mode != 0 || cfg->token_feedback))) return ORCA_ERR_INVALID;
    if (!eng && cfg->kv_slots <= 0) return ORCA_ERR_INVALID;
    orca_sched *s = new (std::nothrow) orca_sched();
    if (!s) return ORCA_ERR_OOM;
    s->cfg = *cfg;
    s->cfg.n_workers = nw;
    s->eng = eng;
    if (!eng) s->own_pool.reset(new orca::KVPool(cfg->kv_slots));
    *out = s;
    return ORCA_OK;
}

int orca_sched_destroy(orca_sched *s) {
    if (!s) return ORCA_ERR_INVALID;
    // return every reservation this scheduler still holds to the engine's pool
    if (s->eng)
        for (auto &kv : s->by_id)
            if (kv.second->kv_off >= 0 && (kv.second->state == W_RUNNING ||
                                           (s->cfg.mode == 1 && kv.second->state == W_FINISHED &&
                                            std::find(s->current_batch.begin(), s->current_batch.end(),
                                                      kv.second.get()) != s->current_batch.end())))
                orca_kv_free(s->eng, kv.first);
    delete s;
    return ORCA_OK;
}

int orca_sched_submit(orca_sched *s, int64_t id, double arrival, const int32_t *prompt, int32_t prompt_len,
                      int32_t out_len, int32_t ctx0, int64_t *out_kv_offset) {
    if (!s || !prompt || prompt_len < 1 || out_len < 1 || ctx0 < 0) return ORCA_ERR_INVALID;
    if (s->by_id.count(id)) return ORCA_ERR_INVALID;
    std::unique_ptr<Request> r(new (std::nothrow) Request());
    if (!r) return ORCA_ERR_OOM;
    r->id = id;
    r->arrival = arrival;
    r->prompt.assign(prompt, prompt + prompt_len);
    r->out_len = out_len;
    r->ctx0 = ctx0;
    int64_t need = ctx0 ? (int64_t)ctx0 + out_len : (int64_t)prompt_len + out_len - 1;
    if ((prompt_len > s->cfg.max_tokens && !s->cfg.chunked_prefill) || need > s->reserve_size(*r))
        return ORCA_ERR_INVALID;
    if (ctx0) {
        if (prompt_len != 1) return ORCA_ERR_INVALID;
        int64_t off = -1;
        int rc = s->kv_alloc(id, s->reserve_size(*r), &off);
        if (rc != ORCA_OK) return rc;
        r->kv_off = off;
        r->ctx = ctx0;
        r->pending = prompt[0];
        r->state = W_RUNNING;
        r->admitted_at = -1;
        if (out_kv_offset) *out_kv_offset = off;
    } else if (out_kv_offset) {
        *out_kv_offset = -1;
    }
    Request *p = r.get();
    s->by_id[id] = std::move(r);
    auto pos = std::upper_bound(s->live.begin(), s->live.end(), p, fcfs_less);
    s->live.insert(pos, p);
    return ORCA_OK;
}

int orca_sched_set_token_feedback(orca_sched *s, int32_t enable) {
    if (!s || (enable && s->cfg.n_workers > 1)) return ORCA_ERR_INVALID;
    if (enable && !s->cfg.token_feedback) s->feedback_since = s->iterations;
    s->cfg.token_feedback = enable ? 1 : 0;
    return ORCA_OK;
}

int orca_sched_next(orca_sched *s, orca_batch *out, int32_t *status) {
    if (!s || !out || !status) return ORCA_ERR_INVALID;
    if ((int32_t)s->open.size() >= s->cfg.n_workers) return ORCA_ERR_INVALID;  // complete one first
    if (s->live.empty() && s->open.empty()) {
        *status = 2;
        return ORCA_OK;
    }
    const double k = (double)s->clock;
    std::vector<Request *> cands;
    for (Request *r : s->live) {
        if (r->arrival > k) break;  // live is sorted by arrival first
        if (r->in_flight) continue;
        if (s->cfg.mode == 1 && r->state != W_WAITING) continue;
        cands.push_back(r);  // (live holds no finished or cancelled request)
    }
    if (s->cfg.mode == 0) {
        s->admit_prefix(cands, s->batch);
    } else {
        if (s->current_batch.empty()) s->admit_prefix(cands, s->current_batch);
        s->batch.clear();
        for (Request *r : s->current_batch)
            if (r->state == W_RUNNING && !r->done()) {
                r->chunk = r->n_input();
                s->batch.push_back(r);
            }
    }
    if (s->batch.empty()) {
        if (!s->open.empty()) {  // all runnable requests are in flight: complete one first
            *status = 3;
            return ORCA_OK;
        }
        s->clock++;
        *status = 0;
        return ORCA_OK;
    }
    size_t B = s->batch.size();
    s->d_id.resize(B);
    s->d_kv.resize(B);
    s->d_phase.resize(B);
    s->d_n.resize(B);
    s->d_ctx.resize(B);
    s->d_tok.clear();
    for (size_t i = 0; i < B; ++i) {
        Request *r = s->batch[i];
        s->d_id[i] = r->id;
        s->d_kv[i] = r->kv_off;
        s->d_phase[i] = r->ctx == 0 ? 0 : 1;
        s->d_n[i] = r->chunk;
        s->d_ctx[i] = r->ctx;
        if (r->in_prompt()) {
            s->d_tok.insert(s->d_tok.end(), r->prompt.begin() + r->ctx, r->prompt.begin() + r->ctx + r->chunk);
        } else if (s->cfg.token_feedback && r->last_iter == s->iterations - 1 && r->last_iter >= s->feedback_since) {
            s->d_tok.push_back(-1 - r->last_index);
        } else {
            s->d_tok.push_back(r->pending);
        }
    }
    out->n_req = (int32_t)B;
    out->request_id = s->d_id.data();
    out->phase = s->d_phase.data();
    out->n_input = s->d_n.data();
    out->ctx_len = s->d_ctx.data();
    out->kv_offset = s->d_kv.data();
    out->tokens = s->d_tok.data();
    OpenBatch ob{s->clock, s->batch, {}};
    for (Request *r : s->batch) {
        r->in_flight = true;
        ob.chunk.push_back(r->chunk);
    }
    s->open.push_back(std::move(ob));
    s->clock++;
    *status = 1;
    return ORCA_OK;
}

int orca_sched_complete(orca_sched *s, const int32_t *next_tokens) {
    if (!s || !next_tokens || s->open.empty()) return ORCA_ERR_INVALID;
    OpenBatch ob = std::move(s->open.front());  // the oldest open batch
    s->open.erase(s->open.begin());
    for (size_t i = 0; i < ob.reqs.size(); ++i) {
        Request *r = ob.reqs[i];
        r->in_flight = false;
        r->ctx += ob.chunk[i];
        r->last_iter = s->iterations;
        r->last_index = (int32_t)i;
        if (r->in_prompt()) continue;  // a prompt chunk before the last: its output is not a token
        r->generated.push_back(next_tokens[i]);
        r->pending = next_tokens[i];
        s->generated++;
        if (r->done()) {
            r->state = W_FINISHED;
            r->finished_at = ob.clock;
            s->finished++;
            if (s->cfg.mode == 0) s->kv_free(r->id);
        }
    }
    s->close_request_batch();
    s->live.erase(std::remove_if(s->live.begin(), s->live.end(), [](Request *r) { return r->state == W_FINISHED; }),
                  s->live.end());
    s->iterations++;
    return ORCA_OK;
}

int orca_sched_cancel(orca_sched *s, int64_t id) {
    if (!s) return ORCA_ERR_INVALID;
    auto it = s->by_id.find(id);
    if (it == s->by_id.end()) return ORCA_ERR_NOT_FOUND;
    Request *r = it->second.get();
    if (r->in_flight) return ORCA_ERR_INVALID;  // its batch is still open
    if (r->state != W_WAITING && r->state != W_RUNNING) return ORCA_ERR_INVALID;
    if (r->kv_off >= 0) s->kv_free(r->id);
    r->state = W_CANCELLED;
    s->cancelled++;
    s->live.erase(std::remove(s->live.begin(), s->live.end(), r), s->live.end());
    s->close_request_batch();
    return ORCA_OK;
}

int orca_sched_stats_get(orca_sched *s, orca_sched_stats *out) {
    if (!s || !out) return ORCA_ERR_INVALID;
    out->clock = s->clock;
    out->iterations = s->iterations;
    out->generated = s->generated;
    out->finished = s->finished;
    out->cancelled = s->cancelled;
    int64_t waiting = 0, running = 0;
    for (Request *r : s->live) (r->state == W_WAITING ? waiting : running)++;
    out->waiting = waiting;
    out->running = running;
    out->kv_reserved = s->kv_reserved();
    return ORCA_OK;
}

int orca_sched_request_get(orca_sched *s, int64_t id, orca_request_info *out) {
    if (!s || !out) return ORCA_ERR_INVALID;
    auto it = s->by_id.find(id);
    if (it == s->by_id.end()) return ORCA_ERR_NOT_FOUND;
    const Request &r = *it->second;
    out->id = r.id;
    out->kv_offset = r.kv_off;
    out->state = r.state;
    out->ctx_len = r.ctx;
    out->n_generated = (int32_t)r.generated.size();
    out->admitted_at = r.admitted_at;
    out->finished_at = r.finished_at;
    return ORCA_OK;
}

int orca_sched_request_tokens(orca_sched *s, int64_t id, int32_t *out, int32_t cap, int32_t *n_out) {
    if (!s || (!out && cap > 0) || !n_out) return ORCA_ERR_INVALID;
    auto it = s->by_id.find(id);
    if (it == s->by_id.end()) return ORCA_ERR_NOT_FOUND;
    const auto &g = it->second->generated;
    int32_t n = (int32_t)std::min<size_t>(g.size(), (size_t)std::max(cap, 0));
    if (n) std::memcpy(out, g.data(), sizeof(int32_t) * n);
    *n_out = (int32_t)g.size();
    return ORCA_OK;
}

int orca_sched_run(orca_sched *s, int64_t max_iterations) {
    if (!s || !s->eng) return ORCA_ERR_INVALID;
    // copies of the open batches' descriptors (the scheduler reuses its arrays)
    struct Desc {
        std::vector<int64_t> id, kv;
        std::vector<int32_t> phase, n, ctx, tok;
        orca_batch view() {
            return orca_batch{(int32_t)id.size(), id.data(), phase.data(), n.data(), ctx.data(), kv.data(), tok.data()};
        }
    };
    std::vector<Desc> queued;  // oldest first
    auto abandon = [&]() {      // the open batches are dropped; the requests keep their state
        for (OpenBatch &ob : s->open)
            for (Request *r : ob.reqs) r->in_flight = false;
        s->open.clear();
    };
    std::vector<int32_t> next;
    int64_t done_iters = 0;
    while (done_iters < max_iterations) {
        // select until n_workers batches are open or nothing more can be selected now
        while ((int32_t)s->open.size() < s->cfg.n_workers &&
               done_iters + (int64_t)queued.size() < max_iterations) {
            orca_batch b{};
            int32_t status = 0;
            int rc = orca_sched_next(s, &b, &status);
            if (rc != ORCA_OK) {
                abandon();
                return rc;
            }
            if (status == 0) continue;  // idle tick
            if (status != 1) break;     // 2: every request finished; 3: wait for an open batch
            const int64_t rows = std::accumulate(b.n_input, b.n_input + b.n_req, (int64_t)0);
            queued.push_back(Desc{{b.request_id, b.request_id + b.n_req}, {b.kv_offset, b.kv_offset + b.n_req},
                                  {b.phase, b.phase + b.n_req}, {b.n_input, b.n_input + b.n_req},
                                  {b.ctx_len, b.ctx_len + b.n_req}, {b.tokens, b.tokens + rows}});
        }
        if (queued.empty()) break;
        orca_batch b = queued.front().view();
        next.resize(b.n_req);
        int rc = orca_run_iteration(s->eng, &b, next.data());
        if (rc != ORCA_OK) {
            abandon();
            return rc;
        }
        rc = orca_sched_complete(s, next.data());
        queued.erase(queued.begin());
        if (rc != ORCA_OK) return rc;
        ++done_iters;
    }
    return ORCA_OK;
}

}  // extern "C"
