// sched.cpp -- request scheduler around Compressed PagedAttention (host).
//
// Zipage paper §4.1 (budget and trigger), §4.2/§4.3 (query slots,
// constrained and hybrid scheduling, Fig. 2), §4.4 (prefix sharing and its
// preemption rule), §4.5 (compressing requests sit out decode), Limitations
// (a budget per request).  The rules and the readings where the pages leave
// a step open are listed in zp_sched.h.  Blocks come from the library's pool
// (lowest free id first) and compaction targets from its planner.
#include <algorithm>
#include <deque>
#include <unordered_map>
#include <vector>

#include "zp_internal.h"
#include "zp_sched.h"

using zp::fail;
using zp::ok;

namespace {

struct Request {
    int32_t id, prompt, output, group, prefix_len, budget;  // budget: N_i
    int32_t state = ZP_REQ_WAITING;
    int32_t len = 0, generated = 0, slot = -1, preemptions = 0;
    bool compressed = false, want_compress = false, holds_prefix = false;
    std::vector<int32_t> table;
    // planned compaction (valid while compressing)
    std::vector<int32_t> new_table, dropped;
};

struct Prefix {
    std::vector<int32_t> blocks;
    int32_t holders = 0;
};

struct Started {
    int32_t id, len, slot, k, first;
    std::vector<int32_t> table, targets;
};

}  // namespace

struct zp_sched {
    zp_sched_config c;
    zp_pool *pool;
    std::deque<Request> reqs;                   // element addresses stay valid as requests are added
    std::unordered_map<int32_t, size_t> index;  // id -> reqs position
    std::deque<Request *> waiting;
    std::vector<Request *> running;  // queue order = admission order
    std::vector<char> slot_used;
    std::unordered_map<int32_t, Prefix> prefix;
    std::unordered_map<int32_t, int32_t> group_len;  // prefix group -> its prefix length
    std::vector<Started> started;
    int last_kind = ZP_STEP_IDLE;
    std::vector<Request *> last;  // requests of the last step

    int32_t free_blocks() const { return zp_pool_num_free(pool); }
    int32_t refcount(int32_t blk) const { return zp_pool_refcount(pool, blk); }

    bool alloc(int32_t n, std::vector<int32_t> &into) {
        if (n <= 0) return true;
        std::vector<int32_t> ids((size_t)n);
        if (zp_pool_alloc(pool, n, ids.data()) != ZP_OK) return false;
        into.insert(into.end(), ids.begin(), ids.end());
        return true;
    }
    void release(const std::vector<int32_t> &blocks) {
        if (!blocks.empty()) zp_pool_release(pool, (int32_t)blocks.size(), blocks.data());
    }

    void leave_prefix(Request *r) {
        if (!r->holds_prefix) return;
        auto it = prefix.find(r->group);
        if (it != prefix.end() && --it->second.holders == 0) prefix.erase(it);
        r->holds_prefix = false;
    }
    void free_slot(Request *r) {
        if (r->slot >= 0) slot_used[(size_t)r->slot] = 0;
        r->slot = -1;
    }
    // Slots go to the foremost requests without one among the first M of the
    // running queue, lowest free slot first.
    void assign_slots() {
        const size_t lim = std::min(running.size(), (size_t)c.query_slots);
        for (size_t i = 0; i < lim; ++i) {
            Request *r = running[i];
            if (r->slot >= 0) continue;
            auto f = std::find(slot_used.begin(), slot_used.end(), 0);
            if (f == slot_used.end()) return;
            *f = 1;
            r->slot = (int32_t)(f - slot_used.begin());
        }
    }
    // Who may be preempted: a running, never-compressed request; with prefix
    // sharing any such request, under hybrid scheduling one without a slot,
    // under constrained scheduling none.
    bool victim_ok(const Request *v) const {
        if (v->state != ZP_REQ_RUNNING || v->compressed) return false;
        if (c.prefix_sharing) return true;
        return c.policy == ZP_SCHED_HYBRID && v->slot < 0;
    }
    void drop_from_running(Request *r) { running.erase(std::find(running.begin(), running.end(), r)); }
    void preempt(Request *v, std::vector<int32_t> &log) {
        release(v->table);
        leave_prefix(v);
        free_slot(v);
        v->table.clear();
        v->len = 0;
        v->want_compress = false;
        v->state = ZP_REQ_WAITING;
        ++v->preemptions;
        drop_from_running(v);
        waiting.push_front(v);
        log.push_back(v->id);
    }
    void finish(Request *r) {
        release(r->table);
        leave_prefix(r);
        free_slot(r);
        r->table.clear();
        r->state = ZP_REQ_FINISHED;
        drop_from_running(r);
    }
    int32_t fresh_needed(const Request *r) const {
        int32_t need = 0;
        for (int32_t t = 0; t < r->budget; ++t) need += refcount(r->table[(size_t)t]) > 1;
        return need;
    }
    // Plans the compaction of r (targets from the pool); with prefix sharing,
    // preempts the last uncompressed requests while the targets do not fit.
    // Leaves r triggered when they still do not fit.
    zp_status try_compress(Request *r, std::vector<int32_t> &log) {
        const int32_t nb = r->len / c.block_size;
        int32_t need = fresh_needed(r);
        while (free_blocks() < need && c.prefix_sharing) {
            Request *victim = nullptr;
            for (auto it = running.rbegin(); it != running.rend(); ++it)
                if (victim_ok(*it)) {
                    victim = *it;
                    break;
                }
            if (!victim) break;
            preempt(victim, log);
            if (victim == r) return ZP_OK;
            need = fresh_needed(r);
        }
        if (free_blocks() < need) return ZP_OK;
        std::vector<int32_t> targets((size_t)r->budget), nt((size_t)r->budget), dropped((size_t)nb);
        int32_t nd = 0, nf = 0;
        zp_status rc = zp_plan_compaction(pool, r->table.data(), nb, r->budget, targets.data(), nt.data(),
                                          dropped.data(), &nd, &nf);
        if (rc != ZP_OK) return rc;
        dropped.resize((size_t)nd);
        targets.resize((size_t)r->budget - 1);
        leave_prefix(r);
        Started s;
        s.id = r->id;
        s.len = r->len;
        s.slot = r->slot;
        s.k = (r->budget - 1) * c.block_size;
        s.first = r->compressed ? 0 : 1;
        s.table.assign(r->table.begin(), r->table.begin() + nb);
        s.targets = targets;
        started.push_back(std::move(s));
        r->new_table = nt;
        r->dropped = dropped;
        r->state = ZP_REQ_COMPRESSING;
        r->want_compress = false;
        return ZP_OK;
    }
    Request *find(int32_t id) {
        auto it = index.find(id);
        return it == index.end() ? nullptr : &reqs[it->second];
    }
};

namespace {

void put_table(const zp_sched *s, const Request *r, int32_t *row) {
    const int32_t stride = s->c.table_stride;
    for (int32_t i = 0; i < stride; ++i) row[i] = i < (int32_t)r->table.size() ? r->table[(size_t)i] : -1;
}

}  // namespace

extern "C" zp_sched *zp_sched_create(const zp_sched_config *cfg, zp_pool *pool) {
    if (!cfg || !pool) {
        fail(ZP_ERR_INVALID_ARG, "sched_create: NULL argument");
        return nullptr;
    }
    const zp_sched_config &c = *cfg;
    if (c.block_size < 1 || c.window < 1 || c.window > c.block_size || c.max_blocks < 2 || c.query_slots < 1 ||
        (c.policy != ZP_SCHED_CONSTRAINED && c.policy != ZP_SCHED_HYBRID) || c.max_running < 1 ||
        c.max_prefill_tokens < 1 || c.table_stride < c.max_blocks) {
        fail(ZP_ERR_INVALID_ARG, "sched_create: bad configuration");
        return nullptr;
    }
    zp_sched *s = new zp_sched;
    s->c = c;
    s->c.prefix_sharing = c.prefix_sharing ? 1 : 0;
    s->pool = pool;
    s->slot_used.assign((size_t)c.query_slots, 0);
    ok();
    return s;
}

extern "C" void zp_sched_destroy(zp_sched *s) { delete s; }

extern "C" zp_status zp_sched_add_request(zp_sched *s, int32_t id, int32_t prompt_len, int32_t output_len,
                                          int32_t prefix_group, int32_t prefix_len, int32_t max_blocks) {
    if (!s) return fail(ZP_ERR_INVALID_ARG, "sched_add_request: NULL scheduler");
    const int32_t b = s->c.block_size;
    const int32_t budget = max_blocks ? max_blocks : s->c.max_blocks;
    if (id < 0 || s->index.count(id)) return fail(ZP_ERR_INVALID_ARG, "sched_add_request: id %d taken or < 0", id);
    if (prompt_len < 1 || output_len < 1 || budget < 2 || budget > s->c.max_blocks)
        return fail(ZP_ERR_INVALID_ARG, "sched_add_request: bad lengths or budget");
    if (prefix_len < 0 || prefix_len % b || prefix_len > prompt_len || (prefix_len && prefix_group < 0))
        return fail(ZP_ERR_INVALID_ARG, "sched_add_request: bad prefix");
    if ((int64_t)prompt_len + output_len - 1 > (int64_t)s->c.table_stride * b)
        return fail(ZP_ERR_INVALID_ARG, "sched_add_request: %d + %d tokens exceed the block table", prompt_len,
                    output_len);
    if (prefix_len) {
        auto g = s->group_len.emplace(prefix_group, prefix_len).first;
        if (g->second != prefix_len)
            return fail(ZP_ERR_INVALID_ARG, "sched_add_request: prefix group %d has prefix length %d, not %d",
                        prefix_group, g->second, prefix_len);
    }
    Request r;
    r.id = id;
    r.prompt = prompt_len;
    r.output = output_len;
    r.group = prefix_len ? prefix_group : -1;
    r.prefix_len = prefix_len;
    r.budget = budget;
    s->index[id] = s->reqs.size();
    s->reqs.push_back(std::move(r));
    s->waiting.push_back(&s->reqs.back());
    return ok();
}

extern "C" zp_status zp_sched_schedule(zp_sched *s, zp_sched_step *out) {
    if (!s || !out || !out->ids || !out->lens || !out->start || !out->slots || !out->tables || !out->preempted)
        return fail(ZP_ERR_INVALID_ARG, "sched_schedule: NULL argument");
    if (s->last_kind != ZP_STEP_IDLE) return fail(ZP_ERR_INVALID_ARG, "sched_schedule: last step not committed");
    const zp_sched_config &c = s->c;
    const int32_t b = c.block_size;
    std::vector<int32_t> preempted;
    s->assign_slots();
    {
        std::vector<Request *> snap = s->running;
        for (Request *r : snap)
            if (r->want_compress && r->state == ZP_REQ_RUNNING) {
                zp_status rc = s->try_compress(r, preempted);
                if (rc != ZP_OK) return rc;
            }
    }
    auto emit_preempted = [&]() {
        out->n_preempted = (int32_t)preempted.size();
        for (size_t i = 0; i < preempted.size(); ++i) out->preempted[i] = preempted[i];
    };
    // ---- admission: first come, first served, no skipping
    std::vector<std::pair<Request *, int32_t>> admitted;
    int64_t tokens = 0;
    while (!s->waiting.empty()) {
        Request *r = s->waiting.front();
        if ((int32_t)s->running.size() >= c.max_running) break;
        if (c.policy == ZP_SCHED_CONSTRAINED && (int32_t)s->running.size() >= c.query_slots) break;
        const int32_t L = r->prompt + r->generated;
        if (!admitted.empty() && tokens + L > c.max_prefill_tokens) break;
        const int32_t nb = (L + b - 1) / b;
        const int32_t pb = c.prefix_sharing ? r->prefix_len / b : 0;
        auto pit = pb > 0 ? s->prefix.find(r->group) : s->prefix.end();
        const bool cached = pit != s->prefix.end();
        const int32_t need = cached ? nb - pb : nb;
        if (need > s->free_blocks()) break;
        s->waiting.pop_front();
        int32_t start = 0;
        r->table.clear();
        if (cached) {
            Prefix &p = pit->second;
            zp_pool_incref(s->pool, (int32_t)p.blocks.size(), p.blocks.data());
            ++p.holders;
            r->table = p.blocks;
            r->holds_prefix = true;
            start = r->prefix_len;
        }
        if (!s->alloc(need, r->table)) return fail(ZP_ERR_INVALID_ARG, "sched: pool allocation failed");
        if (!cached && pb > 0) {
            Prefix p;
            p.blocks.assign(r->table.begin(), r->table.begin() + pb);
            p.holders = 1;
            s->prefix[r->group] = std::move(p);
            r->holds_prefix = true;
        }
        r->len = L;
        ++r->generated;
        r->state = ZP_REQ_RUNNING;
        s->running.push_back(r);
        admitted.emplace_back(r, start);
        tokens += L;
    }
    if (!admitted.empty()) {
        s->assign_slots();
        out->kind = ZP_STEP_PREFILL;
        out->n = (int32_t)admitted.size();
        out->n_blocked = 0;
        s->last.clear();
        for (size_t i = 0; i < admitted.size(); ++i) {
            Request *r = admitted[i].first;
            out->ids[i] = r->id;
            out->lens[i] = r->len;
            out->start[i] = admitted[i].second;
            out->slots[i] = r->slot;
            put_table(s, r, out->tables + i * (size_t)c.table_stride);
            s->last.push_back(r);
        }
        emit_preempted();
        s->last_kind = ZP_STEP_PREFILL;
        return ok();
    }
    // ---- decode: scan the running queue front to back
    std::vector<Request *> batch;
    int32_t blocked = 0;
    size_t idx = 0;
    while (idx < s->running.size()) {
        Request *r = s->running[idx];
        if (r->state != ZP_REQ_RUNNING) {
            ++idx;
            continue;
        }
        if (r->want_compress) {
            ++blocked;
            ++idx;
            continue;
        }
        const int32_t pos = r->len;
        if (r->slot < 0 && pos / b + 1 >= r->budget && pos % b >= b - c.window) {  // window token needs a slot
            ++blocked;
            ++idx;
            continue;
        }
        if (pos % b == 0 && pos / b >= (int32_t)r->table.size()) {
            bool gone = false;
            while (s->free_blocks() == 0) {
                Request *victim = nullptr;
                for (size_t j = s->running.size(); j > idx + 1; --j)
                    if (s->victim_ok(s->running[j - 1])) {
                        victim = s->running[j - 1];
                        break;
                    }
                if (!victim && s->victim_ok(r)) victim = r;
                if (!victim) break;
                s->preempt(victim, preempted);
                if (victim == r) {
                    gone = true;
                    break;
                }
            }
            if (gone) continue;
            if (s->free_blocks() == 0) {
                ++blocked;
                ++idx;
                continue;
            }
            if (!s->alloc(1, r->table)) return fail(ZP_ERR_INVALID_ARG, "sched: pool allocation failed");
        }
        ++r->len;
        batch.push_back(r);
        ++idx;
    }
    emit_preempted();
    out->n_blocked = blocked;
    s->last = batch;
    if (batch.empty()) {
        bool busy = !s->started.empty();
        for (Request *r : s->running) busy |= r->state == ZP_REQ_COMPRESSING;
        out->kind = ZP_STEP_IDLE;
        out->n = 0;
        if (!busy && (!s->running.empty() || !s->waiting.empty()))
            return fail(ZP_ERR_CAPACITY, "sched: deadlock -- no request can run and no compression is in flight");
        return ok();
    }
    out->kind = ZP_STEP_DECODE;
    out->n = (int32_t)batch.size();
    for (size_t i = 0; i < batch.size(); ++i) {
        Request *r = batch[i];
        out->ids[i] = r->id;
        out->lens[i] = r->len;
        out->start[i] = r->len - 1;
        out->slots[i] = r->slot;
        put_table(s, r, out->tables + i * (size_t)c.table_stride);
    }
    s->last_kind = ZP_STEP_DECODE;
    return ok();
}

extern "C" zp_status zp_sched_commit(zp_sched *s, int32_t *finished, int32_t *n_finished, int32_t *preempted,
                                     int32_t *n_preempted) {
    if (!s) return fail(ZP_ERR_INVALID_ARG, "sched_commit: NULL scheduler");
    const int32_t b = s->c.block_size;
    std::vector<int32_t> fin, pre;
    std::vector<Request *> reqs;
    reqs.swap(s->last);
    const int kind = s->last_kind;
    s->last_kind = ZP_STEP_IDLE;
    if (kind == ZP_STEP_PREFILL) {
        for (Request *r : reqs)
            if (r->generated >= r->output) {
                fin.push_back(r->id);
                s->finish(r);
            }
    } else if (kind == ZP_STEP_DECODE) {
        for (Request *r : reqs) {
            ++r->generated;
            if (r->generated >= r->output) {
                fin.push_back(r->id);
                s->finish(r);
            } else if (r->slot >= 0 && r->len % b == 0 && r->len / b >= r->budget) {
                r->want_compress = true;
            }
        }
        for (Request *r : reqs)
            if (r->want_compress && r->state == ZP_REQ_RUNNING) {
                zp_status rc = s->try_compress(r, pre);
                if (rc != ZP_OK) return rc;
            }
    }
    s->assign_slots();
    if (n_finished) *n_finished = (int32_t)fin.size();
    if (finished)
        for (size_t i = 0; i < fin.size(); ++i) finished[i] = fin[i];
    if (n_preempted) *n_preempted = (int32_t)pre.size();
    if (preempted)
        for (size_t i = 0; i < pre.size(); ++i) preempted[i] = pre[i];
    return ok();
}

extern "C" zp_status zp_sched_take_compressions(zp_sched *s, zp_sched_compressions *out) {
    if (!s || !out) return fail(ZP_ERR_INVALID_ARG, "sched_take_compressions: NULL argument");
    const zp_sched_config &c = s->c;
    const size_t n = s->started.size();
    if (n && (!out->ids || !out->lens || !out->slots || !out->k || !out->first || !out->tables || !out->targets))
        return fail(ZP_ERR_INVALID_ARG, "sched_take_compressions: NULL output array");
    out->n = (int32_t)n;
    for (size_t i = 0; i < n; ++i) {
        const Started &st = s->started[i];
        out->ids[i] = st.id;
        out->lens[i] = st.len;
        out->slots[i] = st.slot;
        out->k[i] = st.k;
        out->first[i] = st.first;
        int32_t *tr = out->tables + i * (size_t)c.table_stride;
        for (int32_t j = 0; j < c.table_stride; ++j) tr[j] = j < (int32_t)st.table.size() ? st.table[(size_t)j] : -1;
        int32_t *tg = out->targets + i * (size_t)(c.max_blocks - 1);
        for (int32_t j = 0; j < c.max_blocks - 1; ++j)
            tg[j] = j < (int32_t)st.targets.size() ? st.targets[(size_t)j] : -1;
    }
    s->started.clear();
    return ok();
}

extern "C" zp_status zp_sched_compression_done(zp_sched *s, int32_t id) {
    if (!s) return fail(ZP_ERR_INVALID_ARG, "sched_compression_done: NULL scheduler");
    Request *r = s->find(id);
    if (!r || r->state != ZP_REQ_COMPRESSING)
        return fail(ZP_ERR_INVALID_ARG, "sched_compression_done: request %d is not compressing", id);
    r->table = r->new_table;
    r->len = (r->budget - 1) * s->c.block_size;
    r->compressed = true;
    r->state = ZP_REQ_RUNNING;
    s->release(r->dropped);
    r->new_table.clear();
    r->dropped.clear();
    return ok();
}

extern "C" zp_status zp_sched_counts(const zp_sched *s, int32_t *out) {
    if (!s || !out) return fail(ZP_ERR_INVALID_ARG, "sched_counts: NULL argument");
    int32_t fin = 0;
    for (const Request &r : s->reqs) fin += r.state == ZP_REQ_FINISHED;
    out[0] = (int32_t)s->waiting.size();
    out[1] = (int32_t)s->running.size();
    out[2] = fin;
    out[3] = (int32_t)std::count(s->slot_used.begin(), s->slot_used.end(), 0);
    out[4] = s->free_blocks();
    return ok();
}

extern "C" zp_status zp_sched_request_info(const zp_sched *s, int32_t id, int32_t *out) {
    if (!s || !out) return fail(ZP_ERR_INVALID_ARG, "sched_request_info: NULL argument");
    auto it = s->index.find(id);
    if (it == s->index.end()) return fail(ZP_ERR_INVALID_ARG, "sched_request_info: unknown id %d", id);
    const Request &r = s->reqs[it->second];
    out[0] = r.state;
    out[1] = r.len;
    out[2] = r.generated;
    out[3] = r.slot;
    out[4] = r.preemptions;
    out[5] = r.compressed ? 1 : 0;
    out[6] = (int32_t)r.table.size();
    return ok();
}
