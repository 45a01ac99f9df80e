// pool.cpp -- host block pool and compaction planner (no device work).
//
// Zipage paper §3 (pre-allocated blocks, free blocks), §4.1 (after compression
// the kept entries occupy the first N_max - 1 blocks, the N_max-th block is
// reserved, the rest are released) and §4.4 (reference-counted prefix blocks;
// compression writes into target blocks so shared blocks survive).
#include <algorithm>
#include <set>
#include <vector>

#include "zp_internal.h"

struct zp_pool {
    std::vector<int32_t> ref;
    std::set<int32_t> free_ids;  // ordered: lowest id handed out first
};

using zp::fail;
using zp::ok;

extern "C" zp_pool *zp_pool_create(int32_t n_total) {
    if (n_total <= 0) {
        fail(ZP_ERR_INVALID_ARG, "pool: n_total %d", n_total);
        return nullptr;
    }
    zp_pool *p = new (std::nothrow) zp_pool;
    if (!p) return nullptr;
    p->ref.assign((size_t)n_total, 0);
    for (int32_t i = 0; i < n_total; ++i) p->free_ids.insert(p->free_ids.end(), i);
    return p;
}

extern "C" void zp_pool_destroy(zp_pool *pool) { delete pool; }

extern "C" int32_t zp_pool_num_free(const zp_pool *pool) {
    return pool ? (int32_t)pool->free_ids.size() : -1;
}

extern "C" int32_t zp_pool_refcount(const zp_pool *pool, int32_t block) {
    if (!pool || block < 0 || (size_t)block >= pool->ref.size()) return -1;
    return pool->ref[(size_t)block];
}

static bool valid_ids(const zp_pool *pool, int32_t n, const int32_t *ids) {
    for (int32_t i = 0; i < n; ++i)
        if (ids[i] < 0 || (size_t)ids[i] >= pool->ref.size()) return false;
    return true;
}

extern "C" zp_status zp_pool_alloc(zp_pool *pool, int32_t n, int32_t *ids) {
    if (!pool || n < 0 || (n > 0 && !ids)) return fail(ZP_ERR_INVALID_ARG, "pool_alloc: bad argument");
    if ((size_t)n > pool->free_ids.size())
        return fail(ZP_ERR_CAPACITY, "pool_alloc: %d blocks asked, %zu free", n, pool->free_ids.size());
    for (int32_t i = 0; i < n; ++i) {
        auto it = pool->free_ids.begin();
        ids[i] = *it;
        pool->free_ids.erase(it);
        pool->ref[(size_t)ids[i]] = 1;
    }
    return ok();
}

extern "C" zp_status zp_pool_incref(zp_pool *pool, int32_t n, const int32_t *ids) {
    if (!pool || n < 0 || (n > 0 && !ids)) return fail(ZP_ERR_INVALID_ARG, "pool_incref: bad argument");
    if (!valid_ids(pool, n, ids)) return fail(ZP_ERR_INVALID_ARG, "pool_incref: block id out of range");
    for (int32_t i = 0; i < n; ++i)
        if (pool->ref[(size_t)ids[i]] <= 0) return fail(ZP_ERR_INVALID_ARG, "pool_incref: block %d is free", ids[i]);
    for (int32_t i = 0; i < n; ++i) ++pool->ref[(size_t)ids[i]];
    return ok();
}

extern "C" zp_status zp_pool_release(zp_pool *pool, int32_t n, const int32_t *ids) {
    if (!pool || n < 0 || (n > 0 && !ids)) return fail(ZP_ERR_INVALID_ARG, "pool_release: bad argument");
    if (!valid_ids(pool, n, ids)) return fail(ZP_ERR_INVALID_ARG, "pool_release: block id out of range");
    // check first so that a bad list changes nothing
    std::vector<int32_t> drop((size_t)n);
    for (int32_t i = 0; i < n; ++i) {
        int32_t c = 0;
        for (int32_t j = 0; j < n; ++j) c += ids[j] == ids[i];
        if (pool->ref[(size_t)ids[i]] < c) return fail(ZP_ERR_INVALID_ARG, "pool_release: block %d over-released", ids[i]);
    }
    for (int32_t i = 0; i < n; ++i) {
        int32_t &r = pool->ref[(size_t)ids[i]];
        if (--r == 0) pool->free_ids.insert(ids[i]);
    }
    return ok();
}

extern "C" zp_status zp_plan_compaction(zp_pool *pool, const int32_t *table, int32_t n_blocks,
                                        int32_t max_blocks, int32_t *targets, int32_t *new_table,
                                        int32_t *dropped, int32_t *n_dropped, int32_t *n_fresh) {
    if (!pool || !table || !targets || !new_table || !dropped || !n_dropped || !n_fresh)
        return fail(ZP_ERR_INVALID_ARG, "plan_compaction: NULL argument");
    if (max_blocks < 2 || n_blocks < max_blocks)
        return fail(ZP_ERR_INVALID_ARG, "plan_compaction: needs n_blocks (%d) >= max_blocks (%d) >= 2",
                    n_blocks, max_blocks);
    if (!valid_ids(pool, n_blocks, table)) return fail(ZP_ERR_INVALID_ARG, "plan_compaction: block id out of range");
    for (int32_t i = 0; i < n_blocks; ++i)
        if (pool->ref[(size_t)table[i]] <= 0)
            return fail(ZP_ERR_INVALID_ARG, "plan_compaction: block %d of the table is free", table[i]);
    // how many new blocks: one per shared position among the first max_blocks
    int32_t need = 0;
    for (int32_t t = 0; t < max_blocks; ++t) need += pool->ref[(size_t)table[t]] > 1;
    if ((size_t)need > pool->free_ids.size())
        return fail(ZP_ERR_CAPACITY, "plan_compaction: %d new blocks needed, %zu free", need,
                    pool->free_ids.size());
    std::vector<int32_t> fresh((size_t)need);
    if (need) {
        zp_status rc = zp_pool_alloc(pool, need, fresh.data());
        if (rc != ZP_OK) return rc;
    }
    int32_t used = 0;
    for (int32_t t = 0; t < max_blocks; ++t) {
        const int32_t blk = table[t];
        const int32_t id = pool->ref[(size_t)blk] > 1 ? fresh[(size_t)used++] : blk;
        new_table[t] = id;
        if (t < max_blocks - 1) targets[t] = id;
    }
    // dropped: the table's blocks that the new table does not hold, in table
    // order (a sorted copy of the new table answers each lookup)
    std::vector<int32_t> held(new_table, new_table + max_blocks);
    std::sort(held.begin(), held.end());
    int32_t nd = 0;
    for (int32_t i = 0; i < n_blocks; ++i)
        if (!std::binary_search(held.begin(), held.end(), table[i])) dropped[nd++] = table[i];
    *n_dropped = nd;
    *n_fresh = used;
    return ok();
}

extern "C" zp_status zp_plan_compaction_batch(zp_pool *pool, const int32_t *tables, int32_t table_stride,
                                              const int32_t *n_blocks, int32_t n, int32_t max_blocks,
                                              const int32_t *max_blocks_seq, int32_t *targets,
                                              int32_t *new_tables, int32_t *dropped, int32_t *n_dropped,
                                              int32_t *n_fresh) {
    if (!pool || n < 0 || (n > 0 && (!tables || !n_blocks || !targets || !new_tables || !dropped ||
                                     !n_dropped || !n_fresh)))
        return fail(ZP_ERR_INVALID_ARG, "plan_compaction_batch: NULL argument");
    if (max_blocks < 2 || table_stride < max_blocks)
        return fail(ZP_ERR_INVALID_ARG, "plan_compaction_batch: table_stride %d < max_blocks %d", table_stride,
                    max_blocks);
    for (int32_t i = 0; i < n; ++i) {
        if (n_blocks[i] > table_stride)
            return fail(ZP_ERR_INVALID_ARG, "plan_compaction_batch: sequence %d has %d > %d blocks", i,
                        n_blocks[i], table_stride);
        const int32_t mb = max_blocks_seq ? max_blocks_seq[i] : max_blocks;
        if (mb < 2 || mb > max_blocks)
            return fail(ZP_ERR_INVALID_ARG, "plan_compaction_batch: sequence %d budget %d outside [2, %d]", i, mb,
                        max_blocks);
        int32_t *tg = targets + (size_t)i * (max_blocks - 1);
        int32_t *nt = new_tables + (size_t)i * max_blocks;
        zp_status rc = zp_plan_compaction(pool, tables + (size_t)i * table_stride, n_blocks[i], mb, tg, nt,
                                          dropped + (size_t)i * table_stride, &n_dropped[i], &n_fresh[i]);
        if (rc != ZP_OK) return rc;  // sequences before i stay planned
        for (int32_t t = mb - 1; t < max_blocks - 1; ++t) tg[t] = -1;
        for (int32_t t = mb; t < max_blocks; ++t) nt[t] = -1;
    }
    return ok();
}

// Capacity plan [Zipage §4.2 eq. (1), App. C.3 eq. (2)]: the largest request
// concurrency M and the block count N_total that fit a memory budget,
//     maximise M  s.t.  (1 + extra) m_kv N_total + M m_q <= m_available,
//                       M <= N_total / N_max,  M > 0,  N_total > 0.
// For a given M the least N_total is M N_max, so the optimum is
//     M = floor(m_available / ((1 + extra) m_kv N_max + m_q)),
// and the blocks of the linear program's optimum,
//     N_total = floor(m_available / ((1 + extra) m_kv + m_q / N_max)),
// satisfy both constraints with that M.  Integer arithmetic: extra is given
// as the fraction extra_num / extra_den (the global score cache: 1/(2d) of a
// block's K and V in the paper's element type; 0/1 without it).
extern "C" zp_status zp_plan_capacity(int64_t m_available, int64_t m_kv_block, int64_t m_q_request,
                                      int32_t max_blocks, int64_t extra_num, int64_t extra_den, int64_t *M,
                                      int64_t *N_total) {
    if (!M || !N_total) return fail(ZP_ERR_INVALID_ARG, "plan_capacity: NULL output");
    if (m_available <= 0 || m_kv_block <= 0 || m_q_request < 0 || max_blocks < 1 || extra_num < 0 ||
        extra_den <= 0)
        return fail(ZP_ERR_INVALID_ARG, "plan_capacity: bad sizes");
    // work in units of 1/extra_den byte: block cost (den + num) * m_kv
    const __int128 den = extra_den, blk = (__int128)(extra_den + extra_num) * m_kv_block;
    const __int128 avail = (__int128)m_available * den, q = (__int128)m_q_request * den;
    const __int128 m = avail / (blk * max_blocks + q);
    // N_total = floor(avail / (blk + q / N_max)) = floor(avail * N_max / (blk * N_max + q))
    const __int128 nt = avail * max_blocks / (blk * max_blocks + q);
    if (m <= 0) return fail(ZP_ERR_CAPACITY, "plan_capacity: the budget holds no request of %d blocks", max_blocks);
    *M = (int64_t)m;
    *N_total = (int64_t)nt;
    return ok();
}
