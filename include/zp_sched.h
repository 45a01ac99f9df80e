/* Request scheduler for Compressed PagedAttention: constrained and hybrid
 * scheduling with query slots, preemption and prefix sharing, on the host.
 *
 * Rules [Zipage §4.1, §4.3, §4.4, §4.5, Fig. 2]:
 *   - outside prefill a request holds at most N_max blocks; after a decode
 *     step, N >= N_max with the last block full triggers its compression
 *     (N_max - 1 blocks kept, one reserved, the rest released) [§4.1];
 *   - compressing needs a query slot (M of them, eq. (1)) [§4.2, §4.3];
 *   - constrained: at most M running requests, each holding a slot; a
 *     request that finds no free block is blocked, never preempted [§4.3];
 *   - hybrid: admission needs only the prefill blocks; the first M requests
 *     of the running queue may hold slots and freed slots go to the foremost
 *     request without one; a request without a slot decodes while it holds
 *     fewer than N_max blocks or its new token falls before the last w
 *     positions of its block, and is blocked otherwise; a request that finds
 *     no free block preempts the last running request without a slot, then is
 *     blocked once none is left [§4.3, Fig. 2];
 *   - prefix sharing: blocks of a shared prefix are reference counted and
 *     compaction goes to new targets where a block is shared; a request that
 *     finds no block (to decode or for its targets) preempts the last
 *     uncompressed request, slot or not [§4.4];
 *   - a compressing request sits out decode until its compression completes
 *     (zp_sched_compression_done) [§4.5];
 *   - N_max may be set per request [Zipage, Limitations].
 * Where the pages leave a step open: prefill and decode are separate steps,
 * waiting requests are admitted first, first come first served with no
 * skipping, at most max_prefill_tokens tokens per prefill step (the first
 * request always fits); a preempted request loses its cache, goes back to the
 * front of the waiting queue and re-enters with its generated tokens as part
 * of its prompt (its re-prefill yields one more token); slots are handed out
 * at the start of each step and after each commit; decode scans the running
 * queue front to back and takes victims from the back among the requests not
 * yet scanned in that step, then the scanning request itself; the trigger is
 * checked for the requests that decoded in the step, and a compression that
 * cannot get its target blocks is tried again at the start of later steps.
 *
 * Token accounting: a request of prompt length P and output length O caches
 * P tokens at prefill, which also yields its first token; every decode step
 * caches the previous token and yields the next; it finishes after O tokens.
 *
 * Ownership: the scheduler borrows the pool (which must outlive it) and owns
 * nothing else the caller sees.  Output arrays are caller-owned, sized by
 * max_running (and by table_stride or max_blocks - 1 per row where stated).
 * Errors: ZP_ERR_INVALID_ARG (bad argument or request, unknown id, call out of
 * order), ZP_ERR_CAPACITY (nothing can run and nothing is in flight: the
 * pool or the table cannot hold a waiting request). */
#ifndef ZP_SCHED_H
#define ZP_SCHED_H

#include "zp.h"

#ifdef __cplusplus
extern "C" {
#endif

enum { ZP_SCHED_CONSTRAINED = 0, ZP_SCHED_HYBRID = 1 };
enum { ZP_STEP_IDLE = 0, ZP_STEP_PREFILL = 1, ZP_STEP_DECODE = 2 };
enum { ZP_REQ_WAITING = 0, ZP_REQ_RUNNING = 1, ZP_REQ_COMPRESSING = 2, ZP_REQ_FINISHED = 3 };

typedef struct {
    int32_t block_size;         /* b */
    int32_t window;             /* w, 1 <= w <= b */
    int32_t max_blocks;         /* N_max >= 2 (the largest per-request budget) */
    int32_t query_slots;        /* M >= 1 */
    int32_t policy;             /* ZP_SCHED_CONSTRAINED or ZP_SCHED_HYBRID */
    int32_t prefix_sharing;     /* 1: shared prefixes and the §4.4 preemption rule */
    int32_t max_running;        /* running requests at most (decode batch capacity) */
    int32_t max_prefill_tokens; /* tokens cached by one prefill step */
    int32_t table_stride;       /* block-table entries per request */
} zp_sched_config;

typedef struct zp_sched zp_sched;

/* NULL on a bad configuration (zp_last_error says why). */
zp_sched *zp_sched_create(const zp_sched_config *cfg, zp_pool *pool);
void zp_sched_destroy(zp_sched *s);

/* Queues a request (first come, first served).  id >= 0 and unique; prompt_len
 * >= 1, output_len >= 1, prompt_len + output_len - 1 <= table_stride * b;
 * prefix_group >= 0 names a shared prefix of prefix_len tokens (a multiple of
 * b, <= prompt_len, the same for every request of the group), else -1 and 0;
 * max_blocks: the request's own N_max in
 * [2, N_max], 0 for N_max. */
zp_status zp_sched_add_request(zp_sched *s, int32_t id, int32_t prompt_len, int32_t output_len,
                               int32_t prefix_group, int32_t prefix_len, int32_t max_blocks);

/* One step.  kind: ZP_STEP_PREFILL (requests admitted; lens = tokens cached,
 * start = first position to write, after a cached prefix), ZP_STEP_DECODE
 * (lens = tokens attended, the new one included; start = lens - 1, the new
 * token's position) or ZP_STEP_IDLE (nothing can run until a compression in
 * flight completes).  slots: query slot or -1; tables [n][table_stride]
 * padded with -1; preempted: requests sent back to the waiting queue while
 * planning this step; n_blocked: running requests that sit this step out. */
typedef struct {
    int32_t kind, n, n_preempted, n_blocked;
    int32_t *ids;       /* [max_running] */
    int32_t *lens;      /* [max_running] */
    int32_t *start;     /* [max_running] */
    int32_t *slots;     /* [max_running] */
    int32_t *tables;    /* [max_running][table_stride] */
    int32_t *preempted; /* [max_running] */
} zp_sched_step;

zp_status zp_sched_schedule(zp_sched *s, zp_sched_step *out);

/* Applies the last step (its device work issued): token counts, finishes
 * (blocks and slots released), compression triggers.  finished and preempted
 * are [max_running] arrays (nullable when the counts are not wanted). */
zp_status zp_sched_commit(zp_sched *s, int32_t *finished, int32_t *n_finished, int32_t *preempted,
                          int32_t *n_preempted);

/* Compressions started since the last call (target blocks already taken
 * from the pool): per request its id, length L, slot, budget k = (N_i-1) b,
 * first-compression flag, source table [table_stride] and targets
 * [max_blocks - 1], both padded with -1. */
typedef struct {
    int32_t n;
    int32_t *ids, *lens, *slots, *k, *first; /* [max_running] */
    int32_t *tables;                         /* [max_running][table_stride] */
    int32_t *targets;                        /* [max_running][max_blocks - 1] */
} zp_sched_compressions;

zp_status zp_sched_take_compressions(zp_sched *s, zp_sched_compressions *out);

/* The compaction of request id has completed on the device: its table becomes
 * the planned one, its length (N_i - 1) b, and the blocks it dropped go back
 * to the pool. */
zp_status zp_sched_compression_done(zp_sched *s, int32_t id);

/* out[5] = waiting, running, finished, free slots, free blocks. */
zp_status zp_sched_counts(const zp_sched *s, int32_t *out);

/* out[7] = state, L, generated, slot, preemptions, compressed, blocks held. */
zp_status zp_sched_request_info(const zp_sched *s, int32_t id, int32_t *out);

#ifdef __cplusplus
}
#endif
#endif
