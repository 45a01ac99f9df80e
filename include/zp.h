/*
 * zp.h -- C ABI of the Compressed PagedAttention hot path for one GB300 GPU.
 *
 * The operations follow the paper "Zipage: Maintain High Request Concurrency
 * for LLM Reasoning through Compressed PagedAttention" (Liao et al., arXiv
 * 2603.08743), cited below as [Zipage <section>].
 *
 * Conventions (apply to every call):
 *   Ownership   Every device buffer is owned by the caller.  The library never
 *               allocates device memory: scratch comes from a caller-supplied
 *               workspace whose size the matching *_workspace_size() returns.
 *               The host block pool (zp_pool_*) is owned by the library.
 *   Streams     `stream` is a cudaStream_t passed as void* (NULL = the legacy
 *               default stream).  Device calls only enqueue work on it and
 *               never synchronise the device.
 *   Errors      Every call returns zp_status.  ZP_OK means the arguments were
 *               valid and the work was enqueued; a launch failure returns
 *               ZP_ERR_CUDA.  zp_last_error() gives a message for the calling
 *               thread.  Kernels never trap: a block id outside [0, N_total) or
 *               a failed bounded wait is skipped and recorded in a device status
 *               word that zp_device_status() reads.
 *   Layouts     One layer of the K or V cache is [N_total][b][h_kv][d] ([Zipage
 *               §3]); element (blk, slot, kvh, i) is at ((blk*b+slot)*h_kv+kvh)*d+i.
 *               Several layers sit one after another, `layer_stride` elements
 *               apart.  Per-slot float arrays (the window score S and the global
 *               score cache F of [Zipage App. C.3]) are [N_total][b][h_kv].
 *               Block tables are int32 [B][table_stride]: token t of sequence s
 *               is in block table[s*table_stride + t/b], slot t%b.  Query head h
 *               reads key/value head h/(h_q/h_kv).
 *   Types       ZP_BF16 or ZP_F32 for q, K, V and the attention output; scores
 *               are float32; ids and lengths int32.
 */
#ifndef ZP_H
#define ZP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ZP_OK = 0,
    ZP_ERR_INVALID_ARG = 1, /* NULL pointer, negative size, bad flag */
    ZP_ERR_SHAPE = 2,       /* head / block geometry the library does not support */
    ZP_ERR_DTYPE = 3,       /* unknown element type */
    ZP_ERR_CAPACITY = 4,    /* workspace too small, pool exhausted, budget < window */
    ZP_ERR_CUDA = 5,        /* a CUDA runtime call or launch failed */
    ZP_ERR_TIMEOUT = 6,     /* a bounded device wait gave up (device status) */
    ZP_ERR_DEVICE = 7       /* kernels recorded a bad index (device status) */
} zp_status;

typedef enum { ZP_BF16 = 0, ZP_F32 = 1 } zp_dtype;

/* Geometry of one layer of the paged cache [Zipage §3]. */
typedef struct {
    int32_t h_q;            /* query heads */
    int32_t h_kv;           /* key/value heads; h_q % h_kv == 0 */
    int32_t head_dim;       /* d */
    int32_t block_size;     /* b, tokens per block */
    int32_t n_total_blocks; /* N_total, blocks in the pool */
    int32_t dtype;          /* zp_dtype of q, K, V, out */
} zp_cache_desc;

/* Scoring switches [Zipage App. C.2-C.8].  Recommended values (App. C.8):
 * alpha 0.8, lambda 0.2, tau 0.4, pooling at the first compression only.  The
 * paper gives neither the pooling kernel size nor the similarity threshold p. */
typedef struct {
    int32_t window;         /* w, observation window (1 <= w <= b) */
    int32_t use_global;     /* global score, Alg. 2 */
    float alpha;            /* decay of the global score */
    int32_t pool_kernel;    /* odd max-pool kernel size; <= 1 disables pooling */
    int32_t pool_policy;    /* 0 never, 1 first compression only, 2 every compression */
    int32_t use_similarity; /* redundancy score (eq. 4) */
    int32_t lightning;      /* 1: same-block pairs only (C.7); 0: all pairs (C.5) */
    float threshold;        /* p: similarity above which the newest pair is zeroed */
    float lambda;           /* weight of the redundancy score in eq. (4) */
    float tau;              /* softmax temperature of the redundancy score (C.8) */
} zp_score_params;

/* Rows of lightning redundancy row sums [Zipage App. C.5 (definition), C.7
 * (same-block pairs)]: for each block of b = 16 tokens and each kv head, the
 * cosine matrix of the block's keys with a zero diagonal and, per column, the
 * newest row above the threshold p zeroed; rho[t] is the sum of row t.  Row r
 * of kv head h holds rho[t] at data + l*layer_stride + (r*h_kv + h)*stride + t
 * (t < L of the sequence the row belongs to).
 *   zp_paged_decode_attn_rho writes them: rows[s] (device int32 [B]) is the
 *     row of batch entry s, -1 = none; threshold is p.
 *   zp_compress_layers_rho reads them: rows (nullable, device int32 [n]) is the
 *     row of compressed sequence i (NULL: row i); threshold is not read (the
 *     row sums already hold it).
 * n_rows bounds the rows (a row >= n_rows is recorded as ZP_ERR_DEVICE). */
typedef struct zp_rho_rows {
    float *data;
    int64_t stride;        /* >= L of every sequence with a row */
    int64_t layer_stride;  /* elements between layers (zp_compress_layers_rho) */
    const int32_t *rows;
    int32_t n_rows;
    float threshold;       /* p */
} zp_rho_rows;

/* ---- status ------------------------------------------------------------- */
const char *zp_last_error(void);
const char *zp_status_string(zp_status s);
int32_t zp_version(void);
/* Reads (and, if clear != 0, resets) the device status word of the current
 * device: 0 = clean, else ZP_ERR_DEVICE / ZP_ERR_TIMEOUT with details in
 * *detail (nullable).  Synchronises the current device. */
zp_status zp_device_status(int32_t *code, int32_t *detail, int32_t clear);

/* ---- decode ------------------------------------------------------------- */

/* Bytes of workspace zp_paged_decode_attn needs for B sequences whose tables
 * have table_stride entries.  The workspace is scratch: any content is fine
 * on entry and it need not be kept between calls. */
size_t zp_decode_workspace_size(const zp_cache_desc *D, int32_t B, int32_t table_stride);

/* Paged GQA decode attention fused with window-score accumulation
 * [Zipage §3, §6; App. C.2 for the score].
 *
 * For every sequence s (L = seq_lens[s] >= 1 cached tokens, the newest one
 * included) and query head h:
 *     out[s][h] = sum_{t<L} softmax_t(q[s][h] . k_t / sqrt(d)) v_t
 * q, out: [B][h_q][d] (dtype); k_cache, v_cache: one layer, paged.
 *
 * score_accum (nullable, float [B][h_kv][table_stride*b], 16-byte aligned): the attention
 * score S of each sequence, one row per kv head indexed by token position
 * (row s belongs to batch entry s, as block-table row s does).  When set,
 * sequences whose query position P = L-1 lies in the observation window of
 * its block (P mod b >= b - window) add (1/window) * max over the q heads of
 * each kv head of the attention probability of every token t <= P; at the
 * first window row (P mod b == b - window) and for t == P the value is written
 * instead of added.  After the window steps that fill a block, S equals the
 * observation-window score of App. C.2 computed from those queries.  The
 * score lives with the sequence, not with the block: sequences that share
 * prefix blocks [§4.4] each score those tokens with their own queries.
 * score_rows (nullable, device int32 [B]) maps batch entry s to the row of S
 * it scores into -- the request's query slot [§4.2, §4.3] -- and then S holds
 * n_score_rows rows; -1 marks an entry without a slot, which is decoded but
 * not scored.  A slot >= n_score_rows is recorded as ZP_ERR_DEVICE (detail
 * 0x21) and not scored.  Without the map row s belongs to batch entry s.
 *
 * The workspace needs no clearing between calls.  After a call that left
 * ZP_ERR_TIMEOUT in the device status, clear it (zeros) before reusing it.
 * The kernel allows programmatic dependent launch of the next kernel on the
 * stream (zp_compress_layers uses it); kernels launched without that
 * attribute still start after it has completed.
 * Limits: B <= 4096, h_kv in {2,4,8,16}, h_q/h_kv in {4,8}, d in {64,128},
 * b a power of two >= 16.  Errors: ZP_ERR_INVALID_ARG (NULL buffer, B < 0,
 * window outside [1, b] with score_accum set), ZP_ERR_SHAPE, ZP_ERR_DTYPE,
 * ZP_ERR_CAPACITY (workspace_bytes too small), ZP_ERR_CUDA. */
zp_status zp_paged_decode_attn(const zp_cache_desc *D, const void *q, const void *k_cache,
                               const void *v_cache, const int32_t *block_table,
                               int32_t table_stride, const int32_t *seq_lens, int32_t B,
                               void *out, float *score_accum, const int32_t *score_rows,
                               int32_t n_score_rows, int32_t window, void *workspace,
                               size_t workspace_bytes, void *stream);

/* zp_paged_decode_attn that also computes, for the batch entries with a row
 * in rho (the sequences about to be compressed after this step), the lightning
 * redundancy row sums of every block of their keys [Zipage App. C.5, C.7]
 * from the key tiles the decode already holds on chip (no second read of the
 * keys).  The row sums equal, bit for bit, those zp_score_tokens and
 * zp_compress_layers compute for the same keys and threshold; a compression
 * that runs after this call with the same cache can take them through
 * zp_compress_layers_rho.  Outputs and scores of the decode are unchanged.
 * Requires the bf16 cache and b = 16 (ZP_ERR_SHAPE otherwise); a sequence
 * longer than rho->stride is not given row sums and is recorded as
 * ZP_ERR_DEVICE (detail 0x22).  Other arguments and errors: as
 * zp_paged_decode_attn. */
zp_status zp_paged_decode_attn_rho(const zp_cache_desc *D, const void *q, const void *k_cache,
                                   const void *v_cache, const int32_t *block_table,
                                   int32_t table_stride, const int32_t *seq_lens, int32_t B,
                                   void *out, float *score_accum, const int32_t *score_rows,
                                   int32_t n_score_rows, int32_t window, const zp_rho_rows *rho,
                                   void *workspace, size_t workspace_bytes, void *stream);

/* Same computation and arguments as zp_paged_decode_attn, without the
 * workspace: for callers that cannot allocate device memory when they decode
 * (a serving loop whose device memory is all reserved up front and which may
 * not call cudaMalloc between steps, or a host program, such as a plain C
 * client of this library, that has no device allocator of its own).  The paper has no
 * counterpart; this is an interface convenience.
 *
 * Scratch comes from one 64 MiB array built into the library; every GPU that
 * loads the library holds it until the process exits.  A call whose scratch
 * need (zp_decode_workspace_size) exceeds 64 MiB fails with ZP_ERR_CAPACITY
 * and does nothing.  No device memory is allocated by this call.
 * The first call on a device looks up the array's device address with that
 * device current; make that first call before any stream capture.
 * All calls share the array and it keeps the previous call's contents.  The
 * per-sequence control words of the in-kernel merge (its first B 64-bit
 * words) are read before the kernel writes them; a call that gave up on a
 * bounded wait (ZP_ERR_TIMEOUT) can leave them counting arrivals that never
 * completed.  Every call therefore zeroes those B words on `stream` before
 * its kernel, so a call after a timeout starts clean and the caller has
 * nothing to recover; every other part of the array is written before it is
 * read within a call.  Calls that may overlap on the GPU -- on different
 * streams, or from different threads -- race and must be ordered by the
 * caller. */
zp_status zp_paged_decode_attn_noalloc(const zp_cache_desc *D, const void *q, const void *k_cache,
                                       const void *v_cache, const int32_t *block_table,
                                       int32_t table_stride, const int32_t *seq_lens, int32_t B,
                                       void *out, float *score_accum, const int32_t *score_rows,
                                       int32_t n_score_rows, int32_t window, void *stream);

/* Test hook of zp_paged_decode_attn_noalloc (no counterpart in the paper):
 * writes control word `seq` of the current device's built-in array, as a
 * call that timed out could have left it, so that a test can check that the
 * next call clears it.  Blocking copy; allocates nothing.  ZP_ERR_INVALID_ARG
 * when the word lies outside the array. */
zp_status zp_debug_noalloc_preset_ctl(int32_t seq, uint64_t word);

/* Writes the new token's key and value of each sequence into its slot
 * [Zipage §3: the cache of a block is written into the block's slots]:
 * k_new, v_new [B][h_kv][d] go to slot (L-1) % b of block table[(L-1)/b],
 * where L = seq_lens[s] already counts the new token.  L = 0 skips the
 * sequence (no token this step); zp_paged_decode_attn likewise skips
 * sequences with L = 0 and leaves their output rows untouched. */
zp_status zp_append_kv(const zp_cache_desc *D, const void *k_new, const void *v_new,
                       void *k_cache, void *v_cache, const int32_t *block_table,
                       int32_t table_stride, const int32_t *seq_lens, int32_t B, void *stream);

/* ---- compression -------------------------------------------------------- */

/* Compression trigger [Zipage §4.1]: 1 iff ceil(L/b) >= max_blocks and L%b == 0. */
int32_t zp_needs_compression(int32_t seq_len, int32_t block_size, int32_t max_blocks);

/* zp_needs_compression over n sequences (host arrays, no device work):
 * triggered[0..*n_triggered) receives, ascending, every i with active[i] != 0
 * (active nullable: all) whose trigger holds at seq_lens[i] with the budget
 * max_blocks_seq[i] (nullable: max_blocks for all; per-request budgets,
 * Zipage Limitations).  triggered holds up to n entries. */
zp_status zp_needs_compression_batch(const int32_t *seq_lens, const uint8_t *active, int32_t n,
                                     int32_t block_size, int32_t max_blocks, const int32_t *max_blocks_seq,
                                     int32_t *triggered, int32_t *n_triggered);

/* Explicit observation-window score [Zipage App. C.2, Alg. 1] of n sequences
 * of one layer, for scoring without decode-time accumulation (a long prefill
 * compressed at its first trigger).  q_window [n][window][h_q][d] (dtype)
 * holds the queries of each sequence's `window` newest tokens, oldest first.
 *   A[u,h,t] = q_{u,h} . k_t / sqrt(d), -inf where t > L - window + u (causal;
 *              the mask printed in Alg. 1 is garbled, this is its reading)
 *   S[kvh][t] = (1/window) * sum_u max_{h in group(kvh)} softmax_t(A[u,h,:])[t]
 * scores_out: float [n][h_kv][Lmax], entries t >= L untouched.  Requires
 * window <= L <= Lmax.  bf16 caches: h_kv <= 8, b a multiple of 16 and
 * window * h_q/h_kv a multiple of 16 (ZP_ERR_SHAPE otherwise). */
size_t zp_window_score_workspace_size(const zp_cache_desc *D, int32_t n, int32_t Lmax, int32_t window);
zp_status zp_window_score(const zp_cache_desc *D, const void *q_window, int32_t window,
                          const void *k_cache, const int32_t *block_table, int32_t table_stride,
                          const int32_t *seq_lens, int32_t n, float *scores_out, int32_t Lmax,
                          void *workspace, size_t workspace_bytes, void *stream);

size_t zp_score_workspace_size(const zp_cache_desc *D, int32_t n, int32_t Lmax);

/* Per-sequence score rows: the attention score S written by
 * zp_paged_decode_attn (stride = table_stride*b, rows = the decode batch) or
 * by zp_window_score (stride = Lmax, rows = its n sequences).  Sequence i of a
 * call uses row rows[i] (rows NULL: row i) at
 *     data + l*layer_stride + (row*h_kv + kvh)*stride + t.
 * layer_stride matters only to zp_compact_pages with several layers. */
typedef struct zp_score_rows {
    float *data;
    int64_t stride;        /* >= L of every sequence */
    int64_t layer_stride;  /* elements between layers */
    const int32_t *rows;   /* nullable, int32 [n], device */
} zp_score_rows;

/* Final per-token scores of n sequences of one layer, ready for the top-k
 * [Zipage App. C.2-C.8, §4.2], in the paper's order:
 *   S  <- the sequence's attention-score rows in attn (decode-accumulated or
 *         explicit window score)                        (attention score)
 *   S  <- Alg. 2 with global_F when use_global: S on the first compression,
 *         else max(alpha*F, S) on blocks 0..N-2          (global score)
 *   Sp <- MaxPool1D(S) when pooling applies              (C.4, eq. 3)
 *   R  <- softmax_t(rho_t / (L*tau)) of the key redundancy (C.5 / C.7)
 *   out = Sp - lambda*R, then +inf on the last `window` tokens.
 * first_compression[n] (uint8) says whether each sequence was ever compressed
 * (Alg. 2 branch, pooling policy).  The global score replaces S in attn (t < L)
 * so that zp_compact_pages can store it into F of the kept tokens' new slots;
 * global_F (float [N_total][b][h_kv], paged like K) is only read, and only
 * on compressions after the first, when every block of the sequence is its
 * own [§4.4].  scores_out: float [n][h_kv][Lmax]; entries t >= L are left
 * untouched.  Requires window <= L <= min(Lmax, attn->stride). */
zp_status zp_score_tokens(const zp_cache_desc *D, const zp_score_params *P,
                          const void *k_cache, const int32_t *block_table, int32_t table_stride,
                          const int32_t *seq_lens, const uint8_t *first_compression, int32_t n,
                          const zp_score_rows *attn, const float *global_F, float *scores_out,
                          int32_t Lmax, void *workspace, size_t workspace_bytes, void *stream);

/* Top-k keep set [Zipage §4.2, App. C.6]: for every (sequence, kv head) the k
 * highest scores among t < L, equal scores ranked newer (larger t) first; the
 * kept positions are written ascending to keep_idx [n][h_kv][k].  If L <= k all
 * L positions are kept and keep_idx[L..k-1] = -1.  tie_count (nullable, int32
 * [n][h_kv]) receives how many tokens share the score of the k-th kept token
 * when that score was split between kept and dropped tokens, else 0.
 * Per-request budgets (Zipage, Limitations: N_max as an attribute of each request): k_seq
 * (nullable, device int32 [n]) gives sequence i its own k_i <= k; keep_idx
 * keeps the row stride k and rows are padded with -1 after k_i. */
zp_status zp_select_topk(const float *scores, int32_t h_kv, int32_t Lmax, const int32_t *seq_lens,
                         int32_t n, int32_t k, const int32_t *k_seq, int32_t *keep_idx, int32_t *tie_count,
                         void *stream);

/* KV compaction [Zipage App. C.6, Alg. 4; §4.4 target blocks]: for layers
 * [0, layer_count) (K and V of layer l at base + l*layer_stride elements),
 * every sequence i and kv head h, rank r < min(k, L_i) moves the row at
 * position keep_idx[l][i][h][r] (block src_table[i][pos/b]) to slot r%b of
 * block dst_targets[i][r/b].  The move is order preserving and safe when a
 * target block is the source block of the same index (in place).
 * global_F (nullable, layer l at global_F + l*F_layer_stride) receives at the
 * same slot the global score of the kept token, read from the score rows
 * `scores` left by zp_score_tokens ("compress score"); F is written only in
 * the target blocks.  src_table [n][table_stride], dst_targets
 * [n][target_stride] (at least ceil(k/b) entries), keep_idx
 * [layer_count][n][h_kv][k], seq_lens [n]; k_seq (nullable, device int32 [n])
 * moves min(k_seq[i], L_i) ranks of sequence i (its own budget, <= k). */
zp_status zp_compact_pages(const zp_cache_desc *D, void *k_base, void *v_base,
                           int64_t layer_stride, int32_t layer_count, float *global_F,
                           int64_t F_layer_stride, const zp_score_rows *scores,
                           const int32_t *src_table, int32_t table_stride,
                           const int32_t *dst_targets, int32_t target_stride,
                           const int32_t *seq_lens, const int32_t *keep_idx, int32_t k, const int32_t *k_seq,
                           int32_t n, void *stream);

/* Compression of n sequences over layer_count layers in one call [Zipage
 * App. C.1 (cross-layer parallel compression, layer stride), C.2-C.8, §4.2,
 * App. C.6 Alg. 4, §4.4]: per layer the final scores of zp_score_tokens, the
 * keep sets of zp_select_topk and the moves of zp_compact_pages (K and V rows
 * into dst_targets, F of each target slot <- the kept token's global score),
 * with the same rules and results.  Layer l uses k_base/v_base + l*layer_stride
 * elements, attn rows + l*attn->layer_stride, global_F + l*F_layer_stride,
 * keep_idx [layer_count][n][h_kv][k], tie_count (nullable)
 * [layer_count][n][h_kv] and scores_out (nullable) [layer_count][n][h_kv][Lmax].
 * For bf16 caches with b = 16 and the lightning redundancy, every layer runs
 * in one launch of each of two kernels: the global score and redundancy per
 * (block, sequence, layer), then per (kv head, sequence, layer) one CTA that
 * finishes the scores, selects the keep set and moves the rows from shared
 * memory (while 8*Lmax + 16*k bytes and the table row fit in it); otherwise
 * the three steps run layer by layer.  The workspace
 * (zp_compress_workspace_size) grows with layer_count: the paper's layer
 * stride is the number of layers per call.  k_seq (nullable, device int32
 * [n]): per-request budgets k_i <= k, as in zp_select_topk.
 * Ordering: both kernels of the fused path are launched as programmatic
 * dependents of the kernel before them on the stream.  They read the score
 * rows (and everything the decode may write) only after waiting for that
 * kernel's completion, so results are those of a plain stream-ordered call;
 * when zp_paged_decode_attn immediately precedes on the same stream, the
 * first kernel starts on the SMs the decode's finished CTAs leave and
 * computes the key redundancy while the decode drains.  Anything recorded
 * between the two calls (an event, a copy) only removes that overlap.  No
 * kernel of the call stores to memory before that wait, so its workspace and
 * outputs may be memory the preceding call has just released (the reuse a
 * stream-ordered allocator makes). */
size_t zp_compress_workspace_size(const zp_cache_desc *D, int32_t n, int32_t Lmax, int32_t layer_count);
zp_status zp_compress_layers(const zp_cache_desc *D, const zp_score_params *P, void *k_base, void *v_base,
                             int64_t layer_stride, int32_t layer_count, const int32_t *block_table,
                             int32_t table_stride, const int32_t *seq_lens, const uint8_t *first_compression,
                             int32_t n, const zp_score_rows *attn, float *global_F, int64_t F_layer_stride,
                             const int32_t *dst_targets, int32_t target_stride, int32_t k,
                             const int32_t *k_seq, int32_t *keep_idx,
                             int32_t *tie_count, float *scores_out, int32_t Lmax, void *workspace,
                             size_t workspace_bytes, void *stream);

/* zp_compress_layers with the lightning redundancy row sums given (rho, as
 * written by zp_paged_decode_attn_rho for the same keys) instead of computed:
 * the same scores, keep sets, moves, F and score-row updates, in ONE kernel per
 * call -- per (kv head, sequence, layer) the global score (Alg. 2) of the score
 * row, then the rest as zp_compress_layers; the second read of the keys and
 * the global/lightning kernel drop out.  Requires what the fused path of
 * zp_compress_layers requires (bf16, b = 16, use_similarity and lightning set,
 * the row in shared memory; ZP_ERR_SHAPE otherwise).  Layer l reads rho->data
 * + l*rho->layer_stride.  The workspace is not used (it may be NULL).  The
 * kernel is launched as a programmatic dependent of the kernel before it and
 * reads the score rows and rho only after that kernel has completed. */
/* 1 when zp_compress_layers_rho accepts this cache, these switches, Lmax and k
 * on the current device (the one-kernel path: bf16, b = 16, d 64 or 128,
 * h_kv <= 16, similarity with the lightning redundancy, a row of Lmax scores
 * and k ranks in shared memory), else 0.  No device work. */
int32_t zp_compress_rho_supported(const zp_cache_desc *D, const zp_score_params *P, int32_t Lmax, int32_t k);
zp_status zp_compress_layers_rho(const zp_cache_desc *D, const zp_score_params *P, void *k_base, void *v_base,
                                 int64_t layer_stride, int32_t layer_count, const int32_t *block_table,
                                 int32_t table_stride, const int32_t *seq_lens, const uint8_t *first_compression,
                                 int32_t n, const zp_score_rows *attn, float *global_F, int64_t F_layer_stride,
                                 const int32_t *dst_targets, int32_t target_stride, int32_t k,
                                 const int32_t *k_seq, int32_t *keep_idx, int32_t *tie_count, float *scores_out,
                                 int32_t Lmax, const zp_rho_rows *rho, void *stream);

/* ---- host block pool and planner (no device work) ------------------------ */
typedef struct zp_pool zp_pool;

/* Pool of n_total blocks, all free, reference count 0 [Zipage §3, §4.4]. */
zp_pool *zp_pool_create(int32_t n_total);
void zp_pool_destroy(zp_pool *pool);
int32_t zp_pool_num_free(const zp_pool *pool);
int32_t zp_pool_refcount(const zp_pool *pool, int32_t block);
/* Takes n free blocks (reference count 1), lowest free id first.
 * ZP_ERR_CAPACITY if fewer than n are free (nothing is taken). */
zp_status zp_pool_alloc(zp_pool *pool, int32_t n, int32_t *ids);
/* Adds one reference to each block (prefix sharing). */
zp_status zp_pool_incref(zp_pool *pool, int32_t n, const int32_t *ids);
/* Drops one reference from each block; a block reaching 0 becomes free. */
zp_status zp_pool_release(zp_pool *pool, int32_t n, const int32_t *ids);

/* Target blocks of one compression [Zipage §4.1, §4.4]: target t is a new
 * block when table[t] is shared (reference count > 1), else table[t]; the
 * reserved block is table[max_blocks-1] when not shared, else new.  New blocks
 * are taken from the pool.  Outputs: targets[max_blocks-1], new_table
 * [max_blocks] (targets + reserved), dropped[n_dropped] = the blocks of the old
 * table that the new one no longer holds (own and shared); the caller releases
 * them with zp_pool_release once the compaction that reads them has finished.
 * *n_fresh = new blocks taken.  Requires n_blocks >= max_blocks >= 2. */
zp_status zp_plan_compaction(zp_pool *pool, const int32_t *table, int32_t n_blocks,
                             int32_t max_blocks, int32_t *targets, int32_t *new_table,
                             int32_t *dropped, int32_t *n_dropped, int32_t *n_fresh);

/* zp_plan_compaction for n sequences in one call.  tables [n][table_stride]
 * (sequence i holds n_blocks[i] <= table_stride blocks); outputs per sequence:
 * targets [n][max_blocks-1], new_tables [n][max_blocks], dropped
 * [n][table_stride] (first n_dropped[i] valid), n_fresh [n].  max_blocks_seq
 * (nullable, host int32 [n]): per-request budgets N_max,i <= max_blocks (rows
 * padded with -1 after N_max,i - 1 targets and N_max,i blocks).  Stops at the
 * first sequence that fails (earlier ones stay planned) and returns its error. */
zp_status zp_plan_compaction_batch(zp_pool *pool, const int32_t *tables, int32_t table_stride,
                                   const int32_t *n_blocks, int32_t n, int32_t max_blocks,
                                   const int32_t *max_blocks_seq, int32_t *targets, int32_t *new_tables,
                                   int32_t *dropped, int32_t *n_dropped, int32_t *n_fresh);

/* Capacity plan [Zipage §4.2 eq. (1), App. C.3 eq. (2)] (host only): the
 * largest request concurrency M and the block count N_total for a memory
 * budget, maximising M subject to
 *     (1 + extra) * m_kv_block * N_total + M * m_q_request <= m_available,
 *     M <= N_total / max_blocks,  M > 0,  N_total > 0,
 * with extra = extra_num / extra_den the per-block overhead of the global
 * score cache relative to K and V (the paper's 1/(2d); 0/1 without it).
 * Returns M = floor(m_available / ((1+extra) m_kv N_max + m_q)) and the
 * linear program's N_total = floor(m_available / ((1+extra) m_kv + m_q/N_max)).
 * m_kv_block: bytes of one block's K and V over all layers; m_q_request:
 * per-request bytes that do not depend on N_total (the paper's query cache;
 * here the attention-score rows).  ZP_ERR_CAPACITY when M would be 0. */
zp_status zp_plan_capacity(int64_t m_available, int64_t m_kv_block, int64_t m_q_request, int32_t max_blocks,
                           int64_t extra_num, int64_t extra_den, int64_t *M, int64_t *N_total);

#ifdef __cplusplus
}
#endif
#endif /* ZP_H */
