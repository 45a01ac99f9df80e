/*
 * zp_oracle.c -- plain, slow, fp64 CPU oracle for the Compressed PagedAttention
 * hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call
 * this file: only the tests, the smoke check and the benchmark's CPU-baseline
 * leg use it.  It shares no code, header, table or helper with the CUDA library.
 *
 * Source of every definition below: the paper "Zipage: Maintain High Request
 * Concurrency for LLM Reasoning through Compressed PagedAttention" (Liao et al.,
 * arXiv 2603.08743), cited as [Zipage <section>].  Where the text is silent or
 * garbled the reading taken is written next to the code.
 *
 * Conventions shared by all functions:
 *   - Paged caches have the layout the paper gives for K and V in [Zipage §3]:
 *     one layer is [N_total][b][h_kv][d]; element (blk, slot, kvh, i) sits at
 *     ((blk*b + slot)*h_kv + kvh)*d + i.
 *   - Per-slot score arrays (the accumulated window score S and the global
 *     score cache F of [Zipage App. C.3]) are [N_total][b][h_kv].
 *   - Token t of a sequence lives in block block_table[t / b], slot t % b.
 *   - Query head h uses key/value head h / (h_q / h_kv) (contiguous GQA
 *     groups; the paper does not state the map, this is the usual one).
 *   - Inputs arrive as float (bf16 values are exactly representable in float);
 *     every sum, exponential and division is done in double.
 *
 * Parity status of each function (pins live in tests/test_oracle_pins.py):
 *   orc_decode_attention          pinned (SDPA library, L=1, q=0, permutation)
 *   orc_accumulate_window_score   pinned (equals orc_window_score; closed form
 *                                 and masked brute force fixing the order of
 *                                 the two reductions)
 *   orc_window_score              pinned (row sums, w=1 == decode probabilities,
 *                                 a closed form where max-then-mean and
 *                                 mean-then-max differ, masked brute force)
 *   orc_global_score              pinned (hand-worked example, alpha=0, first)
 *   orc_max_pool                  pinned (torch max_pool1d, kernel 1)
 *   orc_redundancy                pinned (closed forms for identical and
 *                                 orthogonal keys, lightning == full for L<=b)
 *   orc_redundancy_rho            pinned (closed forms for identical and
 *                                 orthogonal keys, pure-Python brute force,
 *                                 softmax of it == orc_redundancy; lightning
 *                                 row sums with p < -1 in closed form)
 *   orc_redundancy_rho_rows       pinned (equals orc_redundancy_rho row by
 *                                 row with planted near-duplicates; closed form)
 *   orc_combine_and_window        pinned (lambda=0, window = +inf, a
 *                                 hand-worked example with lambda=2; the
 *                                 order global score, pooling, combination
 *                                 worked by hand through the step pipeline)
 *   orc_topk_keep                 pinned (exhaustive subsets, Fig. 1 example)
 *   orc_compact_alg4              pinned (Fig. 1 layout, bitwise moves)
 *   orc_plan_targets              pinned (both cases of [Zipage §4.4], Fig. 1)
 *   orc_needs_compression         pinned (Fig. 1 trigger)
 * The threshold p of the redundancy score and the pooling kernel size are not
 * given by the paper; they are parameters here and their default values are
 * unpinned constants (every result is pinned for the value passed in).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_BAD_ARG 1
#define ORC_NO_MEMORY 2

static size_t cache_index(int blk, int slot, int kvh, int b, int h_kv, int d) {
    return (((size_t)blk * (size_t)b + (size_t)slot) * (size_t)h_kv + (size_t)kvh) * (size_t)d;
}

static size_t slot_index(int blk, int slot, int kvh, int b, int h_kv) {
    return ((size_t)blk * (size_t)b + (size_t)slot) * (size_t)h_kv + (size_t)kvh;
}

/* ------------------------------------------------------------------------- */
/* Decode attention over a paged cache [Zipage §3 (paged K, V and block       */
/* table), §6 (attention on the paged cache at decode)].                     */
/*                                                                           */
/* For sequence s with L = seq_lens[s] cached tokens (the newest token, whose */
/* key and value are already in the cache, included) and query head h:        */
/*   a_t  = q_{s,h} . k_{t,kvh} / sqrt(d)          t < L                     */
/*   p_t  = exp(a_t - max a) / sum_j exp(a_j - max a)                          */
/*   out  = sum_t p_t v_{t,kvh}                                               */
/* probs (nullable) receives p_t at probs[(s*h_q + h)*probs_stride + t].      */
/* ------------------------------------------------------------------------- */
int orc_decode_attention(int B, int h_q, int h_kv, int d, int b,
                         const float *q, const float *k_cache, const float *v_cache,
                         const int32_t *block_table, int table_stride,
                         const int32_t *seq_lens,
                         double *out, double *probs, int probs_stride) {
    if (B < 0 || h_q <= 0 || h_kv <= 0 || h_q % h_kv != 0 || d <= 0 || b <= 0)
        return ORC_BAD_ARG;
    const int g = h_q / h_kv;
    const double scale = 1.0 / sqrt((double)d);
    for (int s = 0; s < B; ++s) {
        const int L = seq_lens[s];
        if (L <= 0) return ORC_BAD_ARG;
        if (probs && L > probs_stride) return ORC_BAD_ARG;
        double *a = (double *)malloc(sizeof(double) * (size_t)L);
        if (!a) return ORC_NO_MEMORY;
        for (int h = 0; h < h_q; ++h) {
            const int kvh = h / g;
            const float *qv = q + ((size_t)s * h_q + h) * d;
            double amax = -INFINITY;
            for (int t = 0; t < L; ++t) {
                const int blk = block_table[(size_t)s * table_stride + t / b];
                const float *kv = k_cache + cache_index(blk, t % b, kvh, b, h_kv, d);
                double dot = 0.0;
                for (int i = 0; i < d; ++i) dot += (double)qv[i] * (double)kv[i];
                a[t] = dot * scale;
                if (a[t] > amax) amax = a[t];
            }
            double denom = 0.0;
            for (int t = 0; t < L; ++t) denom += exp(a[t] - amax);
            double *o = out + ((size_t)s * h_q + h) * d;
            for (int i = 0; i < d; ++i) o[i] = 0.0;
            for (int t = 0; t < L; ++t) {
                const double p = exp(a[t] - amax) / denom;
                if (probs) probs[((size_t)s * h_q + h) * probs_stride + t] = p;
                const int blk = block_table[(size_t)s * table_stride + t / b];
                const float *vv = v_cache + cache_index(blk, t % b, kvh, b, h_kv, d);
                for (int i = 0; i < d; ++i) o[i] += p * (double)vv[i];
            }
        }
        free(a);
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* Window score accumulated during decode.                                    */
/*                                                                           */
/* [Zipage App. C.2] scores the cache with the queries of the last w tokens   */
/* of the final block: per query row, softmax over the sequence, max over the */
/* query heads of a KV head, then mean over the w rows.  Under causal decoding */
/* the query of the token at position P sees exactly tokens t <= P, the same  */
/* set the causal mask of Alg. 1 leaves visible, so the window score can be   */
/* accumulated one decode step at a time.  This function is that per-step    */
/* form (a reading, not a separate algorithm of the paper):                   */
/*   window step:  P = L - 1 with P mod b >= b - w                            */
/*   c(t, kvh)  = (1/w) * max_{h in group(kvh)} p_{s,h}(t)        t <= P       */
/*   S[t, kvh]  = c              if P mod b == b - w (first window row) or t==P */
/*              = S[t, kvh] + c  otherwise                                    */
/* Steps that are not window steps leave S untouched.  After the w steps that */
/* end at a full block, S equals orc_window_score for those w queries.        */
/* ------------------------------------------------------------------------- */
int orc_accumulate_window_score(int B, int h_q, int h_kv, int b, int w,
                                const int32_t *block_table, int table_stride,
                                const int32_t *seq_lens,
                                const double *probs, int probs_stride,
                                double *score) {
    if (h_q <= 0 || h_kv <= 0 || h_q % h_kv != 0 || w <= 0 || w > b) return ORC_BAD_ARG;
    const int g = h_q / h_kv;
    for (int s = 0; s < B; ++s) {
        const int L = seq_lens[s];
        const int P = L - 1;
        const int r = P % b;
        if (r < b - w) continue;
        const int first_row = (r == b - w);
        for (int kvh = 0; kvh < h_kv; ++kvh) {
            for (int t = 0; t < L; ++t) {
                double best = 0.0;
                for (int j = 0; j < g; ++j) {
                    const double p = probs[((size_t)s * h_q + kvh * g + j) * probs_stride + t];
                    if (j == 0 || p > best) best = p;
                }
                const double c = best / (double)w;
                const int blk = block_table[(size_t)s * table_stride + t / b];
                const size_t at = slot_index(blk, t % b, kvh, b, h_kv);
                if (first_row || t == P) score[at] = c;
                else score[at] += c;
            }
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* Explicit observation-window attention score [Zipage App. C.2, Alg. 1].     */
/*                                                                           */
/* One sequence of L tokens; q_window[u][h][i] holds the queries of the w    */
/* newest tokens (positions L-w .. L-1), u = 0 oldest.                       */
/*   A[u,h,t] = q_{u,h} . k_t / sqrt(d), set to -inf where t > L - w + u      */
/* The mask printed in Alg. 1 ("-inf if u + b - w > v") is garbled: it would */
/* hide the past and show the future.  The reading taken is the causal mask   */
/* (query u at position L-w+u sees keys t <= L-w+u); for a full last block    */
/* this is "-inf iff v > u + b - w" on the last block, as Alg. 1 intends.     */
/*   P[u,h,:] = softmax over t < L of A[u,h,:]                                */
/*   S[kvh,t] = (1/w) * sum_u max_{h in group(kvh)} P[u,h,t]                  */
/* (max over the heads of a group first, then the mean over the window, in   */
/* the order the text gives them.)  S is [h_kv][L].                          */
/* ------------------------------------------------------------------------- */
int orc_window_score(int h_q, int h_kv, int d, int b, int w,
                     const float *q_window, const float *k_cache,
                     const int32_t *table_row, int L, double *S) {
    if (h_q <= 0 || h_kv <= 0 || h_q % h_kv != 0 || w <= 0 || L < w) return ORC_BAD_ARG;
    const int g = h_q / h_kv;
    const double scale = 1.0 / sqrt((double)d);
    double *P = (double *)malloc(sizeof(double) * (size_t)g * (size_t)L);
    if (!P) return ORC_NO_MEMORY;
    for (int kvh = 0; kvh < h_kv; ++kvh) {
        for (int t = 0; t < L; ++t) S[(size_t)kvh * L + t] = 0.0;
        for (int u = 0; u < w; ++u) {
            const int last_visible = L - w + u;
            for (int j = 0; j < g; ++j) {
                const int h = kvh * g + j;
                const float *qv = q_window + ((size_t)u * h_q + h) * d;
                double *row = P + (size_t)j * L;
                double amax = -INFINITY;
                for (int t = 0; t < L; ++t) {
                    if (t > last_visible) { row[t] = -INFINITY; continue; }
                    const int blk = table_row[t / b];
                    const float *kv = k_cache + cache_index(blk, t % b, kvh, b, h_kv, d);
                    double dot = 0.0;
                    for (int i = 0; i < d; ++i) dot += (double)qv[i] * (double)kv[i];
                    row[t] = dot * scale;
                    if (row[t] > amax) amax = row[t];
                }
                double denom = 0.0;
                for (int t = 0; t <= last_visible; ++t) denom += exp(row[t] - amax);
                for (int t = 0; t < L; ++t)
                    row[t] = (t > last_visible) ? 0.0 : exp(row[t] - amax) / denom;
            }
            for (int t = 0; t < L; ++t) {
                double best = P[t];
                for (int j = 1; j < g; ++j)
                    if (P[(size_t)j * L + t] > best) best = P[(size_t)j * L + t];
                S[(size_t)kvh * L + t] += best / (double)w;
            }
        }
    }
    free(P);
    return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* Global score update [Zipage App. C.3, Alg. 2].                             */
/*                                                                           */
/* S is the sequence's score, [h_kv][L] contiguous; F is the paged global     */
/* score cache [N_total][b][h_kv].  With N = ceil(L/b) blocks:               */
/*   not yet compressed (first != 0):  F[block i] <- S[block i]  for all i    */
/*   compressed before:                for i < N-1: s <- max(alpha*F, s)      */
/*                                     F[block i] <- s; S[block i] <- s        */
/* The last block has no history and keeps its fresh score.                  */
/* ------------------------------------------------------------------------- */
int orc_global_score(int L, int b, int h_kv, int first, double alpha,
                     const int32_t *table_row, double *F, double *S) {
    if (L <= 0 || b <= 0 || h_kv <= 0) return ORC_BAD_ARG;
    const int N = (L + b - 1) / b;
    for (int i = 0; i < N; ++i) {
        for (int j = 0; j < b; ++j) {
            const int t = i * b + j;
            if (t >= L) break;
            for (int kvh = 0; kvh < h_kv; ++kvh) {
                const size_t at = slot_index(table_row[i], j, kvh, b, h_kv);
                double s = S[(size_t)kvh * L + t];
                if (first) {
                    F[at] = s;
                } else {
                    if (i != N - 1) {
                        const double f = F[at];
                        if (alpha * f > s) s = alpha * f;
                    }
                    F[at] = s;
                    S[(size_t)kvh * L + t] = s;
                }
            }
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* Max pooling along the sequence [Zipage App. C.4, eq. (3)]:                */
/*   y[t] = max { x[j] : |j - t| <= r, 0 <= j < L },  kernel = 2r + 1        */
/* i.e. MaxPool1D with stride 1 and same-length output.  The paper does not  */
/* give the kernel size; it is a parameter (odd, >= 1).                      */
/* ------------------------------------------------------------------------- */
int orc_max_pool(int L, int kernel, const double *x, double *y) {
    if (L < 0 || kernel < 1 || kernel % 2 == 0) return ORC_BAD_ARG;
    const int r = kernel / 2;
    for (int t = 0; t < L; ++t) {
        const int lo = t - r < 0 ? 0 : t - r;
        const int hi = t + r > L - 1 ? L - 1 : t + r;
        double m = x[lo];
        for (int j = lo + 1; j <= hi; ++j)
            if (x[j] > m) m = x[j];
        y[t] = m;
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* Redundancy score of the keys [Zipage App. C.5 (full, Fig. 11), C.7        */
/* (lightning, Fig. 15), C.8 (temperature)].                                 */
/*                                                                           */
/* keys is one sequence's keys of one KV head, gathered, [L][d].  The pair  */
/* domain splits the positions into groups: one group [0, L) for the full   */
/* score, the blocks [j*b, min((j+1)*b, L)) for the lightning score (only    */
/* same-block pairs are compared).  Within a group of m positions:           */
/*   C[r][c] = cos(k_r, k_c)                                                 */
/*   C[c][c] = 0                                                             */
/*   for each column c: r* = largest r with C[r][c] > p; C[r*][c] = 0        */
/*   rho[r] = sum_c C[r][c]                                                  */
/* and over the whole sequence                                               */
/*   R = softmax_t( rho[t] / (L * tau) )                                     */
/* A key of zero norm has cosine 0 with every key.  The paper normalises by  */
/* the sequence length for the full score and does not restate it for the    */
/* lightning score; C.7 changes only the pair domain, so the same length     */
/* normalisation is used for both.  Memory is O(m^2) for the largest group.  */
/* ------------------------------------------------------------------------- */
/* The row sums rho[t] (before the normalisation and the softmax) of the     */
/* groups above, for every position.                                        */
int orc_redundancy_rho(int L, int d, int b, const float *keys, double p, int lightning, double *rho) {
    if (L <= 0 || d <= 0 || b <= 0) return ORC_BAD_ARG;
    const int group = lightning ? (b < L ? b : L) : L;
    double *norm = (double *)malloc(sizeof(double) * (size_t)L);
    double *C = (double *)malloc(sizeof(double) * (size_t)group * (size_t)group);
    if (!norm || !C) { free(norm); free(C); return ORC_NO_MEMORY; }
    for (int t = 0; t < L; ++t) {
        double ss = 0.0;
        for (int i = 0; i < d; ++i) ss += (double)keys[(size_t)t * d + i] * (double)keys[(size_t)t * d + i];
        norm[t] = sqrt(ss);
    }
    for (int g0 = 0; g0 < L; g0 += group) {
        const int m = (L - g0 < group) ? L - g0 : group;
        for (int r = 0; r < m; ++r) {
            for (int c = 0; c < m; ++c) {
                const int tr = g0 + r, tc = g0 + c;
                double v = 0.0;
                if (norm[tr] > 0.0 && norm[tc] > 0.0) {
                    double dot = 0.0;
                    for (int i = 0; i < d; ++i)
                        dot += (double)keys[(size_t)tr * d + i] * (double)keys[(size_t)tc * d + i];
                    v = dot / (norm[tr] * norm[tc]);
                }
                C[(size_t)r * m + c] = v;
            }
        }
        for (int c = 0; c < m; ++c) C[(size_t)c * m + c] = 0.0;
        for (int c = 0; c < m; ++c) {
            for (int r = m - 1; r >= 0; --r) {
                if (C[(size_t)r * m + c] > p) { C[(size_t)r * m + c] = 0.0; break; }
            }
        }
        for (int r = 0; r < m; ++r) {
            double acc = 0.0;
            for (int c = 0; c < m; ++c) acc += C[(size_t)r * m + c];
            rho[g0 + r] = acc;
        }
    }
    free(norm); free(C);
    return ORC_OK;
}

int orc_redundancy(int L, int d, int b, const float *keys, double p, double tau,
                   int lightning, double *R) {
    if (L <= 0 || d <= 0 || b <= 0 || !(tau > 0.0)) return ORC_BAD_ARG;
    double *rho = (double *)malloc(sizeof(double) * (size_t)L);
    if (!rho) return ORC_NO_MEMORY;
    const int rc = orc_redundancy_rho(L, d, b, keys, p, lightning, rho);
    if (rc != ORC_OK) { free(rho); return rc; }
    for (int r = 0; r < L; ++r) rho[r] = rho[r] / ((double)L * tau);
    double rmax = -INFINITY;
    for (int r = 0; r < L; ++r)
        if (rho[r] > rmax) rmax = rho[r];
    double denom = 0.0;
    for (int r = 0; r < L; ++r) denom += exp(rho[r] - rmax);
    for (int r = 0; r < L; ++r) R[r] = exp(rho[r] - rmax) / denom;
    free(rho);
    return ORC_OK;
}

/* The all-pairs row sums rho[r] of the definition above for the selected   */
/* rows only, without the L x L matrix (O(L) memory): with C the cosine     */
/* matrix (zero diagonal),                                                  */
/*   rho[r] = sum_c C[r][c] - sum { C[r][c] : r is the largest j with        */
/*                                  C[j][c] > p }                            */
/* and only a column c with C[r][c] > p can have r as that largest index,    */
/* so column c is scanned (newest row first) only for those.  Each cosine is */
/* computed exactly as in orc_redundancy_rho.                               */
static double cosine_at(const float *keys, const double *norm, int d, int tr, int tc) {
    if (tr == tc || !(norm[tr] > 0.0 && norm[tc] > 0.0)) return 0.0;
    double dot = 0.0;
    for (int i = 0; i < d; ++i) dot += (double)keys[(size_t)tr * d + i] * (double)keys[(size_t)tc * d + i];
    return dot / (norm[tr] * norm[tc]);
}

int orc_redundancy_rho_rows(int L, int d, const float *keys, double p, const int32_t *rows, int nrows,
                            double *out) {
    if (L <= 0 || d <= 0 || nrows < 0) return ORC_BAD_ARG;
    double *norm = (double *)malloc(sizeof(double) * (size_t)L);
    if (!norm) return ORC_NO_MEMORY;
    for (int t = 0; t < L; ++t) {
        double ss = 0.0;
        for (int i = 0; i < d; ++i) ss += (double)keys[(size_t)t * d + i] * (double)keys[(size_t)t * d + i];
        norm[t] = sqrt(ss);
    }
    for (int k = 0; k < nrows; ++k) {
        const int r = rows[k];
        if (r < 0 || r >= L) { free(norm); return ORC_BAD_ARG; }
        double sum = 0.0;
        for (int c = 0; c < L; ++c) sum += cosine_at(keys, norm, d, r, c);
        for (int c = 0; c < L; ++c) {
            if (c == r) continue;  /* zeroing the diagonal changes nothing */
            const double v = cosine_at(keys, norm, d, r, c);
            if (!(v > p)) continue;
            int newest = r;
            for (int j = L - 1; j > r; --j)
                if (cosine_at(keys, norm, d, j, c) > p) { newest = j; break; }
            if (newest == r) sum -= v;
        }
        out[k] = sum;
    }
    free(norm);
    return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* Score combination and observation-window protection                        */
/* [Zipage App. C.5 eq. (4); §4.2 and App. C.6 (window set to +inf)]:         */
/*   S[t] <- S[t] - lambda * R[t]          (R nullable: no redundancy term)   */
/*   S[t] <- +inf                          for t >= L - w                     */
/* ------------------------------------------------------------------------- */
int orc_combine_and_window(int L, int w, double lambda, const double *R, double *S) {
    if (L < 0 || w < 0) return ORC_BAD_ARG;
    for (int t = 0; t < L; ++t) {
        if (R) S[t] = S[t] - lambda * R[t];
        if (t >= L - w) S[t] = INFINITY;
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* Top-k keep set [Zipage §4.2 (k = (N_max-1)*b), App. C.6 (top-k tag)].      */
/*                                                                           */
/* Marks the k highest scores of one (sequence, layer, KV head) and returns  */
/* their positions in ascending order (the order Alg. 4 preserves).  The    */
/* paper does not fix the order among equal scores; the reading taken is    */
/* that the newer token (larger position) wins, in the spirit of C.5's      */
/* preference for retaining newer tokens.  If L <= k every token is kept and */
/* keep[L..k-1] = -1.  Returns the number kept.  tag (nullable) receives the */
/* 0/1 tag T of C.6 for t < L.                                              */
/* ------------------------------------------------------------------------- */
typedef struct { double score; int pos; } orc_ranked;

/* qsort order: higher score first; among equal scores the larger position */
static int ranked_before(const void *x, const void *y) {
    const orc_ranked *a = (const orc_ranked *)x, *c = (const orc_ranked *)y;
    if (a->score > c->score) return -1;
    if (a->score < c->score) return 1;
    return (a->pos > c->pos) ? -1 : (a->pos < c->pos);
}

int orc_topk_keep(int L, int k, const double *score, int32_t *keep, uint8_t *tag) {
    if (L < 0 || k < 0) return -1;
    for (int t = 0; t < L; ++t)
        if (score[t] != score[t]) return -1; /* NaN is not a valid score */
    uint8_t *T = (uint8_t *)calloc((size_t)(L > 0 ? L : 1), 1);
    orc_ranked *order = (orc_ranked *)malloc(sizeof(orc_ranked) * (size_t)(L > 0 ? L : 1));
    if (!T || !order) { free(T); free(order); return -1; }
    for (int t = 0; t < L; ++t) { order[t].score = score[t]; order[t].pos = t; }
    qsort(order, (size_t)L, sizeof(orc_ranked), ranked_before);
    for (int j = 0; j < L && j < k; ++j) T[order[j].pos] = 1;
    int n = 0;
    for (int t = 0; t < L; ++t)
        if (T[t]) keep[n++] = t;
    for (int j = n; j < k; ++j) keep[j] = -1;
    if (tag) memcpy(tag, T, (size_t)L);
    free(T);
    free(order);
    return n;
}

/* ------------------------------------------------------------------------- */
/* KV compaction [Zipage App. C.6, Alg. 4] for one sequence, one layer, one  */
/* KV head, as a byte move.                                                 */
/*                                                                           */
/* The read pointer walks every slot of the sequence's N blocks (src_table)  */
/* in order; whenever the tag of the slot is 1 the row is copied to the     */
/* write pointer, which walks the slots of the target blocks (dst_table) in */
/* order.  row_bytes = d * element size for K and V, one element for the    */
/* global score cache F (the "compress score" move of C.6).  With           */
/* dst_table == src_table this is the in-place move of Alg. 4; with the     */
/* target blocks of [Zipage §4.4] it is the redirected move.  Returns the   */
/* number of rows moved.                                                    */
/*   base: the layer's cache, rows addressed as ((blk*b + slot)*h_kv + kvh) */
/* ------------------------------------------------------------------------- */
int orc_compact_alg4(uint8_t *base, size_t row_bytes, int b, int h_kv, int kvh,
                     const int32_t *src_table, int N, const int32_t *dst_table,
                     const uint8_t *tag) {
    int read_block = 0, read_slot = 0;   /* p_r */
    int write_block = 0, write_slot = 0; /* p_w */
    int moved = 0;
    for (int l = 0; read_block < N; ++l) {
        if (tag[l]) {
            const size_t src = slot_index(src_table[read_block], read_slot, kvh, b, h_kv) * row_bytes;
            const size_t dst = slot_index(dst_table[write_block], write_slot, kvh, b, h_kv) * row_bytes;
            memmove(base + dst, base + src, row_bytes);
            ++moved;
            if (moved % b == 0) { ++write_block; write_slot = 0; }
            else ++write_slot;
        }
        if ((l + 1) % b == 0) { ++read_block; read_slot = 0; }
        else ++read_slot;
    }
    return moved;
}

/* ------------------------------------------------------------------------- */
/* Compression trigger [Zipage §4.1]: after a decode step a sequence that    */
/* occupies N >= N_max blocks with its last block full is compressed.        */
/* ------------------------------------------------------------------------- */
int orc_needs_compression(int L, int b, int N_max) {
    if (L <= 0) return 0;
    const int N = (L + b - 1) / b;
    return N >= N_max && L % b == 0;
}

/* ------------------------------------------------------------------------- */
/* Target blocks and the new block table [Zipage §4.1, §4.4, Fig. 1, Fig. 3]. */
/*                                                                           */
/* table[0..N-1]: the sequence's blocks; ref[blk]: reference counts (> 1     */
/* means shared).  fresh[]: free block ids, used in order when a new block   */
/* is needed.  Outputs:                                                      */
/*   targets[0..N_max-2]  where the kept tokens go (Alg. 4 write pointer)    */
/*   new_table[0..N_max-1] = targets followed by the reserved block          */
/*   released[]          own blocks dropped from the table (to the pool)    */
/*   dropped_shared[]    shared blocks left by this sequence (ref - 1)       */
/* Rule ([Zipage §4.4], read position by position): target t is a new block  */
/* if table[t] is shared, else table[t] itself.  This gives the two cases of */
/* the text: N_prefix >= N_max-1 shared blocks -> N_max-1 new targets;      */
/* otherwise N_prefix new blocks plus N_max-1-N_prefix of the sequence's own */
/* blocks.  The reserved N_max-th block is table[N_max-1] when that block is */
/* the sequence's own, else a new block (decode must never write a shared   */
/* block).  Every other own block is released.  Fig. 1 (no sharing) then    */
/* reads: blocks a, b, c are the targets, d is reserved, the rest released. */
/* Returns the number of fresh blocks used, or -1.                          */
/* ------------------------------------------------------------------------- */
int orc_plan_targets(const int32_t *table, int N, int N_max, const int32_t *ref,
                     const int32_t *fresh, int n_fresh,
                     int32_t *targets, int32_t *new_table,
                     int32_t *released, int *n_released,
                     int32_t *dropped_shared, int *n_dropped) {
    if (N_max < 2 || N < N_max) return -1;
    int used = 0;
    for (int t = 0; t < N_max - 1; ++t) {
        if (ref[table[t]] > 1) {
            if (used >= n_fresh) return -1;
            targets[t] = fresh[used++];
        } else {
            targets[t] = table[t];
        }
        new_table[t] = targets[t];
    }
    if (ref[table[N_max - 1]] > 1) {
        if (used >= n_fresh) return -1;
        new_table[N_max - 1] = fresh[used++];
    } else {
        new_table[N_max - 1] = table[N_max - 1];
    }
    *n_released = 0;
    *n_dropped = 0;
    for (int i = 0; i < N; ++i) {
        int kept = 0;
        for (int j = 0; j < N_max; ++j)
            if (new_table[j] == table[i]) kept = 1;
        if (kept) continue;
        if (ref[table[i]] > 1) dropped_shared[(*n_dropped)++] = table[i];
        else released[(*n_released)++] = table[i];
    }
    return used;
}
