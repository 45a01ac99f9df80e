// window_score.cu -- explicit observation-window attention score.
//
// Zipage paper App. C.2 with Alg. 1: for a sequence of L tokens and the
// queries of its w newest tokens (q_window[u], u = 0 oldest, at position
// L - w + u), for every kv head:
//   A[u,h,t] = q_{u,h} . k_t / sqrt(d), -inf where t > L - w + u  (causal; the
//              printed mask of Alg. 1 is garbled, this is its reading)
//   P[u,h,:] = softmax over t of A[u,h,:]
//   S[t]     = (1/w) * sum_u max_{h in the kv head's group} P[u,h,t]
// This is the prefill-then-compress path: after a long prompt the window
// queries exist but no decode step has accumulated the score.
//
// The R = w*g query rows of a kv head against the sequence's keys form a
// dense contraction (64 x 128 x L for the Qwen3-8B shape), run on the
// fifth-generation tensor cores in two passes over K (see the bf16 path
// below: tcgen05.mma with the tokens as the M = 128 operand, accumulators in
// tensor memory, TMA loads of the keys and of the window queries).  fp32
// caches take a plain CUDA-core kernel (the small parity workload, 1e-4).
#include <math.h>

#include "tc05.cuh"

namespace zp {
namespace {


struct WsArgs {
    const void *q;       // [n][w][h_q][d]
    const void *k;
    const int32_t *table;
    int table_stride;
    const int32_t *seq_lens;
    int n, h_q, h_kv, d, b, n_total, w, Lmax;
    float qscale;        // log2(e) / sqrt(d)
    float2 *stats;       // [n][h_kv][w * G] final (max, sum)
    float *out;          // [n][h_kv][Lmax]
    unsigned *err;
};

__device__ __forceinline__ int seq_len(const WsArgs &a, int s) {
    int L = a.seq_lens[s];
    if (L > a.Lmax) L = a.Lmax;
    if (L > a.table_stride * a.b) L = a.table_stride * a.b;
    return L;
}

// ------------------------------------------------------------------ bf16 path
// Per (sequence, kv head) -- a "pair" -- the contraction is D[t][c] = k_t . q_c
// for the R = w*g query rows c = u*g + j of the head (window row u, q head j of
// the group) against every token t: 128 tokens are the M = 128 operand of one
// tcgen05.mma (A: the head's keys, by TMA from the paged cache with the
// 128-byte swizzle), the R query rows the N operand (B: one TMA box of the
// window queries, rows landing in (u, j) order); the accumulator, R fp32
// columns per token, sits in tensor memory, double-buffered.  One persistent
// kernel runs both passes.  Work items (kind, pair, 2048-token chunk) come
// from a grid-wide counter in an order where a pair's pass-2 items follow its
// pass-1 items by `lag` pairs: by then the pass-1 items are done and the
// pair's keys (8.4 MB for the Qwen3-8B shape at 32k tokens) are still in L2
// for the second read.  A producer warp (TMA), an MMA thread and eight
// epilogue warps (two per TMEM lane quarter, each half of the columns); an
// epilogue thread owns one token:
//   pass 1: per column a sum of 2^(x - ref) over the thread's tokens (one
//           exponential per element, the reference raised only when x exceeds
//           it by more than 64), reduced over the warp and the four lane
//           quarters into a partial (max, sum) per (item, column); the last
//           item of a pair to finish a column merges that column's partials
//           into c = max + log2(sum) and counts it ready;
//   pass 2: once all R columns of the pair are ready (bounded wait), per
//           window row u the max over the group of x - c (the probability is
//           monotonic in it), one exponential per (token, u), summed over u
//           and divided by w; the two column halves meet in shared memory.
// x is the logit in log2 units; the causal mask hides token t from window row
// u when t > L - w + u.
constexpr int kWsTile = 128;     // tokens per MMA tile
constexpr int kWsItem = 2048;    // tokens per work item
constexpr int kWsTcStages = 4;
constexpr int kWsEpi = 8;
constexpr int kWsThreads = 32 * (2 + kWsEpi);

template <int D, int R>
struct WsCfg {
    static constexpr int KH = D / 64;
    static constexpr int KS = D / 16;
    static constexpr int HALVES = R >= 32 ? 2 : 1;   // column halves of the epilogue
    static constexpr int RH = R / HALVES;            // columns per epilogue warp
    static constexpr int B_HALF = R * 128;           // query rows, one 64-element half
    static constexpr int B_BYTES = KH * B_HALF;
    static constexpr int A_HALF = kWsTile * 128;
    static constexpr int STAGE = KH * A_HALF;
    static constexpr int A_OFF = (B_BYTES + 1023) / 1024 * 1024;
    static constexpr int BAR_OFF = A_OFF + kWsTcStages * STAGE;
    static constexpr int ZROW_OFF = BAR_OFF + 384;
    static constexpr int RED_OFF = ZROW_OFF + (kWsItem / 16) * 4;
    static constexpr int XCH_OFF = RED_OFF + 2 * 4 * R * 8;
    static constexpr int SMEM = XCH_OFF + 2 * 4 * 32 * 4 + 1024;
    static constexpr uint32_t TMEM_COLS = 2 * R <= 32 ? 32 : (2 * R <= 64 ? 64 : (2 * R <= 128 ? 128 : 256));
    static constexpr uint32_t IDESC = idesc_bf16_f32(128, R);
};

struct WsTcArgs {
    const int32_t *table;
    int table_stride;
    const int32_t *seq_lens;
    int n, h_kv, b, n_total, w, Lmax;
    int items_per_sh;  // chunks per pair (for Lmax)
    int pairs, lag, n_items;
    float qscale;      // log2(e) / sqrt(d)
    float2 *part;      // [pairs][items_per_sh][R] (max, sum) per item (pass 1)
    float *cst;        // [pairs][R] max + log2(sum) per column (pass 2)
    int *done_col;     // [pairs][R] pass-1 items finished per column (zero on entry)
    int *ready;        // [pairs] columns merged (zero on entry)
    float *out;        // [n][h_kv][Lmax]
    int *counter;      // work items taken (zero on entry)
    unsigned *err;
};

__device__ __forceinline__ int ws_len(const WsTcArgs &a, int s) {
    int L = a.seq_lens[s];
    if (L < 0) L = 0;
    if (L > a.Lmax) L = a.Lmax;
    if (L > a.table_stride * a.b) L = a.table_stride * a.b;
    return L;
}


// Work item g -> (pass2, pair, chunk): the first lag*C items are pass 1 of
// pairs 0..lag-1; then per pair j >= lag its C pass-1 items followed by the C
// pass-2 items of pair j - lag; the last lag*C items are pass 2 of the last
// lag pairs (C = chunks per pair).
struct WsItem {
    int pass2, pair, s, h, t0, t1, L;
};

__device__ __forceinline__ WsItem ws_item(const WsTcArgs &a, int g) {
    const int C = a.items_per_sh, P = a.pairs, lag = a.lag;
    WsItem it;
    int chunk;
    if (g < lag * C) {
        it.pass2 = 0;
        it.pair = g / C;
        chunk = g - it.pair * C;
    } else {
        const int g1 = g - lag * C;
        if (g1 < (P - lag) * 2 * C) {
            const int j = lag + g1 / (2 * C);
            const int r = g1 - (j - lag) * 2 * C;
            it.pass2 = r >= C;
            it.pair = it.pass2 ? j - lag : j;
            chunk = it.pass2 ? r - C : r;
        } else {
            const int g2 = g1 - (P - lag) * 2 * C;
            it.pass2 = 1;
            it.pair = P - lag + g2 / C;
            chunk = g2 - (g2 / C) * C;
        }
    }
    it.s = it.pair / a.h_kv;
    it.h = it.pair - it.s * a.h_kv;
    it.L = ws_len(a, it.s);
    it.t0 = chunk * kWsItem;
    it.t1 = min(it.L, it.t0 + kWsItem);
    return it;
}

__device__ __forceinline__ bool ws_item_empty(const WsTcArgs &a, const WsItem &it) {
    return it.t0 >= it.t1 || it.L < a.w;
}

// The RH columns of one epilogue warp in one TMEM load (RH = 16, 32 or 64).
template <int RH>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&v)[RH]) {
    if constexpr (RH == 16) tmem_ld16(taddr, v);
    else if constexpr (RH == 32) tmem_ld32(taddr, v);
    else tmem_ld64(taddr, v);
}

template <int D, int R, int G>
__global__ void __launch_bounds__(kWsThreads, 1)
    ws_tc05_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
                   const WsTcArgs a) {
    using C = WsCfg<D, R>;
    constexpr int RH = C::RH;
    static_assert(R % 16 == 0 && R <= 128 && RH % 16 == 0 && RH % G == 0, "query rows");
    extern __shared__ unsigned char ws_smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(ws_smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    unsigned char *Bs = smem;
    unsigned char *As = smem + C::A_OFF;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::BAR_OFF);
    uint64_t *empty = full + kWsTcStages;
    uint64_t *b_full = empty + kWsTcStages;
    uint64_t *b_empty = b_full + 1;
    uint64_t *acc_full = b_empty + 1;    // [2]
    uint64_t *acc_empty = acc_full + 2;  // [2]
    uint64_t *item_full = acc_empty + 2; // [4]
    uint64_t *item_empty = item_full + 4;
    uint64_t *drain = item_empty + 4;
    uint64_t *xch_full = drain + 1;      // [2] pass 2: the second column half's sums are in xch
    uint64_t *red_full = xch_full + 2;   // [2] pass 1: every warp's statistics are in red
    int *item_slot = reinterpret_cast<int *>(red_full + 2);  // [4]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(item_slot + 4);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *zrow = reinterpret_cast<int *>(smem + C::ZROW_OFF);
    float2 *red = reinterpret_cast<float2 *>(smem + C::RED_OFF);  // [2][4 quarters][R]
    float *xch = reinterpret_cast<float *>(smem + C::XCH_OFF);    // [2][4 quarters][32]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kWsTcStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        mbar_init(b_full, 1);
        mbar_init(b_empty, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_empty[i], kWsEpi);
        }
        for (int i = 0; i < 4; ++i) {
            mbar_init(&item_full[i], 1);
            mbar_init(&item_empty[i], 1 + kWsEpi);
        }
        mbar_init(drain, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&xch_full[i], 4);      // one warp per lane quarter
            mbar_init(&red_full[i], kWsEpi);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---------------- producer: items, the head's query rows (B), token tiles (A);
        // pass-1 keys are kept in L2 for the pass-2 read, pass-2 keys are not needed after
        uint32_t fill = 0, item = 0, b_armed = 0;
        const uint64_t keep_pol = l2_evict_last_policy(), drop_pol = l2_evict_first_policy();
        if (lane == 0) {
            prefetch_tensormap(&kmap);
            prefetch_tensormap(&qmap);
        }
        for (uint32_t k = 0;; ++k) {
            const uint32_t slot = k & 3;
            int g = -1;
            if (lane == 0) {
                if (!*abort_flag &&
                    mbar_wait_bounded(&item_empty[slot], ((k >> 2) & 1) ^ 1, a.err, abort_flag, 0x510)) {
                    g = atomicAdd(a.counter, 1);
                    item_slot[slot] = g < a.n_items ? g : -1;
                    mbar_arrive(&item_full[slot]);
                    if (g >= a.n_items) g = -1;
                } else {
                    g = -2;
                }
            }
            g = __shfl_sync(0xFFFFFFFFu, g, 0);
            if (g < 0) break;
            const WsItem it = ws_item(a, g);
            if (ws_item_empty(a, it)) continue;
            const int ngrp = (it.t1 - it.t0 + 15) / 16;
            for (int q = lane; q < ngrp; q += 32) {
                const int t = it.t0 + 16 * q;
                int z = -16;
                const int blk = a.table[(size_t)it.s * a.table_stride + t / a.b];
                if (blk >= 0 && blk < a.n_total) z = blk * a.b + t % a.b;
                else record_error(a.err, ZP_ERR_DEVICE, 0x511);
                zrow[q] = z;
            }
            __syncwarp();
            if (lane != 0) continue;
            if (!mbar_wait_bounded(b_empty, (item & 1) ^ 1, a.err, abort_flag, 0x512)) continue;
            mbar_arrive_expect_tx(b_full, C::B_BYTES);
            b_armed = item + 1;
#pragma unroll
            for (int kh = 0; kh < C::KH; ++kh)
                tma_load_3d(Bs + kh * C::B_HALF, &qmap, kh * 64, it.h * G, it.s * a.w, b_full);
            const uint64_t pol = it.pass2 ? drop_pol : keep_pol;
            const int ntiles = (it.t1 - it.t0 + kWsTile - 1) / kWsTile;
            for (int j = 0; j < ntiles; ++j) {
                const uint32_t st = fill % kWsTcStages;
                if (!mbar_wait_bounded(&empty[st], ((fill / kWsTcStages) & 1) ^ 1, a.err, abort_flag, 0x513)) break;
                mbar_arrive_expect_tx(&full[st], C::STAGE);
                ++fill;
                unsigned char *dst = As + st * C::STAGE;
#pragma unroll
                for (int q = 0; q < kWsTile / 16; ++q) {
                    const int gi = j * (kWsTile / 16) + q;
                    const int z = gi < ngrp ? zrow[gi] : -16;
#pragma unroll
                    for (int kh = 0; kh < C::KH; ++kh)
                        tma_load_3d_hint(dst + kh * C::A_HALF + q * 2048, &kmap, kh * 64, it.h, z, &full[st], pol);
                }
            }
            ++item;
        }
        if (lane == 0 && *abort_flag) {
            volatile int never = 0;
            for (uint32_t f = fill > kWsTcStages ? fill - kWsTcStages : 0; f < fill; ++f)
                mbar_wait_bounded(&full[f % kWsTcStages], (f / kWsTcStages) & 1, a.err, &never, 0x514);
            if (b_armed > item) mbar_wait_bounded(b_full, item & 1, a.err, &never, 0x515);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer
        if (lane == 0) {
            uint32_t fill = 0, tile = 0, item = 0;
            const uint32_t a_addr = smem_u32(As), b_addr = smem_u32(Bs);
            for (uint32_t k = 0; !*abort_flag; ++k) {
                const uint32_t slot = k & 3;
                if (!mbar_wait_bounded(&item_full[slot], (k >> 2) & 1, a.err, abort_flag, 0x516)) break;
                const int g = item_slot[slot];
                mbar_arrive(&item_empty[slot]);
                if (g < 0) break;
                const WsItem it = ws_item(a, g);
                if (ws_item_empty(a, it)) continue;
                if (!mbar_wait_bounded(b_full, item & 1, a.err, abort_flag, 0x517)) break;
                tc_fence_after();
                const int ntiles = (it.t1 - it.t0 + kWsTile - 1) / kWsTile;
                bool ok_item = true;
                for (int j = 0; j < ntiles; ++j, ++fill, ++tile) {
                    const uint32_t st = fill % kWsTcStages, ab = tile & 1;
                    if (!mbar_wait_bounded(&full[st], (fill / kWsTcStages) & 1, a.err, abort_flag, 0x518) ||
                        !mbar_wait_bounded(&acc_empty[ab], ((tile >> 1) & 1) ^ 1, a.err, abort_flag, 0x519)) {
                        ok_item = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < C::KS; ++ks) {
                        const uint32_t ao = st * C::STAGE + (ks >> 2) * C::A_HALF + (ks & 3) * 32;
                        const uint32_t bo = (ks >> 2) * C::B_HALF + (ks & 3) * 32;
                        tc_mma_bf16(tmem + ab * R, sdesc_k_sw128(a_addr + ao), sdesc_k_sw128(b_addr + bo), C::IDESC,
                                    ks > 0 ? 1u : 0u);
                    }
                    tc_commit(&empty[st]);
                    tc_commit(&acc_full[ab]);
                }
                if (!ok_item) break;
                tc_commit(b_empty);
                ++item;
            }
        }
    } else {
        // ---------------- epilogue: thread = token (lane quarter q), columns [half*RH, half*RH + RH)
        const int e = warp - 2;
        const int q = warp & 3;
        const int half = e >> 2;
        const bool works = half < C::HALVES;
        const int et = threadIdx.x - 64;  // 0..255 over the epilogue warps
        uint32_t tile = 0, eitem = 0, xtile = 0;  // all tiles, pass-1 items, pass-2 tiles
        // every synchronisation here is an mbarrier or a flag with a bounded
        // wait, so a warp that stops after a timeout cannot leave another
        // waiting for ever
        for (uint32_t k = 0;; ++k) {
            const uint32_t slot = k & 3;
            if (!mbar_wait_bounded(&item_full[slot], (k >> 2) & 1, a.err, abort_flag, 0x51A)) break;
            const int g = item_slot[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive(&item_empty[slot]);
            if (g < 0) break;
            const WsItem it = ws_item(a, g);
            if (ws_item_empty(a, it)) continue;
            const int t0 = it.t0, t1 = it.t1, L = it.L;
            const int last0 = L - a.w;  // window row u sees tokens t <= last0 + u
            const size_t pr = (size_t)it.pair;
            // pass 1: m = reference and l = sum per column; pass 2: m = the column's c
            float m[RH], l[RH];
#pragma unroll
            for (int c = 0; c < RH; ++c) {
                m[c] = -1e30f;  // finite: x - m is never NaN
                l[c] = 0.f;
            }
            if (it.pass2) {
                // the pair's R columns merged by the last pass-1 items (bounded wait)
                if (lane == 0) {
                    const volatile int *rd = a.ready + pr;
                    if (*rd < R) {
                        const unsigned long long t_0 = global_ns();
                        while (*rd < R) {
                            if (global_ns() - t_0 > kWaitLimitNs) {
                                record_error(a.err, ZP_ERR_TIMEOUT, 0x51F);
                                *abort_flag = 1;
                                break;
                            }
                            __nanosleep(64);
                        }
                    }
                    __threadfence();
                }
                __syncwarp();
                if (works) {
#pragma unroll
                    for (int c = 0; c < RH; ++c) m[c] = __ldcg(a.cst + pr * R + half * RH + c);
                }
            }
            const int ntiles = (t1 - t0 + kWsTile - 1) / kWsTile;
            bool ok_item = true;
            for (int j = 0; j < ntiles; ++j, ++tile) {
                const uint32_t ab = tile & 1;
                if (!mbar_wait_bounded(&acc_full[ab], (tile >> 1) & 1, a.err, abort_flag, 0x51B)) {
                    ok_item = false;
                    break;
                }
                tc_fence_after();
                const int t = t0 + j * kWsTile + 32 * q + lane;  // this thread's token
                const int tbase = t0 + j * kWsTile;
                // every token of the tile valid and seen by every window row
                const bool full_tile = tbase + kWsTile - 1 <= last0 && tbase + kWsTile <= L;
                float wsum = 0.f;  // pass 2: sum over this half's window rows
                if (works) {
                    uint32_t vall[RH];  // the warp's columns, one load
                    tmem_ld_cols<RH>(tmem + ((uint32_t)(32 * q) << 16) + ab * R + half * RH, vall);
#pragma unroll
                    for (int ch = 0; ch < RH / 16; ++ch) {
                        const uint32_t *v = vall + ch * 16;
                        if (!it.pass2) {
                            // l is the sum of 2^(x - ref): rescaled only when x exceeds
                            // the reference by more than 64 (the first token of an
                            // item, or a jump of 2^64) -- tested once per 16 columns
                            float y[16];
                            float ymax = -INFINITY;
#pragma unroll
                            for (int c2 = 0; c2 < 16; ++c2) {
                                const int c = ch * 16 + c2;
                                const int u = (half * RH + c) / G;
                                const bool vis = full_tile || (t < L && t <= last0 + u);
                                y[c2] = vis ? fmaf(__uint_as_float(v[c2]), a.qscale, -m[c]) : -INFINITY;
                                ymax = fmaxf(ymax, y[c2]);
                            }
                            if (ymax > 64.f) {
#pragma unroll
                                for (int c2 = 0; c2 < 16; ++c2) {
                                    const int c = ch * 16 + c2;
                                    if (y[c2] > 64.f) {
                                        const float x = __uint_as_float(v[c2]) * a.qscale;
                                        l[c] *= ex2_approx(m[c] - x);
                                        m[c] = x;
                                        y[c2] = 0.f;
                                    }
                                }
                            }
#pragma unroll
                            for (int c2 = 0; c2 < 16; ++c2) l[ch * 16 + c2] += ex2_approx(y[c2]);
                        } else {
#pragma unroll
                            for (int u2 = 0; u2 < 16 / G; ++u2) {
                                const int u = (half * RH + ch * 16) / G + u2;
                                float yy = -INFINITY;
#pragma unroll
                                for (int jj = 0; jj < G; ++jj) {
                                    const int c = ch * 16 + u2 * G + jj;
                                    yy = fmaxf(yy, fmaf(__uint_as_float(v[u2 * G + jj]), a.qscale, -m[c]));
                                }
                                if (full_tile || (t < L && t <= last0 + u)) wsum += ex2_approx(yy);
                            }
                        }
                    }
                }
                tc_fence_before();
                if (it.pass2) {
                    // the two column halves of a lane quarter meet in xch; the
                    // first half reads before releasing the accumulator, so the
                    // buffer is free again when the second half reaches it
                    float *xb = xch + ((xtile & 1) * 4 + q) * 32;
                    if (C::HALVES == 2) {
                        if (half == 1) {
                            xb[lane] = wsum;
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&xch_full[xtile & 1]);
                        } else if (mbar_wait_bounded(&xch_full[xtile & 1], (xtile >> 1) & 1, a.err, abort_flag,
                                                     0x51D)) {
                            wsum += xb[lane];
                        }
                    }
                    if (half == 0 && t < L) a.out[((size_t)it.s * a.h_kv + it.h) * a.Lmax + t] = wsum / (float)a.w;
                    ++xtile;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&acc_empty[ab]);
            }
            if (!it.pass2) {
                // (max, sum) per column: over the warp's 32 tokens, then the 4
                // lane quarters (red is double-buffered by pass-1 item; every
                // warp waits for the buffer's completion, so a buffer is
                // rewritten only after every reader of its previous use has
                // moved on)
                float2 *rb = red + (eitem & 1) * 4 * R;
                if (works) {
#pragma unroll
                    for (int c = 0; c < RH; ++c) {
                        // (reference, sum) pairs combine like (max, sum) pairs;
                        // a lane that saw nothing has sum 0 and reference -1e30
                        float M = m[c];
#pragma unroll
                        for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, o));
                        float Ls = l[c] * exp2f(m[c] - M);
#pragma unroll
                        for (int o = 16; o; o >>= 1) Ls += __shfl_xor_sync(0xFFFFFFFFu, Ls, o);
                        if (lane == 0) rb[q * R + half * RH + c] = make_float2(M, Ls);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&red_full[eitem & 1]);
                if (mbar_wait_bounded(&red_full[eitem & 1], (eitem >> 1) & 1, a.err, abort_flag, 0x51E) && et < R) {
                    float M = -INFINITY, Ls = 0.f;
#pragma unroll
                    for (int qq = 0; qq < 4; ++qq) {
                        const float2 p = rb[qq * R + et];
                        if (!(p.y > 0.f)) continue;
                        if (p.x > M) {
                            Ls = Ls * exp2f(M - p.x) + p.y;
                            M = p.x;
                        } else {
                            Ls += p.y * exp2f(p.x - M);
                        }
                    }
                    a.part[(pr * a.items_per_sh + (size_t)(t0 / kWsItem)) * R + et] = make_float2(M, Ls);
                    // the last item of the pair to finish this column merges it
                    // (fence, then count: the partials written before each count
                    // are visible to the thread that sees the last count)
                    __threadfence();
                    const int nitem = (L + kWsItem - 1) / kWsItem;
                    if (atomicAdd(a.done_col + pr * R + et, 1) == nitem - 1) {
                        __threadfence();
                        float MM = -INFINITY, SS = 0.f;
                        for (int i2 = 0; i2 < nitem; ++i2) {
                            const float2 ml = __ldcg(a.part + (pr * a.items_per_sh + i2) * R + et);
                            if (!(ml.y > 0.f)) continue;
                            if (ml.x > MM) {
                                SS = SS * exp2f(MM - ml.x) + ml.y;
                                MM = ml.x;
                            } else {
                                SS += ml.y * exp2f(ml.x - MM);
                            }
                        }
                        a.cst[pr * R + et] = SS > 0.f ? MM + log2f(SS) : INFINITY;
                        __threadfence();
                        atomicAdd(a.ready + pr, 1);
                    }
                }
                ++eitem;
            }
            if (!ok_item) break;
        }
    }

    __syncthreads();
    if (*abort_flag && threadIdx.x == 32) {
        volatile int never = 0;
        tc_commit(drain);
        mbar_wait_bounded(drain, 0, a.err, &never, 0x51C);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
}

// ------------------------------------------------------------------ fp32 path
// (small shapes) pass 1: one block per (sequence, kv head, window row u, q
// head j); pass 2: one thread per (sequence, kv head, token).
__global__ void ws_f32_stats_kernel(const WsArgs a) {
    __shared__ float red[32];
    const int s = blockIdx.z;
    const int kvh = blockIdx.y;
    const int G = a.h_q / a.h_kv;
    const int u = blockIdx.x / G, j = blockIdx.x % G;
    const int L = seq_len(a, s);
    if (L < a.w) return;
    const int last = L - a.w + u;
    const float *qv = static_cast<const float *>(a.q) + (((size_t)s * a.w + u) * a.h_q + kvh * G + j) * a.d;
    const float *K = static_cast<const float *>(a.k);
    float m = -INFINITY;
    for (int t = threadIdx.x; t <= last; t += blockDim.x) {
        const int blk = a.table[(size_t)s * a.table_stride + t / a.b];
        if (blk < 0 || blk >= a.n_total) continue;
        const float *kr = K + (((size_t)blk * a.b + t % a.b) * a.h_kv + kvh) * a.d;
        float dot = 0.f;
        for (int i = 0; i < a.d; ++i) dot = fmaf(qv[i], kr[i], dot);
        m = fmaxf(m, dot * a.qscale);
    }
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    m = -INFINITY;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) m = fmaxf(m, red[i]);
    __syncthreads();
    float sum = 0.f;
    for (int t = threadIdx.x; t <= last; t += blockDim.x) {
        const int blk = a.table[(size_t)s * a.table_stride + t / a.b];
        if (blk < 0 || blk >= a.n_total) continue;
        const float *kr = K + (((size_t)blk * a.b + t % a.b) * a.h_kv + kvh) * a.d;
        float dot = 0.f;
        for (int i = 0; i < a.d; ++i) dot = fmaf(qv[i], kr[i], dot);
        sum += exp2f(dot * a.qscale - m);
    }
    for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = sum;
    __syncthreads();
    if (threadIdx.x == 0) {
        float tot = 0.f;
        for (int i = 0; i < (int)(blockDim.x >> 5); ++i) tot += red[i];
        a.stats[((size_t)s * a.h_kv + kvh) * (a.w * G) + u * G + j] = make_float2(m, tot);
    }
}

__global__ void ws_f32_score_kernel(const WsArgs a) {
    const int s = blockIdx.z;
    const int kvh = blockIdx.y;
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    const int L = seq_len(a, s);
    if (L < a.w || t >= L) return;
    const int G = a.h_q / a.h_kv;
    const int blk = a.table[(size_t)s * a.table_stride + t / a.b];
    if (blk < 0 || blk >= a.n_total) {
        record_error(a.err, ZP_ERR_DEVICE, 0x501);
        return;
    }
    const float *kr = static_cast<const float *>(a.k) + (((size_t)blk * a.b + t % a.b) * a.h_kv + kvh) * a.d;
    float acc = 0.f;
    for (int u = 0; u < a.w; ++u) {
        if (t > L - a.w + u) continue;  // masked: contributes 0
        float best = 0.f;
        for (int j = 0; j < G; ++j) {
            const float *qv = static_cast<const float *>(a.q) + (((size_t)s * a.w + u) * a.h_q + kvh * G + j) * a.d;
            float dot = 0.f;
            for (int i = 0; i < a.d; ++i) dot = fmaf(qv[i], kr[i], dot);
            const float2 ml = a.stats[((size_t)s * a.h_kv + kvh) * (a.w * G) + u * G + j];
            best = fmaxf(best, exp2f(dot * a.qscale - ml.x) / ml.y);
        }
        acc += best;
    }
    a.out[((size_t)s * a.h_kv + kvh) * a.Lmax + t] = acc / (float)a.w;
}

template <int D, int R, int G>
zp_status launch_ws_tc05(WsTcArgs a, const void *k, const void *q, int h_q, const DeviceInfo &dev, cudaStream_t st) {
    using Cfg = WsCfg<D, R>;
    if ((size_t)Cfg::SMEM > (size_t)dev.smem_optin)
        return fail(ZP_ERR_SHAPE, "window score: needs %d B of shared memory", Cfg::SMEM);
    CUtensorMap kmap, qmap;
    {
        const uint64_t dims[3] = {(uint64_t)D, (uint64_t)a.h_kv, (uint64_t)a.n_total * (uint64_t)a.b};
        const uint64_t strides[2] = {(uint64_t)D * 2, (uint64_t)a.h_kv * D * 2};
        const uint32_t box[3] = {64, 1, 16};
        zp_status rc = encode_tmap_bf16_3d(&kmap, k, dims, strides, box, "window score (keys)");
        if (rc != ZP_OK) return rc;
    }
    {
        // the window queries [n][w][h_q][d]: a box is 64 elements of the G q
        // heads of one kv head for the w window rows -> rows in (u, j) order
        const uint64_t dims[3] = {(uint64_t)D, (uint64_t)h_q, (uint64_t)a.n * (uint64_t)a.w};
        const uint64_t strides[2] = {(uint64_t)D * 2, (uint64_t)h_q * D * 2};
        const uint32_t box[3] = {64, (uint32_t)G, (uint32_t)a.w};
        zp_status rc = encode_tmap_bf16_3d(&qmap, q, dims, strides, box, "window score (queries)");
        if (rc != ZP_OK) return rc;
    }
    auto kern = ws_tc05_kernel<D, R, G>;
    zp_status rs = set_max_dynamic_smem(reinterpret_cast<const void *>(kern), Cfg::SMEM, "window score: shared memory");
    if (rs != ZP_OK) return rs;
    const int grid = a.n_items < dev.sm_count ? a.n_items : dev.sm_count;
    // pass 2 of a pair follows its pass 1 by about the items in flight (one
    // or two per CTA, 2 * items_per_sh per pair) plus two pairs: late enough
    // that the pass-1 items are mostly done, early enough that the keys of the
    // pairs in between (lag * 8.4 MB at 32k tokens) stay in L2
    int lag = (grid + 2 * a.items_per_sh - 1) / (2 * a.items_per_sh) + 2;
    if (lag < 1) lag = 1;
    if (lag > a.pairs) lag = a.pairs;
    a.lag = lag;
    cudaError_t e = cudaMemsetAsync(a.done_col, 0, ((size_t)a.pairs * (R + 1) + 1) * 4, st);
    if (e != cudaSuccess) return cuda_fail(e, "window score: clearing the counters");
    kern<<<grid, kWsThreads, Cfg::SMEM, st>>>(kmap, qmap, a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "window score: launch");
    return ZP_OK;
}

}  // namespace
}  // namespace zp

using namespace zp;

extern "C" size_t zp_window_score_workspace_size(const zp_cache_desc *D, int32_t n, int32_t Lmax,
                                                 int32_t window) {
    if (!D || n < 0 || Lmax < 0 || window <= 0 || D->h_kv <= 0) return 0;
    const int G = D->h_q / D->h_kv;
    // fp32 path: final (max, sum) per (sequence, kv head, query row)
    const size_t f32 = align_up((size_t)n * D->h_kv * window * G * 8, 256);
    // bf16 path: (max, sum) per (pass-1 item, query row), max + log2(sum) per
    // query row, per-column and per-pair counters, the item counter
    const size_t R = (size_t)window * G;
    const size_t items = ((size_t)Lmax + kWsItem - 1) / kWsItem;
    const size_t pairs = (size_t)n * D->h_kv;
    const size_t tc = align_up(pairs * items * R * 8, 256) + align_up(pairs * R * 4, 256) +
                      align_up((pairs * (R + 1) + 1) * 4, 256);
    return f32 > tc ? f32 : tc;
}

extern "C" zp_status zp_window_score(const zp_cache_desc *D, const void *q_window, int32_t window,
                                     const void *k_cache, const int32_t *block_table, int32_t table_stride,
                                     const int32_t *seq_lens, int32_t n, float *scores_out, int32_t Lmax,
                                     void *workspace, size_t workspace_bytes, void *stream) {
    zp_status rc = check_desc(D);
    if (rc != ZP_OK) return rc;
    if (n < 0 || Lmax < 0 || table_stride < 1 || window < 1)
        return fail(ZP_ERR_INVALID_ARG, "window score: bad sizes (n=%d Lmax=%d window=%d)", n, Lmax, window);
    if (n == 0 || Lmax == 0) return ok();
    if (!q_window || !k_cache || !block_table || !seq_lens || !scores_out || !workspace)
        return fail(ZP_ERR_INVALID_ARG, "window score: NULL buffer");
    const size_t need = zp_window_score_workspace_size(D, n, Lmax, window);
    if (workspace_bytes < need)
        return fail(ZP_ERR_CAPACITY, "window score: workspace %zu < %zu", workspace_bytes, need);
    DeviceInfo dev;
    rc = device_info(&dev);
    if (rc != ZP_OK) return rc;
    const int G = D->h_q / D->h_kv;
    const int d = D->head_dim;
    WsArgs a;
    a.q = q_window;
    a.k = k_cache;
    a.table = block_table;
    a.table_stride = table_stride;
    a.seq_lens = seq_lens;
    a.n = n;
    a.h_q = D->h_q;
    a.h_kv = D->h_kv;
    a.d = d;
    a.b = D->block_size;
    a.n_total = D->n_total_blocks;
    a.w = window;
    a.Lmax = Lmax;
    a.qscale = (float)(1.4426950408889634 / sqrt((double)d));
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    a.stats = reinterpret_cast<float2 *>(ws);  // fp32 path
    a.out = scores_out;
    a.err = dev.error_word;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (D->dtype == ZP_F32) {
        if (d > 256) return fail(ZP_ERR_SHAPE, "window score: head_dim %d", d);
        ws_f32_stats_kernel<<<dim3(window * G, D->h_kv, n), 256, 0, st>>>(a);
        ws_f32_score_kernel<<<dim3((Lmax + 127) / 128, D->h_kv, n), 128, 0, st>>>(a);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e, "window score: launch");
        return ok();
    }
    // bf16: two passes on the tensor cores (tcgen05)
    if (D->block_size % 16) return fail(ZP_ERR_SHAPE, "window score: block size %d not a multiple of 16", D->block_size);
    const int R = window * G;
    if (!(R == 16 || R == 32 || R == 64 || R == 128) || !(G == 1 || G == 2 || G == 4 || G == 8) || window > 256)
        return fail(ZP_ERR_SHAPE, "window score: window*group = %d (bf16 needs 16, 32, 64 or 128)", R);
    if (((uintptr_t)k_cache | (uintptr_t)q_window) % 16)
        return fail(ZP_ERR_INVALID_ARG, "window score: buffers must be 16-byte aligned");
    WsTcArgs t;
    t.table = block_table;
    t.table_stride = table_stride;
    t.seq_lens = seq_lens;
    t.n = n;
    t.h_kv = D->h_kv;
    t.b = D->block_size;
    t.n_total = D->n_total_blocks;
    t.w = window;
    t.Lmax = Lmax;
    t.items_per_sh = (Lmax + kWsItem - 1) / kWsItem;
    t.pairs = n * D->h_kv;
    const long long n_items = 2LL * t.pairs * t.items_per_sh;  // pass 1 and pass 2
    if (n_items > 0x7FFFFFFF) return fail(ZP_ERR_SHAPE, "window score: too many work items");
    t.n_items = (int)n_items;
    t.lag = 1;  // set by the launcher
    t.qscale = a.qscale;
    t.part = reinterpret_cast<float2 *>(ws);
    const size_t part_bytes = align_up((size_t)t.pairs * t.items_per_sh * R * 8, 256);
    t.cst = reinterpret_cast<float *>(ws + part_bytes);
    // counters, one run that the launcher zeroes: done_col [pairs][R], ready [pairs], the item counter
    t.done_col = reinterpret_cast<int *>(ws + part_bytes + align_up((size_t)t.pairs * R * 4, 256));
    t.ready = t.done_col + (size_t)t.pairs * R;
    t.counter = t.ready + t.pairs;
    t.out = scores_out;
    t.err = dev.error_word;
#define ZP_WS(DD, RR, GG)                                                                        \
    if (d == DD && R == RR && G == GG) {                                                         \
        rc = launch_ws_tc05<DD, RR, GG>(t, k_cache, q_window, D->h_q, dev, st);                  \
        return rc == ZP_OK ? ok() : rc;                                                          \
    }
    ZP_WS(128, 64, 4)
    ZP_WS(128, 32, 4)
    ZP_WS(128, 16, 4)
    ZP_WS(128, 128, 8)
    ZP_WS(128, 64, 8)
    ZP_WS(128, 32, 8)
    ZP_WS(128, 16, 8)
    ZP_WS(128, 128, 4)
    ZP_WS(64, 64, 4)
    ZP_WS(64, 32, 4)
    ZP_WS(64, 16, 4)
    ZP_WS(64, 128, 8)
    ZP_WS(64, 64, 8)
#undef ZP_WS
    return fail(ZP_ERR_SHAPE, "window score: no kernel for d=%d, window*group=%d, group=%d", d, R, G);
}
