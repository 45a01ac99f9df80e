// select.cuh -- block-wide top-k keep set of one score row (Zipage paper
// §4.2: the k = (N_max-1)*b highest-scoring entries are retained; App. C.6).
//
// Order: score descending, then position descending (among equal scores the
// newer token ranks first).  Each score becomes a 32-bit key whose unsigned
// order is the float order (sign-flipped bits).  A most-significant-byte-first
// radix select over the keys finds the threshold key T and how many keys equal
// to T are kept (rem): a 256-bin shared histogram per pass (the lanes of a
// warp that share lane 0's bin add once; two buffers, one cleared while the
// other counts) and an early exit once the bin holding the k-th key is taken
// whole; once that bin holds at most kWarpCand keys, they are gathered into
// shared memory and one warp finishes the passes on them without block
// barriers.  When the passes end inside a run of equal keys, the newest rem
// of them are kept.  One block-wide prefix sum over two counts (keys above T,
// keys equal to T; per thread on short rows, per warp with ballots on long
// ones) then writes the kept positions in ascending order, the order Alg. 4
// preserves.
#pragma once

#include "zp_common.cuh"

namespace zp {

constexpr int kWarpCand = 512;  // candidates a single warp finishes (16 keys per lane)

struct SelectShared {
    int hist2[2][256];
    int wsum[32], weq[32];
    int woff[33], weoff[33];
    int red[32];
    unsigned cand[kWarpCand];  // keys of the bin holding the k-th key, once it is small
    unsigned prefix;
    int shift, need, done;
    int bincount, ncand;
};

static __device__ __forceinline__ unsigned select_key(float f) {
    const unsigned u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// The k highest of sc[0..L) (L > k; sc may be in shared or global memory),
// positions ascending to out_g[0..k) (global, nullable) and out_s (shared,
// nullable).  tie_out (nullable): tokens sharing the score of the lowest kept
// token when that score was split between kept and dropped tokens, else 0.
// Every thread of the block calls it (blockDim.x a multiple of 32, <= 1024).
// WARP_SCAN picks the final scan (per warp: long rows; per thread: short ones)
// at compile time, so that an instance carries one of them: the code runs once
// per block and every instruction line it touches is fetched once.
template <bool WARP_SCAN>
static __device__ void block_select_topk(const float *sc, int L, int k, int32_t *out_g, int *out_s, int32_t *tie_out,
                                         unsigned *err, SelectShared &sh) {
    const int tid = threadIdx.x, nthr = blockDim.x;
    const int lane = tid & 31, wid = tid >> 5;
    if (tid == 0) {
        sh.prefix = 0u;
        sh.shift = 32;
        sh.need = k;
        sh.done = 0;
        sh.bincount = L;
    }
    for (int i = tid; i < 256; i += nthr) sh.hist2[0][i] = 0;
    int hb = 0;  // histogram buffer of the next pass
    bool warp_finish = false;
    for (int pass = 3; pass >= 0; --pass) {
        __syncthreads();
        if (sh.done) break;
        // once the bin holding the k-th key is small, one warp finishes the
        // passes on its keys without block barriers
        if (pass < 3 && sh.bincount <= kWarpCand) {
            warp_finish = true;
            break;
        }
        const int shift = pass * 8;
        int *hist = sh.hist2[hb];
        for (int i = tid; i < 256; i += nthr) sh.hist2[hb ^ 1][i] = 0;  // for the next pass
        const unsigned pre = sh.prefix;
        const int pshift = sh.shift;
        // In the first passes most keys share one or two bins: the lanes of a
        // warp whose bin equals lane 0's add once, through lane 0.
        for (int t0 = 0; t0 < L; t0 += nthr) {
            const int t = t0 + tid;
            int bin = -1;
            if (t < L) {
                const float f = sc[t];
                if (f != f) record_error(err, ZP_ERR_DEVICE, 0x300);
                const unsigned key = select_key(f);
                if (pshift == 32 || (key >> pshift) == pre) bin = (int)((key >> shift) & 255u);
            }
            const int b0 = __shfl_sync(0xFFFFFFFFu, bin, 0);
            const unsigned with0 = __ballot_sync(0xFFFFFFFFu, bin == b0);
            if (lane == 0 && b0 >= 0) atomicAdd(&hist[b0], __popc(with0));
            if (bin >= 0 && bin != b0) atomicAdd(&hist[bin], 1);
        }
        __syncthreads();
        if (tid < 32) {
            // lane l owns bins 8l..8l+7; a suffix scan over the lanes finds the
            // bin where the count from the top reaches `need`
            const int need = sh.need;
            int h8[8], tot = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                h8[j] = hist[8 * tid + j];
                tot += h8[j];
            }
            int incl = tot;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_down_sync(0xFFFFFFFFu, incl, o);
                if (tid + o < 32) incl += y;
            }
            const int above = incl - tot;
            if (above < need && need <= incl) {
                int cum = above, bin = 8 * tid;
                for (int j = 7; j >= 0; --j) {
                    if (cum + h8[j] >= need) {
                        bin = 8 * tid + j;
                        break;
                    }
                    cum += h8[j];
                }
                const int rem = need - cum;
                sh.prefix = (pshift == 32 ? 0u : (pre << 8)) | (unsigned)bin;
                sh.shift = shift;
                sh.need = rem;
                sh.bincount = hist[bin];
                sh.ncand = 0;
                if (hist[bin] == rem) sh.done = 1;
            }
        }
        hb ^= 1;
    }
    if (warp_finish) {
        // gather the bin's keys (sh.bincount <= kWarpCand of them)
        const unsigned pre0 = sh.prefix;
        const int sh0 = sh.shift;
        for (int t = tid; t < L; t += nthr) {
            const unsigned key = select_key(sc[t]);
            if ((key >> sh0) == pre0) {
                const int i = atomicAdd(&sh.ncand, 1);
                if (i < kWarpCand) sh.cand[i] = key;
            }
        }
        __syncthreads();
        if (wid == 0) {
            const int c = min(sh.ncand, kWarpCand);
            unsigned kc[kWarpCand / 32];
#pragma unroll
            for (int j = 0; j < kWarpCand / 32; ++j) kc[j] = lane + 32 * j < c ? sh.cand[lane + 32 * j] : 0u;
            unsigned pre = pre0;
            int shift = sh0, need = sh.need, done = 0;
            int *hist = sh.hist2[0];
            while (shift > 0 && !done) {
                const int lo = shift > 8 ? shift - 8 : 0;
                for (int i = lane; i < 256; i += 32) hist[i] = 0;
                __syncwarp();
#pragma unroll
                for (int j = 0; j < kWarpCand / 32; ++j)
                    if (lane + 32 * j < c && (kc[j] >> shift) == pre)
                        atomicAdd(&hist[(kc[j] >> lo) & ((1u << (shift - lo)) - 1u)], 1);
                __syncwarp();
                // lane l owns bins 8l..8l+7: suffix scan, then the lane holding
                // the need-th key from the top publishes the bin
                int h8[8], tot = 0;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    h8[j] = hist[8 * lane + j];
                    tot += h8[j];
                }
                int incl = tot;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int y = __shfl_down_sync(0xFFFFFFFFu, incl, o);
                    if (lane + o < 32) incl += y;
                }
                const int above = incl - tot;
                const bool mine = above < need && need <= incl;
                int bin = 8 * lane, cum = above, hbin = 0;
                bool found = false;
#pragma unroll
                for (int j = 7; j >= 0; --j) {
                    if (mine && !found) {
                        if (cum + h8[j] >= need) {
                            bin = 8 * lane + j;
                            hbin = h8[j];
                            found = true;
                        } else {
                            cum += h8[j];
                        }
                    }
                }
                const unsigned who = __ballot_sync(0xFFFFFFFFu, mine);
                const int src = who ? __ffs(who) - 1 : 0;
                bin = __shfl_sync(0xFFFFFFFFu, bin, src);
                cum = __shfl_sync(0xFFFFFFFFu, cum, src);
                hbin = __shfl_sync(0xFFFFFFFFu, hbin, src);
                __syncwarp();
                pre = (pre << (shift - lo)) | (unsigned)bin;
                shift = lo;
                need -= cum;
                done = hbin == need ? 1 : 0;
            }
            if (lane == 0) {
                if (sh.ncand > kWarpCand) record_error(err, ZP_ERR_DEVICE, 0x303);
                sh.prefix = pre;
                sh.shift = shift;
                sh.need = need;
                sh.done = done;
            }
        }
    }
    __syncthreads();
    const unsigned thr = sh.prefix;
    const int tsh = sh.shift;
    // whole: keep iff (key >> tsh) >= thr.  Otherwise the passes ended inside a
    // run of keys equal to thr (tsh = 0): keep those above it and the newest
    // `rem` of those equal to it.
    const bool whole = sh.done != 0;
    const int rem = sh.need;
    // Two counts per scan unit (keys above thr -- or at least thr when whole --
    // and keys equal to it), a block-wide prefix over them, then the kept
    // positions written in order.  Per thread (short rows): each thread scans
    // its own consecutive keys (shared-memory conflicts gcd(chunk, 32)-way).
    // Per warp (long rows): warp w owns the positions [w C, w C + C) (C a
    // multiple of 32) and reads them 32 consecutive at a time, so reads are
    // conflict-free (coalesced in global memory), and ballots give each lane
    // the kept and equal keys before it.
    const int chunk = (L + nthr - 1) / nthr;
    constexpr bool per_thread = !WARP_SCAN;
    const int nw = nthr >> 5;
    const int C = ((L + nw - 1) / nw + 31) & ~31;
    const int beg = per_thread ? tid * chunk : wid * C;
    const int end = min(L, beg + (per_thread ? chunk : C));
    const unsigned lower = (1u << lane) - 1u;
    int cnt = 0, ceq = 0;
    if constexpr (per_thread) {
        for (int t = beg; t < end; ++t) {
            const unsigned kt = select_key(sc[t]) >> tsh;
            cnt += whole ? (kt >= thr) : (kt > thr);
            ceq += (!whole && kt == thr) ? 1 : 0;
        }
    } else {
        for (int t0 = beg; t0 < end; t0 += 32) {
            const int t = t0 + lane;
            const unsigned kt = t < end ? select_key(sc[t]) >> tsh : 0u;
            const bool above = t < end && (whole ? kt >= thr : kt > thr);
            const bool equal = t < end && !whole && kt == thr;
            cnt += __popc(__ballot_sync(0xFFFFFFFFu, above));
            ceq += __popc(__ballot_sync(0xFFFFFFFFu, equal));
        }
    }
    // inclusive counts within the warp (per-thread scan units), else the warp's own
    int incl = cnt, ieq = ceq;
    if constexpr (per_thread) {
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            const int ye = __shfl_up_sync(0xFFFFFFFFu, ieq, o);
            if (lane >= o) {
                incl += y;
                ieq += ye;
            }
        }
    }
    if (lane == 31) {
        sh.wsum[wid] = incl;
        sh.weq[wid] = ieq;
    }
    __syncthreads();
    if (wid == 0) {
        const int w = lane < nw ? sh.wsum[lane] : 0;
        const int we = lane < nw ? sh.weq[lane] : 0;
        int wi = w, wie = we;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xFFFFFFFFu, wi, o);
            const int ye = __shfl_up_sync(0xFFFFFFFFu, wie, o);
            if (lane >= o) {
                wi += y;
                wie += ye;
            }
        }
        if (lane < nw) {
            sh.woff[lane] = wi - w;
            sh.weoff[lane] = wie - we;
        }
        if (lane == nw - 1) {
            sh.woff[32] = wi;
            sh.weoff[32] = wie;
        }
    }
    __syncthreads();
    const int eq_total = sh.weoff[32];
    const int eq_drop = whole ? 0 : eq_total - rem;  // the oldest equal keys are dropped
    const int kept_total = sh.woff[32] + (whole ? 0 : rem);
    if (kept_total != k && tid == 0) record_error(err, ZP_ERR_DEVICE, 0x301);
    // equal keys before this scan unit, and its first output position
    int eq_seen = sh.weoff[wid] + (per_thread ? ieq - ceq : 0);
    int pos = sh.woff[wid] + (per_thread ? incl - cnt : 0) + max(0, eq_seen - eq_drop);
    if constexpr (per_thread) {
        for (int t = beg; t < end; ++t) {
            const unsigned kt = select_key(sc[t]) >> tsh;
            bool keep;
            if (whole) {
                keep = kt >= thr;
            } else if (kt == thr) {
                keep = eq_seen >= eq_drop;
                ++eq_seen;
            } else {
                keep = kt > thr;
            }
            if (keep) {
                if (pos < k) {
                    if (out_g) out_g[pos] = t;
                    if (out_s) out_s[pos] = t;
                }
                ++pos;
            }
        }
    } else {
        for (int t0 = beg; t0 < end; t0 += 32) {
            const int t = t0 + lane;
            const unsigned kt = t < end ? select_key(sc[t]) >> tsh : 0u;
            const bool above = t < end && (whole ? kt >= thr : kt > thr);
            const bool equal = t < end && !whole && kt == thr;
            const unsigned be = __ballot_sync(0xFFFFFFFFu, equal);
            const bool keep = above || (equal && eq_seen + __popc(be & lower) >= eq_drop);
            const unsigned bk = __ballot_sync(0xFFFFFFFFu, keep);
            if (keep) {
                const int p = pos + __popc(bk & lower);
                if (p < k) {
                    if (out_g) out_g[p] = t;
                    if (out_s) out_s[p] = t;
                }
            }
            pos += __popc(bk);
            eq_seen += __popc(be);
        }
    }
    // the lowest kept score is split between kept and dropped tokens only when
    // the passes ended inside a run of equal keys with some of it dropped
    if (tie_out && tid == 0) *tie_out = (!whole && eq_drop > 0) ? eq_total : 0;
    __syncthreads();
}

}  // namespace zp
