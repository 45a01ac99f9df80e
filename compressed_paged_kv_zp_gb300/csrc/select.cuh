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
// whole.  When the passes end inside a run of equal keys, the newest rem of
// them are kept.  One block-wide prefix sum over two counts (keys above T,
// keys equal to T) then writes the kept positions in ascending order, the
// order Alg. 4 preserves.
#pragma once

#include "zp_common.cuh"

namespace zp {

struct SelectShared {
    int hist2[2][256];
    int wsum[32], weq[32];
    int woff[33], weoff[33];
    int red[32];
    unsigned prefix;
    int shift, need, done;
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
static __device__ void block_select_topk(const float *sc, int L, int k, int32_t *out_g, int *out_s, int32_t *tie_out,
                                         unsigned *err, SelectShared &sh) {
    const int tid = threadIdx.x, nthr = blockDim.x;
    const int lane = tid & 31, wid = tid >> 5;
    if (tid == 0) {
        sh.prefix = 0u;
        sh.shift = 32;
        sh.need = k;
        sh.done = 0;
    }
    for (int i = tid; i < 256; i += nthr) sh.hist2[0][i] = 0;
    int hb = 0;  // histogram buffer of the next pass
    for (int pass = 3; pass >= 0; --pass) {
        __syncthreads();
        if (sh.done) break;
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
                if (hist[bin] == rem) sh.done = 1;
            }
        }
        hb ^= 1;
    }
    __syncthreads();
    const unsigned thr = sh.prefix;
    const int tsh = sh.shift;
    // whole: keep iff (key >> tsh) >= thr.  Otherwise the passes ended inside a
    // run of keys equal to thr (tsh = 0): keep those above it and the newest
    // `rem` of those equal to it.
    const bool whole = sh.done != 0;
    const int rem = sh.need;
    const int chunk = (L + nthr - 1) / nthr;
    const int beg = tid * chunk;
    const int end = min(L, beg + chunk);
    int cnt = 0, ceq = 0;
    for (int t = beg; t < end; ++t) {
        const unsigned kt = select_key(sc[t]) >> tsh;
        cnt += whole ? (kt >= thr) : (kt > thr);
        ceq += (!whole && kt == thr) ? 1 : 0;
    }
    int incl = cnt, ieq = ceq;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        const int ye = __shfl_up_sync(0xFFFFFFFFu, ieq, o);
        if (lane >= o) {
            incl += y;
            ieq += ye;
        }
    }
    if (lane == 31) {
        sh.wsum[wid] = incl;
        sh.weq[wid] = ieq;
    }
    __syncthreads();
    if (wid == 0) {
        const int nw = nthr >> 5;
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
    int eq_seen = sh.weoff[wid] + ieq - ceq;  // equal keys before this thread's chunk
    int pos = sh.woff[wid] + incl - cnt + max(0, eq_seen - eq_drop);
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
    // the lowest kept score is split between kept and dropped tokens only when
    // the passes ended inside a run of equal keys with some of it dropped
    if (tie_out && tid == 0) *tie_out = (!whole && eq_drop > 0) ? eq_total : 0;
    __syncthreads();
}

}  // namespace zp
