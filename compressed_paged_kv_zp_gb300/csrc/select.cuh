// select.cuh -- block-wide top-k keep set of one score row (Zipage paper
// §4.2: the k = (N_max-1)*b highest-scoring entries are retained; App. C.6).
//
// Each score becomes a 64-bit key: the high word orders floats (sign-flipped
// bits), the low word is the position, so equal scores rank the newer token
// first and all keys are distinct.  A most-significant-byte-first radix
// select (256-bin shared histogram per pass, early exit once the bin holding
// the k-th key is taken whole) finds the threshold key; a block-wide prefix
// sum over the keep flags then writes the kept positions in ascending order,
// the order Alg. 4 preserves.
#pragma once

#include "zp_common.cuh"

namespace zp {

struct SelectShared {
    int hist[256];
    int wsum[32];
    int woff[33];
    int red[32];
    float fmin[32];
    unsigned long long prefix;
    int shift, need, done;
};

static __device__ __forceinline__ unsigned long long select_key(float f, int t) {
    unsigned u = __float_as_uint(f);
    u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((unsigned long long)u << 32) | (unsigned)t;
}

static __device__ __forceinline__ int select_block_sum(int v, SelectShared &sh) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    __syncthreads();
    if (lane == 0) sh.red[warp] = v;
    __syncthreads();
    int tot = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += sh.red[w];
    return tot;
}

// The k highest of sc[0..L) (L > k; sc may be in shared or global memory),
// positions ascending to out_g[0..k) (global, nullable) and out_s (shared,
// nullable).  tie_out (nullable): tokens sharing the score of the lowest kept
// token when that score was split between kept and dropped tokens, else 0.
// Every thread of the block calls it (blockDim.x a multiple of 32, <= 1024).
static __device__ void block_select_topk(const float *sc, int L, int k, int32_t *out_g, int *out_s, int32_t *tie_out,
                                  unsigned *err, SelectShared &sh) {
    const int tid = threadIdx.x, nthr = blockDim.x;
    if (tid == 0) {
        sh.prefix = 0;
        sh.shift = 64;
        sh.need = k;
        sh.done = 0;
    }
    for (int pass = 7; pass >= 0; --pass) {
        __syncthreads();
        if (sh.done) break;
        for (int i = tid; i < 256; i += nthr) sh.hist[i] = 0;
        __syncthreads();
        const int shift = pass * 8;
        const unsigned long long pre = sh.prefix;
        const int pshift = sh.shift;
        for (int t = tid; t < L; t += nthr) {
            const float f = sc[t];
            if (f != f) record_error(err, ZP_ERR_DEVICE, 0x300);
            const unsigned long long key = select_key(f, t);
            if (pshift == 64 || (key >> pshift) == pre) atomicAdd(&sh.hist[(key >> shift) & 255], 1);
        }
        __syncthreads();
        if (tid < 32) {
            // lane l owns bins 8l..8l+7; a suffix scan over the lanes finds the
            // bin where the count from the top reaches `need`
            const int need = sh.need;
            int h8[8], tot = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                h8[j] = sh.hist[8 * tid + j];
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
                sh.prefix = (pshift == 64 ? 0ull : (pre << 8)) | (unsigned long long)bin;
                sh.shift = shift;
                sh.need = rem;
                if (sh.hist[bin] == rem) sh.done = 1;
            }
        }
    }
    __syncthreads();
    const unsigned long long thr = sh.prefix;
    const int tsh = sh.shift;
    // keep iff the key's top (64 - tsh) bits >= thr; ascending positions
    const int chunk = (L + nthr - 1) / nthr;
    const int beg = tid * chunk;
    const int end = min(L, beg + chunk);
    int cnt = 0;
    for (int t = beg; t < end; ++t) cnt += (select_key(sc[t], t) >> tsh) >= thr;
    const int lane = tid & 31, wid = tid >> 5;
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) sh.wsum[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        const int nw = nthr >> 5;
        const int w = lane < nw ? sh.wsum[lane] : 0;
        int wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xFFFFFFFFu, wi, o);
            if (lane >= o) wi += y;
        }
        if (lane < nw) sh.woff[lane] = wi - w;
        if (lane == nw - 1) sh.woff[32] = wi;
    }
    __syncthreads();
    int pos = sh.woff[wid] + incl - cnt;
    if (sh.woff[32] != k && tid == 0) record_error(err, ZP_ERR_DEVICE, 0x301);
    float kept_min = INFINITY;
    for (int t = beg; t < end; ++t) {
        const float f = sc[t];
        if ((select_key(f, t) >> tsh) >= thr) {
            if (pos < k) {
                if (out_g) out_g[pos] = t;
                if (out_s) out_s[pos] = t;
            }
            ++pos;
            kept_min = fminf(kept_min, f);
        }
    }
    if (tie_out) {
        for (int o = 16; o; o >>= 1) kept_min = fminf(kept_min, __shfl_xor_sync(0xFFFFFFFFu, kept_min, o));
        __syncthreads();
        if (lane == 0) sh.fmin[wid] = kept_min;
        __syncthreads();
        float mk = INFINITY;
        for (int w = 0; w < (nthr >> 5); ++w) mk = fminf(mk, sh.fmin[w]);
        int eq_kept = 0, eq_drop = 0;
        for (int t = tid; t < L; t += nthr) {
            const float f = sc[t];
            if (f == mk) {
                if ((select_key(f, t) >> tsh) >= thr) ++eq_kept;
                else ++eq_drop;
            }
        }
        const int a = select_block_sum(eq_kept, sh);
        const int b2 = select_block_sum(eq_drop, sh);
        if (tid == 0) *tie_out = b2 > 0 ? a + b2 : 0;
    }
    __syncthreads();
}

}  // namespace zp
