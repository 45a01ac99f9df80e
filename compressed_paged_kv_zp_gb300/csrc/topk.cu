// topk.cu -- segmented top-k keep sets (Zipage paper §4.2: the k = (N_max-1)*b
// highest-scoring entries are retained; App. C.6: top-k tag).
//
// One CTA per (sequence, kv head).  Each score is turned into a 64-bit key
// whose high word orders floats (sign-flipped bits) and whose low word is the
// position, so equal scores rank the newer token first and all keys are
// distinct.  A most-significant-byte-first radix select (256-bin shared
// histogram per pass, early exit once the bin holding the k-th key is taken
// whole) finds the threshold; a block-wide prefix sum over the keep flags then
// writes the kept positions in ascending order, the order Alg. 4 preserves.
#include <math.h>

#include "zp_common.cuh"

namespace zp {
namespace {

constexpr int kThreads = 1024;

__device__ __forceinline__ unsigned long long make_key(float f, int t) {
    unsigned u = __float_as_uint(f);
    u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((unsigned long long)u << 32) | (unsigned)t;
}

__device__ __forceinline__ int block_sum(int v, int *red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    int tot = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += red[w];
    return tot;
}

// Scores are staged in shared memory when the row fits (kSmemRow floats),
// so the radix passes never go back to global memory.
constexpr int kSmemRow = 32768;

template <bool STAGED>
__global__ void __launch_bounds__(kThreads) topk_kernel(const float *scores, int h_kv, int Lmax,
                                                        const int32_t *seq_lens, int k, int32_t *keep,
                                                        int32_t *tie_count, unsigned *err) {
    extern __shared__ float srow[];
    __shared__ int hist[256];
    __shared__ int red[32];
    __shared__ int scan[kThreads];
    __shared__ unsigned long long s_prefix;
    __shared__ int s_shift, s_need, s_done;
    const int kvh = blockIdx.x;
    const int s = blockIdx.y;
    const int tid = threadIdx.x;
    int L = seq_lens[s];
    if (L < 0) L = 0;
    if (L > Lmax) L = Lmax;
    const float *sc = scores + ((size_t)s * h_kv + kvh) * Lmax;
    int32_t *out = keep + ((size_t)s * h_kv + kvh) * k;
    if constexpr (STAGED) {
        if (L > k) {
            for (int t = tid; t < L; t += blockDim.x) srow[t] = sc[t];
            __syncthreads();
            sc = srow;
        }
    }
    if (L <= k) {
        for (int r = tid; r < k; r += blockDim.x) out[r] = r < L ? r : -1;
        if (tie_count && tid == 0) tie_count[(size_t)s * h_kv + kvh] = 0;
        return;
    }
    if (tid == 0) {
        s_prefix = 0;
        s_shift = 64;
        s_need = k;
        s_done = 0;
    }
    for (int pass = 7; pass >= 0; --pass) {
        __syncthreads();
        if (s_done) break;
        for (int i = tid; i < 256; i += blockDim.x) hist[i] = 0;
        __syncthreads();
        const int shift = pass * 8;
        const unsigned long long pre = s_prefix;
        const int pshift = s_shift;
        for (int t = tid; t < L; t += blockDim.x) {
            const float f = sc[t];
            if (f != f) record_error(err, ZP_ERR_DEVICE, 0x300);
            const unsigned long long key = make_key(f, t);
            if (pshift == 64 || (key >> pshift) == pre) atomicAdd(&hist[(key >> shift) & 255], 1);
        }
        __syncthreads();
        if (tid < 32) {
            // warp 0: lane l owns bins 8l..8l+7; a suffix scan over the lanes
            // finds the bin where the count from the top reaches `need`
            const int need = s_need;
            int h8[8], tot = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                h8[j] = hist[8 * tid + j];
                tot += h8[j];
            }
            int incl = tot;  // bins of lanes >= this one
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
                s_prefix = (pshift == 64 ? 0ull : (pre << 8)) | (unsigned long long)bin;
                s_shift = shift;
                s_need = rem;
                if (hist[bin] == rem) s_done = 1;
            }
        }
    }
    __syncthreads();
    const unsigned long long thr = s_prefix;
    const int tsh = s_shift;
    // keep iff key's top (64 - tsh) bits >= thr; write ascending positions
    const int chunk = (L + blockDim.x - 1) / blockDim.x;
    const int beg = tid * chunk;
    const int end = min(L, beg + chunk);
    int cnt = 0;
    for (int t = beg; t < end; ++t) cnt += (make_key(sc[t], t) >> tsh) >= thr;
    // exclusive block scan of cnt: warp shuffles, then the 32 warp totals
    const int lane = tid & 31, wid = tid >> 5;
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) scan[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        const int nw = blockDim.x >> 5;
        int w = lane < nw ? scan[lane] : 0;
        int wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xFFFFFFFFu, wi, o);
            if (lane >= o) wi += y;
        }
        if (lane < nw) scan[32 + lane] = wi - w;  // exclusive warp offsets
        if (lane == nw - 1) scan[64] = wi;        // total
    }
    __syncthreads();
    int pos = scan[32 + wid] + incl - cnt;
    const int total = scan[64];
    if (total != k && tid == 0) record_error(err, ZP_ERR_DEVICE, 0x301);
    float kept_min = INFINITY;
    for (int t = beg; t < end; ++t) {
        const float f = sc[t];
        if ((make_key(f, t) >> tsh) >= thr) {
            if (pos < k) out[pos] = t;
            ++pos;
            kept_min = fminf(kept_min, f);
        }
    }
    if (tie_count) {
        // score of the lowest kept token; ties split between kept and dropped?
        for (int o = 16; o; o >>= 1) kept_min = fminf(kept_min, __shfl_xor_sync(0xFFFFFFFFu, kept_min, o));
        __shared__ float s_min[32];
        __syncthreads();
        if ((tid & 31) == 0) s_min[tid >> 5] = kept_min;
        __syncthreads();
        float mk = INFINITY;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) mk = fminf(mk, s_min[w]);
        int eq_kept = 0, eq_drop = 0;
        for (int t = tid; t < L; t += blockDim.x) {
            const float f = sc[t];
            if (f == mk) {
                if ((make_key(f, t) >> tsh) >= thr) ++eq_kept;
                else ++eq_drop;
            }
        }
        const int a = block_sum(eq_kept, red);
        const int b2 = block_sum(eq_drop, red);
        if (tid == 0) tie_count[(size_t)s * h_kv + kvh] = b2 > 0 ? a + b2 : 0;
    }
}

}  // namespace
}  // namespace zp

using namespace zp;

extern "C" zp_status zp_select_topk(const float *scores, int32_t h_kv, int32_t Lmax,
                                    const int32_t *seq_lens, int32_t n, int32_t k, int32_t *keep_idx,
                                    int32_t *tie_count, void *stream) {
    if (n < 0 || h_kv <= 0 || Lmax < 0 || k < 0) return fail(ZP_ERR_INVALID_ARG, "topk: bad sizes");
    if (n == 0 || k == 0) return ok();
    if (!scores || !seq_lens || !keep_idx) return fail(ZP_ERR_INVALID_ARG, "topk: NULL buffer");
    DeviceInfo dev;
    zp_status rc = device_info(&dev);
    if (rc != ZP_OK) return rc;
    dim3 grid(h_kv, n);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (Lmax <= kSmemRow) {
        const size_t smem = (size_t)Lmax * 4;
        if (smem > 48 * 1024) {
            cudaError_t e = cudaFuncSetAttribute(topk_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)smem);
            if (e != cudaSuccess) return cuda_fail(e, "topk: cudaFuncSetAttribute");
        }
        topk_kernel<true><<<grid, kThreads, smem, st>>>(scores, h_kv, Lmax, seq_lens, k, keep_idx, tie_count,
                                                        dev.error_word);
    } else {
        topk_kernel<false><<<grid, kThreads, 0, st>>>(scores, h_kv, Lmax, seq_lens, k, keep_idx, tie_count,
                                                      dev.error_word);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "topk: launch");
    return ok();
}
