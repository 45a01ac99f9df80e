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

#include "select.cuh"

namespace zp {
namespace {

constexpr int kThreads = 1024;
// Scores are staged in shared memory when the row fits (kSmemRow floats), so
// the radix passes never go back to global memory.
constexpr int kSmemRow = 32768;

template <bool STAGED, bool WARP_SCAN>
__global__ void __launch_bounds__(kThreads) topk_kernel(const float *scores, int h_kv, int Lmax,
                                                        const int32_t *seq_lens, int k, const int32_t *k_seq,
                                                        int32_t *keep, int32_t *tie_count, unsigned *err) {
    extern __shared__ float srow[];
    __shared__ SelectShared sh;
    const int kvh = blockIdx.x;
    const int s = blockIdx.y;
    const int tid = threadIdx.x;
    int L = seq_lens[s];
    if (L < 0) L = 0;
    if (L > Lmax) L = Lmax;
    const float *sc = scores + ((size_t)s * h_kv + kvh) * Lmax;
    int32_t *out = keep + ((size_t)s * h_kv + kvh) * k;  // row stride k
    int ki = k_seq ? k_seq[s] : k;                       // this request's budget
    if (ki < 0 || ki > k) {
        if (tid == 0) record_error(err, ZP_ERR_DEVICE, 0x302);
        ki = ki < 0 ? 0 : k;
    }
    for (int r = ki + tid; r < k; r += blockDim.x) out[r] = -1;
    if (L <= ki) {
        for (int r = tid; r < ki; r += blockDim.x) out[r] = r < L ? r : -1;
        if (tie_count && tid == 0) tie_count[(size_t)s * h_kv + kvh] = 0;
        return;
    }
    if constexpr (STAGED) {
        for (int t = tid; t < L; t += blockDim.x) srow[t] = sc[t];
        __syncthreads();
        sc = srow;
    }
    block_select_topk<WARP_SCAN>(sc, L, ki, out, nullptr, tie_count ? tie_count + (size_t)s * h_kv + kvh : nullptr, err, sh);
}

}  // namespace
}  // namespace zp

using namespace zp;

extern "C" zp_status zp_select_topk(const float *scores, int32_t h_kv, int32_t Lmax,
                                    const int32_t *seq_lens, int32_t n, int32_t k, const int32_t *k_seq,
                                    int32_t *keep_idx, int32_t *tie_count, void *stream) {
    if (n < 0 || h_kv <= 0 || Lmax < 0 || k < 0) return fail(ZP_ERR_INVALID_ARG, "topk: bad sizes");
    if (n == 0 || k == 0) return ok();
    if (!scores || !seq_lens || !keep_idx) return fail(ZP_ERR_INVALID_ARG, "topk: NULL buffer");
    DeviceInfo dev;
    zp_status rc = device_info(&dev);
    if (rc != ZP_OK) return rc;
    dim3 grid(h_kv, n);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // the final scan per warp once a thread would scan more than four keys
    const bool warp_scan = (Lmax + kThreads - 1) / kThreads > 4;
    if (Lmax <= kSmemRow) {
        const size_t smem = (size_t)Lmax * 4;
        auto kern = warp_scan ? topk_kernel<true, true> : topk_kernel<true, false>;
        zp_status rs = set_max_dynamic_smem(reinterpret_cast<const void *>(kern), smem, "topk: shared-memory attribute");
        if (rs != ZP_OK) return rs;
        kern<<<grid, kThreads, smem, st>>>(scores, h_kv, Lmax, seq_lens, k, k_seq, keep_idx, tie_count, dev.error_word);
    } else {
        topk_kernel<false, true><<<grid, kThreads, 0, st>>>(scores, h_kv, Lmax, seq_lens, k, k_seq, keep_idx,
                                                            tie_count, dev.error_word);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "topk: launch");
    return ok();
}
