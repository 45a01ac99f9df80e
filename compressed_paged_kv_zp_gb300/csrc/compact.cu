// compact.cu -- gather-compaction of the kept rows into the target blocks.
//
// Zipage paper App. C.6, Alg. 4: the kept entries of a sequence are packed, in
// their original order, into the first N_max - 1 blocks (or the target blocks
// of §4.4 when prefix blocks are shared).  Rank r of the keep list goes to
// slot r % b of target block r / b.  The global score cache F of that slot
// receives the kept token's global score ("compress score"), read from the
// sequence's score row where zp_score_tokens left it: F is written only in
// target blocks, never in a source block another sequence may share.
//
// One CTA per (kv head, sequence, layer).  Alg. 4 walks one slot at a time;
// here a CTA moves a chunk of up to 128 ranks at once: every thread first loads
// its share of the chunk's source rows (16-byte vectors) into registers, the
// CTA synchronises, then the rows are stored.  Rank r's source position is
// >= r, so a chunk's stores (positions < chunk end) never overwrite a source
// of a later chunk, and the barrier orders the loads of the chunk before its
// own stores: the move is correct in place as well as into fresh blocks.
#include "zp_common.cuh"

namespace zp {
namespace {

constexpr int kChunkMax = 128;       // ranks per load/store round (at most)
constexpr int kThreads = 256;
constexpr int kMaxVecPerThread = 16;  // registers of 16 bytes per thread and round

struct CompactArgs {
    uint4 *K;
    uint4 *V;
    long long layer_stride_vec;  // in 16-byte vectors
    float *F;
    long long F_layer_stride;
    const float *S;  // score rows: S + layer*S_layer_stride + (row*h_kv + kvh)*S_stride + pos
    long long S_stride, S_layer_stride;
    const int32_t *S_rows;  // nullable
    const int32_t *src_table;
    int table_stride;
    const int32_t *dst;
    int target_stride;
    const int32_t *seq_lens;
    const int32_t *keep;
    const int32_t *k_seq;  // nullable: per-request budgets
    int k, n, h_kv, b, n_total;
    int row_vec;  // vectors per (token, kv head) row = d * elem / 16
    int chunk;    // ranks per round: min(kChunkMax, kThreads * kMaxVecPerThread / (2 * row_vec))
    unsigned *err;
};

__global__ void __launch_bounds__(kThreads) compact_kernel(const CompactArgs a) {
    const int kvh = blockIdx.x;
    const int s = blockIdx.y;
    const int layer = blockIdx.z;
    int L = a.seq_lens[s];
    if (L > a.table_stride * a.b) L = a.table_stride * a.b;
    const int32_t *kp = a.keep + (((size_t)layer * a.n + s) * a.h_kv + kvh) * a.k;
    uint4 *K = a.K + layer * a.layer_stride_vec;
    uint4 *V = a.V + layer * a.layer_stride_vec;
    float *F = a.F ? a.F + layer * a.F_layer_stride : nullptr;
    const float *Srow = nullptr;
    if (F) {
        const int row = a.S_rows ? a.S_rows[s] : s;
        if (row < 0) {
            if (threadIdx.x == 0) record_error(a.err, ZP_ERR_DEVICE, 0x402);
            F = nullptr;
        } else {
            Srow = a.S + layer * a.S_layer_stride + ((size_t)row * a.h_kv + kvh) * a.S_stride;
        }
    }
    if (F && L > a.S_stride) L = (int)a.S_stride;
    const int kk = min(a.k_seq ? min(a.k_seq[s], a.k) : a.k, L);
    const int per_rank = 2 * a.row_vec;  // K then V vectors
    for (int r0 = 0; r0 < kk; r0 += a.chunk) {
        const int nr = min(a.chunk, kk - r0);
        const int items = nr * per_rank;
        uint4 buf[kMaxVecPerThread];
        float fbuf = 0.f;
        // ---- load phase
#pragma unroll
        for (int i = 0; i < kMaxVecPerThread; ++i) {
            const int it = threadIdx.x + i * kThreads;
            if (it < items) {
                const int r = r0 + it / per_rank;
                const int v = it % per_rank;
                const int pos = kp[r];
                int blk = -1;
                if (pos >= 0 && pos < L) blk = a.src_table[(size_t)s * a.table_stride + pos / a.b];
                if (blk < 0 || blk >= a.n_total) {
                    record_error(a.err, ZP_ERR_DEVICE, 0x400);
                    buf[i] = make_uint4(0, 0, 0, 0);
                } else {
                    const size_t row = ((size_t)blk * a.b + pos % a.b) * a.h_kv + kvh;
                    const uint4 *base = v < a.row_vec ? K : V;
                    buf[i] = base[row * a.row_vec + (v % a.row_vec)];
                }
            }
        }
        if (F && threadIdx.x < nr) {  // nr <= kChunkMax <= kThreads
            const int pos = kp[r0 + threadIdx.x];
            if (pos >= 0 && pos < L) fbuf = Srow[pos];
        }
        __syncthreads();
        // ---- store phase
#pragma unroll
        for (int i = 0; i < kMaxVecPerThread; ++i) {
            const int it = threadIdx.x + i * kThreads;
            if (it < items) {
                const int r = r0 + it / per_rank;
                const int v = it % per_rank;
                const int blk = a.dst[(size_t)s * a.target_stride + r / a.b];
                if (blk < 0 || blk >= a.n_total) {
                    record_error(a.err, ZP_ERR_DEVICE, 0x401);
                } else {
                    const size_t row = ((size_t)blk * a.b + r % a.b) * a.h_kv + kvh;
                    uint4 *base = v < a.row_vec ? K : V;
                    base[row * a.row_vec + (v % a.row_vec)] = buf[i];
                }
            }
        }
        if (F && threadIdx.x < nr) {
            const int r = r0 + threadIdx.x;
            const int blk = a.dst[(size_t)s * a.target_stride + r / a.b];
            if (blk >= 0 && blk < a.n_total) F[((size_t)blk * a.b + r % a.b) * a.h_kv + kvh] = fbuf;
        }
        __syncthreads();
    }
}

// Main variant, one CTA per (tensor, kv head, sequence, layer): K and V are
// independent, so each moves in a CTA of its own (twice the CTAs, half the
// bytes each).  The CTA first resolves, in shared memory, every rank's keep
// position, source block, F value and the target blocks (two rounds of
// independent loads); then per chunk of up to kVChunk ranks every thread loads
// its share of the chunk's row pieces (16-byte vectors of this kv head's row
// in its tensor) into registers, the CTA synchronises, and the pieces are
// stored to the target slots; the K CTA also writes F.  A chunk reads positions >= its first rank and earlier
// chunks write slots below it, and a slot shared by a source and a target has
// the same index in both (the target rule): the move is correct in place.
// (Many small bulk copies were measured slower: the copy engine keeps few
// requests in flight per SM.)
constexpr int kVChunk = 512;
constexpr int kVThreads = 1024;  // rounds of 512 ranks for 256-byte row pieces (64 ranks with 256 threads
                                 // took 4x the load-then-store round trips, each one a memory latency)
constexpr int kVPerThread = 8;   // 16-byte registers per thread and chunk (row pieces up to 256 B)

// dynamic shared memory: pos[k], src block[k] (ints), F values[k], target blocks[ceil(k/b)]
__host__ __device__ inline size_t compact_meta_smem(int k, int b) {
    return (size_t)k * 12 + (size_t)((k + b - 1) / b) * 4 + 16;
}

__global__ void __launch_bounds__(kVThreads, 1) compact_vec_kernel(const CompactArgs a) {
    extern __shared__ __align__(16) unsigned char csm[];
    __shared__ int s_L;
    const int kvh = blockIdx.x >> 1;
    const int tensor = blockIdx.x & 1;  // 0: K (and F), 1: V
    const int s = blockIdx.y;
    const int layer = blockIdx.z;
    const int tid = threadIdx.x;
    int *pos_s = reinterpret_cast<int *>(csm);
    int *src_s = pos_s + a.k;
    float *f_s = reinterpret_cast<float *>(src_s + a.k);
    int *dst_s = reinterpret_cast<int *>(f_s + a.k);
    const int32_t *kp = a.keep + (((size_t)layer * a.n + s) * a.h_kv + kvh) * a.k;
    uint4 *X = (tensor ? a.V : a.K) + layer * a.layer_stride_vec;  // this CTA's tensor
    float *F = (a.F && tensor == 0) ? a.F + layer * a.F_layer_stride : nullptr;
    const int nt = (a.k + a.b - 1) / a.b;
    // ---- first loads: length, keep positions, target blocks (independent)
    if (tid == 0) {
        int L = a.seq_lens[s];
        if (L > a.table_stride * a.b) L = a.table_stride * a.b;
        s_L = L;
    }
    for (int r = tid; r < a.k; r += blockDim.x) pos_s[r] = kp[r];
    for (int t = tid; t < nt; t += blockDim.x) dst_s[t] = a.dst[(size_t)s * a.target_stride + t];
    __syncthreads();
    const float *Srow = nullptr;
    int L = s_L;
    if (F) {
        const int row = a.S_rows ? a.S_rows[s] : s;
        if (row < 0) {
            if (tid == 0) record_error(a.err, ZP_ERR_DEVICE, 0x402);
            F = nullptr;
        } else {
            Srow = a.S + layer * a.S_layer_stride + ((size_t)row * a.h_kv + kvh) * a.S_stride;
            if (L > a.S_stride) L = (int)a.S_stride;
        }
    }
    const int kk = min(a.k_seq ? min(a.k_seq[s], a.k) : a.k, L);
    // ---- second loads: source blocks and F values of every rank
    for (int r = tid; r < kk; r += blockDim.x) {
        const int pos = pos_s[r];
        int blk = -1;
        if (pos >= 0 && pos < L) blk = a.src_table[(size_t)s * a.table_stride + pos / a.b];
        if (blk < 0 || blk >= a.n_total) {
            record_error(a.err, ZP_ERR_DEVICE, 0x400);
            blk = -1;
        }
        src_s[r] = blk;
        if (F) f_s[r] = (blk >= 0) ? Srow[pos] : 0.f;
    }
    __syncthreads();
    const int per_rank = a.row_vec;  // vectors of this kv head's row piece in the tensor
    const int chunk = min(kVChunk, kVThreads * kVPerThread / per_rank);
    for (int r0 = 0; r0 < kk; r0 += chunk) {
        const int nr = min(chunk, kk - r0);
        const int items = nr * per_rank;
        uint4 buf[kVPerThread];
#pragma unroll
        for (int i = 0; i < kVPerThread; ++i) {
            const int it = tid + i * kVThreads;
            if (it < items) {
                const int r = r0 + it / per_rank, v = it % per_rank;
                const int blk = src_s[r];
                if (blk >= 0) {
                    const size_t row = ((size_t)blk * a.b + pos_s[r] % a.b) * a.h_kv + kvh;
                    buf[i] = X[row * a.row_vec + v];
                }
            }
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < kVPerThread; ++i) {
            const int it = tid + i * kVThreads;
            if (it < items) {
                const int r = r0 + it / per_rank, v = it % per_rank;
                const int blk = dst_s[r / a.b];
                if (blk < 0 || blk >= a.n_total) {
                    if (tensor == 0) record_error(a.err, ZP_ERR_DEVICE, 0x401);
                } else if (src_s[r] >= 0) {
                    const size_t row = ((size_t)blk * a.b + r % a.b) * a.h_kv + kvh;
                    X[row * a.row_vec + v] = buf[i];
                }
            }
        }
        if (F)
            for (int i = tid; i < nr; i += blockDim.x) {
                const int r = r0 + i;
                const int blk = dst_s[r / a.b];
                if (blk >= 0 && blk < a.n_total) F[((size_t)blk * a.b + r % a.b) * a.h_kv + kvh] = f_s[r];
            }
        __syncthreads();  // the next chunk's loads follow this chunk's stores
    }
}

}  // namespace
}  // namespace zp

using namespace zp;

extern "C" zp_status zp_compact_pages(const zp_cache_desc *D, void *k_base, void *v_base,
                                      int64_t layer_stride, int32_t layer_count, float *global_F,
                                      int64_t F_layer_stride, const zp_score_rows *scores,
                                      const int32_t *src_table,
                                      int32_t table_stride, const int32_t *dst_targets,
                                      int32_t target_stride, const int32_t *seq_lens,
                                      const int32_t *keep_idx, int32_t k, const int32_t *k_seq, int32_t n,
                                      void *stream) {
    zp_status rc = check_desc(D);
    if (rc != ZP_OK) return rc;
    if (n < 0 || k < 0 || layer_count < 0 || table_stride < 1 || target_stride < 1)
        return fail(ZP_ERR_INVALID_ARG, "compact: bad sizes");
    if (n == 0 || k == 0 || layer_count == 0) return ok();
    if (!k_base || !v_base || !src_table || !dst_targets || !seq_lens || !keep_idx)
        return fail(ZP_ERR_INVALID_ARG, "compact: NULL buffer");
    if (global_F && (!scores || !scores->data || scores->stride < 1))
        return fail(ZP_ERR_INVALID_ARG, "compact: global_F needs the score rows");
    if ((long long)target_stride * D->block_size < k)
        return fail(ZP_ERR_CAPACITY, "compact: %d target blocks hold fewer than k=%d rows", target_stride, k);
    const int es = elem_bytes(D->dtype);
    const size_t row_bytes = (size_t)D->head_dim * es;
    if (row_bytes % 16) return fail(ZP_ERR_SHAPE, "compact: row of %zu bytes", row_bytes);
    const long long elems_per_layer = (long long)D->n_total_blocks * D->block_size * D->h_kv * D->head_dim;
    if (layer_count > 1 && layer_stride < elems_per_layer)
        return fail(ZP_ERR_INVALID_ARG, "compact: layer_stride %lld < one layer", (long long)layer_stride);
    if ((layer_stride * es) % 16) return fail(ZP_ERR_INVALID_ARG, "compact: layer_stride not 16-byte aligned");
    if (((uintptr_t)k_base | (uintptr_t)v_base) % 16) return fail(ZP_ERR_INVALID_ARG, "compact: unaligned cache");
    const int row_vec = (int)(row_bytes / 16);
    int chunk = kThreads * kMaxVecPerThread / (2 * row_vec);
    if (chunk > kChunkMax) chunk = kChunkMax;
    if (chunk < 1) return fail(ZP_ERR_SHAPE, "compact: head_dim %d too large", D->head_dim);
    DeviceInfo dev;
    rc = device_info(&dev);
    if (rc != ZP_OK) return rc;
    CompactArgs a;
    a.K = static_cast<uint4 *>(k_base);
    a.V = static_cast<uint4 *>(v_base);
    a.layer_stride_vec = layer_stride * es / 16;
    a.F = global_F;
    a.F_layer_stride = F_layer_stride;
    a.S = global_F ? scores->data : nullptr;
    a.S_stride = global_F ? scores->stride : 1;
    a.S_layer_stride = global_F ? scores->layer_stride : 0;
    a.S_rows = global_F ? scores->rows : nullptr;
    a.src_table = src_table;
    a.table_stride = table_stride;
    a.dst = dst_targets;
    a.target_stride = target_stride;
    a.seq_lens = seq_lens;
    a.keep = keep_idx;
    a.k_seq = k_seq;
    a.k = k;
    a.n = n;
    a.h_kv = D->h_kv;
    a.b = D->block_size;
    a.n_total = D->n_total_blocks;
    a.row_vec = row_vec;
    a.chunk = chunk;
    a.err = dev.error_word;
    const int meta_smem = (int)compact_meta_smem(k, D->block_size);
    if (row_vec <= kVThreads * kVPerThread && meta_smem <= 96 * 1024) {
        zp_status rs = set_max_dynamic_smem(reinterpret_cast<const void *>(compact_vec_kernel), meta_smem,
                                            "compact: shared-memory attribute");
        if (rs != ZP_OK) return rs;
        dim3 grid(2 * D->h_kv, n, layer_count);  // (tensor, kv head) fastest
        compact_vec_kernel<<<grid, kVThreads, meta_smem, static_cast<cudaStream_t>(stream)>>>(a);
    } else {
        dim3 grid(D->h_kv, n, layer_count);
        compact_kernel<<<grid, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(a);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "compact: launch");
    return ok();
}
