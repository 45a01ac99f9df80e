// append_kv.cu -- store the new token's key and value rows into their slots.
//
// Zipage paper §3: the KV cache of each block is written into free blocks of
// the pre-allocated K and V; the block table records where.  The row of one
// token (all kv heads) is contiguous in the [N_total][b][h_kv][d] layout, so
// one CTA per sequence copies it with 16-byte vectors.
#include "zp_common.cuh"

namespace zp {
namespace {

__global__ void append_kv_kernel(const uint4 *k_new, const uint4 *v_new, uint4 *K, uint4 *V,
                                 const int32_t *table, int table_stride, const int32_t *seq_lens,
                                 int b, int n_total, int row_vec, unsigned *err) {
    const int s = blockIdx.x;
    const int L = seq_lens[s];
    if (L == 0) return;  // no token for this sequence in this step
    if (L < 0 || L > table_stride * b) {
        if (threadIdx.x == 0) record_error(err, ZP_ERR_DEVICE, 0x100);
        return;
    }
    const int P = L - 1;
    const int blk = table[(size_t)s * table_stride + P / b];
    if (blk < 0 || blk >= n_total) {
        if (threadIdx.x == 0) record_error(err, ZP_ERR_DEVICE, 0x101);
        return;
    }
    const size_t dst = ((size_t)blk * b + P % b) * row_vec;
    const size_t src = (size_t)s * row_vec;
    for (int i = threadIdx.x; i < row_vec; i += blockDim.x) {
        K[dst + i] = k_new[src + i];
        V[dst + i] = v_new[src + i];
    }
}

}  // namespace
}  // namespace zp

using namespace zp;

extern "C" zp_status zp_append_kv(const zp_cache_desc *D, const void *k_new, const void *v_new,
                                  void *k_cache, void *v_cache, const int32_t *block_table,
                                  int32_t table_stride, const int32_t *seq_lens, int32_t B,
                                  void *stream) {
    zp_status rc = check_desc(D);
    if (rc != ZP_OK) return rc;
    if (B < 0 || table_stride < 1) return fail(ZP_ERR_INVALID_ARG, "append: B=%d table_stride=%d", B, table_stride);
    if (B == 0) return ok();
    if (!k_new || !v_new || !k_cache || !v_cache || !block_table || !seq_lens)
        return fail(ZP_ERR_INVALID_ARG, "append: NULL buffer");
    const size_t row_bytes = (size_t)D->h_kv * D->head_dim * elem_bytes(D->dtype);
    if (row_bytes % 16) return fail(ZP_ERR_SHAPE, "append: row of %zu bytes not a multiple of 16", row_bytes);
    const uintptr_t al = (uintptr_t)k_new | (uintptr_t)v_new | (uintptr_t)k_cache | (uintptr_t)v_cache;
    if (al % 16) return fail(ZP_ERR_INVALID_ARG, "append: buffers must be 16-byte aligned");
    DeviceInfo dev;
    rc = device_info(&dev);
    if (rc != ZP_OK) return rc;
    const int row_vec = (int)(row_bytes / 16);
    const int threads = row_vec >= 128 ? 128 : 32;
    append_kv_kernel<<<B, threads, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4 *>(k_new), static_cast<const uint4 *>(v_new), static_cast<uint4 *>(k_cache),
        static_cast<uint4 *>(v_cache), block_table, table_stride, seq_lens, D->block_size,
        D->n_total_blocks, row_vec, dev.error_word);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "append: launch");
    return ok();
}
