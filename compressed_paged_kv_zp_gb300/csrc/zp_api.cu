// zp_api.cu -- host-side plumbing of libzp: error messages, per-device
// properties, the device status word and small entry points.
#include <stdarg.h>
#include <stdio.h>

#include <map>
#include <mutex>
#include <string>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "zp_common.cuh"

namespace zp {

// Device status word of this module (one per device context).  Kernels get
// its device address from device_info(); host code never dereferences it.
__device__ unsigned g_zp_status_word;

namespace {
thread_local std::string t_last_error;
std::mutex g_dev_mutex;
DeviceInfo g_dev[64];
bool g_dev_ready[64] = {false};
}  // namespace

zp_status fail(zp_status s, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return s;
}

zp_status cuda_fail(cudaError_t e, const char *where) {
    return fail(ZP_ERR_CUDA, "%s: %s (%s)", where, cudaGetErrorString(e), cudaGetErrorName(e));
}

zp_status ok() {
    t_last_error.clear();
    return ZP_OK;
}

zp_status device_info(DeviceInfo *out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return fail(ZP_ERR_CUDA, "device id %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    if (!g_dev_ready[dev]) {
        DeviceInfo d;
        d.device = dev;
        e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
        e = cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(smem opt-in)");
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_zp_status_word);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status word)");
        d.error_word = static_cast<unsigned *>(p);
        g_dev[dev] = d;
        g_dev_ready[dev] = true;
    }
    *out = g_dev[dev];
    return ZP_OK;
}

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
}  // namespace

zp_status encode_tmap_bf16_3d(void *map, const void *base, const uint64_t dims[3], const uint64_t strides[2],
                              const uint32_t box[3], const char *what) {
    std::call_once(g_encode_once, [] {
        cudaDriverEntryPointQueryResult q;
        void *fn = nullptr;
        const cudaError_t e =
            cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (e == cudaSuccess && q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (!g_encode) return fail(ZP_ERR_CUDA, "%s: cuTensorMapEncodeTiled unavailable", what);
    const cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
    const cuuint64_t st[2] = {strides[0], strides[1]};
    const cuuint32_t bx[3] = {box[0], box[1], box[2]};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = g_encode(static_cast<CUtensorMap *>(map), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                                const_cast<void *>(base), d, st, bx, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(ZP_ERR_CUDA, "%s: cuTensorMapEncodeTiled failed (%d)", what, (int)r);
    return ZP_OK;
}

namespace {
std::mutex g_smem_mutex;
std::map<std::pair<const void *, int>, size_t> g_smem_set;  // (kernel, device) -> bytes
}  // namespace

zp_status set_max_dynamic_smem(const void *func, size_t bytes, const char *what) {
    // (set even below 48 KB: that default limit covers a kernel's static and
    // dynamic shared memory together)
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, what);
    std::lock_guard<std::mutex> lock(g_smem_mutex);
    size_t &have = g_smem_set[std::make_pair(func, dev)];
    if (have >= bytes) return ZP_OK;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return cuda_fail(e, what);
    have = bytes;
    return ZP_OK;
}

zp_status check_desc(const zp_cache_desc *D) {
    if (!D) return fail(ZP_ERR_INVALID_ARG, "NULL cache descriptor");
    if (D->dtype != ZP_BF16 && D->dtype != ZP_F32) return fail(ZP_ERR_DTYPE, "unknown dtype %d", D->dtype);
    if (D->h_q <= 0 || D->h_kv <= 0 || D->h_q % D->h_kv != 0)
        return fail(ZP_ERR_SHAPE, "heads h_q=%d h_kv=%d", D->h_q, D->h_kv);
    if (D->head_dim <= 0 || D->head_dim % 16 != 0) return fail(ZP_ERR_SHAPE, "head_dim %d", D->head_dim);
    if (D->block_size <= 0) return fail(ZP_ERR_SHAPE, "block_size %d", D->block_size);
    if (D->n_total_blocks <= 0) return fail(ZP_ERR_SHAPE, "n_total_blocks %d", D->n_total_blocks);
    return ZP_OK;
}

}  // namespace zp

using namespace zp;

extern "C" const char *zp_last_error(void) { return t_last_error.c_str(); }

extern "C" const char *zp_status_string(zp_status s) {
    switch (s) {
        case ZP_OK: return "ZP_OK";
        case ZP_ERR_INVALID_ARG: return "ZP_ERR_INVALID_ARG";
        case ZP_ERR_SHAPE: return "ZP_ERR_SHAPE";
        case ZP_ERR_DTYPE: return "ZP_ERR_DTYPE";
        case ZP_ERR_CAPACITY: return "ZP_ERR_CAPACITY";
        case ZP_ERR_CUDA: return "ZP_ERR_CUDA";
        case ZP_ERR_TIMEOUT: return "ZP_ERR_TIMEOUT";
        case ZP_ERR_DEVICE: return "ZP_ERR_DEVICE";
    }
    return "ZP_ERR_UNKNOWN";
}

extern "C" int32_t zp_version(void) { return 1; }

extern "C" zp_status zp_device_status(int32_t *code, int32_t *detail, int32_t clear) {
    DeviceInfo dev;
    zp_status rc = device_info(&dev);
    if (rc != ZP_OK) return rc;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "zp_device_status: synchronize");
    unsigned w = 0;
    e = cudaMemcpy(&w, dev.error_word, sizeof w, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "zp_device_status: read");
    if (code) *code = (int32_t)(w >> 24);
    if (detail) *detail = (int32_t)(w & 0xFFFFFFu);
    if (clear) {
        e = cudaMemset(dev.error_word, 0, sizeof w);
        if (e != cudaSuccess) return cuda_fail(e, "zp_device_status: clear");
    }
    return ok();
}

extern "C" int32_t zp_needs_compression(int32_t seq_len, int32_t block_size, int32_t max_blocks) {
    if (seq_len <= 0 || block_size <= 0) return 0;
    const int32_t n = (seq_len + block_size - 1) / block_size;
    return (n >= max_blocks && seq_len % block_size == 0) ? 1 : 0;
}

extern "C" zp_status zp_needs_compression_batch(const int32_t *seq_lens, const uint8_t *active, int32_t n,
                                                int32_t block_size, int32_t max_blocks,
                                                const int32_t *max_blocks_seq, int32_t *triggered,
                                                int32_t *n_triggered) {
    if (n < 0 || block_size <= 0 || !n_triggered || (n > 0 && (!seq_lens || !triggered)))
        return fail(ZP_ERR_INVALID_ARG, "needs_compression_batch: bad argument");
    int32_t m = 0;
    for (int32_t i = 0; i < n; ++i) {
        if (active && !active[i]) continue;
        const int32_t nb = max_blocks_seq ? max_blocks_seq[i] : max_blocks;
        if (zp_needs_compression(seq_lens[i], block_size, nb)) triggered[m++] = i;
    }
    *n_triggered = m;
    return ok();
}
