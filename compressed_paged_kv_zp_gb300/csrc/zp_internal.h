// zp_internal.h -- declarations shared by the translation units of libzp.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "zp.h"

namespace zp {

// Host: record a message for zp_last_error() and return the status.
zp_status fail(zp_status s, const char *fmt, ...);
zp_status cuda_fail(cudaError_t e, const char *where);
zp_status ok();

// Host: properties of the current device (cached per device).
struct DeviceInfo {
    int device;
    int sm_count;
    int smem_optin;  // max dynamic shared memory per block
    unsigned *error_word;  // device address of the status word
};
zp_status device_info(DeviceInfo *out);

// Host: raise the dynamic shared-memory limit of kernel `func` on the current
// device to at least `bytes` (one call per kernel, device and larger size;
// safe from several host threads).  A failure
// returns ZP_ERR_CUDA with `what` in the message.
zp_status set_max_dynamic_smem(const void *func, size_t bytes, const char *what);

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline int elem_bytes(int dtype) { return dtype == ZP_BF16 ? 2 : (dtype == ZP_F32 ? 4 : 0); }

zp_status check_desc(const zp_cache_desc *D);

// Host: a 3-D tiled tensor map of bf16 elements with the 128-byte swizzle
// (tensor maps for the TMA loads of tcgen05 operands).  dims innermost first;
// strides (bytes) of dims 1 and 2; box innermost first (box[0] * 2 <= 128).
// Encoded through the driver entry point (no link against libcuda).
zp_status encode_tmap_bf16_3d(void *map /* CUtensorMap */, const void *base, const uint64_t dims[3],
                              const uint64_t strides[2], const uint32_t box[3], const char *what);

// All-pairs key redundancy of one layer (redundancy.cu): rho [n][h_kv][Lmax]
// receives the row sums of the thresholded cosine matrix of every sequence and
// kv head (overwritten).  Lengths are clamped to Lcap.
struct AllPairsArgs {
    const void *k;  // paged keys of the layer
    int dtype;      // ZP_BF16 or ZP_F32
    const int32_t *table;
    int table_stride;
    const int32_t *seq_lens;
    int n, h_kv, d, b, n_total, Lmax, Lcap;
    float p;
    float *rho;
    void *workspace;  // all_pairs_workspace_size bytes
};
size_t all_pairs_workspace_size(int n, int h_kv, int d, int Lmax);
zp_status launch_all_pairs(const AllPairsArgs &a, cudaStream_t st);

}  // namespace zp
