// zp_common.cuh -- device helpers shared by the kernels of libzp (sm_103a).
//
// Inline PTX for the Blackwell pieces used here: mbarrier waits with an
// iteration bound, 1-D bulk copies (cp.async.bulk, TMA engine) with an L2
// eviction hint, and the packed fp32x2 FMA.  Nothing here traps: failures are
// recorded in the library's device status word and the kernel carries on.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "zp_internal.h"

namespace zp {

// ---------------------------------------------------------------- status word
// The first error wins; the word holds (code << 24) | detail.
__device__ __forceinline__ void record_error(unsigned *err, unsigned code, unsigned detail) {
    if (err) atomicCAS(err, 0u, (code << 24) | (detail & 0xFFFFFFu));
}

// ---------------------------------------------------------------- element IO
template <typename T> struct Elem;
template <> struct Elem<float> {
    static constexpr int kBytes = 4;
};
template <> struct Elem<__nv_bfloat16> {
    static constexpr int kBytes = 2;
};

// bf16x2 word -> (low element, high element) as floats: the bf16 bits are the
// high half of the fp32 bits.
__device__ __forceinline__ float2 bf2_to_f2(uint32_t w) {
    float2 r;
    r.x = __uint_as_float(w << 16);
    r.y = __uint_as_float(w & 0xFFFF0000u);
    return r;
}

__device__ __forceinline__ uint32_t f2_to_bf2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// ---------------------------------------------------------------- fp32x2 FMA
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    unsigned long long A = *reinterpret_cast<unsigned long long *>(&a);
    unsigned long long Bv = *reinterpret_cast<unsigned long long *>(&b);
    unsigned long long C = *reinterpret_cast<unsigned long long *>(&c);
    unsigned long long Dv;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(Dv) : "l"(A), "l"(Bv), "l"(C));
    return *reinterpret_cast<float2 *>(&Dv);
}

__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
    unsigned long long A = *reinterpret_cast<unsigned long long *>(&a);
    unsigned long long Bv = *reinterpret_cast<unsigned long long *>(&b);
    unsigned long long Dv;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(Dv) : "l"(A), "l"(Bv));
    return *reinterpret_cast<float2 *>(&Dv);
}

// 2^x by the PTX ISA's approximate base-2 exponential (ex2.approx.ftz.f32,
// relative error ~2^-22; inputs below -126 give 0).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\t"
        "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, unsigned bytes) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\t"
        "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
        "r"(bytes)
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, unsigned parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, 1000000;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase with the given parity to complete.  Gives up after
// about kWaitLimitNs of wall time, records ZP_ERR_TIMEOUT and returns false;
// *abort is then set so that the other waits of the CTA return at once.
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // 1 s

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, unsigned parity, unsigned *err,
                                                  volatile int *abort, unsigned where) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (true) {
        if (*abort) return false;
        if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > kWaitLimitNs) {
            record_error(err, ZP_ERR_TIMEOUT, where);
            *abort = 1;
            return false;
        }
    }
}

// ---------------------------------------------------------------- bulk copy
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Global -> shared 1-D bulk copy completing on `bar` (bytes and both addresses
// multiples of 16).
__device__ __forceinline__ void bulk_g2s(void *dst_smem, const void *src, unsigned bytes,
                                         uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst_smem)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t l2_evict_last_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 4-byte global store with an L2 cache-policy hint.
__device__ __forceinline__ void st_global_hint(float *p, float v, uint64_t policy) {
    asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(p), "f"(v), "l"(policy) : "memory");
}

// Asynchronous prefetch of [src, src + bytes) into L2 (bytes and src multiples of 16).
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, unsigned bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Global -> shared 1-D bulk copy completing on `bar`, default L2 policy.
__device__ __forceinline__ void bulk_g2s_plain(void *dst_smem, const void *src, unsigned bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst_smem)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Shared -> global 1-D bulk copy (bulk-group completion; bytes and both
// addresses multiples of 16).  Before it, fence_proxy_async_smem() makes the
// CTA's ordinary shared-memory writes visible to the copy engine.
__device__ __forceinline__ void bulk_s2g(void *dst, const void *src_smem, unsigned bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
                 "r"(smem_u32(src_smem)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// the shared-memory sources of all committed groups have been read
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ldmatrix: four 8x8 b16 matrices; lane i gives the row address of matrix
// i/8, row i%8.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
                 : "memory");
}

// D += A(16x16 bf16, row) * B(16x8 bf16, col), fp32 accumulate.
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}



__device__ __forceinline__ void named_bar_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}
// the same with the barrier id a constant (so that only the ids used count)
template <int ID>
__device__ __forceinline__ void named_bar_sync_id(int threads) {
    asm volatile("bar.sync %0, %1;" ::"n"(ID), "r"(threads) : "memory");
}

// ---------------------------------------------------------------- misc
__device__ __forceinline__ float warp_max_xor(float v, int mask) {
    return fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, mask));
}

}  // namespace zp
