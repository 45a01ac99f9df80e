// window_score.cu -- explicit observation-window attention score.
//
// Zipage paper App. C.2 with Alg. 1: for a sequence of L tokens and the
// queries of its w newest tokens (q_window[u], u = 0 oldest, at position
// L - w + u), for every kv head:
//   A[u,h,t] = q_{u,h} . k_t / sqrt(d), -inf where t > L - w + u  (causal; the
//              printed mask of Alg. 1 is garbled, this is its reading)
//   P[u,h,:] = softmax over t of A[u,h,:]
//   S[t]     = (1/w) * sum_u max_{h in the kv head's group} P[u,h,t]
// This is the prefill-then-compress path: after a long prompt the window
// queries exist but no decode step has accumulated the score.
//
// The R = w*g query rows of a kv head against the sequence's keys form a
// dense contraction (64 x 128 x L for the Qwen3-8B shape), run on the tensor
// cores (mma.sync m16n8k16, bf16 in, fp32 accumulate) in two passes over K:
//   pass 1: per CTA and row, the max and sum of exp over its chunk of pages;
//   merge:  the chunks' statistics -> per row (M, L);
//   pass 2: logits again, P from (M, L), max over the group, sum over u.
// One CTA per (sequence, chunk of pages); a producer warp copies each token
// row of a page (all kv heads, contiguous in HBM) with one bulk copy into a
// padded staging row; one consumer warp per kv head.  fp32 caches take a
// plain CUDA-core kernel (the small parity workload).
#include <math.h>

#include "zp_common.cuh"

namespace zp {
namespace {

constexpr int kPages = 64;   // pages (16-token units) per CTA chunk
constexpr int kWsStages = 2;
constexpr int kRowPad = 16;

struct WsArgs {
    const void *q;       // [n][w][h_q][d]
    const void *k;
    const int32_t *table;
    int table_stride;
    const int32_t *seq_lens;
    int n, h_q, h_kv, d, b, n_total, w, Lmax;
    float qscale;        // log2(e) / sqrt(d)
    float2 *part;        // [n][chunks][h_kv * R] partial (max, sum)
    float2 *stats;       // [n][h_kv * R] final (max, sum)
    float *out;          // [n][h_kv][Lmax]
    int chunks;          // chunk capacity per sequence
    unsigned *err;
};

__device__ __forceinline__ int seq_len(const WsArgs &a, int s) {
    int L = a.seq_lens[s];
    if (L > a.Lmax) L = a.Lmax;
    if (L > a.table_stride * a.b) L = a.table_stride * a.b;
    return L;
}

// ------------------------------------------------------------------ bf16 path
// smem: bars | Q tiles [h_kv][R rows][D*2 + pad] | stages [kWsStages][16 rows][h_kv*D*2 + pad]
template <int D, int MT, int G, bool PASS2>
__global__ void __launch_bounds__(9 * 32, 1) ws_tc_kernel(const WsArgs a) {
    constexpr int R = MT * 16;
    constexpr int KS = D / 16;
    extern __shared__ __align__(128) unsigned char sm[];
    const int s = blockIdx.y;
    const int chunk = blockIdx.x;
    const int L = seq_len(a, s);
    const int npages = (L + 15) / 16;
    const int p0 = chunk * kPages;
    if (p0 >= npages || L < a.w) return;
    const int p1 = min(npages, p0 + kPages);
    const int h_kv = a.h_kv;
    const int QRS = D * 2 + kRowPad;               // Q row stride
    const int KRS = h_kv * D * 2 + kRowPad;        // staged K row stride
    uint64_t *full = reinterpret_cast<uint64_t *>(sm);
    uint64_t *empty = full + kWsStages;
    unsigned char *qs = sm + 128;
    unsigned char *ks0 = qs + (size_t)h_kv * R * QRS;
    ks0 += (128 - (reinterpret_cast<uintptr_t>(ks0) & 127)) & 127;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int stage_bytes = 16 * KRS;

    if (tid == 0) {
        for (int i = 0; i < kWsStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], h_kv);
        }
        fence_barrier_init();
    }
    // Q rows (u, j) of every kv head: row r = u*G + j, q head kvh*G + j
    const __nv_bfloat16 *qg = static_cast<const __nv_bfloat16 *>(a.q) + (size_t)s * a.w * a.h_q * D;
    for (int c = tid; c < h_kv * R * (D / 8); c += blockDim.x) {
        const int kvh = c / (R * (D / 8));
        const int rem = c % (R * (D / 8));
        const int r = rem / (D / 8);
        const int c16 = rem % (D / 8);
        uint4 v = make_uint4(0, 0, 0, 0);
        const int u = r / G, j = r % G;
        if (u < a.w)
            v = reinterpret_cast<const uint4 *>(qg + ((size_t)u * a.h_q + kvh * G + j) * D)[c16];
        reinterpret_cast<uint4 *>(qs + ((size_t)kvh * R + r) * QRS)[c16] = v;
    }
    __syncthreads();
    volatile int abort_flag = 0;

    if (warp == h_kv) {  // producer
        const uint64_t pol = l2_evict_first_policy();
        const unsigned row_bytes = (unsigned)(h_kv * D * 2);
        const __nv_bfloat16 *kg = static_cast<const __nv_bfloat16 *>(a.k);
        for (int p = p0, i = 0; p < p1; ++p, ++i) {
            const int st = i % kWsStages;
            if (i >= kWsStages &&
                !mbar_wait_bounded(&empty[st], (unsigned)(((i / kWsStages) - 1) & 1), a.err, &abort_flag, 50))
                break;
            const int blk = __ldg(&a.table[(size_t)s * a.table_stride + (p * 16) / a.b]);
            const bool bad = blk < 0 || blk >= a.n_total;
            int valid = L - p * 16;
            if (valid > 16) valid = 16;
            if (lane == 0) {
                if (bad) record_error(a.err, ZP_ERR_DEVICE, 0x500);
                mbar_arrive_expect_tx(&full[st], bad ? 0u : valid * row_bytes);
            }
            __syncwarp();
            if (!bad && lane < valid) {
                const size_t off = ((size_t)blk * a.b + (p * 16) % a.b + lane) * h_kv * D;
                bulk_g2s(ks0 + (size_t)st * stage_bytes + lane * KRS, kg + off, row_bytes, &full[st], pol);
            }
        }
        return;
    }

    // consumer warp = kv head
    const int kvh = warp;
    const int g = lane >> 2, tig = lane & 3;
    const int lm = lane >> 3;
    // K (B operand) matrices: (t0-7,c) (t0-7,c+1) (t8-15,c) (t8-15,c+1)
    const int krow = (lm >> 1) * 8 + (lane & 7), kch = lm & 1;
    // Q (A operand) matrices: (r0-7,c) (r8-15,c) (r0-7,c+1) (r8-15,c+1)
    const int qrow = (lm & 1) * 8 + (lane & 7), qch = lm >> 1;
    const uint32_t qt = smem_u32(qs + (size_t)kvh * R * QRS);
    // rows of this lane: (mt, g) and (mt, g+8); row r = 16*mt + g (+8)
    float m_run[MT][2], l_run[MT][2];
    float2 fin[MT][2];  // pass 2: final (max, 1/sum)
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            m_run[mt][hh] = -INFINITY;
            l_run[mt][hh] = 0.f;
            if constexpr (PASS2) {
                const float2 st2 = a.stats[(size_t)s * h_kv * R + kvh * R + 16 * mt + g + 8 * hh];
                fin[mt][hh] = make_float2(st2.x, st2.y > 0.f ? 1.f / st2.y : 0.f);
            }
        }
    const float inv_w = 1.f / (float)a.w;
    for (int p = p0, i = 0; p < p1; ++p, ++i) {
        const int st = i % kWsStages;
        const bool got = mbar_wait_bounded(&full[st], (unsigned)((i / kWsStages) & 1), a.err, &abort_flag, 60);
        int valid = L - p * 16;
        if (valid > 16) valid = 16;
        if (got) {
            const uint32_t kt = smem_u32(ks0 + (size_t)st * stage_bytes) + kvh * D * 2;
            uint32_t kb[KS][4];
#pragma unroll
            for (int t = 0; t < KS; ++t)
                ldsm_x4(kt + krow * KRS + (2 * t + kch) * 16, kb[t][0], kb[t][1], kb[t][2], kb[t][3]);
            float colsum[2][2] = {{0.f, 0.f}, {0.f, 0.f}};  // pass 2: [n-tile][e] sum over u of max over h
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int t = 0; t < KS; ++t) {
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4(qt + (16 * mt + qrow) * QRS + (2 * t + qch) * 16, a0, a1, a2, a3);
                    mma_16816(c0, a0, a1, a2, a3, kb[t][0], kb[t][1]);
                    mma_16816(c1, a0, a1, a2, a3, kb[t][2], kb[t][3]);
                }
                // c0: rows (g, g+8) x tokens (2tig, 2tig+1); c1: tokens (8+2tig, 9+2tig)
                float x[2][4];  // [row half][token]
                x[0][0] = c0[0]; x[0][1] = c0[1]; x[0][2] = c1[0]; x[0][3] = c1[1];
                x[1][0] = c0[2]; x[1][1] = c0[3]; x[1][2] = c1[2]; x[1][3] = c1[3];
                const int tk[4] = {2 * tig, 2 * tig + 1, 8 + 2 * tig, 9 + 2 * tig};
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int r = 16 * mt + g + 8 * hh;
                    const int u = r / G;
                    const int last = L - a.w + u;  // last key this query sees
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int t = p * 16 + tk[e];
                        x[hh][e] = (u < a.w && tk[e] < valid && t <= last) ? x[hh][e] * a.qscale : -INFINITY;
                    }
                }
                if constexpr (!PASS2) {
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        float mx = fmaxf(fmaxf(x[hh][0], x[hh][1]), fmaxf(x[hh][2], x[hh][3]));
                        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
                        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
                        const float mn = fmaxf(m_run[mt][hh], mx);
                        float sum = 0.f;
#pragma unroll
                        for (int e = 0; e < 4; ++e) sum += (x[hh][e] == -INFINITY) ? 0.f : exp2f(x[hh][e] - mn);
                        sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 1);
                        sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 2);
                        l_run[mt][hh] = (mn == -INFINITY) ? 0.f : l_run[mt][hh] * exp2f(m_run[mt][hh] - mn) + sum;
                        m_run[mt][hh] = mn;
                    }
                } else {
                    // P, then the max over the G rows of a window query: rows
                    // r = u*G + j with j in the low bits of g
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            float pv = (x[hh][e] == -INFINITY) ? 0.f : exp2f(x[hh][e] - fin[mt][hh].x) * fin[mt][hh].y;
#pragma unroll
                            for (int o = 4; o < 4 * G && o < 32; o <<= 1)
                                pv = fmaxf(pv, __shfl_xor_sync(0xFFFFFFFFu, pv, o));
                            // one lane per (u) group adds it: rows with j == 0
                            if ((g % G) == 0) colsum[e >> 1][e & 1] += pv;
                        }
                }
            }
            if constexpr (PASS2) {
                // sum over the u's held by different g (lanes with j == 0) and
                // both row halves: add across the g bits above the group bits
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        float v = ((g % G) == 0) ? colsum[nt][e] : 0.f;
                        v += __shfl_xor_sync(0xFFFFFFFFu, v, 4);
                        v += __shfl_xor_sync(0xFFFFFFFFu, v, 8);
                        v += __shfl_xor_sync(0xFFFFFFFFu, v, 16);
                        const int t = nt * 8 + 2 * tig + e;
                        if (g == 0 && t < valid)
                            a.out[((size_t)s * h_kv + kvh) * a.Lmax + p * 16 + t] = v * inv_w;
                    }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
    }
    if constexpr (!PASS2) {
        if (tig == 0) {
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh)
                    a.part[((size_t)s * a.chunks + chunk) * h_kv * R + kvh * R + 16 * mt + g + 8 * hh] =
                        make_float2(m_run[mt][hh], l_run[mt][hh]);
        }
    }
}

// merge of the chunks' (max, sum) per (sequence, row); one thread per row
__global__ void ws_merge_kernel(const WsArgs a, int rows) {
    const int s = blockIdx.y;
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= rows) return;
    const int L = seq_len(a, s);
    const int nchunk = ((L + 15) / 16 + kPages - 1) / kPages;
    float M = -INFINITY, S = 0.f;
    for (int c = 0; c < nchunk; ++c) {
        const float2 ml = a.part[((size_t)s * a.chunks + c) * rows + r];
        if (ml.x == -INFINITY) continue;
        if (ml.x > M) {
            S = S * exp2f(M - ml.x) + ml.y;
            M = ml.x;
        } else {
            S += ml.y * exp2f(ml.x - M);
        }
    }
    a.stats[(size_t)s * rows + r] = make_float2(M, S);
}

// ------------------------------------------------------------------ fp32 path
// (small shapes) pass 1: one block per (sequence, kv head, window row u, q
// head j); pass 2: one thread per (sequence, kv head, token).
__global__ void ws_f32_stats_kernel(const WsArgs a) {
    __shared__ float red[32];
    const int s = blockIdx.z;
    const int kvh = blockIdx.y;
    const int G = a.h_q / a.h_kv;
    const int u = blockIdx.x / G, j = blockIdx.x % G;
    const int L = seq_len(a, s);
    if (L < a.w) return;
    const int last = L - a.w + u;
    const float *qv = static_cast<const float *>(a.q) + (((size_t)s * a.w + u) * a.h_q + kvh * G + j) * a.d;
    const float *K = static_cast<const float *>(a.k);
    float m = -INFINITY;
    for (int t = threadIdx.x; t <= last; t += blockDim.x) {
        const int blk = a.table[(size_t)s * a.table_stride + t / a.b];
        if (blk < 0 || blk >= a.n_total) continue;
        const float *kr = K + (((size_t)blk * a.b + t % a.b) * a.h_kv + kvh) * a.d;
        float dot = 0.f;
        for (int i = 0; i < a.d; ++i) dot = fmaf(qv[i], kr[i], dot);
        m = fmaxf(m, dot * a.qscale);
    }
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    m = -INFINITY;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) m = fmaxf(m, red[i]);
    __syncthreads();
    float sum = 0.f;
    for (int t = threadIdx.x; t <= last; t += blockDim.x) {
        const int blk = a.table[(size_t)s * a.table_stride + t / a.b];
        if (blk < 0 || blk >= a.n_total) continue;
        const float *kr = K + (((size_t)blk * a.b + t % a.b) * a.h_kv + kvh) * a.d;
        float dot = 0.f;
        for (int i = 0; i < a.d; ++i) dot = fmaf(qv[i], kr[i], dot);
        sum += exp2f(dot * a.qscale - m);
    }
    for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = sum;
    __syncthreads();
    if (threadIdx.x == 0) {
        float tot = 0.f;
        for (int i = 0; i < (int)(blockDim.x >> 5); ++i) tot += red[i];
        a.stats[((size_t)s * a.h_kv + kvh) * (a.w * G) + u * G + j] = make_float2(m, tot);
    }
}

__global__ void ws_f32_score_kernel(const WsArgs a) {
    const int s = blockIdx.z;
    const int kvh = blockIdx.y;
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    const int L = seq_len(a, s);
    if (L < a.w || t >= L) return;
    const int G = a.h_q / a.h_kv;
    const int blk = a.table[(size_t)s * a.table_stride + t / a.b];
    if (blk < 0 || blk >= a.n_total) {
        record_error(a.err, ZP_ERR_DEVICE, 0x501);
        return;
    }
    const float *kr = static_cast<const float *>(a.k) + (((size_t)blk * a.b + t % a.b) * a.h_kv + kvh) * a.d;
    float acc = 0.f;
    for (int u = 0; u < a.w; ++u) {
        if (t > L - a.w + u) continue;  // masked: contributes 0
        float best = 0.f;
        for (int j = 0; j < G; ++j) {
            const float *qv = static_cast<const float *>(a.q) + (((size_t)s * a.w + u) * a.h_q + kvh * G + j) * a.d;
            float dot = 0.f;
            for (int i = 0; i < a.d; ++i) dot = fmaf(qv[i], kr[i], dot);
            const float2 ml = a.stats[((size_t)s * a.h_kv + kvh) * (a.w * G) + u * G + j];
            best = fmaxf(best, exp2f(dot * a.qscale - ml.x) / ml.y);
        }
        acc += best;
    }
    a.out[((size_t)s * a.h_kv + kvh) * a.Lmax + t] = acc / (float)a.w;
}

template <int D, int MT, int G>
zp_status launch_ws_tc(const WsArgs &a, cudaStream_t st, const DeviceInfo &dev, size_t smem) {
    auto k1 = ws_tc_kernel<D, MT, G, false>;
    auto k2 = ws_tc_kernel<D, MT, G, true>;
    zp_status rs = set_max_dynamic_smem(reinterpret_cast<const void *>(k1), smem,
                                        "window score: shared-memory attribute");
    if (rs == ZP_OK)
        rs = set_max_dynamic_smem(reinterpret_cast<const void *>(k2), smem, "window score: shared-memory attribute");
    if (rs != ZP_OK) return rs;
    const dim3 grid(a.chunks, a.n);
    const int threads = (a.h_kv + 1) * 32;
    k1<<<grid, threads, smem, st>>>(a);
    const int rows = a.h_kv * MT * 16;
    ws_merge_kernel<<<dim3((rows + 127) / 128, a.n), 128, 0, st>>>(a, rows);
    k2<<<grid, threads, smem, st>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "window score: launch");
    return ZP_OK;
}

}  // namespace
}  // namespace zp

using namespace zp;

extern "C" size_t zp_window_score_workspace_size(const zp_cache_desc *D, int32_t n, int32_t Lmax,
                                                 int32_t window) {
    if (!D || n < 0 || Lmax < 0 || window <= 0 || D->h_kv <= 0) return 0;
    const int G = D->h_q / D->h_kv;
    const size_t rows = (size_t)D->h_kv * ((window * G + 15) / 16) * 16;
    const size_t chunks = ((size_t)(Lmax + 15) / 16 + kPages - 1) / kPages;
    return align_up((size_t)n * chunks * rows * 8, 256) + align_up((size_t)n * rows * 8, 256) + 256;
}

extern "C" zp_status zp_window_score(const zp_cache_desc *D, const void *q_window, int32_t window,
                                     const void *k_cache, const int32_t *block_table, int32_t table_stride,
                                     const int32_t *seq_lens, int32_t n, float *scores_out, int32_t Lmax,
                                     void *workspace, size_t workspace_bytes, void *stream) {
    zp_status rc = check_desc(D);
    if (rc != ZP_OK) return rc;
    if (n < 0 || Lmax < 0 || table_stride < 1 || window < 1)
        return fail(ZP_ERR_INVALID_ARG, "window score: bad sizes (n=%d Lmax=%d window=%d)", n, Lmax, window);
    if (n == 0 || Lmax == 0) return ok();
    if (!q_window || !k_cache || !block_table || !seq_lens || !scores_out || !workspace)
        return fail(ZP_ERR_INVALID_ARG, "window score: NULL buffer");
    const size_t need = zp_window_score_workspace_size(D, n, Lmax, window);
    if (workspace_bytes < need)
        return fail(ZP_ERR_CAPACITY, "window score: workspace %zu < %zu", workspace_bytes, need);
    DeviceInfo dev;
    rc = device_info(&dev);
    if (rc != ZP_OK) return rc;
    const int G = D->h_q / D->h_kv;
    const int d = D->head_dim;
    WsArgs a;
    a.q = q_window;
    a.k = k_cache;
    a.table = block_table;
    a.table_stride = table_stride;
    a.seq_lens = seq_lens;
    a.n = n;
    a.h_q = D->h_q;
    a.h_kv = D->h_kv;
    a.d = d;
    a.b = D->block_size;
    a.n_total = D->n_total_blocks;
    a.w = window;
    a.Lmax = Lmax;
    a.qscale = (float)(1.4426950408889634 / sqrt((double)d));
    a.chunks = (int)(((size_t)(Lmax + 15) / 16 + kPages - 1) / kPages);
    const size_t rows = (size_t)D->h_kv * ((window * G + 15) / 16) * 16;
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    a.part = reinterpret_cast<float2 *>(ws);
    a.stats = reinterpret_cast<float2 *>(ws + align_up((size_t)n * a.chunks * rows * 8, 256));
    a.out = scores_out;
    a.err = dev.error_word;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (D->dtype == ZP_F32) {
        if (d > 256) return fail(ZP_ERR_SHAPE, "window score: head_dim %d", d);
        ws_f32_stats_kernel<<<dim3(window * G, D->h_kv, n), 256, 0, st>>>(a);
        ws_f32_score_kernel<<<dim3((Lmax + 127) / 128, D->h_kv, n), 128, 0, st>>>(a);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e, "window score: launch");
        return ok();
    }
    // bf16: tensor-core passes
    if (D->h_kv > 8) return fail(ZP_ERR_SHAPE, "window score: h_kv %d > 8", D->h_kv);
    if (D->block_size % 16) return fail(ZP_ERR_SHAPE, "window score: block size %d not a multiple of 16", D->block_size);
    if ((window * G) % 16) return fail(ZP_ERR_SHAPE, "window score: window*group %d not a multiple of 16", window * G);
    const int MT = window * G / 16;
    if (((uintptr_t)k_cache | (uintptr_t)q_window) % 16)
        return fail(ZP_ERR_INVALID_ARG, "window score: buffers must be 16-byte aligned");
    const size_t smem = 128 + (size_t)D->h_kv * MT * 16 * (d * 2 + kRowPad) + 128 +
                        (size_t)kWsStages * 16 * (D->h_kv * d * 2 + kRowPad);
    if (smem > (size_t)dev.smem_optin) return fail(ZP_ERR_SHAPE, "window score: needs %zu B of shared memory", smem);
#define ZP_WS(DD, MM, GG)                                               \
    if (d == DD && MT == MM && G == GG) {                               \
        rc = launch_ws_tc<DD, MM, GG>(a, st, dev, smem);                \
        return rc == ZP_OK ? ok() : rc;                                 \
    }
    ZP_WS(128, 4, 4)
    ZP_WS(128, 2, 4)
    ZP_WS(128, 1, 4)
    ZP_WS(128, 8, 8)
    ZP_WS(128, 4, 8)
    ZP_WS(64, 4, 4)
    ZP_WS(64, 2, 4)
    ZP_WS(64, 1, 4)
#undef ZP_WS
    return fail(ZP_ERR_SHAPE, "window score: no kernel for d=%d, window*group/16=%d, group=%d", d, MT, G);
}
