// redundancy.cu -- the all-pairs ("flash") key redundancy of one layer
// [Zipage App. C.5, Fig. 11, Alg. 3], in O(L) memory.
//
// Definition (per sequence and kv head, keys k_0..k_{L-1}): C[r][c] =
// cos(k_r, k_c) with C[c][c] = 0; in every column c the entry of the largest
// row r*(c) with C[r][c] > p is set to zero; rho[r] = sum_c C[r][c].  The
// cosine matrix is symmetric, so r*(c) is the largest index j with
// cos(k_c, k_j) > p (j = c itself counts when 0 > p, and then nothing is
// zeroed), and
//     rho[r] = khat_r . (Shat - khat_r) - sum_{c : r*(c) = r, r != c} cos(k_c, k_r),
// with khat = k / |k| (0 for a zero key) and Shat = sum_c khat_c: the row sums
// are a linear function of the keys, and only the threshold search needs the
// Gram matrix.  Three kernels:
//   prep    1/|k| per token, Shat per (sequence, kv head), candidate words;
//   gram    the threshold search over every pair j > i once (the upper
//           triangle of the Gram matrix): bf16 keys on the tensor cores
//           (tcgen05.mma, accumulators in tensor memory, key tiles by TMA),
//           fp32 keys on the CUDA cores;
//   finish  rho = the row sums minus the zeroed entries.
// The candidate word of token c holds the largest key among j + L for hits
// j > c (c + L for the diagonal when 0 > p) and j for hits j < c, so that one
// atomicMax keeps the largest index above p, and a word >= L names a newer
// token than any word < L.
#include <math.h>

#include "tc05.cuh"

namespace zp {
namespace {

struct ApArgs {
    const void *k;  // paged keys of the layer [N_total][b][h_kv][d]
    const int32_t *table;
    int table_stride;
    const int32_t *seq_lens;
    int n, h_kv, d, b, n_total;
    int Lcap;   // lengths are clamped to this (Lmax, table capacity, score-row stride)
    int Lmax;   // row stride of rho
    int Lpad;   // row stride of inv and cand (a multiple of 128, >= Lmax)
    float p;
    float *inv;   // [n][h_kv][Lpad]
    float *cmax;  // [n][h_kv][Lpad / 32]: the largest 1/|k| of each 32-token chunk
    int *cand;    // [n][h_kv][Lpad]
    float *shat;  // [n][h_kv][d]
    float *rho;   // [n][h_kv][Lmax], zero on entry to the finish
    int *counter; // work-item counter of the tensor-core kernel, zero on entry
    unsigned *err;
};

__device__ __forceinline__ int ap_len(const ApArgs &a, int s) {
    int L = a.seq_lens[s];
    if (L < 0) L = 0;
    if (L > a.Lcap) L = a.Lcap;
    return L;
}

// Block of token t, or -1 (recorded) when the table entry is not a block.
__device__ __forceinline__ int ap_block(const ApArgs &a, int s, int t, unsigned detail) {
    const int blk = a.table[(size_t)s * a.table_stride + t / a.b];
    if (blk < 0 || blk >= a.n_total) {
        record_error(a.err, ZP_ERR_DEVICE, detail);
        return -1;
    }
    return blk;
}

// The D / 32 key elements of lane `lane` of token row `row` (nullptr: zeros).
template <typename T, int D>
__device__ __forceinline__ void load_lane(const T *row, int lane, float (&x)[D / 32]) {
    constexpr int E = D / 32;
    if (!row) {
#pragma unroll
        for (int e = 0; e < E; ++e) x[e] = 0.f;
        return;
    }
    if constexpr (sizeof(T) == 2) {
        const __nv_bfloat16 *r = reinterpret_cast<const __nv_bfloat16 *>(row) + lane * E;
        if constexpr (E == 4) {
            const uint2 w = *reinterpret_cast<const uint2 *>(r);
            const float2 a = bf2_to_f2(w.x), b = bf2_to_f2(w.y);
            x[0] = a.x, x[1] = a.y, x[2] = b.x, x[3] = b.y;
        } else {
            const float2 a = bf2_to_f2(*reinterpret_cast<const uint32_t *>(r));
            x[0] = a.x, x[1] = a.y;
        }
    } else {
        const float *r = reinterpret_cast<const float *>(row) + lane * E;
        if constexpr (E == 4) {
            const float4 w = *reinterpret_cast<const float4 *>(r);
            x[0] = w.x, x[1] = w.y, x[2] = w.z, x[3] = w.w;
        } else {
            const float2 w = *reinterpret_cast<const float2 *>(r);
            x[0] = w.x, x[1] = w.y;
        }
    }
}

template <typename T, int D>
__device__ __forceinline__ const T *ap_row(const ApArgs &a, int s, int h, int t, unsigned detail) {
    const int blk = ap_block(a, s, t, detail);
    if (blk < 0) return nullptr;
    return static_cast<const T *>(a.k) + (((size_t)blk * a.b + t % a.b) * a.h_kv + h) * D;
}

// ------------------------------------------------------------------ prep
// grid (Lpad / 128, h_kv, n), 128 threads: a warp per token row (lanes split
// the head dimension, so each row is one coalesced read).
template <typename T, int D>
__global__ void __launch_bounds__(128) ap_prep_kernel(const ApArgs a) {
    constexpr int E = D / 32;
    __shared__ float part[4][D];
    const int s = blockIdx.z, h = blockIdx.y;
    const int t0 = blockIdx.x * 128;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int L = ap_len(a, s);
    const size_t base = ((size_t)s * a.h_kv + h) * a.Lpad;
    {
        const int t = t0 + threadIdx.x;
        a.cand[base + t] = (t < L && a.p < 0.f) ? t + L : -1;
    }
    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    float chunk_max = 0.f;  // the warp's 32 tokens are one chunk
    for (int r = 0; r < 32; ++r) {
        const int t = t0 + warp * 32 + r;
        if (t >= a.Lpad) break;
        float inv = 0.f;
        if (t < L) {
            float x[E];
            load_lane<T, D>(ap_row<T, D>(a, s, h, t, 0x210), lane, x);
            float ss = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) ss = fmaf(x[e], x[e], ss);
#pragma unroll
            for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
            inv = ss > 0.f ? rsqrtf(ss) : 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) acc[e] = fmaf(x[e], inv, acc[e]);
        }
        if (lane == 0) a.inv[base + t] = inv;
        chunk_max = fmaxf(chunk_max, inv);
    }
    if (lane == 0) a.cmax[base / 32 + (t0 >> 5) + warp] = chunk_max;
#pragma unroll
    for (int e = 0; e < E; ++e) part[warp][lane * E + e] = acc[e];
    __syncthreads();
    if (t0 < L) {
        for (int i = threadIdx.x; i < D; i += blockDim.x) {
            const float v = part[0][i] + part[1][i] + part[2][i] + part[3][i];
            atomicAdd(a.shat + ((size_t)s * a.h_kv + h) * D + i, v);
        }
    }
}

// ------------------------------------------------------------------ finish
// grid (ceil(Lmax / 128), h_kv, n), 128 threads, a warp per token row c:
// rho[c] += khat_c . (Shat - khat_c); rho[r*(c)] -= cos(k_c, k_r*) when the
// candidate word names another token.
template <typename T, int D>
__global__ void __launch_bounds__(128) ap_finish_kernel(const ApArgs a) {
    constexpr int E = D / 32;
    const int s = blockIdx.z, h = blockIdx.y;
    const int t0 = blockIdx.x * 128;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int L = ap_len(a, s);
    if (t0 >= L) return;
    const size_t base = ((size_t)s * a.h_kv + h) * a.Lpad;
    float *rho = a.rho + ((size_t)s * a.h_kv + h) * a.Lmax;
    float sh[E];
#pragma unroll
    for (int e = 0; e < E; ++e) sh[e] = a.shat[((size_t)s * a.h_kv + h) * D + lane * E + e];
    for (int r = 0; r < 32; ++r) {
        const int c = t0 + warp * 32 + r;
        if (c >= L) break;
        float x[E];
        load_lane<T, D>(ap_row<T, D>(a, s, h, c, 0x211), lane, x);
        const float ic = a.inv[base + c];
        float part = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const float kh = x[e] * ic;
            part = fmaf(kh, sh[e] - kh, part);
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) part += __shfl_xor_sync(0xFFFFFFFFu, part, o);
        if (lane == 0) atomicAdd(rho + c, part);
        const int key = a.cand[base + c];
        const int rs = key >= L ? key - L : key;
        if (rs >= 0 && rs != c && rs < L) {
            float y[E];
            load_lane<T, D>(ap_row<T, D>(a, s, h, rs, 0x212), lane, y);
            float dot = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) dot = fmaf(x[e], y[e], dot);
#pragma unroll
            for (int o = 16; o; o >>= 1) dot += __shfl_xor_sync(0xFFFFFFFFu, dot, o);
            if (lane == 0) atomicAdd(rho + rs, -(dot * ic * a.inv[base + rs]));
        }
    }
}

// ------------------------------------------------------------------ gram, fp32 keys
// grid (ceil(Lmax / 128), h_kv, n), 128 threads: thread i owns row i (its key
// in registers) and scans every other column (the whole matrix: the row's own
// hits decide its candidate word alone).  Column tiles of 32 keys are staged
// in shared memory and read by all threads at once (broadcast).
template <int D>
__global__ void __launch_bounds__(128) ap_gram_f32_kernel(const ApArgs a) {
    __shared__ float colk[32][D];
    __shared__ float colinv[32];
    const int s = blockIdx.z, h = blockIdx.y;
    const int t0 = blockIdx.x * 128;
    const int L = ap_len(a, s);
    if (t0 >= L) return;
    const size_t base = ((size_t)s * a.h_kv + h) * a.Lpad;
    const int i = t0 + threadIdx.x;
    const bool valid = i < L;
    float r[D];
    {
        const float *row = valid ? ap_row<float, D>(a, s, h, i, 0x213) : nullptr;
#pragma unroll
        for (int e = 0; e < D; e += 4) {
            const float4 w = row ? *reinterpret_cast<const float4 *>(row + e) : make_float4(0.f, 0.f, 0.f, 0.f);
            r[e] = w.x, r[e + 1] = w.y, r[e + 2] = w.z, r[e + 3] = w.w;
        }
    }
    const float inv_i = valid ? a.inv[base + i] : 0.f;
    const float thr = inv_i > 0.f ? a.p / inv_i : (a.p < 0.f ? -INFINITY : INFINITY);
    int best = -1;
    for (int j0 = 0; j0 < L; j0 += 32) {
        __syncthreads();
        for (int q = threadIdx.x; q < 32 * (D / 4); q += blockDim.x) {
            const int jj = q / (D / 4), e = (q % (D / 4)) * 4;
            const int j = j0 + jj;
            float4 w = make_float4(0.f, 0.f, 0.f, 0.f);
            if (j < L) {
                const float *row = ap_row<float, D>(a, s, h, j, 0x214);
                if (row) w = *reinterpret_cast<const float4 *>(row + e);
            }
            *reinterpret_cast<float4 *>(&colk[jj][e]) = w;
        }
        if (threadIdx.x < 32) colinv[threadIdx.x] = j0 + threadIdx.x < L ? a.inv[base + j0 + threadIdx.x] : 0.f;
        __syncthreads();
        if (!valid) continue;
        for (int jj = 0; jj < 32; ++jj) {
            const int j = j0 + jj;
            if (j >= L) break;
            float dot = 0.f;
#pragma unroll
            for (int e = 0; e < D; ++e) dot = fmaf(r[e], colk[jj][e], dot);
            if (j != i && fmaf(dot, colinv[jj], -thr) > 0.f) {
                const int key = j > i ? j + L : j;
                best = key > best ? key : best;
            }
        }
    }
    if (valid && best >= 0) atomicMax(a.cand + base + i, best);
}

// ------------------------------------------------------------------ gram, bf16 keys on tcgen05
// Persistent kernel, one CTA per SM (all 512 TMEM columns, ~193 KB of shared
// memory).  A work item is (sequence, kv head, row super-tile of ROWS = RT*128
// tokens, up to kItemCols columns starting at or after the super-tile's first
// row); items are taken from a grid-wide counter (one atomic per item by the
// producer, handed to the other roles through a small ring in shared memory),
// in (sequence, kv head)-major order so that the CTAs at work share the keys
// of one head in L2, and the small items come last.  The rows' keys stay in
// shared memory (A) while the columns' keys stream through a ring of
// kStages tiles of N = 256/RT keys (B).  For each column tile one thread
// issues RT x (D/16) MMAs of M = 128, N, K = 16 into one of two accumulator
// buffers (RT*N = 256 TMEM columns each); eight epilogue warps read the other
// buffer.  Row i hits column j when acc_ij * (1/|k_j|) > p*|k_i| (> 0 for
// p > 0); since 1/|k_j| <= the chunk's largest, a 32-column chunk whose
// largest acc times that bound stays at or below p*|k_i| has no hit -- nearly
// every chunk -- so the common path is one three-way max per two elements.
// Chunks that may hold a hit, chunks on the diagonal or past L, and rows with
// p*|k_i| <= 0 take the exact path: per column the hit mask of the warp's 32
// rows (ballot) gives the column's largest row i < j (atomicMax into j's
// word), and each row keeps its largest column j > i (one atomicMax per item).
constexpr int kApStages = 4;
constexpr int kItemCols = 8192;
constexpr int kEpiWarps = 8;
constexpr int kApThreads = 32 * (2 + kEpiWarps);
constexpr int kItemRing = 4;

template <int D, int RT>
struct GramCfg {
    static constexpr int N = 256 / RT;               // columns per tile (MMA N)
    static constexpr int KH = D / 64;                // 128-byte halves of a key row
    static constexpr int KS = D / 16;                // MMA K steps
    static constexpr int ROWS = RT * 128;            // rows per work item
    static constexpr int A_HALF = ROWS * 128;        // bytes of one half of A
    static constexpr int A_BYTES = KH * A_HALF;
    static constexpr int B_HALF = N * 128;
    static constexpr int STAGE = KH * B_HALF;
    static constexpr int BAR_OFF = A_BYTES + kApStages * STAGE;
    static constexpr int BLK_OFF = BAR_OFF + 512;     // block rows of the current item
    static constexpr int NBLK = ROWS / 16 + kItemCols / 16;
    static constexpr int SMEM = BLK_OFF + NBLK * 4 + 1024;  // + alignment slack
    static constexpr uint32_t IDESC = idesc_bf16_f32(128, N);
};

// Work item g of the grid-wide list: (s, h) major, then super-tiles, then
// column chunks, for the largest length Lmax (items past a sequence's own
// length are empty).
template <int ROWS>
__device__ __forceinline__ bool ap_item(const ApArgs &a, int g, int items_per_sh, int &s, int &h, int &r0, int &c0,
                                        int &c1, int &L) {
    const int sh = g / items_per_sh;
    int loc = g - sh * items_per_sh;
    s = sh / a.h_kv;
    h = sh - s * a.h_kv;
    int P = 0;
    while (true) {
        const int nc = (a.Lmax - P * ROWS + kItemCols - 1) / kItemCols;
        if (loc < nc) break;
        loc -= nc;
        ++P;
    }
    r0 = P * ROWS;
    c0 = r0 + loc * kItemCols;
    L = ap_len(a, s);
    c1 = min(L, c0 + kItemCols);
    return c0 < L;
}

__device__ __forceinline__ float max3f(float x, float y, float z) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(x), "f"(y), "f"(z));
    return r;
}

// Exact test of one 32-column chunk (v: raw products, columns j0..j0+31) for
// the warp's rows (see the kernel).
__device__ __forceinline__ void ap_chunk_exact(const uint32_t *v, const float *inv_row, int i, bool valid,
                                               float nthr, int j0, int L, int rowbase, int *best, int *cand_row,
                                               int lane) {
    float ic[32];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const float4 w = *reinterpret_cast<const float4 *>(inv_row + j0 + 4 * u);
        ic[4 * u] = w.x, ic[4 * u + 1] = w.y, ic[4 * u + 2] = w.z, ic[4 * u + 3] = w.w;
    }
#pragma unroll
    for (int jj = 0; jj < 32; ++jj) {
        const int j = j0 + jj;
        const float y = fmaf(__uint_as_float(v[jj]), ic[jj], nthr);
        const bool hit = valid && j < L && j > i && y > 0.f;
        if (hit) *best = j;
        const unsigned bal = __ballot_sync(0xFFFFFFFFu, hit);
        if (lane == 0 && bal) atomicMax(cand_row + j, rowbase + 31 - __clz(bal));
    }
}

template <int D, int RT>
__global__ void __launch_bounds__(kApThreads, 1)
    ap_gram_tc_kernel(const __grid_constant__ CUtensorMap tmap, const ApArgs a, int items_per_sh, int n_items) {
    using C = GramCfg<D, RT>;
    constexpr int N = C::N;
    static_assert(N % 32 == 0, "tiles are whole 32-column chunks");
    extern __shared__ unsigned char ap_smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(ap_smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    unsigned char *As = smem;
    unsigned char *Bs = smem + C::A_BYTES;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::BAR_OFF);
    uint64_t *empty = full + kApStages;
    uint64_t *a_full = empty + kApStages;
    uint64_t *a_empty = a_full + 1;
    uint64_t *acc_full = a_empty + 1;    // [2]
    uint64_t *acc_empty = acc_full + 2;  // [2]
    uint64_t *item_full = acc_empty + 2; // [kItemRing]
    uint64_t *item_empty = item_full + kItemRing;
    uint64_t *drain = item_empty + kItemRing;
    int *item_slot = reinterpret_cast<int *>(drain + 1);  // [kItemRing]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(item_slot + kItemRing);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *zrow = reinterpret_cast<int *>(smem + C::BLK_OFF);  // TMA row of each 16-token group, -16 = zeros
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kApStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        mbar_init(a_full, 1);
        mbar_init(a_empty, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_empty[i], kEpiWarps);
        }
        for (int i = 0; i < kItemRing; ++i) {
            mbar_init(&item_full[i], 1);
            mbar_init(&item_empty[i], 1 + kEpiWarps);  // the MMA thread and every epilogue warp
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---------------- producer: takes the items, TMA loads of A and of the B tiles.
        // The whole warp looks up the item's block ids (one table read per 16
        // tokens) into shared memory first; lane 0 then issues the copies.
        uint32_t fill = 0, item = 0, item_armed = 0;
        if (lane == 0) prefetch_tensormap(&tmap);
        for (uint32_t k = 0;; ++k) {
            const uint32_t slot = k % kItemRing;
            int g = -1;
            if (lane == 0) {
                if (!*abort_flag &&
                    mbar_wait_bounded(&item_empty[slot], ((k / kItemRing) & 1) ^ 1, a.err, abort_flag, 0x22B)) {
                    g = atomicAdd(a.counter, 1);
                    item_slot[slot] = g < n_items ? g : -1;
                    mbar_arrive(&item_full[slot]);  // releases the slot's value to the other roles
                    if (g >= n_items) g = -1;
                } else {
                    g = -2;  // aborted: nothing published
                }
            }
            g = __shfl_sync(0xFFFFFFFFu, g, 0);
            if (g < 0) break;
            int s, h, r0, c0, c1, L;
            if (!ap_item<C::ROWS>(a, g, items_per_sh, s, h, r0, c0, c1, L)) continue;
            const int nrow = C::ROWS / 16, ncol = (c1 - c0 + 15) / 16;
            __syncwarp();  // lane 0 is done with the previous item's rows
            for (int G = lane; G < nrow + ncol; G += 32) {
                const int t = G < nrow ? r0 + 16 * G : c0 + 16 * (G - nrow);
                int z = -16;  // past the sequence: a box of zeros
                if (t < L) {
                    const int blk = ap_block(a, s, t, G < nrow ? 0x221 : 0x223);
                    if (blk >= 0) z = blk * a.b + t % a.b;
                }
                zrow[G] = z;
            }
            __syncwarp();
            if (lane != 0) continue;
            // a wait that gives up sets the abort flag: lane 0 goes back to the
            // top, where the other lanes learn it from the broadcast
            if (!mbar_wait_bounded(a_empty, (item & 1) ^ 1, a.err, abort_flag, 0x220)) continue;
            mbar_arrive_expect_tx(a_full, C::A_BYTES);
            item_armed = item + 1;
            for (int G = 0; G < nrow; ++G) {
#pragma unroll
                for (int kh = 0; kh < C::KH; ++kh)
                    tma_load_3d(As + kh * C::A_HALF + G * 2048, &tmap, kh * 64, h, zrow[G], a_full);
            }
            const int ntiles = (c1 - c0 + N - 1) / N;
            for (int j = 0; j < ntiles; ++j) {
                const uint32_t st = fill % kApStages;
                if (!mbar_wait_bounded(&empty[st], ((fill / kApStages) & 1) ^ 1, a.err, abort_flag, 0x222)) break;
                mbar_arrive_expect_tx(&full[st], C::STAGE);
                ++fill;
                unsigned char *dst = Bs + st * C::STAGE;
#pragma unroll
                for (int G = 0; G < N / 16; ++G) {
                    const int gi = nrow + j * (N / 16) + G;
                    const int z = gi < nrow + ncol ? zrow[gi] : -16;
#pragma unroll
                    for (int kh = 0; kh < C::KH; ++kh)
                        tma_load_3d(dst + kh * C::B_HALF + G * 2048, &tmap, kh * 64, h, z, &full[st]);
                }
            }
            ++item;
        }
        if (lane == 0 && *abort_flag) {
            // let the loads already armed land before the CTA releases its
            // shared memory: the newest armed phase of each stage and of A
            volatile int never = 0;
            for (uint32_t f = fill > kApStages ? fill - kApStages : 0; f < fill; ++f)
                mbar_wait_bounded(&full[f % kApStages], (f / kApStages) & 1, a.err, &never, 0x229);
            if (item_armed > item) mbar_wait_bounded(a_full, item & 1, a.err, &never, 0x22A);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer
        if (lane == 0) {
            uint32_t fill = 0, tile = 0, item = 0;
            const uint32_t a_addr = smem_u32(As), b_addr = smem_u32(Bs);
            for (uint32_t k = 0; !*abort_flag; ++k) {
                const uint32_t slot = k % kItemRing;
                if (!mbar_wait_bounded(&item_full[slot], (k / kItemRing) & 1, a.err, abort_flag, 0x22C)) break;
                const int g = item_slot[slot];
                mbar_arrive(&item_empty[slot]);
                if (g < 0) break;
                int s, h, r0, c0, c1, L;
                if (!ap_item<C::ROWS>(a, g, items_per_sh, s, h, r0, c0, c1, L)) continue;
                if (!mbar_wait_bounded(a_full, item & 1, a.err, abort_flag, 0x224)) break;
                tc_fence_after();
                const int ntiles = (c1 - c0 + N - 1) / N;
                bool ok_item = true;
                for (int j = 0; j < ntiles; ++j, ++fill, ++tile) {
                    const uint32_t st = fill % kApStages, ab = tile & 1;
                    if (!mbar_wait_bounded(&full[st], (fill / kApStages) & 1, a.err, abort_flag, 0x225) ||
                        !mbar_wait_bounded(&acc_empty[ab], ((tile >> 1) & 1) ^ 1, a.err, abort_flag, 0x226)) {
                        ok_item = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int rt = 0; rt < RT; ++rt) {
                        const uint32_t d_tmem = tmem + ab * 256 + rt * N;
#pragma unroll
                        for (int ks = 0; ks < C::KS; ++ks) {
                            const uint32_t ao = (ks >> 2) * C::A_HALF + rt * 128 * 128 + (ks & 3) * 32;
                            const uint32_t bo = st * C::STAGE + (ks >> 2) * C::B_HALF + (ks & 3) * 32;
                            tc_mma_bf16(d_tmem, sdesc_k_sw128(a_addr + ao), sdesc_k_sw128(b_addr + bo), C::IDESC,
                                        ks > 0 ? 1u : 0u);
                        }
                    }
                    tc_commit(&empty[st]);
                    tc_commit(&acc_full[ab]);
                }
                if (!ok_item) break;
                tc_commit(a_empty);
                ++item;
            }
        }
    } else {
        // ---------------- epilogue: eight warps, two per TMEM lane quarter
        const int e = warp - 2;
        const int q = warp & 3;      // TMEM lanes 32q..32q+31 (fixed by the warp's position)
        const int half = e >> 2;     // row tiles half, half + 2, ...
        uint32_t tile = 0;
        for (uint32_t k = 0; !*abort_flag; ++k) {
            const uint32_t slot = k % kItemRing;
            if (!mbar_wait_bounded(&item_full[slot], (k / kItemRing) & 1, a.err, abort_flag, 0x22D)) break;
            const int g = item_slot[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive(&item_empty[slot]);
            if (g < 0) break;
            int s, h, r0, c0, c1, L;
            if (!ap_item<C::ROWS>(a, g, items_per_sh, s, h, r0, c0, c1, L)) continue;
            const size_t base = ((size_t)s * a.h_kv + h) * a.Lpad;
            const float *inv_row = a.inv + base;
            const float *cmax_row = a.cmax + base / 32;
            int *cand_row = a.cand + base;
            constexpr int M = RT / 2;  // rows per thread
            int rowi[M], best[M];
            bool valid[M];
            float thr[M];
#pragma unroll
            for (int m = 0; m < M; ++m) {
                rowi[m] = r0 + (half + 2 * m) * 128 + 32 * q + lane;
                valid[m] = rowi[m] < L;
                const float iv = valid[m] ? inv_row[rowi[m]] : 0.f;
                thr[m] = iv > 0.f ? a.p / iv : (a.p < 0.f ? -INFINITY : INFINITY);
                best[m] = -1;
            }
            const int ntiles = (c1 - c0 + N - 1) / N;
            bool ok_item = true;
            for (int j = 0; j < ntiles; ++j, ++tile) {
                const uint32_t ab = tile & 1;
                const int cb = c0 + j * N;
                float cm[N / 32];  // chunk bounds of 1/|k_j|, fetched before the wait
#pragma unroll
                for (int ch = 0; ch < N / 32; ++ch) cm[ch] = cmax_row[(cb >> 5) + ch];
                if (!mbar_wait_bounded(&acc_full[ab], (tile >> 1) & 1, a.err, abort_flag, 0x227)) {
                    ok_item = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int m = 0; m < M; ++m) {
                    const int rt = half + 2 * m;
                    const int rowbase = r0 + rt * 128 + 32 * q;
#pragma unroll
                    for (int c2 = 0; c2 < N / 64; ++c2) {
                        uint32_t v[64];
                        tmem_ld64(tmem + ((uint32_t)(32 * q) << 16) + ab * 256 + rt * N + c2 * 64, v);
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            const int ch = c2 * 2 + hh;
                            const int j0 = cb + ch * 32;
                            const uint32_t *vc = v + hh * 32;
                            bool exact = !(j0 > rowbase + 31 && j0 + 31 < L && rowbase + 31 < L);
                            if (!exact) {
                                float mx = __uint_as_float(vc[0]);
#pragma unroll
                                for (int jj = 1; jj < 31; jj += 2)
                                    mx = max3f(mx, __uint_as_float(vc[jj]), __uint_as_float(vc[jj + 1]));
                                mx = fmaxf(mx, __uint_as_float(vc[31]));
                                // no hit possible iff thr > 0 and mx * bound <= thr
                                const bool maybe = !(thr[m] > 0.f) || fmaf(mx, cm[ch], -thr[m]) > 0.f;
                                exact = __any_sync(0xFFFFFFFFu, maybe);
                            }
                            if (exact)
                                ap_chunk_exact(vc, inv_row, rowi[m], valid[m], -thr[m], j0, L, rowbase, &best[m],
                                               cand_row, lane);
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acc_empty[ab]);
            }
#pragma unroll
            for (int m = 0; m < M; ++m)
                if (valid[m] && best[m] >= 0) atomicMax(cand_row + rowi[m], best[m] + L);
            if (!ok_item) break;
        }
    }

    // ---------------- teardown: after a timeout, let the products in flight
    // land before the tensor memory is released
    __syncthreads();
    if (*abort_flag && threadIdx.x == 32) {
        volatile int never = 0;
        tc_commit(drain);
        mbar_wait_bounded(drain, 0, a.err, &never, 0x228);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

// ------------------------------------------------------------------ host
// The layer's keys as a 3-D tensor (element of the head, kv head, token row);
// a box is 64 elements of one kv head for 16 tokens.
zp_status encode_key_map(CUtensorMap *map, const void *k, int d, int h_kv, int b, int n_total) {
    const uint64_t dims[3] = {(uint64_t)d, (uint64_t)h_kv, (uint64_t)n_total * (uint64_t)b};
    const uint64_t strides[2] = {(uint64_t)d * 2, (uint64_t)h_kv * d * 2};
    const uint32_t box[3] = {64, 1, 16};
    return encode_tmap_bf16_3d(map, k, dims, strides, box, "all-pairs redundancy");
}

template <int D, int RT>
zp_status launch_gram_tc(const ApArgs &a, const DeviceInfo &dev, cudaStream_t st) {
    using C = GramCfg<D, RT>;
    CUtensorMap map;
    zp_status rc = encode_key_map(&map, a.k, D, a.h_kv, a.b, a.n_total);
    if (rc != ZP_OK) return rc;
    if ((size_t)C::SMEM > (size_t)dev.smem_optin)
        return fail(ZP_ERR_SHAPE, "all-pairs redundancy: needs %d B of shared memory", C::SMEM);
    rc = set_max_dynamic_smem(reinterpret_cast<const void *>(ap_gram_tc_kernel<D, RT>), C::SMEM,
                              "all-pairs redundancy: shared-memory attribute");
    if (rc != ZP_OK) return rc;
    int items_per_sh = 0;
    for (int P = 0; P * C::ROWS < a.Lmax; ++P) items_per_sh += (a.Lmax - P * C::ROWS + kItemCols - 1) / kItemCols;
    const long long n_items = (long long)a.n * a.h_kv * items_per_sh;
    if (n_items <= 0) return ZP_OK;
    if (n_items > 0x7FFFFFFF) return fail(ZP_ERR_SHAPE, "all-pairs redundancy: too many work items");
    const int grid = (int)(n_items < dev.sm_count ? n_items : dev.sm_count);
    ap_gram_tc_kernel<D, RT><<<grid, kApThreads, C::SMEM, st>>>(map, a, items_per_sh, (int)n_items);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "all-pairs redundancy: tensor-core kernel launch");
    return ZP_OK;
}

template <typename T, int D>
zp_status launch_typed(const ApArgs &a, const DeviceInfo &dev, cudaStream_t st) {
    cudaError_t e = cudaMemsetAsync(a.shat, 0, (size_t)a.n * a.h_kv * D * 4, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(a.counter, 0, 4, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(a.rho, 0, (size_t)a.n * a.h_kv * a.Lmax * 4, st);
    if (e != cudaSuccess) return cuda_fail(e, "all-pairs redundancy: clearing the sums");
    ap_prep_kernel<T, D><<<dim3(a.Lpad / 128, a.h_kv, a.n), 128, 0, st>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "all-pairs redundancy: prep launch");
    zp_status rc = ZP_OK;
    if constexpr (sizeof(T) == 2) {
        rc = launch_gram_tc<D, 2>(a, dev, st);  // two 128-row tiles, N = 128 (measured best)
    } else {
        ap_gram_f32_kernel<D><<<dim3((a.Lmax + 127) / 128, a.h_kv, a.n), 128, 0, st>>>(a);
        e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e, "all-pairs redundancy: fp32 kernel launch");
    }
    if (rc != ZP_OK) return rc;
    ap_finish_kernel<T, D><<<dim3((a.Lmax + 127) / 128, a.h_kv, a.n), 128, 0, st>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "all-pairs redundancy: finish launch");
    return ZP_OK;
}

}  // namespace

size_t all_pairs_workspace_size(int n, int h_kv, int d, int Lmax) {
    const size_t Lpad = align_up((size_t)(Lmax > 0 ? Lmax : 1), 128);
    return 2 * align_up((size_t)n * h_kv * Lpad * 4, 256) + align_up((size_t)n * h_kv * d * 4, 256) +
           align_up((size_t)n * h_kv * (Lpad / 32) * 4, 256) + 256;
}

zp_status launch_all_pairs(const AllPairsArgs &in, cudaStream_t st) {
    if (!(in.d == 64 || in.d == 128)) return fail(ZP_ERR_SHAPE, "all-pairs redundancy: head_dim %d", in.d);
    if (in.dtype == ZP_BF16 && in.b % 16)
        return fail(ZP_ERR_SHAPE, "all-pairs redundancy: bf16 keys need a block size multiple of 16 (b=%d)", in.b);
    if (reinterpret_cast<uintptr_t>(in.k) % 16) return fail(ZP_ERR_INVALID_ARG, "all-pairs redundancy: keys unaligned");
    DeviceInfo dev;
    zp_status rc = device_info(&dev);
    if (rc != ZP_OK) return rc;
    ApArgs a;
    a.k = in.k;
    a.table = in.table;
    a.table_stride = in.table_stride;
    a.seq_lens = in.seq_lens;
    a.n = in.n;
    a.h_kv = in.h_kv;
    a.d = in.d;
    a.b = in.b;
    a.n_total = in.n_total;
    a.Lmax = in.Lmax;
    a.Lcap = in.Lcap;
    a.Lpad = (int)align_up((size_t)in.Lmax, 128);
    a.p = in.p;
    unsigned char *ws = static_cast<unsigned char *>(in.workspace);
    const size_t arr = align_up((size_t)in.n * in.h_kv * a.Lpad * 4, 256);
    a.inv = reinterpret_cast<float *>(ws);
    a.cand = reinterpret_cast<int *>(ws + arr);
    a.shat = reinterpret_cast<float *>(ws + 2 * arr);
    const size_t sh_bytes = align_up((size_t)in.n * in.h_kv * in.d * 4, 256);
    a.cmax = reinterpret_cast<float *>(ws + 2 * arr + sh_bytes);
    a.counter = reinterpret_cast<int *>(ws + 2 * arr + sh_bytes + align_up((size_t)in.n * in.h_kv * (a.Lpad / 32) * 4, 256));
    a.rho = in.rho;
    a.err = dev.error_word;
    if (in.n == 0 || in.Lmax == 0) return ZP_OK;
    if (in.dtype == ZP_BF16) {
        if (in.d == 128) return launch_typed<__nv_bfloat16, 128>(a, dev, st);
        return launch_typed<__nv_bfloat16, 64>(a, dev, st);
    }
    if (in.d == 128) return launch_typed<float, 128>(a, dev, st);
    return launch_typed<float, 64>(a, dev, st);
}

}  // namespace zp
