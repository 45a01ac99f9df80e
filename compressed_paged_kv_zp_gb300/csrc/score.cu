// score.cu -- per-token eviction scores of the sequences being compressed.
//
// Zipage paper App. C.2-C.8 and §4.2, in the order of the paper's per-op
// timing figure (Figs. 13/14): attention score -> global score -> pooling ->
// redundancy score -> window mask.  Three launches:
//   1. gather_global: the attention score S of each (sequence, kv head) is
//      read from its score row and, if enabled, run through Alg. 2 against
//      the paged global score cache F (read only).  The global score goes
//      back into the score row (the compaction stores it into F of the kept
//      tokens) and to X [n][h_kv][Lmax].
//   2. lightning: one CTA per (sequence, block): the block's keys of every kv
//      head are staged in shared memory, each warp forms the b x b cosine
//      matrix of one kv head, zeroes the diagonal and, per column, the newest
//      entry above the threshold p (C.5, restricted to the block as in C.7),
//      and writes the row sums rho [n][h_kv][Lmax].
//   3. finalize: one CTA per (sequence, kv head): max-pool X (C.4) when the
//      policy says so, R = softmax(rho / (L * tau)) (C.5, C.8), out = Xp -
//      lambda * R (eq. 4), last w tokens -> +inf (§4.2, App. C.6).
#include <math.h>

#include "zp_common.cuh"

namespace zp {
namespace {

constexpr int kTile = 64;  // tokens per gather tile

struct ScoreArgs {
    const int32_t *table;
    int table_stride;
    const int32_t *seq_lens;
    const uint8_t *first;
    int n, h_kv, b, n_total, Lmax, d;
    float *S;               // score rows: S + (row * h_kv + kvh) * S_stride + t
    long long S_stride;
    const int32_t *S_rows;  // nullable: row of sequence i
    const float *F;         // paged [N_total][b][h_kv], nullable
    float *X;         // [n][h_kv][Lmax]
    float *rho;       // [n][h_kv][Lmax]
    float *out;       // [n][h_kv][Lmax]
    const void *k;    // paged keys of this layer
    int use_global;
    float alpha;
    int pool_kernel, pool_policy;
    int use_sim;
    float p, lambda, tau;
    int window;
    unsigned *err;
};

__device__ __forceinline__ int clamp_len(const ScoreArgs &a, int s) {
    int L = a.seq_lens[s];
    if (L < 0) L = 0;
    if (L > a.Lmax) L = a.Lmax;
    if (L > a.table_stride * a.b) L = a.table_stride * a.b;
    if (L > a.S_stride) L = (int)a.S_stride;
    return L;
}

// grid (ceil(Lmax / kTile), n), 256 threads.  Phase 1 stages the tile's F
// values (paged, (slot, kv head) fastest) in shared memory when Alg. 2 reads
// them; phase 2 walks (kv head, token) so the score rows are read and written
// along tokens.
__global__ void gather_global_kernel(const ScoreArgs a) {
    __shared__ float tile[16][kTile + 1];  // h_kv <= 16
    const int s = blockIdx.y;
    const int t0 = blockIdx.x * kTile;
    const int L = clamp_len(a, s);
    if (t0 >= L) return;
    const int N = (L + a.b - 1) / a.b;
    const bool first = a.first ? a.first[s] != 0 : true;
    const bool read_F = a.use_global && !first;
    const int items = kTile * a.h_kv;
    const int row = a.S_rows ? a.S_rows[s] : s;
    if (row < 0) {
        if (threadIdx.x == 0) record_error(a.err, ZP_ERR_DEVICE, 0x202);
        return;
    }
    if (read_F) {
        for (int it = threadIdx.x; it < items; it += blockDim.x) {
            const int tl = it / a.h_kv;
            const int kvh = it % a.h_kv;
            const int t = t0 + tl;
            float f = 0.f;
            if (t < L && t / a.b != N - 1) {
                const int blk = a.table[(size_t)s * a.table_stride + t / a.b];
                if (blk < 0 || blk >= a.n_total)
                    record_error(a.err, ZP_ERR_DEVICE, 0x200);
                else
                    f = a.F[((size_t)blk * a.b + t % a.b) * a.h_kv + kvh];
            }
            tile[kvh][tl] = f;
        }
        __syncthreads();
    }
    for (int it = threadIdx.x; it < items; it += blockDim.x) {
        const int kvh = it / kTile;
        const int tl = it % kTile;
        const int t = t0 + tl;
        if (t >= L) continue;
        float *sp = a.S + ((size_t)row * a.h_kv + kvh) * a.S_stride + t;
        float v = *sp;
        if (read_F && t / a.b != N - 1) {
            v = fmaxf(a.alpha * tile[kvh][tl], v);
            *sp = v;
        }
        a.X[((size_t)s * a.h_kv + kvh) * a.Lmax + t] = v;
    }
}

// grid (ceil(Lmax / b), n), h_kv warps; dynamic smem: h_kv * b * (d + 1) floats
// + b * h_kv norms.  Keys are converted to fp32 once; the padded row stride
// (d + 1) keeps the 16 lanes that read 16 different rows on 16 banks.
template <typename T>
__global__ void lightning_kernel(const ScoreArgs a) {
    extern __shared__ float kf[];
    const int s = blockIdx.y;
    const int bi = blockIdx.x;
    const int L = clamp_len(a, s);
    const int tb0 = bi * a.b;
    if (tb0 >= L) return;
    const int nvalid = min(a.b, L - tb0);
    const int blk = a.table[(size_t)s * a.table_stride + bi];
    if (blk < 0 || blk >= a.n_total) {
        if (threadIdx.x == 0) record_error(a.err, ZP_ERR_DEVICE, 0x201);
        return;
    }
    const int d = a.d;
    const int ld = d + 1;
    const T *src = static_cast<const T *>(a.k) + (size_t)blk * a.b * a.h_kv * d;
    const int total = nvalid * a.h_kv * d;
    for (int i = threadIdx.x; i < total; i += blockDim.x) {
        const int r = i / (a.h_kv * d);
        const int rem = i % (a.h_kv * d);
        const int kvh = rem / d;
        const int dd = rem % d;
        float x;
        if constexpr (sizeof(T) == 2) x = __bfloat162float(src[i]);
        else x = src[i];
        kf[((size_t)kvh * a.b + r) * ld + dd] = x;
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int kvh = warp;
    if (kvh >= a.h_kv) return;
    const float *kh = kf + (size_t)kvh * a.b * ld;
    // one warp per kv head; b <= 32 rows; lane = (row r, column half)
    // Rows/columns beyond nvalid are outside the sequence and excluded.
    const int b = a.b;
    for (int rbase = 0; rbase < b; rbase += 16) {
        const int r = rbase + (lane & 15);
        const int chalf = lane >> 4;
        // columns c = cb*16 + chalf*8 + j, processed 8 at a time
        float rowsum = 0.f;
        const float nr2 = [&] {
            float acc = 0.f;
            if (r < nvalid)
                for (int dd = 0; dd < d; ++dd) acc = fmaf(kh[r * ld + dd], kh[r * ld + dd], acc);
            return acc;
        }();
        const float nr = sqrtf(nr2);
        for (int cb = 0; cb < b; cb += 16) {
            float dot[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) dot[j] = 0.f;
            const int c0 = cb + chalf * 8;
            if (r < nvalid) {
                for (int dd = 0; dd < d; ++dd) {
                    const float x = kh[r * ld + dd];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int c = c0 + j;
                        if (c < nvalid) dot[j] = fmaf(x, kh[c * ld + dd], dot[j]);
                    }
                }
            }
            // cosine, diagonal, threshold: for column c the newest row r* with
            // cos > p is zeroed.  Rows of this column live in lanes with the
            // same chalf across the 16-row groups; with b <= 16 one group.
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int c = c0 + j;
                float cosv = 0.f;
                if (r < nvalid && c < nvalid && r != c) {
                    float nc2 = 0.f;
                    for (int dd = 0; dd < d; ++dd) nc2 = fmaf(kh[c * ld + dd], kh[c * ld + dd], nc2);
                    const float nc = sqrtf(nc2);
                    if (nr > 0.f && nc > 0.f) cosv = dot[j] / (nr * nc);
                }
                const unsigned above = __ballot_sync(0xFFFFFFFFu, cosv > a.p);
                const unsigned mine = (above >> (chalf * 16)) & 0xFFFFu;
                const int rstar = mine ? (31 - __clz(mine)) : -1;
                if ((lane & 15) == rstar) cosv = 0.f;
                rowsum += cosv;
            }
        }
        rowsum += __shfl_xor_sync(0xFFFFFFFFu, rowsum, 16);
        if (chalf == 0 && r < nvalid)
            a.rho[((size_t)s * a.h_kv + kvh) * a.Lmax + tb0 + r] = rowsum;
    }
}

// Tensor-core variant for bf16 keys and b = 16 (one 16 x 16 Gram per block and
// kv head).  grid (ceil(Lmax / 16), n), one warp per kv head.  The block's
// keys (all kv heads: one contiguous page) are copied with coalesced 16-byte
// loads into shared memory, each head's 16 rows of 128 dims as two 16 x 128 B
// tiles whose 16-byte chunks are XOR-swizzled by (row % 8), so that ldmatrix
// reads conflict-free.  G = K K^T takes 16 mma.sync (8 k-steps x 2 n-tiles);
// one ldmatrix.x4 per k-step feeds both operands.  Then, on the accumulator
// fragments: cosine (zero-norm keys give 0), zero diagonal, per column the
// newest row above p zeroed (a ballot over the column's lanes), row sums.
template <int D>
__global__ void __launch_bounds__(512) lightning_tc_kernel(const ScoreArgs a) {
    constexpr int HALVES = D / 64;
    constexpr int KS = D / 16;
    extern __shared__ __align__(128) unsigned char lsm[];
    const int s = blockIdx.y;
    const int bi = blockIdx.x;
    const int L = clamp_len(a, s);
    const int tb0 = bi * 16;
    if (tb0 >= L) return;
    const int nvalid = min(16, L - tb0);
    const int blk = a.table[(size_t)s * a.table_stride + bi];
    if (blk < 0 || blk >= a.n_total) {
        if (threadIdx.x == 0) record_error(a.err, ZP_ERR_DEVICE, 0x202);
        return;
    }
    const int h_kv = a.h_kv;
    // ---- page -> swizzled tiles [head][half][16 rows][8 chunks of 16 B]
    const uint4 *src = reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(a.k) +
                                                       (size_t)blk * 16 * h_kv * D);
    const int chunks_per_row = D / 8;  // 16-byte chunks in one (token, head) row
    const int total = nvalid * h_kv * chunks_per_row;
    for (int i = threadIdx.x; i < total; i += blockDim.x) {
        const int t = i / (h_kv * chunks_per_row);
        const int rem = i % (h_kv * chunks_per_row);
        const int h = rem / chunks_per_row;
        const int c = rem % chunks_per_row;
        const int hf = c >> 3, cc = c & 7;
        reinterpret_cast<uint4 *>(lsm + ((h * HALVES + hf) * 16 + t) * 128)[cc ^ (t & 7)] = src[i];
    }
    // rows past the sequence end: zeros (excluded again below)
    for (int i = threadIdx.x; i < (16 - nvalid) * h_kv * chunks_per_row; i += blockDim.x) {
        const int t = nvalid + i / (h_kv * chunks_per_row);
        const int rem = i % (h_kv * chunks_per_row);
        const int h = rem / chunks_per_row;
        const int c = rem % chunks_per_row;
        reinterpret_cast<uint4 *>(lsm + ((h * HALVES + (c >> 3)) * 16 + t) * 128)[(c & 7) ^ (t & 7)] =
            make_uint4(0, 0, 0, 0);
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp >= h_kv) return;
    const int kvh = warp;
    const int g = lane >> 2, tig = lane & 3;
    const int lm = lane >> 3;
    const int lrow = (lm & 1) * 8 + (lane & 7);  // matrices: (t0-7,c) (t8-15,c) (t0-7,c+1) (t8-15,c+1)
    const int lchunk = lm >> 1;
    const uint32_t tile0 = smem_u32(lsm + (size_t)kvh * HALVES * 16 * 128);
    float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int t = 0; t < KS; ++t) {
        const uint32_t tile = tile0 + (t >> 2) * 16 * 128;
        const int chunk = (t & 3) * 2 + lchunk;
        uint32_t r0, r1, r2, r3;  // (t0-7,c) (t8-15,c) (t0-7,c+1) (t8-15,c+1)
        ldsm_x4(tile + lrow * 128 + ((chunk ^ (lrow & 7)) << 4), r0, r1, r2, r3);
        // A = K rows (a0a1 row g / c, a2a3 row g+8 / c, a4a5 row g / c+1, a6a7 row g+8 / c+1)
        // B = K^T: n-tile 0 = tokens 0-7 (b0 = chunk c, b1 = chunk c+1), n-tile 1 = tokens 8-15
        mma_16816(c0, r0, r1, r2, r3, r0, r2);
        mma_16816(c1, r0, r1, r2, r3, r1, r3);
    }
    // lane holds G[g][2tig+e] (c0[e]), G[g+8][2tig+e] (c0[2+e]), G[g][8+2tig+e] (c1[e]), G[g+8][8+2tig+e] (c1[2+e])
    __shared__ float nrm[16][16];  // per warp: the 16 norms
    float *myn = nrm[warp];
    if (tig == (g >> 1)) myn[g] = c0[g & 1];               // G[g][g], g < 8
    if (tig == (g >> 1)) myn[g + 8] = c1[2 + (g & 1)];     // G[g+8][g+8]
    __syncwarp();
    const int rows[2] = {g, g + 8};
    const int cols[4] = {2 * tig, 2 * tig + 1, 8 + 2 * tig, 9 + 2 * tig};
    float v[2][4];  // [row][col]
    v[0][0] = c0[0]; v[0][1] = c0[1]; v[0][2] = c1[0]; v[0][3] = c1[1];
    v[1][0] = c0[2]; v[1][1] = c0[3]; v[1][2] = c1[2]; v[1][3] = c1[3];
#pragma unroll
    for (int ri = 0; ri < 2; ++ri) {
        const float nr = sqrtf(fmaxf(myn[rows[ri]], 0.f));
#pragma unroll
        for (int ci = 0; ci < 4; ++ci) {
            const float nc = sqrtf(fmaxf(myn[cols[ci]], 0.f));
            const bool ok = rows[ri] < nvalid && cols[ci] < nvalid && rows[ri] != cols[ci] && nr > 0.f && nc > 0.f;
            v[ri][ci] = ok ? v[ri][ci] / (nr * nc) : 0.f;
        }
    }
    // per column: the newest row with cos > p loses its entry
#pragma unroll
    for (int ci = 0; ci < 4; ++ci) {
        const unsigned blo = __ballot_sync(0xFFFFFFFFu, v[0][ci] > a.p);
        const unsigned bhi = __ballot_sync(0xFFFFFFFFu, v[1][ci] > a.p);
        // bits of the lanes sharing this lane's column: lanes tig + 4 g', g' = 0..7
        unsigned mlo = 0, mhi = 0;
#pragma unroll
        for (int gg = 0; gg < 8; ++gg) {
            mlo |= ((blo >> (tig + 4 * gg)) & 1u) << gg;
            mhi |= ((bhi >> (tig + 4 * gg)) & 1u) << gg;
        }
        int rstar = -1;
        if (mhi) rstar = 8 + (31 - __clz(mhi));
        else if (mlo) rstar = 31 - __clz(mlo);
        if (rstar == rows[0]) v[0][ci] = 0.f;
        if (rstar == rows[1]) v[1][ci] = 0.f;
    }
    float rs0 = v[0][0] + v[0][1] + v[0][2] + v[0][3];
    float rs1 = v[1][0] + v[1][1] + v[1][2] + v[1][3];
    rs0 += __shfl_xor_sync(0xFFFFFFFFu, rs0, 1);
    rs0 += __shfl_xor_sync(0xFFFFFFFFu, rs0, 2);
    rs1 += __shfl_xor_sync(0xFFFFFFFFu, rs1, 1);
    rs1 += __shfl_xor_sync(0xFFFFFFFFu, rs1, 2);
    if (tig == 0) {
        float *out = a.rho + ((size_t)s * a.h_kv + kvh) * a.Lmax + tb0;
        if (g < nvalid) out[g] = rs0;
        if (g + 8 < nvalid) out[g + 8] = rs1;
    }
}

// grid (h_kv, n), 1024 threads
__global__ void finalize_kernel(const ScoreArgs a) {
    __shared__ float red[32];
    const int kvh = blockIdx.x;
    const int s = blockIdx.y;
    const int L = clamp_len(a, s);
    if (L <= 0) return;
    const size_t row = ((size_t)s * a.h_kv + kvh) * a.Lmax;
    const float *X = a.X + row;
    const float *rho = a.rho + row;
    float *out = a.out + row;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
    const bool first = a.first ? a.first[s] != 0 : true;
    const bool pool = a.pool_kernel > 1 && (a.pool_policy == 2 || (a.pool_policy == 1 && first));
    const int r = a.pool_kernel / 2;
    float rmax = -INFINITY, rsum = 0.f;
    const float inv = 1.f / ((float)L * a.tau);
    if (a.use_sim) {
        float m = -INFINITY;
        for (int t = tid; t < L; t += blockDim.x) m = fmaxf(m, rho[t] * inv);
        for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        if (lane == 0) red[warp] = m;
        __syncthreads();
        if (warp == 0) {
            float x = lane < nw ? red[lane] : -INFINITY;
            for (int o = 16; o; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xFFFFFFFFu, x, o));
            if (lane == 0) red[0] = x;
        }
        __syncthreads();
        rmax = red[0];
        __syncthreads();
        float sum = 0.f;
        for (int t = tid; t < L; t += blockDim.x) sum += expf(rho[t] * inv - rmax);
        for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
        if (lane == 0) red[warp] = sum;
        __syncthreads();
        if (warp == 0) {
            float x = lane < nw ? red[lane] : 0.f;
            for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, o);
            if (lane == 0) red[0] = x;
        }
        __syncthreads();
        rsum = red[0];
    }
    for (int t = tid; t < L; t += blockDim.x) {
        float v;
        if (pool) {
            const int lo = max(0, t - r), hi = min(L - 1, t + r);
            v = X[lo];
            for (int j = lo + 1; j <= hi; ++j) v = fmaxf(v, X[j]);
        } else {
            v = X[t];
        }
        if (a.use_sim) v -= a.lambda * (expf(rho[t] * inv - rmax) / rsum);
        if (t >= L - a.window) v = INFINITY;
        out[t] = v;
    }
}

}  // namespace
}  // namespace zp

using namespace zp;

extern "C" size_t zp_score_workspace_size(const zp_cache_desc *D, int32_t n, int32_t Lmax) {
    if (!D || n < 0 || Lmax < 0) return 0;
    return 2 * align_up((size_t)n * D->h_kv * Lmax * 4, 256);
}

extern "C" zp_status zp_score_tokens(const zp_cache_desc *D, const zp_score_params *P,
                                     const void *k_cache, const int32_t *block_table,
                                     int32_t table_stride, const int32_t *seq_lens,
                                     const uint8_t *first_compression, int32_t n,
                                     const zp_score_rows *attn, const float *global_F,
                                     float *scores_out,
                                     int32_t Lmax, void *workspace, size_t workspace_bytes,
                                     void *stream) {
    zp_status rc = check_desc(D);
    if (rc != ZP_OK) return rc;
    if (!P) return fail(ZP_ERR_INVALID_ARG, "score: NULL params");
    if (n < 0 || Lmax < 0 || table_stride < 1) return fail(ZP_ERR_INVALID_ARG, "score: bad sizes");
    if (n == 0 || Lmax == 0) return ok();
    if (!block_table || !seq_lens || !scores_out || !workspace)
        return fail(ZP_ERR_INVALID_ARG, "score: NULL buffer");
    if (!attn || !attn->data) return fail(ZP_ERR_INVALID_ARG, "score: NULL attention-score rows");
    if (attn->stride < 1) return fail(ZP_ERR_INVALID_ARG, "score: score row stride %lld", (long long)attn->stride);
    if (P->use_global && !global_F) return fail(ZP_ERR_INVALID_ARG, "score: use_global needs global_F");
    if (P->use_similarity && !k_cache) return fail(ZP_ERR_INVALID_ARG, "score: similarity needs k_cache");
    if (P->window < 0) return fail(ZP_ERR_INVALID_ARG, "score: window %d", P->window);
    if (P->pool_kernel > 1 && P->pool_kernel % 2 == 0)
        return fail(ZP_ERR_INVALID_ARG, "score: pool kernel %d must be odd", P->pool_kernel);
    if (P->pool_policy < 0 || P->pool_policy > 2) return fail(ZP_ERR_INVALID_ARG, "score: pool policy");
    if (P->use_similarity && !(P->tau > 0.f)) return fail(ZP_ERR_INVALID_ARG, "score: tau must be > 0");
    if (D->h_kv > 16) return fail(ZP_ERR_SHAPE, "score: h_kv %d > 16", D->h_kv);
    if (P->use_similarity && !P->lightning)
        return fail(ZP_ERR_SHAPE, "score: the all-pairs redundancy score is not built; use lightning");
    if (P->use_similarity && D->block_size > 16)
        return fail(ZP_ERR_SHAPE, "score: lightning kernel supports b <= 16 (b=%d)", D->block_size);
    const size_t need = zp_score_workspace_size(D, n, Lmax);
    if (workspace_bytes < need) return fail(ZP_ERR_CAPACITY, "score: workspace %zu < %zu", workspace_bytes, need);
    DeviceInfo dev;
    rc = device_info(&dev);
    if (rc != ZP_OK) return rc;
    ScoreArgs a;
    a.table = block_table;
    a.table_stride = table_stride;
    a.seq_lens = seq_lens;
    a.first = first_compression;
    a.n = n;
    a.h_kv = D->h_kv;
    a.b = D->block_size;
    a.n_total = D->n_total_blocks;
    a.Lmax = Lmax;
    a.d = D->head_dim;
    a.S = attn->data;
    a.S_stride = attn->stride;
    a.S_rows = attn->rows;
    a.F = global_F;
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    a.X = reinterpret_cast<float *>(ws);
    a.rho = reinterpret_cast<float *>(ws + align_up((size_t)n * D->h_kv * Lmax * 4, 256));
    a.out = scores_out;
    a.k = k_cache;
    a.use_global = P->use_global;
    a.alpha = P->alpha;
    a.pool_kernel = P->pool_kernel;
    a.pool_policy = P->pool_policy;
    a.use_sim = P->use_similarity;
    a.p = P->threshold;
    a.lambda = P->lambda;
    a.tau = P->tau;
    a.window = P->window;
    a.err = dev.error_word;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    dim3 g1((Lmax + kTile - 1) / kTile, n);
    gather_global_kernel<<<g1, 256, 0, st>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "score: gather launch");
    if (a.use_sim) {
        dim3 g2((Lmax + a.b - 1) / a.b, n);
        const size_t smem = (size_t)a.h_kv * a.b * (a.d + 1) * 4;
        if (smem > (size_t)dev.smem_optin) return fail(ZP_ERR_SHAPE, "score: block of keys too large");
        if (D->dtype == ZP_BF16 && a.b == 16 && (a.d == 64 || a.d == 128)) {
            const size_t smem_tc = (size_t)a.h_kv * (a.d / 64) * 16 * 128;
            if (a.d == 128) {
                if (smem_tc > 48 * 1024)
                    cudaFuncSetAttribute(lightning_tc_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem_tc);
                lightning_tc_kernel<128><<<g2, a.h_kv * 32, smem_tc, st>>>(a);
            } else {
                if (smem_tc > 48 * 1024)
                    cudaFuncSetAttribute(lightning_tc_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem_tc);
                lightning_tc_kernel<64><<<g2, a.h_kv * 32, smem_tc, st>>>(a);
            }
        } else if (D->dtype == ZP_BF16) {
            cudaFuncSetAttribute(lightning_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
            lightning_kernel<__nv_bfloat16><<<g2, a.h_kv * 32, smem, st>>>(a);
        } else {
            cudaFuncSetAttribute(lightning_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
            lightning_kernel<float><<<g2, a.h_kv * 32, smem, st>>>(a);
        }
        e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e, "score: lightning launch");
    }
    dim3 g3(a.h_kv, n);
    finalize_kernel<<<g3, 1024, 0, st>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "score: finalize launch");
    return ok();
}
