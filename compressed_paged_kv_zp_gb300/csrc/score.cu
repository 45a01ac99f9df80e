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

#include "lightning.cuh"
#include "select.cuh"

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
    // layers of one call (blockIdx.z of the fused kernels): strides in bytes (K)
    // and elements (S, F, X / rho / out)
    long long k_layer_bytes, S_layer, F_layer, X_layer;
    // lightning row sums given by the caller (zp_compress_layers_rho), else null
    const float *rho_in;     // rho_in + (row * h_kv + kvh) * rho_stride + t
    long long rho_stride, rho_layer;
    const int32_t *rho_rows;  // nullable [n]
    int n_rho_rows;
};

// The arguments of layer z: every per-layer pointer advanced by its stride.
__device__ __forceinline__ ScoreArgs at_layer(const ScoreArgs &a0, int z) {
    ScoreArgs a = a0;
    a.k = static_cast<const char *>(a0.k) + z * a0.k_layer_bytes;
    a.S = a0.S + z * a0.S_layer;
    if (a0.F) a.F = a0.F + z * a0.F_layer;
    a.X = a0.X + z * a0.X_layer;
    a.rho = a0.rho + z * a0.X_layer;
    if (a0.out) a.out = a0.out + z * a0.X_layer;
    if (a0.rho_in) a.rho_in = a0.rho_in + z * a0.rho_layer;
    return a;
}

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
            // cosine, diagonal, threshold: for column c the newest row r* < nvalid
            // with cos > p is zeroed (rows past the block's end take no part,
            // also when p < 0 makes their zero entries exceed it).  Rows of this
            // column live in lanes with the same chalf across the 16-row groups;
            // with b <= 16 one group.
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
                const unsigned above = __ballot_sync(0xFFFFFFFFu, r < nvalid && cosv > a.p);
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
    // rows >= nvalid hold zeros: every entry they touch is masked
    const float2 rs = lightning_rowsums<false>(c0, c1, nvalid, a.p, lane);
    const float rs0 = rs.x, rs1 = rs.y;
    if (tig == 0) {
        float *out = a.rho + ((size_t)s * a.h_kv + kvh) * a.Lmax + tb0;
        if (g < nvalid) out[g] = rs0;
        if (g + 8 < nvalid) out[g + 8] = rs1;
    }
}

// Lightning redundancy of one block for kv head `kvh` (one warp).  The
// block's token rows (all kv heads) are in shared memory in the decode's
// staged layout (lightning.cuh: groups of kStageRows rows, group stride GS =
// kStageRows RB + 16, RB = bytes of a row).  G = K K^T on the tensor cores
// (16 mma.sync) with the same fragments as the decode's Gram -- operand tile
// 0 as the first 8 rows / columns, tile 1 as the second -- then the rule on
// the accumulator fragments (lightning_rowsums).  Returns the row sums of
// fragment rows g and g + 8 (store_block_rho writes them).
template <int D>
__device__ __forceinline__ float2 lightning_block(const ScoreArgs &a, const unsigned char *gsm, int GS, int nvalid,
                                                  int kvh, int lane) {
    const int h_kv = a.h_kv;
    constexpr int KS = D / 16;
    const int lm = lane >> 3;
    const int li = lane & 7;
    const int RB = h_kv * D * 2;
    // matrices: (tile 0, chunk c) (tile 1, c) (tile 0, c + 1) (tile 1, c + 1)
    const uint32_t base =
        smem_u32(gsm) + (uint32_t)((li / (kStageRows / 2)) * GS + (li % (kStageRows / 2) + (lm & 1) * (kStageRows / 2)) * RB +
                                   (lm >> 1) * 16 + kvh * D * 2);
    float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int t = 0; t < KS; ++t) {
        uint32_t r0, r1, r2, r3;
        ldsm_x4(base + (uint32_t)(32 * t), r0, r1, r2, r3);
        mma_16816(c0, r0, r1, r2, r3, r0, r2);
        mma_16816(c1, r0, r1, r2, r3, r1, r3);
    }
    // rows >= nvalid were not copied: every entry they touch is masked
    return lightning_rowsums<true>(c0, c1, nvalid, a.p, lane);
}

// Row sums of lightning_block to rho: fragment rows g, g + 8 are row g of
// operand tiles 0 and 1.
__device__ __forceinline__ void store_block_rho(const ScoreArgs &a, float2 rs, int nvalid, int s, int tb0, int kvh,
                                                int lane) {
    const int g = lane >> 2, tig = lane & 3;
    if (tig == 0) {
        float *out = a.rho + ((size_t)s * a.h_kv + kvh) * a.Lmax + tb0;
        const int t0 = staged_token(0, g), t1 = staged_token(1, g);
        if (t0 < nvalid) out[t0] = rs.x;
        if (t1 < nvalid) out[t1] = rs.y;
    }
}

// Redundancy and global score of one 16-token block in one CTA (bf16 keys,
// b = 16, the path zp_compress_layers takes).  grid (ceil(Lmax / 16), n), one
// warp per kv head.  The block's token rows (all kv heads, contiguous in HBM)
// come by one bulk copy per pair of rows into shared memory pairs padded by 16
// bytes; while they are in flight, the CTA computes the block's global score
// (Alg. 2, as gather_global_kernel) from the score rows and F.  Then the
// lightning rule per head (lightning_block).
template <int D>
__global__ void __launch_bounds__(512) global_lightning_kernel(const ScoreArgs a0) {
    const ScoreArgs a = at_layer(a0, blockIdx.z);
    extern __shared__ __align__(128) unsigned char gsm[];
    __shared__ __align__(8) uint64_t bar;
    __shared__ int s_blk, s_abort;
    const int s = blockIdx.y;
    const int bi = blockIdx.x;
    const int L = clamp_len(a, s);
    const int tb0 = bi * 16;
    if (tb0 >= L) return;
    const int nvalid = min(16, L - tb0);
    const int h_kv = a.h_kv;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const unsigned row_bytes = (unsigned)(h_kv * D * 2);
    const int GS = kStageRows * (int)row_bytes + 16;  // staged group of rows
    if (tid == 0) {
        const int blk = a.table[(size_t)s * a.table_stride + bi];
        s_blk = blk;
        s_abort = 0;
        mbar_init(&bar, 1);
        fence_barrier_init();
        if (blk < 0 || blk >= a.n_total) {
            record_error(a.err, ZP_ERR_DEVICE, 0x202);
        } else {
            mbar_arrive_expect_tx(&bar, row_bytes * (unsigned)nvalid);
            const char *src = static_cast<const char *>(a.k) + (size_t)blk * 16 * row_bytes;
            for (int j = 0; kStageRows * j < nvalid; ++j)
                bulk_g2s_plain(gsm + j * GS, src + (size_t)kStageRows * j * row_bytes,
                               (unsigned)min(kStageRows, nvalid - kStageRows * j) * row_bytes, &bar);
        }
    }
    __syncthreads();
    const int blk = s_blk;
    if (blk < 0 || blk >= a.n_total) return;
    // This kernel is launched as a programmatic dependent of the preceding one
    // (the decode call, when it precedes), which writes the score rows but not
    // the lengths, the block table, the keys or F: everything but the score
    // rows is read, and the redundancy computed, before griddepcontrol.wait.
    // Nothing is stored to global memory before the wait: the caller may have
    // given this call memory that the preceding kernel still uses (a scratch
    // buffer freed after that call was queued and handed out again, which
    // stream order alone makes safe).
    // Global score (Alg. 2) of this thread's (kv head, token) of the block:
    // F read now, the score row after the wait.
    const int N = (L + a.b - 1) / a.b;
    const bool first = a.first ? a.first[s] != 0 : true;
    const bool read_F = a.use_global && !first && bi != N - 1;
    const int row = a.S_rows ? a.S_rows[s] : s;
    const int g_kvh = tid / nvalid, g_tl = tid % nvalid;  // one item per thread: 16 * h_kv <= blockDim
    const bool g_on = tid < nvalid * h_kv;
    const float fv = (g_on && read_F) ? a.F[((size_t)blk * a.b + g_tl) * h_kv + g_kvh] : 0.f;
    mbar_wait_bounded(&bar, 0, a.err, &s_abort, 0x203);
    __syncthreads();
    // the finish kernel may be scheduled once every CTA of this grid is this
    // far (late, so that its waiting CTAs do not take the SM slots of this
    // grid's later CTAs); it waits for this grid's completion before reading
    // its output
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (s_abort) return;
    const float2 rs = lightning_block<D>(a, gsm, GS, nvalid, warp, lane);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    store_block_rho(a, rs, nvalid, s, tb0, warp, lane);
    if (g_on) {
        if (row < 0) {
            record_error(a.err, ZP_ERR_DEVICE, 0x202);
        } else {
            float *sp = a.S + ((size_t)row * h_kv + g_kvh) * a.S_stride + tb0 + g_tl;
            float v = *sp;
            if (read_F) {
                v = fmaxf(a.alpha * fv, v);
                *sp = v;
            }
            a.X[((size_t)s * h_kv + g_kvh) * a.Lmax + tb0 + g_tl] = v;
        }
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


// ---------------------------------------------------------------------------
// Fused finish of one layer's compression (zp_compress_layers): per (sequence,
// kv head) one CTA takes the global score X and the row sums rho into shared
// memory, finalises the scores there (as finalize_kernel), selects the keep
// set (block_select_topk) and moves this kv head's kept rows of K and V into
// the target blocks, F of each target slot receiving the kept token's global
// score (as the compaction).  The keep set never leaves the CTA before the
// move (it is also written out).
struct MoveArgs {
    uint4 *K, *V;
    int row_vec;         // 16-byte vectors per (token, kv head) row
    const int32_t *dst;  // [n][target_stride]
    int target_stride;
    int k;               // row stride of keep (the largest budget)
    const int32_t *k_seq;  // nullable: per-request budgets k_i <= k
    int32_t *keep;       // [n][h_kv][k]
    int32_t *tie;        // nullable [n][h_kv]
    float *F;            // nullable, paged
    long long kv_layer_vec;  // 16-byte vectors between layers of K (and V)
    long long F_layer;       // elements between layers of F
};

constexpr int kFsThreads = 1024;
constexpr int kFsChunk = 128;      // ranks per move round
constexpr int kFsVecPerThread = 4; // 16-byte registers per thread and round (row pieces up to 256 B)

// xs, fs [Lmax]; keep, source row, F value, target row [k]; target blocks
// [ceil(k / b)]; the sequence's table row [ceil(Lmax / b)]
__host__ __device__ inline size_t fused_smem(int Lmax, int k, int b) {
    return (size_t)Lmax * 8 + (size_t)k * 16 + (size_t)((k + b - 1) / b) * 4 + (size_t)((Lmax + b - 1) / b) * 4 + 64;
}

// Whether the one-kernel finish (scores, selection, move per (kv head,
// sequence, layer)) covers this cache, these switches, Lmax and k: its dynamic
// shared memory and its static part (the select's state, the reductions) fit.
inline bool fused_finish_fits(const zp_cache_desc *D, const zp_score_params *P, int Lmax, int k, size_t optin) {
    const int row_vec = D->head_dim * elem_bytes(D->dtype) / 16;
    const size_t static_bytes = sizeof(SelectShared) + 64 * sizeof(float) + 256;
    return D->dtype == ZP_BF16 && D->block_size == 16 && (D->head_dim == 64 || D->head_dim == 128) &&
           D->h_kv <= 16 && P && P->use_similarity && P->lightning && 2 * row_vec <= kFsThreads * kFsVecPerThread &&
           fused_smem(Lmax, k, D->block_size) + static_bytes <= optin;
}

// Block-wide combination of per-thread online-softmax pairs (max m, sum s of
// 2^(y - m)): M = max m, S = sum s * 2^(m - M).  red: 64 floats.
__device__ __forceinline__ float2 block_reduce_maxsum(float m, float s, float *red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    for (int o = 16; o; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xFFFFFFFFu, m, o);
        const float s2 = __shfl_xor_sync(0xFFFFFFFFu, s, o);
        const float M = fmaxf(m, m2);
        s = (M == -INFINITY) ? 0.f : s * exp2f(m - M) + s2 * exp2f(m2 - M);
        m = M;
    }
    __syncthreads();
    if (lane == 0) {
        red[warp] = m;
        red[32 + warp] = s;
    }
    __syncthreads();
    // every warp combines the per-warp pairs by the same shuffle tree
    m = lane < nw ? red[lane] : -INFINITY;
    s = lane < nw ? red[32 + lane] : 0.f;
    for (int o = 16; o; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xFFFFFFFFu, m, o);
        const float s2 = __shfl_xor_sync(0xFFFFFFFFu, s, o);
        const float M = fmaxf(m, m2);
        s = (M == -INFINITY) ? 0.f : s * exp2f(m - M) + s2 * exp2f(m2 - M);
        m = M;
    }
    return make_float2(m, s);
}

// OWN_X: the global score (Alg. 2, as global_lightning_kernel) is formed here
// from the score row and F, and rho comes from the caller's rows (a.rho_in);
// otherwise both are read from X and rho of the preceding scores kernel.
template <bool OWN_X>
__global__ void __launch_bounds__(kFsThreads) finalize_select_move_kernel(const ScoreArgs a0, const MoveArgs m0) {
    const int z = blockIdx.z;
    const ScoreArgs a = at_layer(a0, z);
    MoveArgs m = m0;
    m.K = m0.K + z * m0.kv_layer_vec;
    m.V = m0.V + z * m0.kv_layer_vec;
    if (m0.F) m.F = m0.F + z * m0.F_layer;
    m.keep = m0.keep + (size_t)z * a0.n * a0.h_kv * m0.k;
    if (m0.tie) m.tie = m0.tie + (size_t)z * a0.n * a0.h_kv;
    extern __shared__ __align__(16) unsigned char fsm[];
    __shared__ SelectShared sh;
    __shared__ float red[64];
    const int kvh = blockIdx.x, s = blockIdx.y, tid = threadIdx.x, nthr = blockDim.x;
    const int L = clamp_len(a, s);
    float *xs = reinterpret_cast<float *>(fsm);
    float *fs = xs + a.Lmax;
    int *keep_s = reinterpret_cast<int *>(fs + a.Lmax);
    int *src_s = keep_s + m.k;                              // source row (token, kv head) of rank i, -1: none
    float *fv_s = reinterpret_cast<float *>(src_s + m.k);  // global score of rank i
    int *drow_s = reinterpret_cast<int *>(fv_s + m.k);     // target row of rank i, -1: bad target
    int *dst_s = drow_s + m.k;
    const int nt = (m.k + a.b - 1) / a.b;
    int *tbl_s = dst_s + nt;
    const int nb = (L + a.b - 1) / a.b;
    for (int t = tid; t < nt; t += nthr) dst_s[t] = m.dst[(size_t)s * m.target_stride + t];
    for (int t = tid; t < nb; t += nthr) tbl_s[t] = a.table[(size_t)s * a.table_stride + t];
    const bool first = a.first ? a.first[s] != 0 : true;
    const size_t row = ((size_t)s * a.h_kv + kvh) * a.Lmax;
    if constexpr (OWN_X) {
        // Global score (Alg. 2): max(alpha * F, S) on blocks 0..N-2 after the
        // first compression, else S.  alpha * F first (F is not written by the
        // kernel this one may follow), the score row after the wait.
        const bool read_F = a.use_global && !first;
        if (read_F) {
            __syncthreads();
            for (int t = tid; t < L; t += nthr) {
                if ((t >> 4) == nb - 1) continue;
                const int blk = tbl_s[t >> 4];
                float f = 0.f;
                if (blk < 0 || blk >= a.n_total) record_error(a.err, ZP_ERR_DEVICE, 0x202);
                else f = a.F[((size_t)blk * 16 + (t & 15)) * a.h_kv + kvh];
                xs[t] = a.alpha * f;
            }
        }
        // launched as a programmatic dependent of the decode: the score rows
        // and rho are read after its completion (a no-op for a plain launch)
        asm volatile("griddepcontrol.wait;" ::: "memory");
        const int srow = a.S_rows ? a.S_rows[s] : s;
        int rrow = a.rho_rows ? a.rho_rows[s] : s;
        if (a.use_sim && (rrow < 0 || rrow >= a.n_rho_rows || L > a.rho_stride)) {
            if (tid == 0) record_error(a.err, ZP_ERR_DEVICE, 0x203);
            rrow = -1;
        }
        if (srow < 0) {
            if (tid == 0) record_error(a.err, ZP_ERR_DEVICE, 0x202);
        } else {
            float *sp = a.S + ((size_t)srow * a.h_kv + kvh) * a.S_stride;
            const float *rp = rrow >= 0 ? a.rho_in + ((size_t)rrow * a.h_kv + kvh) * a.rho_stride : nullptr;
            for (int t0 = tid; t0 < L; t0 += 4 * nthr) {  // four elements' loads in flight per thread
                float sv[4], rv4[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int t = t0 + i * nthr;
                    sv[i] = t < L ? sp[t] : 0.f;
                    rv4[i] = (t < L && rp) ? rp[t] : 0.f;
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int t = t0 + i * nthr;
                    if (t < L) {
                        float v = sv[i];
                        if (read_F && (t >> 4) != nb - 1) {
                            v = fmaxf(xs[t], v);
                            sp[t] = v;
                        }
                        xs[t] = v;
                        fs[t] = rv4[i];
                    }
                }
            }
        }
    } else {
    // launched as a programmatic dependent of the scores kernel: X, rho and the
    // score rows are read after its completion (a no-op for a plain launch)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    for (int t0 = tid; t0 < L; t0 += 4 * nthr) {  // four elements' loads in flight per thread
        float xv[4], rv4[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int t = t0 + i * nthr;
            xv[i] = t < L ? a.X[row + t] : 0.f;
            rv4[i] = (t < L && a.use_sim) ? a.rho[row + t] : 0.f;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int t = t0 + i * nthr;
            if (t < L) {
                xs[t] = xv[i];
                fs[t] = rv4[i];
            }
        }
    }
    }
    __syncthreads();
    // ---- final scores (App. C.4-C.8, eq. 4, window), in place of rho
    const bool pool = a.pool_kernel > 1 && (a.pool_policy == 2 || (a.pool_policy == 1 && first));
    const int r = a.pool_kernel / 2;
    // R = softmax(rho / (L tau)) in base 2: one pass for the max and the sum
    // (online), one block reduction of the (max, sum) pairs
    const float inv2 = 1.4426950408889634f / ((float)L * a.tau);
    float rmax = 0.f, rinv = 1.f;
    if (a.use_sim && L > 0) {
        float mx = -INFINITY, sm = 0.f;
        for (int t = tid; t < L; t += nthr) {
            const float y = fs[t] * inv2;
            if (y > mx) {
                sm = sm * exp2f(mx - y) + 1.f;
                mx = y;
            } else {
                sm += exp2f(y - mx);
            }
        }
        const float2 ms = block_reduce_maxsum(mx, sm, red);
        rmax = ms.x;
        rinv = 1.f / ms.y;
    }
    for (int t = tid; t < L; t += nthr) {
        float v = xs[t];
        if (pool && r <= 8) {
            // the window's loads unrolled (clamped indices repeat an element,
            // which leaves the max unchanged)
#pragma unroll
            for (int j = 1; j <= 8; ++j)
                if (j <= r) v = fmaxf(v, fmaxf(xs[max(t - j, 0)], xs[min(t + j, L - 1)]));
        } else if (pool) {
            const int lo = max(0, t - r), hi = min(L - 1, t + r);
            for (int j = lo; j <= hi; ++j) v = fmaxf(v, xs[j]);
        }
        if (a.use_sim) v -= a.lambda * (exp2f(fs[t] * inv2 - rmax) * rinv);
        if (t >= L - a.window) v = INFINITY;
        fs[t] = v;
        if (a.out) a.out[row + t] = v;
    }
    __syncthreads();
    // ---- keep set (this request's budget ki; the row is padded with -1)
    int32_t *kout = m.keep + ((size_t)s * a.h_kv + kvh) * m.k;
    int ki = m.k_seq ? m.k_seq[s] : m.k;
    if (ki < 0 || ki > m.k) {
        if (tid == 0) record_error(a.err, ZP_ERR_DEVICE, 0x302);
        ki = ki < 0 ? 0 : m.k;
    }
    for (int i = ki + tid; i < m.k; i += nthr) kout[i] = -1;
    if (L <= ki) {
        for (int i = tid; i < ki; i += nthr) {
            keep_s[i] = i < L ? i : -1;
            kout[i] = i < L ? i : -1;
        }
        if (m.tie && tid == 0) m.tie[(size_t)s * a.h_kv + kvh] = 0;
        __syncthreads();
    } else {
        block_select_topk<false>(fs, L, ki, kout, keep_s, m.tie ? m.tie + (size_t)s * a.h_kv + kvh : nullptr, a.err, sh);
    }
    // ---- move this kv head's kept rows (Alg. 4 with the target blocks).
    // Rank i: source row (block of its token, from the table row in shared
    // memory), target row (slot i of target block i / b) and its global score
    // (X, the value the compaction stores into F).  b = 16 and the 16-byte
    // vectors per row piece are a power of two on this path, so the item
    // indices below are shifts.
    const int kk = min(ki, L);
    float *F = m.F;
    if (F && a.S_rows && a.S_rows[s] < 0) {
        if (tid == 0) record_error(a.err, ZP_ERR_DEVICE, 0x402);
        F = nullptr;
    }
    for (int i = tid; i < kk; i += nthr) {
        const int pos = keep_s[i];
        int blk = (pos >= 0 && pos < L) ? tbl_s[pos >> 4] : -1;
        if (blk < 0 || blk >= a.n_total) {
            record_error(a.err, ZP_ERR_DEVICE, 0x400);
            blk = -1;
        }
        src_s[i] = blk >= 0 ? (blk * 16 + (pos & 15)) * a.h_kv + kvh : -1;
        fv_s[i] = blk >= 0 ? xs[pos] : 0.f;
        const int tblk = dst_s[i >> 4];
        if (tblk < 0 || tblk >= a.n_total) {
            record_error(a.err, ZP_ERR_DEVICE, 0x401);
            drow_s[i] = -1;
        } else {
            drow_s[i] = (tblk * 16 + (i & 15)) * a.h_kv + kvh;
        }
    }
    __syncthreads();
    const int rv = m.row_vec, rv_sh = 31 - __clz(rv);
    const int pr_sh = rv_sh + 1;  // 16-byte vectors per rank (K and V pieces)
    const int chunk = min(kFsChunk, (kFsThreads * kFsVecPerThread) >> pr_sh);
    for (int r0 = 0; r0 < kk; r0 += chunk) {
        const int nr = min(chunk, kk - r0);
        const int items = nr << pr_sh;
        uint4 buf[kFsVecPerThread];
#pragma unroll
        for (int i = 0; i < kFsVecPerThread; ++i) {
            const int it = tid + i * kFsThreads;
            if (it < items) {
                const int rr = r0 + (it >> pr_sh), v = it & ((rv << 1) - 1);
                const int sr = src_s[rr];
                if (sr >= 0) buf[i] = (v < rv ? m.K : m.V)[(size_t)sr * rv + (v & (rv - 1))];
            }
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < kFsVecPerThread; ++i) {
            const int it = tid + i * kFsThreads;
            if (it < items) {
                const int rr = r0 + (it >> pr_sh), v = it & ((rv << 1) - 1);
                const int dr = drow_s[rr];
                if (dr >= 0 && src_s[rr] >= 0) (v < rv ? m.K : m.V)[(size_t)dr * rv + (v & (rv - 1))] = buf[i];
            }
        }
        if (F)
            for (int i = tid; i < nr; i += nthr) {
                const int dr = drow_s[r0 + i];
                if (dr >= 0) F[dr] = fv_s[r0 + i];
            }
        __syncthreads();  // the next round's loads follow this round's stores
    }
}
}  // namespace
}  // namespace zp

using namespace zp;

extern "C" size_t zp_score_workspace_size(const zp_cache_desc *D, int32_t n, int32_t Lmax) {
    if (!D || n < 0 || Lmax < 0) return 0;
    // X and rho, then the all-pairs redundancy's scratch
    return 2 * align_up((size_t)n * D->h_kv * Lmax * 4, 256) + all_pairs_workspace_size(n, D->h_kv, D->head_dim, Lmax);
}

// Validates the scoring arguments, fills `a` and launches the global-score and
// redundancy kernels (X and rho in the workspace); the caller launches the
// finish.  *launched = false when there is nothing to do (n or Lmax zero).
// With rho_in (lightning row sums given by the caller) nothing is launched and
// the workspace is not needed: the finish kernel forms X itself.
static zp_status launch_scores(const zp_cache_desc *D, const zp_score_params *P, const void *k_cache,
                               const int32_t *block_table, int32_t table_stride, const int32_t *seq_lens,
                               const uint8_t *first_compression, int32_t n, const zp_score_rows *attn,
                               const float *global_F, float *scores_out, int32_t Lmax, void *workspace,
                               size_t workspace_bytes, cudaStream_t st, ScoreArgs &a, DeviceInfo &dev,
                               bool *launched, int layers = 1, long long k_layer_elems = 0,
                               long long F_layer = 0, const zp_rho_rows *rho_in = nullptr) {
    *launched = false;
    zp_status rc = check_desc(D);
    if (rc != ZP_OK) return rc;
    if (!P) return fail(ZP_ERR_INVALID_ARG, "score: NULL params");
    if (n < 0 || Lmax < 0 || table_stride < 1) return fail(ZP_ERR_INVALID_ARG, "score: bad sizes");
    if (n == 0 || Lmax == 0) return ok();
    if (!block_table || !seq_lens || (!workspace && !rho_in))
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
    const bool all_pairs = P->use_similarity && !P->lightning;
    if (all_pairs && !(D->head_dim == 64 || D->head_dim == 128))
        return fail(ZP_ERR_SHAPE, "score: the all-pairs redundancy needs head_dim 64 or 128");
    if (all_pairs && D->dtype == ZP_BF16 && D->block_size % 16)
        return fail(ZP_ERR_SHAPE, "score: the all-pairs redundancy of bf16 keys needs b a multiple of 16");
    if (P->use_similarity && P->lightning && D->block_size > 16)
        return fail(ZP_ERR_SHAPE, "score: lightning kernel supports b <= 16 (b=%d)", D->block_size);
    const size_t need = (size_t)layers * zp_score_workspace_size(D, n, Lmax);
    if (!rho_in && workspace_bytes < need)
        return fail(ZP_ERR_CAPACITY, "score: workspace %zu < %zu", workspace_bytes, need);
    if (rho_in) {
        if (!(P->use_similarity && P->lightning && D->dtype == ZP_BF16 && D->block_size == 16))
            return fail(ZP_ERR_SHAPE, "score: given row sums need bf16 keys, b = 16 and the lightning redundancy");
        if (!rho_in->data || rho_in->stride < 1 || rho_in->n_rows < 1 ||
            (layers > 1 && rho_in->layer_stride < (long long)rho_in->n_rows * D->h_kv * rho_in->stride))
            return fail(ZP_ERR_INVALID_ARG, "score: bad redundancy rows");
    }
    rc = device_info(&dev);
    if (rc != ZP_OK) return rc;
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
    a.X_layer = (long long)n * D->h_kv * Lmax;
    a.X = reinterpret_cast<float *>(ws);
    a.rho = reinterpret_cast<float *>(ws + align_up((size_t)layers * a.X_layer * 4, 256));
    a.rho_in = rho_in ? rho_in->data : nullptr;
    a.rho_stride = rho_in ? rho_in->stride : 0;
    a.rho_layer = rho_in ? rho_in->layer_stride : 0;
    a.rho_rows = rho_in ? rho_in->rows : nullptr;
    a.n_rho_rows = rho_in ? rho_in->n_rows : 0;
    a.k_layer_bytes = k_layer_elems * elem_bytes(D->dtype);
    a.S_layer = attn->layer_stride;
    a.F_layer = F_layer;
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
    if (rho_in) {
        *launched = true;
        return ok();
    }
    if (a.use_sim && P->lightning && D->dtype == ZP_BF16 && a.b == 16 && (a.d == 64 || a.d == 128) &&
        a.h_kv <= 16 && reinterpret_cast<uintptr_t>(k_cache) % 16 == 0) {
        // global score and redundancy of each block in one kernel
        const size_t smem = (size_t)(16 / kStageRows) * (kStageRows * a.h_kv * a.d * 2 + 16);  // staged groups
        dim3 g2((Lmax + 15) / 16, n, layers);
        auto kern = a.d == 128 ? global_lightning_kernel<128> : global_lightning_kernel<64>;
        zp_status rs = set_max_dynamic_smem(reinterpret_cast<const void *>(kern), smem,
                                            "score: global/lightning shared-memory attribute");
        if (rs != ZP_OK) return rs;
        // programmatic dependent launch: the CTAs may start on SMs that the
        // preceding kernel has left and fetch their keys while it drains
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = g2;
        cfg.blockDim = dim3(a.h_kv * 32);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a);
        if (e != cudaSuccess) return cuda_fail(e, "score: global/lightning launch");
        *launched = true;
        return ok();
    }
    if (layers != 1) return fail(ZP_ERR_SHAPE, "score: several layers per call need bf16 keys and b = 16");
    dim3 g1((Lmax + kTile - 1) / kTile, n);
    gather_global_kernel<<<g1, 256, 0, st>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "score: gather launch");
    if (all_pairs) {
        AllPairsArgs ap;
        ap.k = k_cache;
        ap.dtype = D->dtype;
        ap.table = block_table;
        ap.table_stride = table_stride;
        ap.seq_lens = seq_lens;
        ap.n = n;
        ap.h_kv = a.h_kv;
        ap.d = a.d;
        ap.b = a.b;
        ap.n_total = a.n_total;
        ap.Lmax = Lmax;
        long long cap = Lmax;
        if ((long long)table_stride * a.b < cap) cap = (long long)table_stride * a.b;
        if (a.S_stride < cap) cap = a.S_stride;
        ap.Lcap = (int)cap;
        ap.p = a.p;
        ap.rho = a.rho;
        ap.workspace = reinterpret_cast<unsigned char *>(a.rho) + align_up((size_t)a.X_layer * 4, 256);
        zp_status rs = launch_all_pairs(ap, st);
        if (rs != ZP_OK) return rs;
    } else if (a.use_sim) {
        dim3 g2((Lmax + a.b - 1) / a.b, n);
        const size_t smem = (size_t)a.h_kv * a.b * (a.d + 1) * 4;
        if (smem > (size_t)dev.smem_optin) return fail(ZP_ERR_SHAPE, "score: block of keys too large");
        if (D->dtype == ZP_BF16 && a.b == 16 && (a.d == 64 || a.d == 128)) {
            const size_t smem_tc = (size_t)a.h_kv * (a.d / 64) * 16 * 128;
            const void *lk = a.d == 128 ? reinterpret_cast<const void *>(lightning_tc_kernel<128>)
                                        : reinterpret_cast<const void *>(lightning_tc_kernel<64>);
            zp_status rs = set_max_dynamic_smem(lk, smem_tc, "score: lightning shared-memory attribute");
            if (rs != ZP_OK) return rs;
            if (a.d == 128) lightning_tc_kernel<128><<<g2, a.h_kv * 32, smem_tc, st>>>(a);
            else lightning_tc_kernel<64><<<g2, a.h_kv * 32, smem_tc, st>>>(a);
        } else if (D->dtype == ZP_BF16) {
            zp_status rs = set_max_dynamic_smem(reinterpret_cast<const void *>(lightning_kernel<__nv_bfloat16>), smem,
                                                "score: lightning shared-memory attribute");
            if (rs != ZP_OK) return rs;
            lightning_kernel<__nv_bfloat16><<<g2, a.h_kv * 32, smem, st>>>(a);
        } else {
            zp_status rs = set_max_dynamic_smem(reinterpret_cast<const void *>(lightning_kernel<float>), smem,
                                                "score: lightning shared-memory attribute");
            if (rs != ZP_OK) return rs;
            lightning_kernel<float><<<g2, a.h_kv * 32, smem, st>>>(a);
        }
        e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e, "score: lightning launch");
    }
    *launched = true;
    return ok();
}

extern "C" zp_status zp_score_tokens(const zp_cache_desc *D, const zp_score_params *P,
                                     const void *k_cache, const int32_t *block_table,
                                     int32_t table_stride, const int32_t *seq_lens,
                                     const uint8_t *first_compression, int32_t n,
                                     const zp_score_rows *attn, const float *global_F,
                                     float *scores_out,
                                     int32_t Lmax, void *workspace, size_t workspace_bytes,
                                     void *stream) {
    if (!scores_out && n > 0 && Lmax > 0) return fail(ZP_ERR_INVALID_ARG, "score: NULL scores_out");
    ScoreArgs a;
    DeviceInfo dev;
    bool launched;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    zp_status rc = launch_scores(D, P, k_cache, block_table, table_stride, seq_lens, first_compression, n, attn,
                                 global_F, scores_out, Lmax, workspace, workspace_bytes, st, a, dev, &launched);
    if (rc != ZP_OK || !launched) return rc;
    dim3 g3(a.h_kv, n);
    finalize_kernel<<<g3, 1024, 0, st>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "score: finalize launch");
    return ok();
}

extern "C" size_t zp_compress_workspace_size(const zp_cache_desc *D, int32_t n, int32_t Lmax,
                                             int32_t layer_count) {
    if (layer_count < 1) return 0;
    return (size_t)layer_count * zp_score_workspace_size(D, n, Lmax);
}


static zp_status compress_impl(const zp_cache_desc *D, const zp_score_params *P, void *k_base, void *v_base,
                               int64_t layer_stride, int32_t layer_count, const int32_t *block_table,
                               int32_t table_stride, const int32_t *seq_lens, const uint8_t *first_compression,
                               int32_t n, const zp_score_rows *attn, float *global_F, int64_t F_layer_stride,
                               const int32_t *dst_targets, int32_t target_stride, int32_t k, const int32_t *k_seq,
                               int32_t *keep_idx, int32_t *tie_count, float *scores_out, int32_t Lmax,
                               void *workspace, size_t workspace_bytes, void *stream, const zp_rho_rows *rho) {
    zp_status rc = check_desc(D);
    if (rc != ZP_OK) return rc;
    if (n < 0 || k < 0 || Lmax < 0 || target_stride < 1 || layer_count < 0)
        return fail(ZP_ERR_INVALID_ARG, "compress: bad sizes");
    if (n == 0 || k == 0 || layer_count == 0) return ok();
    if (!k_base || !v_base || !dst_targets || !keep_idx || !attn)
        return fail(ZP_ERR_INVALID_ARG, "compress: NULL buffer");
    if ((long long)target_stride * D->block_size < k)
        return fail(ZP_ERR_CAPACITY, "compress: %d target blocks hold fewer than k=%d rows", target_stride, k);
    const int es = elem_bytes(D->dtype);
    const size_t row_bytes = (size_t)D->head_dim * es;
    if (row_bytes % 16) return fail(ZP_ERR_SHAPE, "compress: row of %zu bytes", row_bytes);
    const long long per_layer = (long long)D->n_total_blocks * D->block_size * D->h_kv * D->head_dim;
    if (layer_count > 1 && (layer_stride < per_layer || (layer_stride * es) % 16))
        return fail(ZP_ERR_INVALID_ARG, "compress: layer_stride %lld", (long long)layer_stride);
    if (((uintptr_t)k_base | (uintptr_t)v_base) % 16) return fail(ZP_ERR_INVALID_ARG, "compress: unaligned cache");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t ws_layer = zp_score_workspace_size(D, n, Lmax);
    const size_t out_layer = (size_t)n * D->h_kv * Lmax;
    const size_t keep_layer = (size_t)n * D->h_kv * k;
    DeviceInfo dev;
    rc = device_info(&dev);
    if (rc != ZP_OK) return rc;
    const int row_vec = (int)(row_bytes / 16);
    const size_t smem = fused_smem(Lmax, k, D->block_size);
    const bool fused_ok = fused_finish_fits(D, P, Lmax, k, (size_t)dev.smem_optin);
    if (rho && !fused_ok)
        return fail(ZP_ERR_SHAPE, "compress: given row sums need the one-kernel path (bf16, b = 16, lightning, "
                                  "%zu bytes of shared memory per row)", smem);
    if (fused_ok) {
        // every layer in one launch of each kernel (blockIdx.z = layer)
        ScoreArgs a;
        bool launched;
        rc = launch_scores(D, P, k_base, block_table, table_stride, seq_lens, first_compression, n, attn, global_F,
                           scores_out, Lmax, workspace, workspace_bytes, st, a, dev, &launched, layer_count,
                           layer_stride, F_layer_stride, rho);
        if (rc != ZP_OK || !launched) return rc;
        MoveArgs m;
        m.K = static_cast<uint4 *>(k_base);
        m.V = static_cast<uint4 *>(v_base);
        m.row_vec = row_vec;
        m.dst = dst_targets;
        m.target_stride = target_stride;
        m.k = k;
        m.k_seq = k_seq;
        m.keep = keep_idx;
        m.tie = tie_count;
        m.F = global_F;
        m.kv_layer_vec = layer_stride * es / 16;
        m.F_layer = F_layer_stride;
        auto kfin = rho ? finalize_select_move_kernel<true> : finalize_select_move_kernel<false>;
        zp_status rs = set_max_dynamic_smem(reinterpret_cast<const void *>(kfin), smem,
                                            "compress: shared-memory attribute");
        if (rs != ZP_OK) return rs;
        // programmatic dependent launch: the finish grid may start while the
        // kernel before it (the scores kernel, or with given row sums the
        // decode) drains; it reads that kernel's output only after
        // griddepcontrol.wait
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(a.h_kv, n, layer_count);
        cfg.blockDim = dim3(kFsThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cudaError_t e = cudaLaunchKernelEx(&cfg, kfin, a, m);
        if (e != cudaSuccess) return cuda_fail(e, "compress: launch");
        return ok();
    }
    // otherwise the three steps, one layer at a time (scores land in scores_out,
    // else in place of the row sums)
    if (workspace_bytes < (size_t)layer_count * ws_layer)
        return fail(ZP_ERR_CAPACITY, "compress: workspace %zu < %zu", workspace_bytes, (size_t)layer_count * ws_layer);
    for (int l = 0; l < layer_count; ++l) {
        zp_score_rows at = *attn;
        at.data = attn->data + (size_t)l * attn->layer_stride;
        at.layer_stride = 0;
        unsigned char *ws = static_cast<unsigned char *>(workspace) + (size_t)l * ws_layer;
        char *kl = static_cast<char *>(k_base) + (size_t)l * layer_stride * es;
        char *vl = static_cast<char *>(v_base) + (size_t)l * layer_stride * es;
        float *Fl = global_F ? global_F + (size_t)l * F_layer_stride : nullptr;
        ScoreArgs a;
        bool launched;
        rc = launch_scores(D, P, kl, block_table, table_stride, seq_lens, first_compression, n, &at, Fl,
                           scores_out ? scores_out + l * out_layer : nullptr, Lmax, ws, ws_layer, st, a, dev,
                           &launched);
        if (rc != ZP_OK) return rc;
        if (!launched) continue;
        if (!a.out) a.out = a.rho;
        finalize_kernel<<<dim3(a.h_kv, n), 1024, 0, st>>>(a);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e, "compress: finalize launch");
        rc = zp_select_topk(a.out, a.h_kv, Lmax, seq_lens, n, k, k_seq, keep_idx + l * keep_layer,
                            tie_count ? tie_count + (size_t)l * n * D->h_kv : nullptr, stream);
        if (rc != ZP_OK) return rc;
        rc = zp_compact_pages(D, kl, vl, 0, 1, Fl, 0, &at, block_table, table_stride, dst_targets, target_stride,
                              seq_lens, keep_idx + l * keep_layer, k, k_seq, n, stream);
        if (rc != ZP_OK) return rc;
    }
    return ok();
}

extern "C" int32_t zp_compress_rho_supported(const zp_cache_desc *D, const zp_score_params *P, int32_t Lmax,
                                             int32_t k) {
    if (check_desc(D) != ZP_OK || !P || Lmax < 0 || k < 0) return 0;
    DeviceInfo dev;
    if (device_info(&dev) != ZP_OK) return 0;
    return fused_finish_fits(D, P, Lmax, k, (size_t)dev.smem_optin);
}

extern "C" zp_status zp_compress_layers(const zp_cache_desc *D, const zp_score_params *P, void *k_base,
                                        void *v_base, int64_t layer_stride, int32_t layer_count,
                                        const int32_t *block_table, int32_t table_stride, const int32_t *seq_lens,
                                        const uint8_t *first_compression, int32_t n, const zp_score_rows *attn,
                                        float *global_F, int64_t F_layer_stride, const int32_t *dst_targets,
                                        int32_t target_stride, int32_t k, const int32_t *k_seq,
                                        int32_t *keep_idx, int32_t *tie_count,
                                        float *scores_out, int32_t Lmax, void *workspace, size_t workspace_bytes,
                                        void *stream) {
    return compress_impl(D, P, k_base, v_base, layer_stride, layer_count, block_table, table_stride, seq_lens,
                         first_compression, n, attn, global_F, F_layer_stride, dst_targets, target_stride, k, k_seq,
                         keep_idx, tie_count, scores_out, Lmax, workspace, workspace_bytes, stream, nullptr);
}

extern "C" zp_status zp_compress_layers_rho(const zp_cache_desc *D, const zp_score_params *P, void *k_base,
                                            void *v_base, int64_t layer_stride, int32_t layer_count,
                                            const int32_t *block_table, int32_t table_stride,
                                            const int32_t *seq_lens, const uint8_t *first_compression, int32_t n,
                                            const zp_score_rows *attn, float *global_F, int64_t F_layer_stride,
                                            const int32_t *dst_targets, int32_t target_stride, int32_t k,
                                            const int32_t *k_seq, int32_t *keep_idx, int32_t *tie_count,
                                            float *scores_out, int32_t Lmax, const zp_rho_rows *rho, void *stream) {
    if (!rho) return fail(ZP_ERR_INVALID_ARG, "compress: NULL redundancy rows");
    return compress_impl(D, P, k_base, v_base, layer_stride, layer_count, block_table, table_stride, seq_lens,
                         first_compression, n, attn, global_F, F_layer_stride, dst_targets, target_stride, k, k_seq,
                         keep_idx, tie_count, scores_out, Lmax, nullptr, 0, stream, rho);
}
