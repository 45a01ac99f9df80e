// decode_attn.cu -- paged GQA decode attention fused with the window score.
//
// Computes, for every sequence s and query head h (Zipage paper §3 paged
// cache, §6 decode attention on it):
//     out[s][h] = sum_{t<L_s} softmax_t(q[s][h] . k_t / sqrt(d)) v_t
// and, on observation-window steps, the per-token window score of App. C.2
// accumulated one decode step at a time (see zp_paged_decode_attn in zp.h).
//
// Design (HBM bound: ~4 flop per byte of K/V at a group of 4), common to both
// paths:
//   * Work unit = up to T tokens of one block of one sequence, all kv heads:
//     in the [N_total][b][h_kv][d] layout these are T*h_kv*d contiguous
//     elements, fetched by 1-D bulk copies (TMA engine) into a shared-memory
//     ring of S stages guarded by mbarriers.  K/V loads carry an L2
//     evict-first hint so the small scratch arrays stay resident.
//   * Stream-K split: the units of all sequences are concatenated and every
//     CTA (one per SM, persistent) takes an equal contiguous range, so ragged
//     lengths cannot unbalance the grid.  A sequence cut between CTAs leaves
//     per-CTA partial (max, sum, accumulator) records that are merged later.
//   * Warp specialisation: one producer warp issues the copies, consumer
//     warps do the products with an online softmax in base 2.
//   * Score: on window steps the logits (already in log2 units) go to a
//     scratch array; once a sequence's final max and sum are known they become
//     probabilities, the max over the GQA group is taken and 1/w of it is
//     added to (or at the first window row written into) the score row.
// bf16 caches (decode_tc_kernel): 16-token units copied a pair of token rows
// at a time, S = Q K^T and O^T += V^T P^T on the tensor cores (mma.sync), one
// cooperative launch whose epilogue merges the cut sequences and forms the
// window score (see the epilogue notes below), optionally with the lightning
// row sums of the sequences about to be compressed.
// fp32 caches (decode_main_kernel, small parity workloads): a half-warp per
// token row, packed fp32x2 FMAs and a butterfly reduce-scatter, then two more
// launches: decode_merge_kernel (one merger per cut sequence) and
// decode_score_kernel (the window score).
#include <math.h>

#include <mutex>

#include "lightning.cuh"
#include "zp_common.cuh"

namespace zp {
namespace {

constexpr int kMaxConsumerWarps = 16;
constexpr int kStageBytesCap = 32768;  // per tensor and stage
constexpr int kMaxB = 4096;
// A unit whose block also gets its lightning row sums costs the consumer warps
// about this much more than a plain one (sixteenths; per-CTA loop times of
// the 64-sequence Qwen3-8B layer fit 1.15-1.18); the stream-K split weighs
// such units accordingly so that the CTAs holding them finish with the rest.
constexpr int kRhoUnitWeight16 = 19;

struct DecodeArgs {
    const void *q;
    const void *k;
    const void *v;
    void *out;
    const int32_t *table;
    int table_stride;
    const int32_t *seq_lens;
    int B;
    int h_q, h_kv, b, n_total;
    int T;     // tokens per unit
    int upb;   // units per block = b / T
    int wph;   // consumer warps per kv head
    int ncw;   // consumer warps
    int stages;
    float qscale;  // log2(e) / sqrt(d)
    int want_score;
    int window;
    float *score;
    long long score_stride;  // elements between kv-head rows of S: table_stride * b
    const int32_t *score_rows;  // nullable [B]: row of S (query slot) of each batch entry, -1 = none
    int n_score_rows;           // rows of S when score_rows is set
    float *logits;     // [units * T][h_q]
    float2 *stats;     // [B][h_q] final (max, sum), log2 units
    float *part_acc;   // [2*grid][h_q][D]
    float2 *part_ml;   // [2*grid][h_q]
    int *unit_prefix;  // [B+1]
    int4 *unit_info;   // [units]: (sequence, first token, length, window flags) of every unit
    long long logits_units;  // capacity of `logits` in units
    unsigned long long *ctl;  // [B] per-sequence control words of the in-kernel merge (tensor-core path)
    // lightning redundancy of the sequences about to be compressed (tensor-core
    // path, b = 16): row sums of each block's cosine matrix per kv head
    float *rho;               // nullable: rho + (row * h_kv + kvh) * rho_stride + t
    long long rho_stride;
    const int32_t *rho_rows;  // [B]: row of each batch entry, -1 = none
    int n_rho_rows;
    float rho_p;              // similarity threshold p
    int rho_weight16;         // stream-K weight of a unit with row sums, in sixteenths of a plain unit
    unsigned *err;
};

// Reduce-scatter of V per-lane values over the 16 lanes of a half-warp (lane
// bits 3..0, high bit first).  Afterwards lane l holds in v[0..max(V/16,1))
// the full sums of indices l*(V/16)+i (V >= 16) or l/(16/V) (V < 16).
template <int N, int BIT>
struct ReduceScatter16 {
    template <int V>
    static __device__ __forceinline__ void run(float (&v)[V], int lane) {
        if constexpr (BIT >= 0) {
            if constexpr (N > 1) {
                constexpr int H = N / 2;
                const bool up = (lane >> BIT) & 1;
#pragma unroll
                for (int i = 0; i < H; ++i) {
                    const float send = up ? v[i] : v[i + H];
                    const float keep = up ? v[i + H] : v[i];
                    v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 1 << BIT);
                }
                ReduceScatter16<H, BIT - 1>::run(v, lane);
            } else {
                v[0] += __shfl_xor_sync(0xFFFFFFFFu, v[0], 1 << BIT);
                ReduceScatter16<1, BIT - 1>::run(v, lane);
            }
        }
    }
};

// DPL elements of a row (this lane's dims) as DPL/2 float pairs.
template <typename T, int DPL>
__device__ __forceinline__ void load_row(const T *p, float2 (&o)[DPL / 2]) {
    if constexpr (sizeof(T) == 2) {
        if constexpr (DPL == 8) {
            const uint4 w = *reinterpret_cast<const uint4 *>(p);
            o[0] = bf2_to_f2(w.x);
            o[1] = bf2_to_f2(w.y);
            o[2] = bf2_to_f2(w.z);
            o[3] = bf2_to_f2(w.w);
        } else {
            static_assert(DPL == 4, "bf16 rows: d in {64, 128}");
            const uint2 w = *reinterpret_cast<const uint2 *>(p);
            o[0] = bf2_to_f2(w.x);
            o[1] = bf2_to_f2(w.y);
        }
    } else {
#pragma unroll
        for (int i = 0; i < DPL / 4; ++i) {
            const float4 w = reinterpret_cast<const float4 *>(p)[i];
            o[2 * i] = make_float2(w.x, w.y);
            o[2 * i + 1] = make_float2(w.z, w.w);
        }
    }
}

template <typename T, int DPL>
__device__ __forceinline__ void store_row(T *p, const float2 (&o)[DPL / 2], float scale) {
    if constexpr (sizeof(T) == 2) {
        uint32_t w[DPL / 2];
#pragma unroll
        for (int i = 0; i < DPL / 2; ++i) w[i] = f2_to_bf2(o[i].x * scale, o[i].y * scale);
        if constexpr (DPL == 8) {
            *reinterpret_cast<uint4 *>(p) = make_uint4(w[0], w[1], w[2], w[3]);
        } else {
            *reinterpret_cast<uint2 *>(p) = make_uint2(w[0], w[1]);
        }
    } else {
#pragma unroll
        for (int i = 0; i < DPL / 4; ++i)
            reinterpret_cast<float4 *>(p)[i] = make_float4(o[2 * i].x * scale, o[2 * i].y * scale,
                                                           o[2 * i + 1].x * scale,
                                                           o[2 * i + 1].y * scale);
    }
}

__device__ __forceinline__ long long cta_start(int c, long long U, int G) {
    return (long long)c * U / G;
}

// CTA whose range [start(c), start(c+1)) holds unit u.
__device__ __forceinline__ int cta_of(long long u, long long U, int G) {
    int c = (int)((u * G) / U);
    if (c >= G) c = G - 1;
    while (c + 1 < G && cta_start(c + 1, U, G) <= u) ++c;
    while (c > 0 && cta_start(c, U, G) > u) --c;
    return c;
}

// Row of S that batch entry s scores into: its query slot when a slot map is
// given (-1: the entry holds no slot and is not scored), else s.  A slot
// outside [0, n_score_rows) is recorded as an error and not scored.
__device__ __forceinline__ int score_row_of(const DecodeArgs &a, int s) {
    if (!a.score_rows) return s;
    const int r = __ldg(&a.score_rows[s]);
    if (r >= a.n_score_rows) {
        record_error(a.err, ZP_ERR_DEVICE, 0x21);
        return -1;
    }
    return r < 0 ? -1 : r;
}

// Record of one unit for the score epilogue: sequence, first token, length
// and flags (bit 0: the sequence is on a window step, bit 1: first window row).
__device__ __forceinline__ int4 unit_record(const DecodeArgs &a, int s, int tok0, int L) {
    const int P = L - 1;
    const int r = P >= 0 ? P % a.b : -1;
    const int win = (P >= 0 && r >= a.b - a.window && score_row_of(a, s) >= 0) ? 1 : 0;
    const int first = (win && r == a.b - a.window) ? 2 : 0;
    return make_int4(s, tok0, L, win | first);
}

// Shared-memory layout (dynamic).
struct SmemLayout {
    int bar_off;      // 2*stages mbarriers
    int ctl_off;      // small ints: abort flag, last-arriver flag
    int stage_off;    // stages * 2 * stage_bytes
    int warp_off;     // per consumer warp: p[8][G], m_new[G], alpha[G], l[G]
    int merge_off;    // (ncw - h_kv) * (G*D + 2G) floats
    int prefix_off;   // B+1 ints
    int lens_off;     // B ints
    int total;
};

__host__ __device__ inline SmemLayout make_layout(int stages, int stage_bytes, int ncw, int h_kv,
                                                  int G, int D, int B) {
    SmemLayout L;
    int off = 0;
    L.bar_off = off;
    off += 2 * stages * 8;
    L.ctl_off = off;
    off += 16;
    off = (off + 127) / 128 * 128;
    L.stage_off = off;
    off += stages * 2 * stage_bytes;
    L.warp_off = off;
    off += ncw * (8 * G + 3 * G) * 4;
    off = (off + 15) / 16 * 16;
    L.merge_off = off;
    off += (ncw - h_kv) * (G * D + 2 * G) * 4;
    off = (off + 15) / 16 * 16;
    L.prefix_off = off;
    off += (B + 1) * 4;
    L.lens_off = off;
    off += B * 4;
    L.total = (off + 127) / 128 * 128;
    return L;
}

template <typename T, int D, int G>
__global__ void __launch_bounds__(kMaxConsumerWarps * 32, 1)
    decode_main_kernel(const DecodeArgs a) {
    constexpr int DPL = D / 16;  // dims per lane (16 lanes per token row)
    constexpr int V = 4 * G;     // (token, head) partial sums per lane per half-warp step
    constexpr int NV = V >= 16 ? V / 16 : 1;
    extern __shared__ __align__(128) unsigned char smem[];

    const int B = a.B;
    const int TU = a.T;
    const int stage_bytes = TU * a.h_kv * D * (int)sizeof(T);
    const SmemLayout lay = make_layout(a.stages, stage_bytes, a.ncw, a.h_kv, G, D, B);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + lay.bar_off);
    uint64_t *empty = full + a.stages;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + lay.ctl_off);
    int *prefix = reinterpret_cast<int *>(smem + lay.prefix_off);
    int *lens = reinterpret_cast<int *>(smem + lay.lens_off);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;

    // ---- unit prefix over sequences: n_units(s) = ceil(L_s / T)
    for (int s = tid; s < B; s += blockDim.x) {
        int L = a.seq_lens[s];
        if (L < 0) {
            record_error(a.err, ZP_ERR_DEVICE, 1);
            L = 0;
        }
        const int maxL = a.table_stride * a.b;
        if (L > maxL) {
            record_error(a.err, ZP_ERR_DEVICE, 2);
            L = maxL;
        }
        lens[s] = L;
    }
    if (tid == 0) {
        abort_flag[0] = 0;
        abort_flag[1] = 0;
        for (int i = 0; i < a.stages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], a.ncw);
        }
        fence_barrier_init();
    }
    __syncthreads();
    // block-wide exclusive scan of unit counts (B <= 4096, serial chunks per warp 0)
    if (warp == 0) {
        int carry = 0;
        for (int base = 0; base < B; base += 32) {
            const int s = base + lane;
            const int n = s < B ? (lens[s] + TU - 1) / TU : 0;
            int x = n;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
                if (lane >= o) x += y;
            }
            if (s < B) prefix[s] = carry + x - n;
            carry += __shfl_sync(0xFFFFFFFFu, x, 31);
        }
        if (lane == 0) prefix[B] = carry;
    }
    __syncthreads();
    const long long U = prefix[B];
    if (blockIdx.x == 0) {
        for (int s = tid; s <= B; s += blockDim.x) a.unit_prefix[s] = prefix[s];
    }
    if (a.want_score && U > a.logits_units) {
        if (tid == 0) record_error(a.err, ZP_ERR_DEVICE, 3);
        return;
    }
    const int Gd = gridDim.x;
    const long long u0 = cta_start(blockIdx.x, U, Gd);
    const long long u1 = cta_start(blockIdx.x + 1, U, Gd);
    if (u0 >= u1) return;

    // first sequence of the range: largest s with prefix[s] <= u0
    int s_first = 0;
    {
        int lo = 0, hi = B - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (prefix[mid] <= u0) lo = mid;
            else hi = mid - 1;
        }
        s_first = lo;
    }

    unsigned char *stage_base = smem + lay.stage_off;
    const int row_elems = a.h_kv * D;

    // =====================================================================
    // Copies are issued by lane 0 of warp 0 (no dedicated producer warp: a
    // 17th warp would cap every thread at 96 registers).  Unit i of the range
    // goes to stage i % stages; the stage is refilled once all consumer warps
    // have released it (empty barrier), so up to stages-1 units are in flight
    // ahead of the slowest warp.
    const uint64_t pol = l2_evict_first_policy();
    int ps = s_first;  // sequence of the next unit to issue (lane 0 of warp 0 only)
    auto issue = [&](long long i) {
        const long long u = u0 + i;
        while (u >= prefix[ps + 1]) ++ps;
        const int st = (int)(i % a.stages);
        const int j = (int)(u - prefix[ps]);
        const int tok0 = j * TU;
        int valid = lens[ps] - tok0;
        if (valid > TU) valid = TU;
        const int blk = __ldg(&a.table[(size_t)ps * a.table_stride + tok0 / a.b]);
        if (a.want_score) a.unit_info[u] = unit_record(a, ps, tok0, lens[ps]);
        unsigned char *ks = stage_base + (size_t)st * 2 * stage_bytes;
        unsigned char *vs = ks + stage_bytes;
        if (blk < 0 || blk >= a.n_total) {
            record_error(a.err, ZP_ERR_DEVICE, 4);
            mbar_arrive_expect_tx(&full[st], 0);
        } else {
            const unsigned bytes = (unsigned)(valid * row_elems * (int)sizeof(T));
            const size_t off = ((size_t)blk * a.b + (tok0 % a.b)) * row_elems;
            mbar_arrive_expect_tx(&full[st], 2 * bytes);
            bulk_g2s(ks, static_cast<const T *>(a.k) + off, bytes, &full[st], pol);
            bulk_g2s(vs, static_cast<const T *>(a.v) + off, bytes, &full[st], pol);
        }
    };
    const long long n_units = u1 - u0;
    if (tid == 0) {
        for (long long i = 0; i < n_units && i < a.stages; ++i) issue(i);
    }

    // =====================================================================
    // consumer warps
    const int ncw_threads = a.ncw * 32;
    const int kvh = warp / a.wph;
    const int wih = warp % a.wph;
    const int lane16 = lane & 15;
    const int half = lane >> 4;
    const int TPW = TU / a.wph;
    float *wsm = reinterpret_cast<float *>(smem + lay.warp_off) + warp * (11 * G);
    float *sp = wsm;               // p[8][G]
    float *ctl_m = wsm + 8 * G;    // m_new[G]
    float *ctl_a = ctl_m + G;      // alpha[G]
    float *ctl_l = ctl_a + G;      // l[G]
    float *merge = reinterpret_cast<float *>(smem + lay.merge_off);
    const int h0 = kvh * G;

    // value i of this lane: head index and "writer / owner" roles
    int jv[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int idx = V >= 16 ? lane16 * NV + i : lane16 / (16 / V);
        jv[i] = idx % G;
    }
    const bool writer = V >= 16 ? true : (lane16 % (16 / V)) == 0;
    const bool owner = writer && ((lane & 0x1C) == 0);
    const int tok_in_step = half * 4 + (lane16 >> 2);

    float2 qv[G][DPL / 2];
    float2 acc[G][DPL / 2];
    float m[G];
    float l_own[NV];

    auto reset_state = [&]() {
#pragma unroll
        for (int j = 0; j < G; ++j) {
            m[j] = -INFINITY;
#pragma unroll
            for (int p = 0; p < DPL / 2; ++p) acc[j][p] = make_float2(0.f, 0.f);
        }
#pragma unroll
        for (int i = 0; i < NV; ++i) l_own[i] = 0.f;
    };
    auto load_q = [&](int s) {
        const T *qg = static_cast<const T *>(a.q) + ((size_t)s * a.h_q + h0) * D + lane16 * DPL;
#pragma unroll
        for (int j = 0; j < G; ++j) {
            float2 t2[DPL / 2];
            load_row<T, DPL>(qg + (size_t)j * D, t2);
#pragma unroll
            for (int p = 0; p < DPL / 2; ++p)
                qv[j][p] = make_float2(t2[p].x * a.qscale, t2[p].y * a.qscale);
        }
    };

    int s = s_first;
    long long seg_begin = u0;
    reset_state();
    load_q(s);
    bool window_step = false;
    auto compute_window = [&](int seq) {
        const int P = lens[seq] - 1;
        return a.want_score && P >= 0 && (P % a.b) >= a.b - a.window && score_row_of(a, seq) >= 0;
    };
    window_step = compute_window(s);

    for (long long u = u0, i = 0; u < u1; ++u, ++i) {
        const int st = (int)(i % a.stages);
        const bool got = mbar_wait_bounded(&full[st], (unsigned)((i / a.stages) & 1), a.err,
                                           abort_flag, 20);
        const int j_unit = (int)(u - prefix[s]);
        int valid = lens[s] - j_unit * TU;
        if (valid > TU) valid = TU;
        if (!got) valid = 0;
        const T *ks = reinterpret_cast<const T *>(stage_base + (size_t)st * 2 * stage_bytes);
        const T *vs = reinterpret_cast<const T *>(stage_base + (size_t)st * 2 * stage_bytes +
                                                  stage_bytes);

        for (int step = 0; step < TPW / 8; ++step) {
            const int tok_base = wih * TPW + step * 8;  // token index within the unit
            if (tok_base >= valid) break;  // warp-uniform
            // ---- logits for 4 tokens of this half-warp
            float v[V];
#pragma unroll
            for (int i4 = 0; i4 < 4; ++i4) {
                const int tok = tok_base + half * 4 + i4;
                float2 kk[DPL / 2];
                load_row<T, DPL>(ks + ((size_t)tok * a.h_kv + kvh) * D + lane16 * DPL, kk);
#pragma unroll
                for (int j = 0; j < G; ++j) {
                    float2 acc2 = make_float2(0.f, 0.f);
#pragma unroll
                    for (int p = 0; p < DPL / 2; ++p) acc2 = ffma2(qv[j][p], kk[p], acc2);
                    v[i4 * G + j] = acc2.x + acc2.y;
                }
            }
            ReduceScatter16<V, 3>::run(v, lane16);
            const int tok = tok_base + tok_in_step;
            const bool tvalid = tok < valid;
            float sc[NV], mx[NV];
#pragma unroll
            for (int i2 = 0; i2 < NV; ++i2) {
                sc[i2] = tvalid ? v[i2] : -INFINITY;
                mx[i2] = sc[i2];
                mx[i2] = warp_max_xor(mx[i2], 4);
                mx[i2] = warp_max_xor(mx[i2], 8);
                mx[i2] = warp_max_xor(mx[i2], 16);
            }
            if (window_step && writer && tvalid) {
                float *lg = a.logits + ((size_t)u * TU + tok) * a.h_q + h0;
#pragma unroll
                for (int i2 = 0; i2 < NV; ++i2) lg[jv[i2]] = sc[i2];
            }
            if (owner) {
#pragma unroll
                for (int i2 = 0; i2 < NV; ++i2) {
                    const int j = jv[i2];
                    const float mo = m[j];
                    const float mn = fmaxf(mo, mx[i2]);
                    ctl_m[j] = mn;
                    ctl_a[j] = (mn == -INFINITY) ? 1.f : exp2f(mo - mn);
                }
            }
            __syncwarp();
            float alpha[G];
#pragma unroll
            for (int j = 0; j < G; ++j) {
                m[j] = ctl_m[j];
                alpha[j] = ctl_a[j];
            }
            float pr[NV], ps[NV];
#pragma unroll
            for (int i2 = 0; i2 < NV; ++i2) {
                pr[i2] = (sc[i2] == -INFINITY) ? 0.f : exp2f(sc[i2] - m[jv[i2]]);
                ps[i2] = pr[i2];
                ps[i2] += __shfl_xor_sync(0xFFFFFFFFu, ps[i2], 4);
                ps[i2] += __shfl_xor_sync(0xFFFFFFFFu, ps[i2], 8);
                ps[i2] += __shfl_xor_sync(0xFFFFFFFFu, ps[i2], 16);
                if (owner) l_own[i2] = l_own[i2] * alpha[jv[i2]] + ps[i2];
                if (writer) sp[tok_in_step * G + jv[i2]] = pr[i2];
            }
            __syncwarp();
            // ---- P V
#pragma unroll
            for (int j = 0; j < G; ++j) {
                const float2 a2 = make_float2(alpha[j], alpha[j]);
#pragma unroll
                for (int p = 0; p < DPL / 2; ++p) acc[j][p] = fmul2(acc[j][p], a2);
            }
#pragma unroll
            for (int i4 = 0; i4 < 4; ++i4) {
                const int tl = half * 4 + i4;
                if (tok_base + tl < valid) {
                    float2 vv[DPL / 2];
                    load_row<T, DPL>(vs + ((size_t)(tok_base + tl) * a.h_kv + kvh) * D + lane16 * DPL,
                                     vv);
#pragma unroll
                    for (int j = 0; j < G; ++j) {
                        const float pj = sp[tl * G + j];
                        const float2 p2 = make_float2(pj, pj);
#pragma unroll
                        for (int p = 0; p < DPL / 2; ++p) acc[j][p] = ffma2(vv[p], p2, acc[j][p]);
                    }
                }
            }
            __syncwarp();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
        if (tid == 0 && i + a.stages < n_units) {
            if (mbar_wait_bounded(&empty[st], (unsigned)((i / a.stages) & 1), a.err, abort_flag, 10))
                issue(i + a.stages);
        }

        // ---- end of a segment: this sequence ends here, or the CTA range ends
        const bool seq_ends = (u + 1 == prefix[s + 1]);
        if (seq_ends || u + 1 == u1) {
            // halves -> lanes 0..15
#pragma unroll
            for (int j = 0; j < G; ++j)
#pragma unroll
                for (int p = 0; p < DPL / 2; ++p) {
                    acc[j][p].x += __shfl_xor_sync(0xFFFFFFFFu, acc[j][p].x, 16);
                    acc[j][p].y += __shfl_xor_sync(0xFFFFFFFFu, acc[j][p].y, 16);
                }
            if (owner) {
#pragma unroll
                for (int i2 = 0; i2 < NV; ++i2) ctl_l[jv[i2]] = l_own[i2];
            }
            __syncwarp();
            float l[G];
#pragma unroll
            for (int j = 0; j < G; ++j) l[j] = ctl_l[j];

            // merge the WPH warps of a kv head into its leader (wih == 0)
            if (a.wph > 1) {
                if (wih > 0) {
                    float *mw = merge + (size_t)(kvh * (a.wph - 1) + (wih - 1)) * (G * D + 2 * G);
                    if (lane < 16) {
#pragma unroll
                        for (int j = 0; j < G; ++j)
#pragma unroll
                            for (int p = 0; p < DPL / 2; ++p)
                                reinterpret_cast<float2 *>(mw + j * D + lane16 * DPL)[p] = acc[j][p];
                    }
                    if (lane == 0) {
#pragma unroll
                        for (int j = 0; j < G; ++j) {
                            mw[G * D + j] = m[j];
                            mw[G * D + G + j] = l[j];
                        }
                    }
                }
                named_bar_sync(1, ncw_threads);
                if (wih == 0) {
                    for (int w2 = 1; w2 < a.wph; ++w2) {
                        const float *mw = merge + (size_t)(kvh * (a.wph - 1) + (w2 - 1)) * (G * D + 2 * G);
#pragma unroll
                        for (int j = 0; j < G; ++j) {
                            const float mo = mw[G * D + j];
                            const float lo = mw[G * D + G + j];
                            const float mn = fmaxf(m[j], mo);
                            const float f_self = (mn == -INFINITY) ? 0.f : exp2f(m[j] - mn);
                            const float f_oth = (mn == -INFINITY) ? 0.f : exp2f(mo - mn);
                            l[j] = l[j] * f_self + lo * f_oth;
                            m[j] = mn;
                            const float2 fs = make_float2(f_self, f_self);
                            const float2 fo = make_float2(f_oth, f_oth);
#pragma unroll
                            for (int p = 0; p < DPL / 2; ++p) {
                                const float2 ov =
                                    reinterpret_cast<const float2 *>(mw + j * D + lane16 * DPL)[p];
                                acc[j][p] = ffma2(ov, fo, fmul2(acc[j][p], fs));
                            }
                        }
                    }
                }
                named_bar_sync(1, ncw_threads);
            }

            const bool whole = (prefix[s] >= seg_begin) && seq_ends;
            if (whole) {
                if (wih == 0 && lane < 16) {
                    T *og = static_cast<T *>(a.out) + ((size_t)s * a.h_q + h0) * D + lane16 * DPL;
#pragma unroll
                    for (int j = 0; j < G; ++j) {
                        const float inv = l[j] > 0.f ? 1.f / l[j] : 0.f;
                        store_row<T, DPL>(og + (size_t)j * D, acc[j], inv);
                    }
                    if (a.want_score && lane == 0) {
#pragma unroll
                        for (int j = 0; j < G; ++j) a.stats[(size_t)s * a.h_q + h0 + j] = make_float2(m[j], l[j]);
                    }
                }
            } else {
                // partial record of this CTA for sequence s
                const int slot = 2 * blockIdx.x + ((prefix[s] <= u0) ? 0 : 1);
                if (wih == 0 && lane < 16) {
                    float *pa = a.part_acc + ((size_t)slot * a.h_q + h0) * D + lane16 * DPL;
#pragma unroll
                    for (int j = 0; j < G; ++j)
#pragma unroll
                        for (int p = 0; p < DPL / 2; ++p)
                            reinterpret_cast<float2 *>(pa + (size_t)j * D)[p] = acc[j][p];
                    if (lane == 0) {
#pragma unroll
                        for (int j = 0; j < G; ++j)
                            a.part_ml[(size_t)slot * a.h_q + h0 + j] = make_float2(m[j], l[j]);
                    }
                }
            }
            // next sequence (skipping empty ones)
            if (u + 1 < u1) {
                while (u + 1 >= prefix[s + 1]) ++s;
                seg_begin = u + 1;
                reset_state();
                load_q(s);
                window_step = compute_window(s);
            }
        }
    }

}

// Window-score epilogue: one block per unit, one thread per (kv head, token)
// of window-step sequences.  p_h(t) = 2^(logit - m_h) / l_h;
// S += (1/w) max over the group of p_h(t) (written instead of added at the
// first window row and for the newest token).  (m_h, l_h) are the sequence's
// final softmax statistics, written by the main kernel (sequences one CTA saw
// whole) or by the merge kernel (cut sequences).  S is the sequence's own row
// per kv head, indexed by token position: consecutive threads take
// consecutive tokens of one row.
template <int G>
__global__ void __launch_bounds__(128) decode_score_kernel(const DecodeArgs a) {
    const int u = blockIdx.x;
    const int U = __ldg(&a.unit_prefix[a.B]);
    const int4 info = a.unit_info[u];
    if (u >= U || !(info.w & 1)) return;
    const int s = info.x;
    const int L = info.z;
    const int P = L - 1;
    const bool first_row = (info.w & 2) != 0;
    const float inv_w = 1.f / (float)a.window;
    for (int it = threadIdx.x; it < a.T * a.h_kv; it += blockDim.x) {
        const int tl = it % a.T;
        const int kvh = it / a.T;
        const int tok = info.y + tl;
        if (tok >= L) continue;
        const float *lg = a.logits + ((size_t)u * a.T + tl) * a.h_q + kvh * G;
        const float2 *st = a.stats + (size_t)s * a.h_q + kvh * G;
        float x[G];
        float2 ml[G];
        if constexpr (G % 4 == 0) {
#pragma unroll
            for (int q4 = 0; q4 < G / 4; ++q4) {
                const float4 v = reinterpret_cast<const float4 *>(lg)[q4];
                x[4 * q4] = v.x;
                x[4 * q4 + 1] = v.y;
                x[4 * q4 + 2] = v.z;
                x[4 * q4 + 3] = v.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < G; ++j) x[j] = lg[j];
        }
#pragma unroll
        for (int j = 0; j < G; ++j) ml[j] = st[j];
        float best = 0.f;
#pragma unroll
        for (int j = 0; j < G; ++j) best = fmaxf(best, exp2f(x[j] - ml[j].x) / ml[j].y);
        const float c = best * inv_w;
        float *dst = a.score + ((size_t)score_row_of(a, s) * a.h_kv + kvh) * a.score_stride + tok;
        *dst = (first_row || tok == P) ? c : (*dst + c);
    }
}

// ===========================================================================
// Tensor-core decode for bf16 caches.
//
// Same stream-K unit distribution, merge and score epilogue as the kernel
// above, with both products on the tensor cores (mma.sync m16n8k16, bf16 in,
// fp32 accumulate):
//   S  = Q_g K^T : A = the group's queries (rows = q heads, padded to 16),
//                  B = 16 tokens of K (from shared memory by ldmatrix);
//   O^T += V^T P^T: A = V^T (ldmatrix.trans), B = P^T, which is exactly the
//                  fragment the first product leaves in each lane, so P never
//                  leaves the registers.
// Operands come from shared memory filled by a producer warp with 1-D bulk
// copies (TMA engine), one per PAIR of token rows of a unit: the row of one
// token holds all kv heads and is contiguous in HBM, so each unit is read in
// address order (per-head tensor boxes of 128-byte rows 2 KB apart measured
// ~20 % slower, 16-byte cp.async copies slower still), and a copy engine
// streams two-row copies ~4 % faster than one-row copies.  Pair j (tokens 2j,
// 2j + 1) lands at j * (2 row_bytes + 16): the eight even tokens (or the
// eight odd ones) an ldmatrix reads fall on eight different bank groups, so
// each 8-token operand tile is every other token -- the even tokens in the
// first n-tile of S, the odd in the second, and the k order of V^T P^T the
// same.  One consumer warp per kv head.  P is rounded to bf16 for the second
// product; the scores and the softmax statistics stay in fp32.
constexpr int kTcTokens = 16;     // tokens per unit
// Epilogue region of shared memory: 8 ints, an mbarrier, the CTA's last
// sequence (for the announcement), (max, 1/sum) of up to 64 q heads (before
// the announcement: the control words read ahead), up to kMaxSeg window
// segments {sequence, first token, end token, byte offset}, then the first
// unit of every CTA (grid + 1 long longs).
constexpr int kEpiStatsHeads = 64;  // q heads of one statistics slot; two slots (the two cut sequences)
constexpr int kEpiBar = 32, kEpiSLast = 40, kEpiStats = 48, kEpiSeg = 48 + 2 * kEpiStatsHeads * 8, kMaxSeg = 32;
constexpr int kEpiCst = kEpiSeg + kMaxSeg * 16;
constexpr int kTcPad = 16;        // bytes of padding after each staged group of token rows

// Staged unit: K then V, each as kTcTokens / kStageRows groups of kStageRows
// consecutive token rows of the block (one bulk copy each) followed by 16
// bytes of pad.  Token t sits at (t / kStageRows) * group_stride +
// (t % kStageRows) * row_bytes.
__host__ __device__ inline int tc_group_stride(int h_kv, int d) { return kStageRows * h_kv * d * 2 + kTcPad; }
constexpr int kTcGroups = kTcTokens / kStageRows;

__host__ __device__ inline SmemLayout make_tc_layout(int stages, int h_kv, int halves, int B, int grid) {
    SmemLayout L;
    int off = 0;
    L.bar_off = off;
    off += 2 * stages * 8;
    L.ctl_off = off;
    off += 16;
    off = (off + 1023) / 1024 * 1024;
    L.stage_off = off;
    off += stages * 2 * kTcGroups * tc_group_stride(h_kv, halves * 64);
    L.warp_off = off;
    L.merge_off = off;  // epilogue: see kEpi* offsets
    off += kEpiCst + (grid + 1) * 8;
    L.prefix_off = off;
    off += (B + 1) * 4;
    L.lens_off = off;
    off += B * 4;
    L.total = (off + 127) / 128 * 128 + 1024;  // + slack to align the base at run time
    return L;
}

// ---------------------------------------------------------------------------
// In-kernel epilogue of the tensor-core path (cooperative launch: every CTA is
// resident).  After its main loop a CTA announces its parts of the sequences
// cut between CTAs (at most its first and its last); the last arrival
// publishes the sequence.  Every CTA then works through its sequences: the
// final statistics of a cut sequence come from the part records once it is
// published (a bounded wait unless this CTA published it), each part-holder
// combines its slice of the output, and every CTA computes the window score
// of its own units.  An arrival never waits, so every publication happens.
//
// Per-sequence control word (64 bits): (kCtlTag << 16) | phase << 15 | count.
// Phase 0 counts arrivals; the last arrival sets phase 1 ("published": every
// part's record is written).
// A word without the tag -- zero, or memory never written -- and a published
// word left by an earlier call read as phase 0, count 0, so the workspace
// needs no clearing between calls.
constexpr unsigned long long kCtlTag = 0xC0DE5EC7A11Dull;  // 48 bits

__device__ __forceinline__ unsigned long long ctl_word(int phase, int count) {
    return (kCtlTag << 16) | ((unsigned long long)phase << 15) | (unsigned long long)count;
}
__device__ __forceinline__ bool ctl_valid(unsigned long long w) { return (w >> 16) == kCtlTag; }

// Release / acquire at GPU scope around the control words (the part records
// written before a release are visible to a thread after its acquire).
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
__device__ __forceinline__ unsigned long long ld_volatile_u64(const unsigned long long *p) {
    return *reinterpret_cast<const volatile unsigned long long *>(p);
}

// CTA owning unit u, from the table cst[0..G] of first units (binary search).
__device__ __forceinline__ int owner_of(long long u, const long long *cst, int G) {
    int lo = 0, hi = G - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (cst[mid] <= u) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// The CTAs that own units of [p0, p1): c_lo..c_hi, of which the returned
// number own at least one.
__device__ __forceinline__ int parts_of(long long p0, long long p1, const long long *cst, int G, int *c_lo,
                                        int *c_hi) {
    *c_lo = owner_of(p0, cst, G);
    *c_hi = owner_of(p1 - 1, cst, G);
    int n = 0;
    for (int c = *c_lo; c <= *c_hi; ++c) n += cst[c + 1] > cst[c] ? 1 : 0;
    return n;
}

// Announces one part; true for the last of n_parts, whose update publishes
// the sequence (every part's record is then in place).  A word left
// published by an earlier call counts as zero.  `cur` is the caller's guess
// of the word's value (read before the main loop): when no other part has
// arrived since, the first compare-and-swap succeeds -- one round trip.
__device__ bool ctl_arrive(unsigned long long *w, int n_parts, unsigned long long cur, unsigned *err) {
    for (int it = 0; it < 4096; ++it) {
        const int have = (ctl_valid(cur) && ((cur >> 15) & 1) == 0) ? (int)(cur & 0x7FFF) : 0;
        const bool last = have + 1 == n_parts;
        const unsigned long long prev = atomicCAS(w, cur, last ? ctl_word(1, 0) : ctl_word(0, have + 1));
        if (prev == cur) return last;
        cur = prev;
    }
    record_error(err, ZP_ERR_DEVICE, 6);
    return false;
}

// Waits (bounded) for the publication of the part records of up to two
// sequences (w0, w1; nullptr: none), polling both words together.  A word
// stays published after the call: the next call's first arrival counts a
// published word as zero.  Returns bit i set when word i is published (or
// absent); a timeout records an error.
__device__ unsigned ctl_wait_published2(const unsigned long long *w0, const unsigned long long *w1, unsigned *err) {
    const unsigned long long t0 = global_ns();
    bool p0 = w0 == nullptr, p1 = w1 == nullptr;
    while (true) {
        const unsigned long long v0 = p0 ? 0ull : ld_volatile_u64(w0);
        const unsigned long long v1 = p1 ? 0ull : ld_volatile_u64(w1);
        p0 = p0 || (ctl_valid(v0) && ((v0 >> 15) & 1));
        p1 = p1 || (ctl_valid(v1) && ((v1 >> 15) & 1));
        if (p0 && p1) break;
        if (global_ns() - t0 > kWaitLimitNs) {
            record_error(err, ZP_ERR_TIMEOUT, 50);
            break;
        }
        __nanosleep(32);
    }
    return (p0 ? 1u : 0u) | (p1 ? 2u : 0u);
}

// Merge of the partial records of the cut sequences this CTA finished last
// (at most two, ms[0..1], -1 when absent), in two phases so that the final
// statistics can be published before the outputs are combined:
//     M = max_j m_j,  w_j = 2^(m_j - M),  L = sum_j w_j l_j,  out = sum_j w_j acc_j / L.
// CTA c's record of s is slot 2c when s is the first sequence of c's range,
// else 2c + 1.  Other CTAs wrote the records: read through L2 (ld.cg).

// Part j of sequence s (p0 = its first unit): slot, or -1 for a CTA without units.
__device__ __forceinline__ int part_slot(int c_lo, int j, long long p0, const long long *cst) {
    const int c = c_lo + j;
    return cst[c + 1] > cst[c] ? 2 * c + (p0 > cst[c] ? 1 : 0) : -1;
}

// Final statistics of every head of cut sequence s from its part records, as
// c = M + log2 L into shared memory (one head per thread; the records are
// published; +inf for an empty sum).  Up to eight records are loaded
// together, then combined.
__device__ void part_stats(const DecodeArgs &a, int s, const int *prefix, const long long *cst, int Gd,
                           float *out, int ctid, int nthr) {
    const int h_q = a.h_q;
    for (int h = ctid; h < h_q; h += nthr) {
        const long long p0 = prefix[s];
        int c_lo, c_hi;
        parts_of(p0, prefix[s + 1], cst, Gd, &c_lo, &c_hi);
        const int nc = c_hi - c_lo + 1;
        float M = -INFINITY, Lsum = 0.f;
        for (int j0 = 0; j0 < nc; j0 += 8) {
            float2 v[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int sl = j0 + q < nc ? part_slot(c_lo, j0 + q, p0, cst) : -1;
                v[q] = sl < 0 ? make_float2(-INFINITY, 0.f) : __ldcg(&a.part_ml[(size_t)sl * h_q + h]);
            }
            float Mn = M;
#pragma unroll
            for (int q = 0; q < 8; ++q) Mn = fmaxf(Mn, v[q].x);
            if (Mn == -INFINITY) continue;
            Lsum = (M == -INFINITY) ? 0.f : Lsum * exp2f(M - Mn);
#pragma unroll
            for (int q = 0; q < 8; ++q)
                if (v[q].x != -INFINITY) Lsum += v[q].y * exp2f(v[q].x - Mn);
            M = Mn;
        }
        out[h] = Lsum > 0.f ? M + log2f(Lsum) : INFINITY;
    }
}

// Output of cut sequence s from its part records, the share of this CTA:
// the (head, 16 dims) items of the sequence are split evenly over the CTAs
// that hold a part of it (in CTA order), so every part-holder combines a
// slice once the sequence is published and no CTA combines the whole
// sequence alone.  Each item derives its head's statistics from the records
// it loads (online rescaling, four parts per round), so the merge needs no
// shared statistics and runs beside part_stats: threads [t0, nthr) take the
// items.  With all_items the CTA combines the whole output (used without the
// window score, where only the last arrival merges and nobody waits).
//     M = max_j m_j,  w_j = 2^(m_j - M),  out = sum_j w_j acc_j / sum_j w_j l_j.
template <int D>
__device__ void merge_slice(const DecodeArgs &a, int s, const int *prefix, const long long *cst, int Gd,
                            bool all_items, int ctid, int t0, int nthr) {
    if (ctid < t0) return;
    const int h_q = a.h_q;
    constexpr int CH = 16;
    const long long p0 = prefix[s];
    int c_lo, c_hi;
    int np = parts_of(p0, prefix[s + 1], cst, Gd, &c_lo, &c_hi);
    const int nc = c_hi - c_lo + 1;
    int j = 0;  // this CTA's index among the parts that hold units
    for (int c = c_lo; c < (int)blockIdx.x; ++c) j += cst[c + 1] > cst[c] ? 1 : 0;
    if (all_items) j = 0, np = 1;
    const int items = h_q * (D / CH);
    const int it_b = (int)((long long)j * items / np), it_e = (int)((long long)(j + 1) * items / np);
    for (int it = it_b + ctid - t0; it < it_e; it += nthr - t0) {
        const int h = it / (D / CH);
        const int d0 = (it % (D / CH)) * CH;
        float acc[CH];
#pragma unroll
        for (int k = 0; k < CH; ++k) acc[k] = 0.f;
        float M = -INFINITY, Lsum = 0.f;
        for (int j0 = 0; j0 < nc; j0 += 4) {  // four parts' loads in flight
            float2 ml[4];
            float4 x4[4][CH / 4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int sl = j0 + q < nc ? part_slot(c_lo, j0 + q, p0, cst) : -1;
                if (sl >= 0) {
                    ml[q] = __ldcg(&a.part_ml[(size_t)sl * h_q + h]);
                    const float4 *src =
                        reinterpret_cast<const float4 *>(a.part_acc + ((size_t)sl * h_q + h) * D + d0);
#pragma unroll
                    for (int q4 = 0; q4 < CH / 4; ++q4) x4[q][q4] = __ldcg(src + q4);
                } else {
                    ml[q] = make_float2(-INFINITY, 0.f);
#pragma unroll
                    for (int q4 = 0; q4 < CH / 4; ++q4) x4[q][q4] = make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
            float Mn = M;
#pragma unroll
            for (int q = 0; q < 4; ++q) Mn = fmaxf(Mn, ml[q].x);
            if (Mn == -INFINITY) continue;
            const float r = (M == -INFINITY) ? 0.f : exp2f(M - Mn);  // rescale of what is summed so far
            Lsum *= r;
#pragma unroll
            for (int k = 0; k < CH; ++k) acc[k] *= r;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float w = (ml[q].x == -INFINITY) ? 0.f : exp2f(ml[q].x - Mn);
                Lsum += w * ml[q].y;
#pragma unroll
                for (int q4 = 0; q4 < CH / 4; ++q4) {
                    acc[4 * q4] += w * x4[q][q4].x;
                    acc[4 * q4 + 1] += w * x4[q][q4].y;
                    acc[4 * q4 + 2] += w * x4[q][q4].z;
                    acc[4 * q4 + 3] += w * x4[q][q4].w;
                }
            }
            M = Mn;
        }
        const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
        uint32_t w4[CH / 2];
#pragma unroll
        for (int k = 0; k < CH / 2; ++k) w4[k] = f2_to_bf2(acc[2 * k] * inv, acc[2 * k + 1] * inv);
        uint4 *og = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(a.out) + ((size_t)s * h_q + h) * D + d0);
        og[0] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        og[1] = make_uint4(w4[4], w4[5], w4[6], w4[7]);
    }
}

// Window score of n tokens whose logits (lg_s [n16][HQ], log2 units, n16 the
// token count rounded up to 16) and score pieces (sc_s [HKV][RSF], token t of
// kv head h at h * RSF + t; RSF a multiple of 4, sc_s 16-byte aligned) are in
// shared memory; the pieces are updated in place:
//     piece[t] (+)= (1/w) max_{h in group} 2^(logit_h(t) - M_h) / L_h,
// written instead of added at the first window row and for the newest token
// (tok0 + t == P).  2^(x - M) / L = 2^(x - c) with c = M + log2 L (sm_c, one
// per q head; +inf gives a zero score), so the max over the group is taken on
// x - c and each (token, kv head) needs one exponential (the ISA's
// approximate one).  nthr is a multiple of HKV, so each thread keeps one kv
// head and its group's c in registers; it takes four consecutive tokens at a
// time (their logits rows exist up to n16), so that the four rows' loads and
// the pieces' one 16-byte load are in flight together.
template <int G, int HKV>
__device__ __forceinline__ void score_tokens_smem(const float *lg_s, float *sc_s, int RSF, int n, int tok0, int P,
                                                  bool first_row, float inv_w, const float *sm_c, int ctid,
                                                  int nthr) {
    constexpr int HQ = G * HKV;
    const int kvh = ctid % HKV;
    const int TS = nthr / HKV;
    float c[G];
#pragma unroll
    for (int j = 0; j < G; ++j) c[j] = sm_c[kvh * G + j];
    const float keep_old = first_row ? 0.f : 1.f;  // 0: the piece is written, not added to
    float *row = sc_s + kvh * RSF;
    for (int t4 = (ctid / HKV) * 4; t4 < n; t4 += 4 * TS) {
        float x[4][G];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float *lg = lg_s + (size_t)(t4 + u) * HQ + kvh * G;
            if constexpr (G % 4 == 0) {
#pragma unroll
                for (int q4 = 0; q4 < G / 4; ++q4) {
                    const float4 v = reinterpret_cast<const float4 *>(lg)[q4];
                    x[u][4 * q4] = v.x;
                    x[u][4 * q4 + 1] = v.y;
                    x[u][4 * q4 + 2] = v.z;
                    x[u][4 * q4 + 3] = v.w;
                }
            } else {
#pragma unroll
                for (int j = 0; j < G; ++j) x[u][j] = lg[j];
            }
        }
        const float4 old4 = *reinterpret_cast<const float4 *>(row + t4);
        float o[4] = {old4.x, old4.y, old4.z, old4.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            float e = -INFINITY;
#pragma unroll
            for (int j = 0; j < G; ++j) e = fmaxf(e, x[u][j] - c[j]);
            const int t = t4 + u;
            const float k = tok0 + t == P ? 0.f : keep_old;
            const float v = fmaf(ex2_approx(e), inv_w, o[u] * k);
            o[u] = t < n ? v : o[u];
        }
        *reinterpret_cast<float4 *>(row + t4) = make_float4(o[0], o[1], o[2], o[3]);
    }
}

// Window score of tokens [tb, te) of sequence s (tb a multiple of 16):
//     S[kvh][t] (+)= (1/w) max_{h in group(kvh)} 2^(logit_h(t) - M_h) / L_h
// written instead of added at the first window row and for t = P.  Chunks of
// CT tokens: the logits rows (contiguous) and the h_kv score-row pieces come
// into shared memory by bulk copies, are combined there, and the score pieces
// go back by bulk copies.  buf: shared memory of buf_bytes (16-aligned);
// sm_c: the sequence's c_h = M_h + log2 L_h, filled by the caller.
template <int G, int HKV>
__device__ void score_segment(const DecodeArgs &a, int s, int L, long long p0, int tb, int te, unsigned char *buf,
                              int buf_bytes, uint64_t *bar, unsigned &bar_phase, volatile int *abort,
                              const float *sm_c, int ctid, int nthr) {
    constexpr int HQ = G * HKV;
    const int P = L - 1;
    const bool first_row = (P % a.b) == a.b - a.window;
    const float inv_w = 1.f / (float)a.window;
    // chunk capacity: CT tokens of logits (HQ floats each) + HKV score pieces of CT + 4 floats
    int CT = (buf_bytes - HKV * 16) / (HQ * 4 + HKV * 4);
    CT &= ~15;
    const int RSF = CT + 4;  // score piece stride in floats (bank shift of 4 per kv head)
    float *lg_s = reinterpret_cast<float *>(buf);
    float *sc_s = lg_s + (size_t)CT * HQ;
    float *srow0 = a.score + (size_t)score_row_of(a, s) * HKV * a.score_stride;
    const float *lg_g = a.logits + ((size_t)p0 * kTcTokens) * HQ;
    fence_proxy_async_smem();  // earlier ordinary writes to buf precede the copies into it
    named_bar_sync(1, nthr);
    for (int c0 = tb; c0 < te; c0 += CT) {
        const int n = min(CT, te - c0);
        const int n16 = (n + 15) & ~15;  // whole units: in bounds of the logits and score rows
        if (ctid == 0) {
            mbar_arrive_expect_tx(bar, (unsigned)(n16 * HQ * 4 + HKV * n16 * 4));
            bulk_g2s_plain(lg_s, lg_g + (size_t)c0 * HQ, (unsigned)(n16 * HQ * 4), bar);
#pragma unroll
            for (int kvh = 0; kvh < HKV; ++kvh)
                bulk_g2s_plain(sc_s + kvh * RSF, srow0 + (size_t)kvh * a.score_stride + c0, (unsigned)(n16 * 4), bar);
        }
        const bool got = mbar_wait_bounded(bar, bar_phase, a.err, abort, 60);
        bar_phase ^= 1u;
        if (got) score_tokens_smem<G, HKV>(lg_s, sc_s, RSF, n, c0, P, first_row, inv_w, sm_c, ctid, nthr);
        fence_proxy_async_smem();
        named_bar_sync(1, nthr);
        if (ctid == 0) {
            if (got) {
#pragma unroll
                for (int kvh = 0; kvh < HKV; ++kvh)
                    bulk_s2g(srow0 + (size_t)kvh * a.score_stride + c0, sc_s + kvh * RSF, (unsigned)(n16 * 4));
                bulk_commit();
            }
            bulk_wait_read_all();  // the pieces may be overwritten by the next chunk
        }
        named_bar_sync(1, nthr);
    }
}

// Window score of a prefetched segment: tokens [tb, tb + n) of sequence s,
// logits lg_s [n16][HQ] and the score pieces sc_s [HKV][n16 + 4] already in
// shared memory; the pieces are updated there and written back by bulk
// copies (committed, not waited for) by thread ctid 0.  sm_c holds
// c_h = M_h + log2 L_h.  nthr threads (a multiple of HKV) take part; BAR is
// the named barrier they share.
template <int G, int HKV, int BAR = 1>
__device__ void score_prefetched(const DecodeArgs &a, int s, int L, int tb, int n, int n16, const float *lg_s,
                                 float *sc_s, const float *sm_c, int ctid, int nthr) {
    const int P = L - 1;
    const bool first_row = (P % a.b) == a.b - a.window;
    const float inv_w = 1.f / (float)a.window;
    const int RSF = n16 + 4;
    score_tokens_smem<G, HKV>(lg_s, sc_s, RSF, n, tb, P, first_row, inv_w, sm_c, ctid, nthr);
    fence_proxy_async_smem();
    named_bar_sync_id<BAR>(nthr);
    if (ctid == 0) {
        float *srow0 = a.score + (size_t)score_row_of(a, s) * HKV * a.score_stride;
#pragma unroll
        for (int kvh = 0; kvh < HKV; ++kvh)
            bulk_s2g(srow0 + (size_t)kvh * a.score_stride + tb, sc_s + kvh * RSF, (unsigned)(n16 * 4));
        bulk_commit();
    }
}

// A sequence cut between CTAs, as one CTA of its parts sees it in the epilogue:
// its tokens [tb, te) in this CTA, window segment kk, whether another CTA
// publishes it (wait) and whether this CTA scores tokens of it (seg).
struct CutSeq {
    int sq, L, tb, te, kk;
    long long pb;
    bool seg, wait;
};

template <int D, int G>
__global__ void __launch_bounds__(9 * 32, 1) decode_tc_kernel(const DecodeArgs a) {
    constexpr int HALVES = D / 64;
    constexpr int KS = D / 16;  // k-steps of Q K^T = m-tiles of V^T P^T
    static_assert(G >= 1 && G <= 8, "group of at most 8 q heads");
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    // A kernel launched after this one as its programmatic dependent (the
    // compression's first kernel) may be scheduled on the SMs this grid
    // leaves; it reads nothing this kernel writes before waiting for it.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int B = a.B;
    const int h_kv = a.h_kv;
    const SmemLayout lay = make_tc_layout(a.stages, h_kv, HALVES, B, gridDim.x);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + lay.bar_off);
    uint64_t *empty = full + a.stages;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + lay.ctl_off);
    int *prefix = reinterpret_cast<int *>(smem + lay.prefix_off);
    int *lens = reinterpret_cast<int *>(smem + lay.lens_off);
    // [0] -, [1..2] sequences to merge (-1: none), [3] broadcast, [4] cut parts, [5..6] their
    // sequences, [7] window segments (negative: not prefetched)
    int *mlist = reinterpret_cast<int *>(smem + lay.merge_off);
    uint64_t *ebar = reinterpret_cast<uint64_t *>(smem + lay.merge_off + kEpiBar);  // epilogue copies
    // per q head c = M + log2 L of the sequence being scored (two slots); before
    // the epilogue the same bytes hold the guessed control words
    float *sm_c = reinterpret_cast<float *>(smem + lay.merge_off + kEpiStats);
    unsigned long long *guess_words = reinterpret_cast<unsigned long long *>(smem + lay.merge_off + kEpiStats);
    int4 *segs = reinterpret_cast<int4 *>(smem + lay.merge_off + kEpiSeg);
    long long *cst = reinterpret_cast<long long *>(smem + lay.merge_off + kEpiCst);
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int RB = h_kv * D * 2;                       // bytes of one token row (every kv head)
    const int GS = tc_group_stride(h_kv, D);           // staged group stride
    const int stage_bytes = 2 * kTcGroups * GS;        // K groups then V groups
    // Weighted stream-K split (row sums requested): the weighted prefix
    // wpre[0..B] and the per-sequence unit weights wgt[0..B) sit in the stage
    // area, which no copy writes before the split is done.
    const bool weighted = a.rho && a.rho_weight16 != 16;
    int *wpre = reinterpret_cast<int *>(smem + lay.stage_off);
    int *wgt = wpre + (B + 1);

    for (int s = tid; s < B; s += blockDim.x) {
        int L = a.seq_lens[s];
        if (L < 0) {
            record_error(a.err, ZP_ERR_DEVICE, 1);
            L = 0;
        }
        const int maxL = a.table_stride * a.b;
        if (L > maxL) {
            record_error(a.err, ZP_ERR_DEVICE, 2);
            L = maxL;
        }
        lens[s] = L;
        if (weighted) wgt[s] = a.rho_rows[s] >= 0 ? a.rho_weight16 : 16;
    }
    if (tid == 0) {
        abort_flag[0] = 0;
        abort_flag[1] = 0;
        mlist[0] = 0;
        mlist[4] = 0;
        mbar_init(ebar, 1);
        for (int i = 0; i < a.stages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], h_kv);
        }
        fence_barrier_init();
    }
    __syncthreads();
    if (warp == 0) {
        // unit prefix, and with a weighted split the weighted prefix, in one pass
        int carry = 0, wcarry = 0;
        for (int base = 0; base < B; base += 32) {
            const int s = base + lane;
            const int n = s < B ? (lens[s] + kTcTokens - 1) / kTcTokens : 0;
            const int nw = (weighted && s < B) ? n * wgt[s] : 0;
            int x = n, xw = nw;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
                const int yw = __shfl_up_sync(0xFFFFFFFFu, xw, o);
                if (lane >= o) {
                    x += y;
                    xw += yw;
                }
            }
            if (s < B) {
                prefix[s] = carry + x - n;
                if (weighted) wpre[s] = wcarry + xw - nw;
            }
            carry += __shfl_sync(0xFFFFFFFFu, x, 31);
            wcarry += __shfl_sync(0xFFFFFFFFu, xw, 31);
        }
        if (lane == 0) {
            prefix[B] = carry;
            if (weighted) wpre[B] = wcarry;
        }
    }
    __syncthreads();
    const long long U = prefix[B];
    if (blockIdx.x == 0)
        for (int s = tid; s <= B; s += blockDim.x) a.unit_prefix[s] = prefix[s];
    if (weighted) {
        // Stream-K over weighted units: a unit of a sequence with row sums
        // weighs rho_weight16, a plain one 16.
        const long long W = wpre[B];
        for (int c = tid; c <= (int)gridDim.x; c += blockDim.x) {
            const long long target = (long long)c * W / gridDim.x;
            int lo = 0, hi = B;  // the last sequence whose weighted start is <= target
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (wpre[mid] <= target) lo = mid;
                else hi = mid - 1;
            }
            long long v = U;
            if (lo < B) {
                const int w = wgt[lo];
                v = prefix[lo] + (target - wpre[lo] + w - 1) / w;
                if (v > prefix[lo + 1]) v = prefix[lo + 1];
            }
            cst[c] = v;
        }
        fence_proxy_async_smem();  // these reads of the stage area precede the copies into it
    } else {
        for (int c = tid; c <= (int)gridDim.x; c += blockDim.x) cst[c] = cta_start(c, U, gridDim.x);
    }
    __syncthreads();
    if (a.want_score && U > a.logits_units) {
        if (tid == 0) record_error(a.err, ZP_ERR_DEVICE, 3);
        return;
    }
    const int Gd = gridDim.x;
    const long long u0 = cst[blockIdx.x];
    const long long u1 = cst[blockIdx.x + 1];
    if (u0 >= u1) return;
    int s_first = 0;
    {
        int lo = 0, hi = B - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (prefix[mid] <= u0) lo = mid;
            else hi = mid - 1;
        }
        s_first = lo;
    }
    unsigned char *stage_base = smem + lay.stage_off;

    // =====================================================================
    // producer warp: one bulk copy per token row (K rows by lanes 0..15, V rows
    // by lanes 16..31), after lane 0 has announced the unit's bytes
    if (warp == h_kv) {
        const uint64_t pol = l2_evict_first_policy();
        const unsigned row_bytes = (unsigned)(h_kv * D * 2);
        const __nv_bfloat16 *kg = static_cast<const __nv_bfloat16 *>(a.k);
        const __nv_bfloat16 *vg = static_cast<const __nv_bfloat16 *>(a.v);
        // the next unit's block id is loaded one iteration ahead
        int ns = s_first;
        while (u0 >= prefix[ns + 1]) ++ns;
        int cur_s = ns;
        int ntok0 = (int)(u0 - prefix[ns]) * kTcTokens;
        int nblk = __ldg(&a.table[(size_t)ns * a.table_stride + ntok0 / a.b]);
        for (long long u = u0, i = 0; u < u1; ++u, ++i) {
            const int tok0 = ntok0;
            const int blk = nblk;
            const int useq = cur_s;
            if (u + 1 < u1) {
                while (u + 1 >= prefix[ns + 1]) ++ns;
                ntok0 = (int)(u + 1 - prefix[ns]) * kTcTokens;
                nblk = __ldg(&a.table[(size_t)ns * a.table_stride + ntok0 / a.b]);
            }
            cur_s = ns;
            const int st = (int)(i % a.stages);
            if (i >= a.stages &&
                !mbar_wait_bounded(&empty[st], (unsigned)(((i / a.stages) - 1) & 1), a.err, abort_flag, 30))
                break;
            int valid = lens[useq] - tok0;
            if (valid > kTcTokens) valid = kTcTokens;
            const bool bad = blk < 0 || blk >= a.n_total;
            if (a.want_score && (u == u0 || tok0 == 0) && lane < h_kv) {
                // first unit of a segment on a window step: bring its score pieces into L2
                const int L = lens[useq], P = L - 1;
                const int row = score_row_of(a, useq);
                if ((P % a.b) >= a.b - a.window && row >= 0) {
                    const long long ue = prefix[useq + 1] < u1 ? prefix[useq + 1] : u1;
                    int te = (int)(ue - prefix[useq]) * kTcTokens;
                    if (te > L) te = L;
                    const unsigned bytes = (unsigned)(((te - tok0) * 4 + 15) & ~15);
                    bulk_prefetch_l2(a.score + ((size_t)row * h_kv + lane) * a.score_stride + tok0, bytes);
                }
            }
            if (lane == 0) {
                if (bad) record_error(a.err, ZP_ERR_DEVICE, 4);
                mbar_arrive_expect_tx(&full[st], bad ? 0u : 2u * valid * row_bytes);
            }
            __syncwarp();
            // lanes [0, kTcGroups): K groups, then V groups; group j holds
            // tokens [j R, j R + R) (fewer when the unit ends inside it)
            const int j = lane % kTcGroups;
            const int nrows = min(kStageRows, valid - kStageRows * j);
            if (!bad && lane < 2 * kTcGroups && nrows > 0) {
                const size_t off = ((size_t)blk * a.b + (tok0 % a.b) + kStageRows * j) * h_kv * D;
                unsigned char *dst = stage_base + (size_t)st * stage_bytes + (lane / kTcGroups) * kTcGroups * GS + j * GS;
                bulk_g2s(dst, (lane < kTcGroups ? kg : vg) + off, (unsigned)nrows * row_bytes, &full[st], pol);
            }
        }
        return;
    }

    // =====================================================================
    // consumer warp `warp` = kv head
    const int kvh = warp;
    const int g = lane >> 2;    // fragment row group
    const int tig = lane & 3;   // thread in group
    const int h0 = kvh * G;
    // ldmatrix address of this lane: matrix m = lane / 8 is operand tile
    // m / 2 (staged_token) at 16-byte chunk +(m & 1); its row i = lane % 8.
    const int lm = lane >> 3;
    const int li = lane & 7;
    const uint32_t loff = (uint32_t)((li / (kStageRows / 2)) * GS +
                                     (li % (kStageRows / 2) + (lm >> 1) * (kStageRows / 2)) * RB + (lm & 1) * 16);

    uint32_t qa[KS][2];
    float acc[KS][4];
    float m_run, l_run;
    auto reset_state = [&]() {
        m_run = -INFINITY;
        l_run = 0.f;
#pragma unroll
        for (int t = 0; t < KS; ++t)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[t][e] = 0.f;
    };
    auto load_q = [&](int s) {
        const uint32_t *qg = reinterpret_cast<const uint32_t *>(static_cast<const __nv_bfloat16 *>(a.q) +
                                                              ((size_t)s * a.h_q + h0 + g) * D);
#pragma unroll
        for (int t = 0; t < KS; ++t) {
            qa[t][0] = g < G ? qg[(16 * t + 2 * tig) / 2] : 0u;
            qa[t][1] = g < G ? qg[(16 * t + 8 + 2 * tig) / 2] : 0u;
        }
    };
    auto compute_window = [&](int seq) {
        const int P = lens[seq] - 1;
        return a.want_score && P >= 0 && (P % a.b) >= a.b - a.window && score_row_of(a, seq) >= 0;
    };
    // this sequence's row of lightning row sums, -1: none
    auto rho_row_of = [&](int seq) {
        if (!a.rho) return -1;
        const int r = a.rho_rows[seq];
        if (r >= a.n_rho_rows || (r >= 0 && lens[seq] > a.rho_stride)) {
            if (lane == 0) record_error(a.err, ZP_ERR_DEVICE, 0x22);
            return -1;
        }
        return r;
    };

    int s = s_first;
    long long seg_begin = u0;
    const uint64_t keep_pol = l2_evict_last_policy();
    reset_state();
    load_q(s);
    bool window_step = compute_window(s);
    int rho_row = rho_row_of(s);
    // The control words of the CTA's first and last sequence are read now (into
    // the epilogue's statistics area, unused until after the announcement), so
    // that announcing a part after the loop is usually one compare-and-swap.
    if (warp == 0 && lane < 2) {
        int s_last = s_first;
        while (u1 > prefix[s_last + 1]) ++s_last;
        if (lane == 0) *reinterpret_cast<int *>(smem + lay.merge_off + kEpiSLast) = s_last;
        guess_words[lane] = ld_volatile_u64(a.ctl + (lane ? s_last : s_first));
    }

    for (long long u = u0, i = 0; u < u1; ++u, ++i) {
        const int st = (int)(i % a.stages);
        const bool got = mbar_wait_bounded(&full[st], (unsigned)((i / a.stages) & 1), a.err, abort_flag, 40);
        int valid = lens[s] - (int)(u - prefix[s]) * kTcTokens;
        if (valid > kTcTokens) valid = kTcTokens;
        if (!got) valid = 0;
        unsigned char *ks = stage_base + (size_t)st * stage_bytes + kvh * D * 2;  // this head's columns
        unsigned char *vs = ks + kTcGroups * GS;
        if (valid > 0) {
            if (valid < kTcTokens) {
                // rows past the sequence end were not copied and hold stale
                // data: zero this head's part of them in V so that
                // 0 * garbage cannot produce a NaN
                for (int c = lane; c < (kTcTokens - valid) * (D / 8); c += 32) {
                    const int row = valid + c / (D / 8);
                    reinterpret_cast<uint4 *>(vs + (row / kStageRows) * GS + (row % kStageRows) * RB)[c % (D / 8)] =
                        make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();  // ordered before later bulk copies into this stage
                __syncwarp();
            }
            const uint32_t kt = smem_u32(ks);
            const uint32_t vt = smem_u32(vs);
            // ---- S = Q K^T for 16 tokens (two n-tiles of 8)
            float sc0[4] = {0.f, 0.f, 0.f, 0.f}, sc1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int t = 0; t < KS; ++t) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4(kt + loff + 32 * t, b0, b1, b2, b3);
                mma_16816(sc0, qa[t][0], 0u, qa[t][1], 0u, b0, b1);
                mma_16816(sc1, qa[t][0], 0u, qa[t][1], 0u, b2, b3);
            }
            // the n-tiles are the two operand tiles: lane holds S[head g] of
            // tile 0 rows 2tig, 2tig+1 (sc0) and tile 1 rows 2tig, 2tig+1
            // (sc1).  The k order of V^T P^T below is the same (tile 0, then
            // tile 1), so P goes to it in these registers unchanged.
            float x[4];
            x[0] = sc0[0] * a.qscale;
            x[1] = sc0[1] * a.qscale;
            x[2] = sc1[0] * a.qscale;
            x[3] = sc1[1] * a.qscale;
            const int tk[4] = {staged_token(0, 2 * tig), staged_token(0, 2 * tig + 1), staged_token(1, 2 * tig),
                               staged_token(1, 2 * tig + 1)};
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (g >= G || tk[e] >= valid) x[e] = -INFINITY;
            if (window_step && g < G) {  // kept in L2 for the epilogue
                float *lg = a.logits + ((size_t)u * kTcTokens) * a.h_q + h0 + g;
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (tk[e] < valid) st_global_hint(lg + (size_t)tk[e] * a.h_q, x[e], keep_pol);
            }
            float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
            mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
            const float m_new = fmaxf(m_run, mx);
            const float alpha = (m_new == -INFINITY) ? 1.f : exp2f(m_run - m_new);
            float p[4], rs = 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                p[e] = (x[e] == -INFINITY) ? 0.f : exp2f(x[e] - m_new);
                rs += p[e];
            }
            rs += __shfl_xor_sync(0xFFFFFFFFu, rs, 1);
            rs += __shfl_xor_sync(0xFFFFFFFFu, rs, 2);
            l_run = l_run * alpha + rs;
            m_run = m_new;
            const uint32_t pb0 = f2_to_bf2(p[0], p[1]);
            const uint32_t pb1 = f2_to_bf2(p[2], p[3]);
            // accumulator columns are heads 2tig, 2tig+1: their rescale factors
            const float a_lo = __shfl_sync(0xFFFFFFFFu, alpha, (2 * tig) * 4);
            const float a_hi = __shfl_sync(0xFFFFFFFFu, alpha, (2 * tig + 1) * 4);
            // ---- O^T += V^T P^T, one m-tile of 16 dims at a time
#pragma unroll
            for (int t = 0; t < KS; ++t) {
                acc[t][0] *= a_lo;
                acc[t][1] *= a_hi;
                acc[t][2] *= a_lo;
                acc[t][3] *= a_hi;
                uint32_t v0, v1, v2, v3;
                ldsm_x4_t(vt + loff + 32 * t, v0, v1, v2, v3);
                mma_16816(acc[t], v0, v1, v2, v3, pb0, pb1);
            }
            if (rho_row >= 0) {
                // A sequence about to be compressed: the unit is one block
                // (b = 16), and the key fragments of Q K^T, loaded again, are
                // both operands of its Gram K K^T (A = {b0, b2, b1, b3}: tile
                // 0, then tile 1; B of tile 0 = {b0, b1}, of tile 1 = {b2,
                // b3}), in the
                // fragment order and k-step order of the compression's own
                // Gram, so the lightning row sums carry the same bits.  K rows
                // >= valid hold stale data: lightning_rowsums masks every
                // entry they touch.
                float g0[4] = {0.f, 0.f, 0.f, 0.f}, g1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int t = 0; t < KS; ++t) {
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(kt + loff + 32 * t, b0, b1, b2, b3);
                    mma_16816(g0, b0, b2, b1, b3, b0, b1);
                    mma_16816(g1, b0, b2, b1, b3, b2, b3);
                }
                const float2 rsum = lightning_rowsums<true>(g0, g1, valid, a.rho_p, lane);
                if (tig == 0) {  // fragment rows g, g + 8: row g of tiles 0 and 1
                    float *ro = a.rho + ((size_t)rho_row * h_kv + kvh) * a.rho_stride + (u - prefix[s]) * kTcTokens;
                    const int t0 = staged_token(0, g), t1 = staged_token(1, g);
                    if (t0 < valid) ro[t0] = rsum.x;
                    if (t1 < valid) ro[t1] = rsum.y;
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);

        const bool seq_ends = (u + 1 == prefix[s + 1]);
        if (seq_ends || u + 1 == u1) {
            // l and m of the heads 2tig, 2tig+1 owned by this lane's columns
            const float l_lo = __shfl_sync(0xFFFFFFFFu, l_run, (2 * tig) * 4);
            const float l_hi = __shfl_sync(0xFFFFFFFFu, l_run, (2 * tig + 1) * 4);
            const int hc0 = 2 * tig, hc1 = 2 * tig + 1;  // column heads
            const bool whole = (prefix[s] >= seg_begin) && seq_ends;
            if (whole) {
                __nv_bfloat16 *og = static_cast<__nv_bfloat16 *>(a.out) + ((size_t)s * a.h_q + h0) * D;
                const float i0 = l_lo > 0.f ? 1.f / l_lo : 0.f;
                const float i1 = l_hi > 0.f ? 1.f / l_hi : 0.f;
#pragma unroll
                for (int t = 0; t < KS; ++t) {
                    const int d0 = 16 * t + g;
                    if (hc0 < G) {
                        og[(size_t)hc0 * D + d0] = __float2bfloat16_rn(acc[t][0] * i0);
                        og[(size_t)hc0 * D + d0 + 8] = __float2bfloat16_rn(acc[t][2] * i0);
                    }
                    if (hc1 < G) {
                        og[(size_t)hc1 * D + d0] = __float2bfloat16_rn(acc[t][1] * i1);
                        og[(size_t)hc1 * D + d0 + 8] = __float2bfloat16_rn(acc[t][3] * i1);
                    }
                }
                if (a.want_score && g < G && tig == 0)
                    a.stats[(size_t)s * a.h_q + h0 + g] = make_float2(m_run, l_run);
            } else {
                const int slot = 2 * blockIdx.x + ((prefix[s] <= u0) ? 0 : 1);
                float *pa = a.part_acc + ((size_t)slot * a.h_q + h0) * D;
#pragma unroll
                for (int t = 0; t < KS; ++t) {
                    const int d0 = 16 * t + g;
                    if (hc0 < G) {
                        pa[(size_t)hc0 * D + d0] = acc[t][0];
                        pa[(size_t)hc0 * D + d0 + 8] = acc[t][2];
                    }
                    if (hc1 < G) {
                        pa[(size_t)hc1 * D + d0] = acc[t][1];
                        pa[(size_t)hc1 * D + d0 + 8] = acc[t][3];
                    }
                }
                if (g < G && tig == 0) a.part_ml[(size_t)slot * a.h_q + h0 + g] = make_float2(m_run, l_run);
                if (tid == 0) mlist[5 + mlist[4]++] = s;  // announced after the loop
            }
            if (u + 1 < u1) {
                while (u + 1 >= prefix[s + 1]) ++s;
                seg_begin = u + 1;
                reset_state();
                load_q(s);
                window_step = compute_window(s);
                rho_row = rho_row_of(s);
            }
        }
    }

    // =====================================================================
    // epilogue (consumer warps; the producer has returned and every stage has
    // been consumed, so the stage area is free scratch)
    const int nthr = h_kv * 32;
    unsigned char *scratch = stage_base;
    const int scratch_bytes = a.stages * stage_bytes;
    const int HQ = a.h_q;
    // this thread's partial records and logits are visible to other CTAs and
    // to the copy engine; the stage area may be overwritten by copies
    asm volatile("fence.proxy.async.global;" ::: "memory");
    fence_proxy_async_smem();
    named_bar_sync(1, nthr);
    if (warp == 0) {
        if (lane == 0) {
            // window segments of this CTA and, if they all fit, their prefetch
            int nseg = 0, off = 0, tx = 0;
            bool fits = a.want_score != 0;
            if (a.want_score) {
                for (int sq = s_first; sq <= s && nseg < kMaxSeg; ++sq) {
                    if (!compute_window(sq)) continue;
                    const long long pb = prefix[sq], pe = prefix[sq + 1];
                    const long long ub = pb > u0 ? pb : u0, ue = pe < u1 ? pe : u1;
                    const int tb = (int)(ub - pb) * kTcTokens;
                    int te = (int)(ue - pb) * kTcTokens;
                    if (te > lens[sq]) te = lens[sq];
                    if (te <= tb) continue;
                    const int n16 = (te - tb + 15) & ~15;
                    segs[nseg++] = make_int4(sq, tb, te, off);
                    off += n16 * HQ * 4 + h_kv * (n16 + 4) * 4;  // score pieces padded by 4 floats
                    tx += n16 * HQ * 4 + h_kv * n16 * 4;         // bytes the copies deliver
                }
                bool all = true;  // every window sequence of the range got a segment entry
                for (int sq = s_first, k2 = 0; sq <= s; ++sq)
                    if (compute_window(sq) && lens[sq] > 0) {
                        const long long pb = prefix[sq], pe = prefix[sq + 1];
                        const long long ub = pb > u0 ? pb : u0, ue = pe < u1 ? pe : u1;
                        if (ue > ub) all &= (k2++ < kMaxSeg);
                    }
                // room left for the merge's part list (at most one entry per CTA)
                fits = all && off + 4 * (Gd + 16) <= scratch_bytes;
            }
            if (fits && nseg) {
                mbar_arrive_expect_tx(ebar, (unsigned)tx);
                for (int i = 0; i < nseg; ++i) {
                    const int4 g = segs[i];
                    const int n16 = (g.z - g.y + 15) & ~15;
                    float *lg_s = reinterpret_cast<float *>(scratch + g.w);
                    float *sc_s = lg_s + (size_t)n16 * HQ;
                    bulk_g2s_plain(lg_s, a.logits + ((size_t)prefix[g.x] * kTcTokens + g.y) * HQ,
                                   (unsigned)(n16 * HQ * 4), ebar);
                    const float *srow0 = a.score + (size_t)score_row_of(a, g.x) * h_kv * a.score_stride + g.y;
                    for (int kvh = 0; kvh < h_kv; ++kvh)
                        bulk_g2s_plain(sc_s + kvh * (n16 + 4), srow0 + (size_t)kvh * a.score_stride,
                                       (unsigned)(n16 * 4), ebar);
                }
            }
            mlist[7] = fits ? nseg : -1;
            mlist[0] = fits ? off : 0;
        }
    }
    // announce this CTA's parts of cut sequences (another warp than the
    // prefetch when there is one); the last arrival publishes.  The barrier
    // above ordered every thread's partial records before this fence.
    const int ann_lane0 = h_kv > 1 ? 0 : 1;  // warp 0 lane 0 issues the prefetch when h_kv == 1
    if (warp == (h_kv > 1 ? 1 : 0) && lane >= ann_lane0 && lane < ann_lane0 + 2) {
        const int i = lane - ann_lane0;
        mlist[1 + i] = -1;
        if (i < mlist[4]) {
            const int sc = mlist[5 + i];
            int c_lo, c_hi;
            const int n_parts = parts_of(prefix[sc], prefix[sc + 1], cst, Gd, &c_lo, &c_hi);
            const unsigned long long *guess_w = guess_words;
            const unsigned long long guess =
                sc == s_first ? guess_w[0]
                              : (sc == *reinterpret_cast<const int *>(smem + lay.merge_off + kEpiSLast) ? guess_w[1] : 0ull);
            fence_acq_rel_gpu();  // release: the CTA's part records (ordered by the barrier above)
            if (ctl_arrive(a.ctl + sc, n_parts, guess, a.err)) {
                fence_acq_rel_gpu();  // acquire: the other parts' records
                mlist[1 + i] = sc;
            }
        }
    }
    named_bar_sync(1, nthr);
    const int nseg = mlist[7];
    const int n_cut = mlist[4];  // this CTA's parts of cut sequences: mlist[5..6]; mlist[1 + i]: published by us
    bool waited_copies = false;
    unsigned ebar_phase = 0;
    float *sm_c1 = sm_c + kEpiStatsHeads;  // statistics of the second cut sequence
    // The window score of this CTA's tokens [tb, te) of sequence sq (window
    // segment kk when prefetched) with the statistics st; false on abort.
    auto score_own = [&](int sq, int L, long long pb, int tb, int te, int kk, const float *st) -> bool {
        if (nseg >= 0) {
            if (!waited_copies) {
                waited_copies = true;
                mbar_wait_bounded(ebar, 0, a.err, abort_flag, 61);  // every thread observes the copies
            }
            named_bar_sync(1, nthr);
            if (abort_flag[0]) return false;
            const int4 g = segs[kk];
            const int n = te - tb, n16 = (n + 15) & ~15;
            float *lg_s = reinterpret_cast<float *>(scratch + g.w);
            float *sc_s = lg_s + (size_t)n16 * HQ;
            if (h_kv == 8) score_prefetched<G, 8>(a, sq, L, tb, n, n16, lg_s, sc_s, st, tid, nthr);
            else if (h_kv == 4) score_prefetched<G, 4>(a, sq, L, tb, n, n16, lg_s, sc_s, st, tid, nthr);
            else if (h_kv == 2) score_prefetched<G, 2>(a, sq, L, tb, n, n16, lg_s, sc_s, st, tid, nthr);
            else score_prefetched<G, 1>(a, sq, L, tb, n, n16, lg_s, sc_s, st, tid, nthr);
        } else {
            if (h_kv == 8)
                score_segment<G, 8>(a, sq, L, pb, tb, te, scratch, scratch_bytes, ebar, ebar_phase, abort_flag, st,
                                    tid, nthr);
            else if (h_kv == 4)
                score_segment<G, 4>(a, sq, L, pb, tb, te, scratch, scratch_bytes, ebar, ebar_phase, abort_flag, st,
                                    tid, nthr);
            else if (h_kv == 2)
                score_segment<G, 2>(a, sq, L, pb, tb, te, scratch, scratch_bytes, ebar, ebar_phase, abort_flag, st,
                                    tid, nthr);
            else
                score_segment<G, 1>(a, sq, L, pb, tb, te, scratch, scratch_bytes, ebar, ebar_phase, abort_flag, st,
                                    tid, nthr);
        }
        return true;
    };
    // Whole sequences first (their statistics are this CTA's own), one at a
    // time; then the cut sequences -- at most two, the first and the last of
    // the range -- together: one bounded wait for the publication of those
    // another CTA publishes, the final statistics from the part records and
    // this CTA's slice of each output with the loads of both in flight (two
    // halves of the threads), then the scores of this CTA's tokens of each.
    int cut_kk0 = 0, cut_kk1 = 0;  // window segment index of the cut sequences
    {
        int kseg = 0;  // index of the next window segment in segs
        for (int sq = s_first; sq <= s; ++sq) {
            if (abort_flag[0]) break;  // set before a barrier by a thread that gave up: uniform
            const long long pb = prefix[sq], pe = prefix[sq + 1];
            const long long ub = pb > u0 ? pb : u0, ue = pe < u1 ? pe : u1;
            if (ue <= ub) continue;
            const int L = lens[sq];
            const int tb = (int)(ub - pb) * kTcTokens;
            int te = (int)(ue - pb) * kTcTokens;
            if (te > L) te = L;
            const bool has_seg = compute_window(sq) && te > tb;  // the same rule that built segs
            const int kk = kseg;
            if (has_seg) ++kseg;
            const bool whole = pb >= u0 && pe <= u1;
            if (!whole) {
                if (n_cut > 0 && mlist[5] == sq) cut_kk0 = kk;
                if (n_cut > 1 && mlist[6] == sq) cut_kk1 = kk;
                continue;
            }
            if (!has_seg) continue;
            for (int h = tid; h < HQ; h += nthr) {
                const float2 ml = __ldcg(&a.stats[(size_t)sq * HQ + h]);
                sm_c[h] = ml.y > 0.f ? ml.x + log2f(ml.y) : INFINITY;
            }
            if (!score_own(sq, L, pb, tb, te, kk, sm_c)) break;
            named_bar_sync(1, nthr);  // sm_c reused by the next sequence
        }
    }
    if (!abort_flag[0] && n_cut > 0) {
        // cut sequence i of the range (mlist[5 + i]); wait: published by another CTA
        auto cut_seq = [&](int i) -> CutSeq {
            CutSeq c;
            c.sq = mlist[5 + i];
            const long long pb = prefix[c.sq], pe = prefix[c.sq + 1];
            const long long ub = pb > u0 ? pb : u0, ue = pe < u1 ? pe : u1;
            c.L = lens[c.sq];
            c.pb = pb;
            c.tb = (int)(ub - pb) * kTcTokens;
            c.te = (int)(ue - pb) * kTcTokens;
            if (c.te > c.L) c.te = c.L;
            c.seg = compute_window(c.sq) && c.te > c.tb;
            c.wait = mlist[1 + i] != c.sq;
            c.kk = i ? cut_kk1 : cut_kk0;
            return c;
        };
        CutSeq cs0 = cut_seq(0);
        CutSeq cs1 = n_cut > 1 ? cut_seq(1) : cs0;
        // without the score only the last arrival works
        bool use0 = a.want_score || !cs0.wait;
        bool use1 = n_cut > 1 && (a.want_score || !cs1.wait);
        if (!use0) {
            cs0 = cs1;
            use0 = use1;
            use1 = false;
        }
        const int nc = (use0 ? 1 : 0) + (use1 ? 1 : 0);
        named_bar_sync(1, nthr);  // mlist[1..2] read by every thread before tid 0 reuses them
        if (tid == 0) {
            const bool w0 = nc > 0 && cs0.wait, w1 = nc > 1 && cs1.wait;
            unsigned okm = 3u;
            if (w0 || w1) {
                okm = ctl_wait_published2(w0 ? a.ctl + cs0.sq : nullptr, w1 ? a.ctl + cs1.sq : nullptr, a.err);
                fence_acq_rel_gpu();  // the part records are read after the publication
            }
            mlist[1] = okm & 1u;
            mlist[2] = (okm >> 1) & 1u;
        }
        named_bar_sync(1, nthr);
        const bool cok0 = mlist[1] != 0, cok1 = mlist[2] != 0;
        // the statistics for the score (the first HQ threads of a group) and this
        // CTA's slice of the output (the others); with two sequences and at
        // least 128 threads each half of the threads takes one
        const bool split = nc == 2 && nthr >= 128;
        const int gsz = split ? nthr / 2 : nthr;
        for (int r = 0; r < (split ? 1 : nc); ++r) {
            const int j = split ? tid / gsz : r;
            const int gt = split ? tid - j * gsz : tid;
            const CutSeq c = j ? cs1 : cs0;
            if (j ? cok1 : cok0) {
                const int t0 = c.seg && gsz - HQ >= 64 ? HQ : 0;
                if (c.seg) part_stats(a, c.sq, prefix, cst, Gd, j ? sm_c1 : sm_c, gt, t0 ? t0 : gsz);
                merge_slice<D>(a, c.sq, prefix, cst, Gd, !a.want_score, gt, t0, gsz);
            }
        }
        if (split && nseg >= 0 && cok0 && cok1 && cs0.seg && cs1.seg) {
            // both segments prefetched: each half of the threads scores its own
            // sequence's tokens (named barrier 2 + half)
            if (!waited_copies) {
                waited_copies = true;
                mbar_wait_bounded(ebar, 0, a.err, abort_flag, 61);  // every thread observes the copies
            }
            named_bar_sync(1, nthr);  // both halves' statistics are in place
            if (!abort_flag[0]) {
                const int j = tid / gsz;
                const CutSeq c = j ? cs1 : cs0;
                const int4 g = segs[c.kk];
                const int n = c.te - c.tb, n16 = (n + 15) & ~15;
                const float *lg_s = reinterpret_cast<const float *>(scratch + g.w);
                float *sc_s = reinterpret_cast<float *>(scratch + g.w) + (size_t)n16 * HQ;
                const float *st = j ? sm_c1 : sm_c;
                const int gt = tid - j * gsz;
                if (h_kv == 8) {
                    if (j) score_prefetched<G, 8, 3>(a, c.sq, c.L, c.tb, n, n16, lg_s, sc_s, st, gt, gsz);
                    else score_prefetched<G, 8, 2>(a, c.sq, c.L, c.tb, n, n16, lg_s, sc_s, st, gt, gsz);
                } else {
                    if (j) score_prefetched<G, 4, 3>(a, c.sq, c.L, c.tb, n, n16, lg_s, sc_s, st, gt, gsz);
                    else score_prefetched<G, 4, 2>(a, c.sq, c.L, c.tb, n, n16, lg_s, sc_s, st, gt, gsz);
                }
            }
        } else {
            for (int j = 0; j < nc; ++j) {
                if (abort_flag[0]) break;
                const CutSeq c = j ? cs1 : cs0;
                if (!(j ? cok1 : cok0) || !c.seg) continue;
                if (!score_own(c.sq, c.L, c.pb, c.tb, c.te, c.kk, j ? sm_c1 : sm_c)) break;
                named_bar_sync(1, nthr);
            }
        }
    }
    if (nseg > 0 && !waited_copies && tid == 0) mbar_wait_bounded(ebar, 0, a.err, abort_flag, 62);
    // shared-memory sources read (the score pieces' copies are issued by
    // threads 0 and nthr / 2); the writes complete on their own
    if (tid == 0 || tid == nthr / 2) bulk_wait_read_all();
}

// ===========================================================================
// Merge of the sequences that the stream-K split cut between CTAs.
//
// Every CTA of the main kernel leaves, for a sequence it did not see whole, a
// partial record: its running max m and sum l per q head (log2 units) and its
// unnormalised accumulator.  Block c of this kernel merges the sequence whose
// last unit lies in CTA c's range and which began in an earlier CTA, so every
// cut sequence has exactly one merger and all merges run in parallel:
//     M = max_j m_j,  w_j = 2^(m_j - M),  L = sum_j w_j l_j,
//     out = sum_j w_j acc_j / L.
template <typename T, int D>
__global__ void __launch_bounds__(256) decode_merge_kernel(const DecodeArgs a, int grid_main) {
    extern __shared__ float2 msm[];  // [grid_main][h_q] (m, l) then weights; then slots, L
    const int c = blockIdx.x;
    const int B = a.B;
    const int *pre = a.unit_prefix;
    const long long U = pre[B];
    const long long cs = cta_start(c, U, grid_main), ce = cta_start(c + 1, U, grid_main);
    if (cs >= ce) return;
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pre[mid] <= cs) lo = mid;
        else hi = mid - 1;
    }
    const int s = lo;
    if (!(pre[s] < cs && pre[s + 1] <= ce)) return;  // not cut, or not this block's
    const int h_q = a.h_q;
    const int c_lo = cta_of(pre[s], U, grid_main);
    const int nc = c - c_lo + 1;
    int *slot = reinterpret_cast<int *>(msm + (size_t)grid_main * h_q);
    float *Lh = reinterpret_cast<float *>(slot + grid_main);
    for (int j = threadIdx.x; j < nc; j += blockDim.x) {
        const int cj = c_lo + j;
        const long long sj = cta_start(cj, U, grid_main);
        slot[j] = (sj == cta_start(cj + 1, U, grid_main)) ? -1 : 2 * cj + (pre[s] > sj ? 1 : 0);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < nc * h_q; e += blockDim.x) {
        const int j = e / h_q, h = e % h_q;
        msm[e] = slot[j] < 0 ? make_float2(-INFINITY, 0.f) : __ldcg(&a.part_ml[(size_t)slot[j] * h_q + h]);
    }
    __syncthreads();
    for (int h = threadIdx.x; h < h_q; h += blockDim.x) {
        float M = -INFINITY;
        for (int j = 0; j < nc; ++j) M = fmaxf(M, msm[j * h_q + h].x);
        float L = 0.f;
        for (int j = 0; j < nc; ++j) {
            const float2 ml = msm[j * h_q + h];
            const float w = (ml.x == -INFINITY) ? 0.f : exp2f(ml.x - M);
            L += w * ml.y;
            msm[j * h_q + h].x = w;  // weight in place of the max
        }
        Lh[h] = L;
        if (a.want_score) a.stats[(size_t)s * h_q + h] = make_float2(M, L);
    }
    __syncthreads();
    constexpr int CH = 16;  // dims per item
    for (int it = threadIdx.x; it < h_q * (D / CH); it += blockDim.x) {
        const int h = it / (D / CH);
        const int d0 = (it % (D / CH)) * CH;
        float acc[CH];
#pragma unroll
        for (int i = 0; i < CH; ++i) acc[i] = 0.f;
        for (int j = 0; j < nc; ++j) {
            if (slot[j] < 0) continue;
            const float w = msm[j * h_q + h].x;
            const float4 *src = reinterpret_cast<const float4 *>(a.part_acc + ((size_t)slot[j] * h_q + h) * D + d0);
#pragma unroll
            for (int q4 = 0; q4 < CH / 4; ++q4) {
                const float4 v = __ldcg(src + q4);
                acc[4 * q4] += w * v.x;
                acc[4 * q4 + 1] += w * v.y;
                acc[4 * q4 + 2] += w * v.z;
                acc[4 * q4 + 3] += w * v.w;
            }
        }
        const float inv = Lh[h] > 0.f ? 1.f / Lh[h] : 0.f;
        T *og = static_cast<T *>(a.out) + ((size_t)s * h_q + h) * D + d0;
        if constexpr (sizeof(T) == 2) {
            uint32_t w4[CH / 2];
#pragma unroll
            for (int i = 0; i < CH / 2; ++i) w4[i] = f2_to_bf2(acc[2 * i] * inv, acc[2 * i + 1] * inv);
            reinterpret_cast<uint4 *>(og)[0] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
            reinterpret_cast<uint4 *>(og)[1] = make_uint4(w4[4], w4[5], w4[6], w4[7]);
        } else {
#pragma unroll
            for (int q4 = 0; q4 < CH / 4; ++q4)
                reinterpret_cast<float4 *>(og)[q4] =
                    make_float4(acc[4 * q4] * inv, acc[4 * q4 + 1] * inv, acc[4 * q4 + 2] * inv, acc[4 * q4 + 3] * inv);
        }
    }
}

// Merge kernel, then (window steps) the score epilogue.  (Programmatic
// dependent launches of these two were measured slightly slower.)
template <typename T, int D, int G>
zp_status launch_finish(const DecodeArgs &a, int grid, long long units_cap, cudaStream_t st) {
    const size_t smem = (size_t)grid * a.h_q * 8 + (size_t)grid * 4 + (size_t)a.h_q * 4;
    zp_status rs = set_max_dynamic_smem(reinterpret_cast<const void *>(decode_merge_kernel<T, D>), smem,
                                        "decode: merge shared-memory attribute");
    if (rs != ZP_OK) return rs;
    decode_merge_kernel<T, D><<<grid, 256, smem, st>>>(a, grid);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "decode: merge kernel launch");
    if (a.want_score) {
        decode_score_kernel<G><<<(unsigned)units_cap, 128, 0, st>>>(a);
        e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e, "decode: score kernel launch");
    }
    return ZP_OK;
}

struct Plan {
    bool tc;  // tensor-core kernel (bf16) or CUDA-core kernel
    int T, wph, ncw, threads, stages, smem, grid;
    size_t off_count, off_prefix, off_stats, off_pml, off_pacc, off_info, off_logits, total;
    long long logits_units;
};

zp_status make_plan(const zp_cache_desc *D, int B, int table_stride, const DeviceInfo &dev,
                    Plan *p) {
    const int es = elem_bytes(D->dtype);
    const int d = D->head_dim, b = D->block_size, h_kv = D->h_kv;
    const int G = D->h_q / D->h_kv;
    if (!(d == 64 || d == 128)) return fail(ZP_ERR_SHAPE, "decode: head_dim %d not in {64,128}", d);
    if (b < 16 || (b & (b - 1))) return fail(ZP_ERR_SHAPE, "decode: block size %d", b);
    if (B > kMaxB) return fail(ZP_ERR_SHAPE, "decode: B %d > %d", B, kMaxB);
    p->grid = dev.sm_count;
    p->tc = D->dtype == ZP_BF16 && (h_kv == 1 || h_kv == 2 || h_kv == 4 || h_kv == 8) &&
            (G == 1 || G == 2 || G == 4 || G == 8);
    if (p->tc) {
        p->T = kTcTokens;
        p->wph = 1;
        p->ncw = h_kv;
        p->threads = (h_kv + 1) * 32;
        int stages = 4;
        while (stages > 2 && make_tc_layout(stages, h_kv, d / 64, B, p->grid).total > dev.smem_optin) --stages;
        p->stages = stages;
        p->smem = make_tc_layout(stages, h_kv, d / 64, B, p->grid).total;
    } else {
        if (!(G == 4 || G == 8)) return fail(ZP_ERR_SHAPE, "decode: group size %d not in {4,8}", G);
        if (!(h_kv == 2 || h_kv == 4 || h_kv == 8 || h_kv == 16))
            return fail(ZP_ERR_SHAPE, "decode: h_kv %d not in {2,4,8,16}", h_kv);
        const int row = h_kv * d * es;
        int T = b;
        while (T > 8 && T * row > kStageBytesCap) T >>= 1;
        if (T * row > kStageBytesCap) return fail(ZP_ERR_SHAPE, "decode: row of %d bytes too large", row);
        int wph = T / 8;
        if (wph > kMaxConsumerWarps / h_kv) wph = kMaxConsumerWarps / h_kv;
        if (wph < 1) wph = 1;
        p->T = T;
        p->wph = wph;
        p->ncw = h_kv * wph;
        p->threads = p->ncw * 32;
        const int stage_bytes = T * row;
        int stages = 4;
        while (stages > 2 &&
               make_layout(stages, stage_bytes, p->ncw, h_kv, G, d, B).total > dev.smem_optin)
            --stages;
        p->stages = stages;
        p->smem = make_layout(stages, stage_bytes, p->ncw, h_kv, G, d, B).total;
    }
    if (p->smem > dev.smem_optin) return fail(ZP_ERR_SHAPE, "decode: needs %d B of shared memory", p->smem);
    const long long units_cap = (long long)B * table_stride * (b / p->T);
    p->logits_units = units_cap;
    size_t off = 0;
    p->off_count = off;  // per-sequence arrival counters (tensor-core path)
    off = align_up(off + (size_t)B * 8, 256);
    p->off_prefix = off;
    off = align_up(off + (size_t)(B + 1) * 4, 256);
    p->off_stats = off;
    off = align_up(off + (size_t)B * D->h_q * 8, 256);
    p->off_pml = off;
    off = align_up(off + (size_t)2 * p->grid * D->h_q * 8, 256);
    p->off_pacc = off;
    off = align_up(off + (size_t)2 * p->grid * D->h_q * d * 4, 256);
    p->off_info = off;
    off = align_up(off + (size_t)units_cap * 16, 256);
    p->off_logits = off;
    off = align_up(off + (size_t)units_cap * p->T * D->h_q * 4, 256);
    p->total = off;
    return ZP_OK;
}

template <int Dd, int G>
zp_status launch_tc(const DecodeArgs &a, const Plan &p, const DeviceInfo &dev, cudaStream_t st,
                    const zp_cache_desc *D) {
    auto kmain = decode_tc_kernel<Dd, G>;
    zp_status rs = set_max_dynamic_smem(reinterpret_cast<const void *>(kmain), (size_t)p.smem,
                                        "decode: shared-memory attribute");
    if (rs != ZP_OK) return rs;
    if ((reinterpret_cast<uintptr_t>(a.k) | reinterpret_cast<uintptr_t>(a.v)) % 16)
        return fail(ZP_ERR_INVALID_ARG, "decode: caches must be 16-byte aligned");
    // cooperative: CTAs wait (bounded) for the merges of other CTAs
    DecodeArgs args = a;
    void *params[] = {&args};
    cudaError_t e = cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(kmain), dim3(p.grid), dim3(p.threads), params,
                                    (size_t)p.smem, st);
    if (e != cudaSuccess) return cuda_fail(e, "decode: tensor-core kernel launch");
    return ok();  // merges and the window score run inside the kernel
}

template <typename T, int Dd, int G>
zp_status launch_t(const DecodeArgs &a, const Plan &p, const DeviceInfo &dev, cudaStream_t st) {
    auto kmain = decode_main_kernel<T, Dd, G>;
    zp_status rs = set_max_dynamic_smem(reinterpret_cast<const void *>(kmain), (size_t)p.smem,
                                        "decode: shared-memory attribute");
    if (rs != ZP_OK) return rs;
    kmain<<<p.grid, p.threads, p.smem, st>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "decode: main kernel launch");
    return launch_finish<T, Dd, G>(a, p.grid, p.logits_units, st);
}

}  // namespace
}  // namespace zp

using namespace zp;

extern "C" size_t zp_decode_workspace_size(const zp_cache_desc *D, int32_t B, int32_t table_stride) {
    if (check_desc(D) != ZP_OK || B < 0 || table_stride < 0) return 0;
    DeviceInfo dev;
    if (device_info(&dev) != ZP_OK) return 0;
    Plan p;
    if (make_plan(D, B, table_stride, dev, &p) != ZP_OK) return 0;
    return p.total;
}

static zp_status decode_impl(const zp_cache_desc *D, const void *q, const void *k_cache, const void *v_cache,
                             const int32_t *block_table, int32_t table_stride, const int32_t *seq_lens, int32_t B,
                             void *out, float *score_accum, const int32_t *score_rows, int32_t n_score_rows,
                             int32_t window, void *workspace, size_t workspace_bytes, void *stream,
                             const zp_rho_rows *rho) {
    zp_status rc = check_desc(D);
    if (rc != ZP_OK) return rc;
    if (B < 0 || table_stride < 0) return fail(ZP_ERR_INVALID_ARG, "decode: B or table_stride negative");
    if (B == 0) return ok();
    if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !out || !workspace)
        return fail(ZP_ERR_INVALID_ARG, "decode: NULL buffer");
    if (table_stride < 1) return fail(ZP_ERR_INVALID_ARG, "decode: table_stride < 1");
    if (score_accum && (window < 1 || window > D->block_size))
        return fail(ZP_ERR_INVALID_ARG, "decode: window %d outside [1, b=%d]", window, D->block_size);
    if (reinterpret_cast<uintptr_t>(score_accum) % 16)
        return fail(ZP_ERR_INVALID_ARG, "decode: score_accum must be 16-byte aligned");
    if (score_accum && score_rows && n_score_rows < 1)
        return fail(ZP_ERR_INVALID_ARG, "decode: a slot map needs n_score_rows >= 1");
    DeviceInfo dev;
    rc = device_info(&dev);
    if (rc != ZP_OK) return rc;
    Plan p;
    rc = make_plan(D, B, table_stride, dev, &p);
    if (rc != ZP_OK) return rc;
    if (workspace_bytes < p.total)
        return fail(ZP_ERR_CAPACITY, "decode: workspace %zu < %zu bytes", workspace_bytes, p.total);
    if (rho) {
        if (!rho->data || !rho->rows) return fail(ZP_ERR_INVALID_ARG, "decode: redundancy rows need data and rows");
        if (rho->stride < 1 || rho->n_rows < 1)
            return fail(ZP_ERR_INVALID_ARG, "decode: redundancy rows: stride %lld, %d rows", (long long)rho->stride,
                        rho->n_rows);
        if (!p.tc || D->block_size != 16)
            return fail(ZP_ERR_SHAPE, "decode: the lightning redundancy needs the bf16 tensor-core path and b = 16");
    }
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    DecodeArgs a;
    a.q = q;
    a.k = k_cache;
    a.v = v_cache;
    a.out = out;
    a.table = block_table;
    a.table_stride = table_stride;
    a.seq_lens = seq_lens;
    a.B = B;
    a.h_q = D->h_q;
    a.h_kv = D->h_kv;
    a.b = D->block_size;
    a.n_total = D->n_total_blocks;
    a.T = p.T;
    a.upb = D->block_size / p.T;
    a.wph = p.wph;
    a.ncw = p.ncw;
    a.stages = p.stages;
    a.qscale = (float)(1.4426950408889634 / sqrt((double)D->head_dim));
    a.want_score = score_accum != nullptr;
    a.window = window;
    a.score = score_accum;
    a.score_stride = (long long)table_stride * D->block_size;
    a.score_rows = score_accum ? score_rows : nullptr;
    a.n_score_rows = n_score_rows;
    a.logits = reinterpret_cast<float *>(ws + p.off_logits);
    a.stats = reinterpret_cast<float2 *>(ws + p.off_stats);
    a.part_acc = reinterpret_cast<float *>(ws + p.off_pacc);
    a.part_ml = reinterpret_cast<float2 *>(ws + p.off_pml);
    a.unit_prefix = reinterpret_cast<int *>(ws + p.off_prefix);
    a.unit_info = reinterpret_cast<int4 *>(ws + p.off_info);
    a.logits_units = p.logits_units;
    a.ctl = reinterpret_cast<unsigned long long *>(ws + p.off_count);
    a.rho = rho ? rho->data : nullptr;
    a.rho_stride = rho ? rho->stride : 0;
    a.rho_rows = rho ? rho->rows : nullptr;
    a.n_rho_rows = rho ? rho->n_rows : 0;
    a.rho_p = rho ? rho->threshold : 0.f;
    // weighted split only while the weighted unit count fits in 32 bits and
    // its two arrays (2B + 1 ints) fit in the stage area
    const double max_units = (double)B * table_stride * D->block_size / 16.0;
    const long long stage_area = (long long)p.stages * 2 * kTcGroups * tc_group_stride(D->h_kv, D->head_dim);
    a.rho_weight16 = (rho && p.tc && max_units * kRhoUnitWeight16 < 2.0e9 && (2LL * B + 1) * 4 <= stage_area)
                         ? kRhoUnitWeight16 : 16;
    a.err = dev.error_word;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int G = D->h_q / D->h_kv;
    const int d = D->head_dim;
    if (p.tc) {
        if (d == 128 && G == 4) return launch_tc<128, 4>(a, p, dev, st, D);
        if (d == 128 && G == 8) return launch_tc<128, 8>(a, p, dev, st, D);
        if (d == 128 && G == 2) return launch_tc<128, 2>(a, p, dev, st, D);
        if (d == 128 && G == 1) return launch_tc<128, 1>(a, p, dev, st, D);
        if (d == 64 && G == 4) return launch_tc<64, 4>(a, p, dev, st, D);
        if (d == 64 && G == 8) return launch_tc<64, 8>(a, p, dev, st, D);
        if (d == 64 && G == 2) return launch_tc<64, 2>(a, p, dev, st, D);
        if (d == 64 && G == 1) return launch_tc<64, 1>(a, p, dev, st, D);
    }
    if (D->dtype == ZP_BF16) {
        if (d == 128 && G == 4) return launch_t<__nv_bfloat16, 128, 4>(a, p, dev, st);
        if (d == 128 && G == 8) return launch_t<__nv_bfloat16, 128, 8>(a, p, dev, st);
        if (d == 64 && G == 4) return launch_t<__nv_bfloat16, 64, 4>(a, p, dev, st);
        if (d == 64 && G == 8) return launch_t<__nv_bfloat16, 64, 8>(a, p, dev, st);
    } else {
        if (d == 128 && G == 4) return launch_t<float, 128, 4>(a, p, dev, st);
        if (d == 128 && G == 8) return launch_t<float, 128, 8>(a, p, dev, st);
        if (d == 64 && G == 4) return launch_t<float, 64, 4>(a, p, dev, st);
        if (d == 64 && G == 8) return launch_t<float, 64, 8>(a, p, dev, st);
    }
    return fail(ZP_ERR_SHAPE, "decode: no kernel for d=%d, group=%d", d, G);
}

extern "C" zp_status zp_paged_decode_attn(const zp_cache_desc *D, const void *q, const void *k_cache,
                                          const void *v_cache, const int32_t *block_table,
                                          int32_t table_stride, const int32_t *seq_lens, int32_t B,
                                          void *out, float *score_accum, const int32_t *score_rows,
                                          int32_t n_score_rows, int32_t window, void *workspace,
                                          size_t workspace_bytes, void *stream) {
    return decode_impl(D, q, k_cache, v_cache, block_table, table_stride, seq_lens, B, out, score_accum, score_rows,
                       n_score_rows, window, workspace, workspace_bytes, stream, nullptr);
}

extern "C" zp_status zp_paged_decode_attn_rho(const zp_cache_desc *D, const void *q, const void *k_cache,
                                              const void *v_cache, const int32_t *block_table,
                                              int32_t table_stride, const int32_t *seq_lens, int32_t B,
                                              void *out, float *score_accum, const int32_t *score_rows,
                                              int32_t n_score_rows, int32_t window, const zp_rho_rows *rho,
                                              void *workspace, size_t workspace_bytes, void *stream) {
    return decode_impl(D, q, k_cache, v_cache, block_table, table_stride, seq_lens, B, out, score_accum, score_rows,
                       n_score_rows, window, workspace, workspace_bytes, stream, rho);
}

// ---------------------------------------------------------------------------
// Decode attention without any allocation.
//
// For callers that cannot allocate device memory at the point where they
// decode: for example a serving loop whose device memory is all reserved up
// front and which may not call cudaMalloc between steps, or a plain C client
// of this library that owns no device allocator at all.  The scratch that zp_paged_decode_attn takes from the
// caller's workspace comes instead from one fixed array compiled into this
// library.  Every GPU that loads the library holds that array until the
// process exits.
constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;  // 64 MiB
static __device__ __align__(256) unsigned char g_decode_noalloc_scratch[kNoAllocScratchBytes];

namespace {
std::mutex g_noalloc_mutex;
void *g_noalloc_ptr[64] = {nullptr};
}  // namespace

extern "C" zp_status zp_paged_decode_attn_noalloc(const zp_cache_desc *D, const void *q,
                                                  const void *k_cache, const void *v_cache,
                                                  const int32_t *block_table, int32_t table_stride,
                                                  const int32_t *seq_lens, int32_t B, void *out,
                                                  float *score_accum, const int32_t *score_rows,
                                                  int32_t n_score_rows, int32_t window, void *stream) {
    zp_status rc = check_desc(D);
    if (rc != ZP_OK) return rc;
    if (B < 0 || table_stride < 0) return fail(ZP_ERR_INVALID_ARG, "decode_noalloc: B or table_stride negative");
    if (B == 0) return ok();
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "decode_noalloc: cudaGetDevice");
    if (dev < 0 || dev >= 64) return fail(ZP_ERR_CUDA, "decode_noalloc: device id %d out of range", dev);
    void *scratch = nullptr;
    {
        // First call on a device: look up the device address of the array
        // with that device current.  The host-side name of the array is not
        // a device address and must never be passed to a kernel.
        std::lock_guard<std::mutex> lock(g_noalloc_mutex);
        if (!g_noalloc_ptr[dev]) {
            void *p = nullptr;
            e = cudaGetSymbolAddress(&p, g_decode_noalloc_scratch);
            if (e != cudaSuccess) return cuda_fail(e, "decode_noalloc: cudaGetSymbolAddress");
            g_noalloc_ptr[dev] = p;
        }
        scratch = g_noalloc_ptr[dev];
    }
    const size_t need = zp_decode_workspace_size(D, B, table_stride);
    if (need == 0) return fail(ZP_ERR_SHAPE, "decode_noalloc: %s", zp_last_error());
    if (need > kNoAllocScratchBytes)
        return fail(ZP_ERR_CAPACITY,
                    "decode_noalloc: this call needs %zu bytes of scratch; the built-in buffer holds "
                    "%zu (reduce B or table_stride, or use zp_paged_decode_attn with a workspace)",
                    need, kNoAllocScratchBytes);
    // The per-sequence control words of the in-kernel merge (the first B
    // 64-bit words) persist from call to call.  A call that gave up on a
    // bounded wait (ZP_ERR_TIMEOUT) can leave a word counting arrivals that
    // never completed; a caller with a workspace clears it, but this array is
    // out of a caller's reach, so every call zeroes those words on its own
    // stream first (a zero word reads as "no arrival yet").  Every other part
    // of the scratch is written before it is read within the call.
    e = cudaMemsetAsync(scratch, 0, (size_t)B * 8, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "decode_noalloc: clearing the control words");
    return zp_paged_decode_attn(D, q, k_cache, v_cache, block_table, table_stride, seq_lens, B, out,
                                score_accum, score_rows, n_score_rows, window, scratch, kNoAllocScratchBytes,
                                stream);
}

// Test hook: writes one control word of the built-in array of the current
// device, as a call that timed out could have left it.  Allocates nothing.
extern "C" zp_status zp_debug_noalloc_preset_ctl(int32_t seq, uint64_t word) {
    if (seq < 0 || (size_t)(seq + 1) * 8 > kNoAllocScratchBytes)
        return fail(ZP_ERR_INVALID_ARG, "noalloc_preset_ctl: sequence %d outside the array", seq);
    const unsigned long long w = word;
    cudaError_t e = cudaMemcpyToSymbol(g_decode_noalloc_scratch, &w, 8, (size_t)seq * 8, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e, "noalloc_preset_ctl: cudaMemcpyToSymbol");
    return ok();
}
