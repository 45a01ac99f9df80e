// lightning.cuh -- the lightning redundancy rule of one 16-token block of one
// kv head, applied to its Gram matrix G = K K^T held in mma.sync accumulator
// fragments (Zipage paper App. C.5 definition, C.7 same-block pairs).
//
// Shared by every kernel that forms such a Gram -- the compression's
// global/lightning kernel and the decode kernel, which forms it from the key
// fragments it already holds for Q K^T -- so that both give the same bits.
#pragma once

#include "zp_common.cuh"

namespace zp {

// Staged layout of a 16-token block shared by the decode and the
// compression's Gram: kStageRows consecutive token rows per bulk copy, each
// group of them followed by 16 bytes of pad.  An 8-token operand tile h
// (h = 0, 1) takes rows [h R/2, (h + 1) R/2) of every group, so that its
// eight rows fall on as many bank groups as there are groups of rows.
constexpr int kStageRows = 2;

// Token of row i (0..7) of operand tile h in that layout.
__host__ __device__ constexpr int staged_token(int h, int i) {
    return (i / (kStageRows / 2)) * kStageRows + i % (kStageRows / 2) + h * (kStageRows / 2);
}

// Token order of the fragments.  Natural: fragment row (and column) r is
// token r.  Staged (STAGED = true): fragment row r < 8 is row r of tile 0,
// row r >= 8 row r - 8 of tile 1 (staged_token).
template <bool STAGED>
__device__ __forceinline__ int lightning_token(int r) {
    return STAGED ? (r < 8 ? staged_token(0, r) : staged_token(1, r - 8)) : r;
}

// One column `col` (fragment index) of a lane's fragment: its entries of
// fragment rows g (va) and g + 8 (vb), the reciprocal norm of the column and
// of the two rows (0 for a missing row or column, or a zero key).  Forms both
// cosines, then zeroes the entry of the newest existing token whose cosine
// exceeds p; colmask selects the eight lanes that hold this column (lanes
// tig + 4 g'), and the highest set bit of a ballot over them, shifted right
// by two, is the fragment row g' within its half.
template <bool STAGED>
__device__ __forceinline__ void lightning_column(float &va, float &vb, int col, float inv_c, float inv_a,
                                                 float inv_b, bool rva, bool rvb, int g, unsigned colmask, float p) {
    // a zero reciprocal norm masks the entry (stale rows past the block's
    // end may hold anything, so select rather than multiply by zero)
    va = (inv_a > 0.f && inv_c > 0.f && g != col) ? va * inv_a * inv_c : 0.f;
    vb = (inv_b > 0.f && inv_c > 0.f && g + 8 != col) ? vb * inv_b * inv_c : 0.f;
    // rows past the block's end take no part, also when p < 0 makes their
    // zero entries exceed it
    const unsigned blo = __ballot_sync(0xFFFFFFFFu, rva && va > p) & colmask;
    const unsigned bhi = __ballot_sync(0xFFFFFFFFu, rvb && vb > p) & colmask;
    const int glo = blo ? (31 - __clz(blo)) >> 2 : -1;  // newest hit among fragment rows 0..7
    const int ghi = bhi ? (31 - __clz(bhi)) >> 2 : -1;  // among rows 8..15
    // within each half the token grows with the row; across the halves the
    // newer of the two candidates wins
    int rstar;
    if (ghi < 0) rstar = glo;
    else if (glo < 0) rstar = 8 + ghi;
    else rstar = lightning_token<STAGED>(8 + ghi) > lightning_token<STAGED>(glo) ? 8 + ghi : glo;
    if (rstar == g) va = 0.f;
    if (rstar == g + 8) vb = 0.f;
}

// 1/|k| from the squared norm, 0 for a missing row or a zero key.
__device__ __forceinline__ float lightning_inv_norm(float n_sq, bool exists) {
    return (exists && n_sq > 0.f) ? rsqrtf(n_sq) : 0.f;
}

// Fragment layout (m16n8k16 accumulators, lane = 4 g + tig): c0[e] = G[g][2tig+e],
// c0[2+e] = G[g+8][2tig+e], c1[e] = G[g][8+2tig+e], c1[2+e] = G[g+8][8+2tig+e]
// (fragment indices; lightning_token gives the tokens).
//
// The rule, on the tokens r, c < nvalid (the block's tokens that exist):
//     C[r][c] = G[r][c] / (|k_r| |k_c|), 0 when either norm is 0
//     C[c][c] = 0
//     per column c: the largest (newest) r with C[r][c] > p loses its entry
//     rho[r] = sum_c C[r][c]
// The squared norms are the diagonal of G; C[r][c] is formed as
// G[r][c] * (1/|k_r|) * (1/|k_c|) with the reciprocal square root.  Returns
// (rho of fragment row g, rho of fragment row g + 8), complete in every lane
// of the warp (whole warp must call).
template <bool STAGED>
__device__ __forceinline__ float2 lightning_rowsums(const float (&c0)[4], const float (&c1)[4], int nvalid, float p,
                                                    int lane) {
    const int g = lane >> 2, tig = lane & 3;
    // G[r][r] sits in lane 4 (r % 8) + (r % 8) / 2: c0[r & 1] for r < 8,
    // c1[2 + (r & 1)] for r >= 8.  Each lane turns its own diagonal candidate
    // into a reciprocal norm first, so the shuffles move finished values.
    const int c_lo = 2 * tig, c_hi = 8 + 2 * tig;
    const bool rva = lightning_token<STAGED>(g) < nvalid, rvb = lightning_token<STAGED>(g + 8) < nvalid;
    const float i0 = lightning_inv_norm((g & 1) ? c0[1] : c0[0], rva);
    const float i1 = lightning_inv_norm((g & 1) ? c1[3] : c1[2], rvb);
    const int src_row = 4 * g + (g >> 1);
    const float inv_a = __shfl_sync(0xFFFFFFFFu, i0, src_row);  // row g
    const float inv_b = __shfl_sync(0xFFFFFFFFu, i1, src_row);  // row g + 8
    const float inv0 = __shfl_sync(0xFFFFFFFFu, i0, 9 * tig);  // column 2 tig
    const float inv1 = __shfl_sync(0xFFFFFFFFu, i0, 9 * tig + 4);
    const float inv2 = __shfl_sync(0xFFFFFFFFu, i1, 9 * tig);  // column 8 + 2 tig
    const float inv3 = __shfl_sync(0xFFFFFFFFu, i1, 9 * tig + 4);
    const unsigned colmask = 0x11111111u << tig;
    float a0 = c0[0], a1 = c0[1], a2 = c1[0], a3 = c1[1];  // row g
    float b0 = c0[2], b1 = c0[3], b2 = c1[2], b3 = c1[3];  // row g + 8
    lightning_column<STAGED>(a0, b0, c_lo, inv0, inv_a, inv_b, rva, rvb, g, colmask, p);
    lightning_column<STAGED>(a1, b1, c_lo + 1, inv1, inv_a, inv_b, rva, rvb, g, colmask, p);
    lightning_column<STAGED>(a2, b2, c_hi, inv2, inv_a, inv_b, rva, rvb, g, colmask, p);
    lightning_column<STAGED>(a3, b3, c_hi + 1, inv3, inv_a, inv_b, rva, rvb, g, colmask, p);
    float rs0 = a0 + a1 + a2 + a3;
    float rs1 = b0 + b1 + b2 + b3;
    rs0 += __shfl_xor_sync(0xFFFFFFFFu, rs0, 1);
    rs0 += __shfl_xor_sync(0xFFFFFFFFu, rs0, 2);
    rs1 += __shfl_xor_sync(0xFFFFFFFFu, rs1, 1);
    rs1 += __shfl_xor_sync(0xFFFFFFFFu, rs1, 2);
    return make_float2(rs0, rs1);
}

}  // namespace zp
