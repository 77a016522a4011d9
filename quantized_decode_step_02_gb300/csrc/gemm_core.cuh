// gemm_core.cuh -- the per-stage Q4_K x activation arithmetic of the
// projection kernel (gemm.cu): the stage buffer layout, the tile-block decode
// into mma A fragments, and one warp's contribution of a 16-row tile block
// times the staged activations.
#pragma once
#include "zdec_kernels.cuh"

namespace zdec {

constexpr uint32_t FULL = 0xFFFFFFFFu;
constexpr uint32_t LO_SKEW = 64;   // bytes between the hi and lo planes of a stage

// Stage layout for a kernel covering BR = 4*NT batch rows (B of them real):
//   [0, GROUP_BYTES)                 tile blocks of the group
//   hi plane  BR x 512 bytes, LO_SKEW gap, lo plane BR x 512 bytes,
//   sums BR x 32 bytes, then BR x 32 zero bytes (the lo lanes' min-term slots).
// The bulk copies fill the first B rows of each plane; rows B..BR-1 are zeroed
// once per stage buffer, so every lane reads its rows unconditionally.
struct StageLayout {
    uint32_t hi, lo, sums, zero, bytes;
    __host__ __device__ StageLayout(int BR) {
        hi = GROUP_BYTES;
        lo = hi + (uint32_t)BR * 512u + LO_SKEW;
        sums = lo + (uint32_t)BR * 512u;
        zero = sums + (uint32_t)BR * 32u;
        bytes = (zero + (uint32_t)BR * 32u + 127u) & ~127u;
    }
};

// ------------------------------------------------------- tile decoding ---
struct TileMeta {
    __half2 cg0, cg1, c80, c81;   // (sc, sc) for row g / g+8, sub-block j1 (0) / j2 (1)
    __half2 og0, og1, o80, o81;   // (-1024 sc, -1024 sc)
    uint32_t mg, m8;              // (m_j1, m_j2) of row g / g+8 as fp16 pairs
    float dg, dming, d8, dmin8;
};

__device__ __forceinline__ void decode_meta(uint2 mt, int tig, TileMeta &t) {
    const __half2 k1024 = __float2half2_rn(1024.0f), kneg = __float2half2_rn(-1024.0f);
    uint32_t lo = mt.x, hi = mt.y;
    __half2 scg = __hsub2(u32_as_h2(lop3_and_or(lo, 0x003F003Fu, 0x64006400u)), k1024);
    __half2 sc8 = __hsub2(u32_as_h2(lop3_and_or(hi, 0x003F003Fu, 0x64006400u)), k1024);
    t.cg0 = __low2half2(scg); t.cg1 = __high2half2(scg);
    t.c80 = __low2half2(sc8); t.c81 = __high2half2(sc8);
    t.og0 = __hmul2(t.cg0, kneg); t.og1 = __hmul2(t.cg1, kneg);
    t.o80 = __hmul2(t.c80, kneg); t.o81 = __hmul2(t.c81, kneg);
    t.mg = h2_as_u32(__hsub2(u32_as_h2(lop3_and_or(lo >> 6, 0x003F003Fu, 0x64006400u)), k1024));
    t.m8 = h2_as_u32(__hsub2(u32_as_h2(lop3_and_or(hi >> 6, 0x003F003Fu, 0x64006400u)), k1024));
    uint32_t dq = ((lo >> 12) & 0xFu) | ((lo >> 24) & 0xF0u) | ((hi >> 4) & 0xF00u) |
                  ((hi >> 16) & 0xF000u);
    uint32_t other = __shfl_xor_sync(FULL, dq, 1);
    uint32_t pair = (tig & 1) ? (other | (dq << 16)) : (dq | (other << 16));   // (d, dmin)
    uint32_t pair2 = __shfl_xor_sync(FULL, pair, 2);
    float2 fg = __half22float2(u32_as_h2(tig < 2 ? pair : pair2));
    float2 f8 = __half22float2(u32_as_h2(tig < 2 ? pair2 : pair));
    t.dg = fg.x; t.dming = fg.y; t.d8 = f8.x; t.dmin8 = f8.y;
}

// The eight A-operand pairs of one code word: lo/lo16 from offsets (0,1)/(4,5),
// hi/hi16 from offsets (2,3)/(6,7), all as exact q*sc (16*q*sc for *16).
__device__ __forceinline__ void decode_word(uint32_t w, __half2 c, __half2 o, uint32_t &lo,
                                            uint32_t &lo16, uint32_t &hi, uint32_t &hi16) {
    uint32_t ws = w >> 8;
    lo = h2_as_u32(__hfma2(u32_as_h2(lop3_and_or(w, 0x000F000Fu, 0x64006400u)), c, o));
    lo16 = h2_as_u32(__hfma2(u32_as_h2(lop3_and_or(w, 0x00F000F0u, 0x64006400u)), c, o));
    hi = h2_as_u32(__hfma2(u32_as_h2(lop3_and_or(ws, 0x000F000Fu, 0x64006400u)), c, o));
    hi16 = h2_as_u32(__hfma2(u32_as_h2(lop3_and_or(ws, 0x00F000F0u, 0x64006400u)), c, o));
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }

__device__ __forceinline__ float dot2(uint32_t a, uint32_t x) {
    float2 fa = __half22float2(u32_as_h2(a)), fx = __half22float2(u32_as_h2(x));
    return fmaf(fa.x, fx.x, fa.y * fx.y);
}

// ------------------------------------------------------- stage compute ---
// Stage layout: [GROUP_BYTES tile blocks][hi rows B x 512][lo rows][sums B x 32].
//
// MMA columns are "virtual": column 2c of n-tile nt multiplies the hi plane of
// batch row b = 4nt + c, column 2c+1 its lo plane, so one 8-wide N tile carries
// four batch rows at full (hi + lo) precision and the lane holding C-fragment
// columns (2tig, 2tig+1) owns both halves of batch row 4nt + tig.
// acc[nt][0..3] = (row g, hi), (row g, lo), (row g+8, hi), (row g+8, lo).
// CHAINS: independent MMA accumulator chains per n-tile: 4 (two word pairs,
// and the x1 and x16 nibbles apart), 2 (word pairs) or 1; fewer chains free
// registers for more CTAs per SM, where the n-tiles already interleave.
template <int NT, int CHAINS = 4>
__device__ __forceinline__ void stage_mma(const uint8_t *st, int warp, int lane, uint32_t act_off,
                                          uint32_t sum_off, uint32_t swz, float (&acc)[NT][4]) {
    const int tig = lane & 3;
    const uint8_t *tile = st + warp * TILE_BYTES;
    const uint8_t *act = st + act_off;   // this lane's B column of n-tile 0 (see gemm_kernel)
    TileMeta tm;
    decode_meta(*reinterpret_cast<const uint2 *>(tile + TILE_CODE_BYTES + 8 * lane), tig, tm);
    // independent accumulator chains per n-tile, so a warp always has MMAs
    // whose inputs are ready
    constexpr int PP = CHAINS >= 2 ? 2 : 1;
    constexpr bool S16 = CHAINS >= 4;
    float tq[PP][NT][4], t16[S16 ? PP : 1][NT][4], tmin[NT][4];
    const float zero4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int k = 0; k < PP; k++)
#pragma unroll
        for (int nt = 0; nt < NT; nt++)
#pragma unroll
            for (int i = 0; i < 4; i++) tq[k][nt][i] = 0.0f;
#pragma unroll
    for (int k = 0; k < (S16 ? PP : 1); k++)
#pragma unroll
        for (int nt = 0; nt < NT; nt++)
#pragma unroll
            for (int i = 0; i < 4; i++) t16[k][nt][i] = 0.0f;
#pragma unroll
    for (int c = 0; c < 4; c++) {
        const int h = c >> 1;
        const __half2 cg = h ? tm.cg1 : tm.cg0, og = h ? tm.og1 : tm.og0;
        const __half2 c8 = h ? tm.c81 : tm.c80, o8 = h ? tm.o81 : tm.o80;
        const uint4 qc = *reinterpret_cast<const uint4 *>(tile + c * 512 + 16 * lane);   // codes of chunk c
#pragma unroll
        for (int pp = 0; pp < 2; pp++) {
            const int pidx = (c & 1) * 2 + pp;
            uint32_t w0 = pp ? qc.z : qc.x, w1 = pp ? qc.w : qc.y;
            uint32_t at[4], at16[4];
            decode_word(w0, cg, og, at[0], at16[0], at[2], at16[2]);
            decode_word(w1, c8, o8, at[1], at16[1], at[3], at16[3]);
            const uint32_t off = ((uint32_t)(h * 4 + pidx) ^ swz) * 16;
            const int k = PP == 2 ? pp : 0;
#pragma unroll
            for (int nt = 0; nt < NT; nt++) {
                const uint4 xv = *reinterpret_cast<const uint4 *>(act + nt * 2048 + off);
                mma16816(tq[k][nt], at, xv.x, xv.y, tq[k][nt]);
                if (S16) mma16816(t16[k][nt], at16, xv.z, xv.w, t16[k][nt]);
                else mma16816(tq[k][nt], at16, xv.z, xv.w, tq[k][nt]);
            }
        }
    }
    const uint32_t am[4] = {tm.mg, tm.m8, tm.mg, tm.m8};
#pragma unroll
    for (int nt = 0; nt < NT; nt++) {
        // the min term goes to the hi column only: lo lanes read a zero slot
        const uint2 s = *reinterpret_cast<const uint2 *>(st + sum_off + nt * 128);
        mma16816(tmin[nt], am, s.x, s.y, zero4);
        float sq[4];
#pragma unroll
        for (int i = 0; i < 4; i++) {
            sq[i] = tq[0][nt][i];
            if (PP == 2) sq[i] += tq[PP - 1][nt][i];
            if (S16) sq[i] += t16[0][nt][i] + t16[S16 ? PP - 1 : 0][nt][i];
        }
        acc[nt][0] += tm.dg * sq[0] - tm.dming * tmin[nt][0];
        acc[nt][1] += tm.dg * sq[1] - tm.dming * tmin[nt][1];
        acc[nt][2] += tm.d8 * sq[2] - tm.dmin8 * tmin[nt][2];
        acc[nt][3] += tm.d8 * sq[3] - tm.dmin8 * tmin[nt][3];
    }
}

// ------------------------------------------------------ batch of one ---
// B = 1: the mma as a dot-product engine with one column per sub-block.
//   A: the raw codes as fp16 subnormals, q * 2^-24 (one AND per two codes;
//      the high nibbles give 16q * 2^-24, their activations being stored
//      divided by 16), so no bias and no scale enter the operand;
//   B: column n = 2t + e of an mma carries the activations of sub-block
//      2t + h (e = 0: hi plane, 1: lo plane) in the k-slots of lane group
//      tig = t and zeros elsewhere.  A lane (g, tig) loads real activations
//      only when g = 2 tig (hi) or g = 2 tig + 1 (lo); the other lanes read a
//      zero row.
// D[row][2t + e] is then 2^-24 times the code-times-activation sum of one
// sub-block, and the C fragment hands lane (g, tig) exactly its own two
// sub-blocks for rows g and g + 8.
// Lane offsets inside a stage, fixed for the whole kernel.
struct MvOff {
    uint32_t codes;    // warp's tile block + 16 * lane
    uint32_t meta;     // warp's tile block + 2048 + 8 * lane
    uint32_t act[4];   // B-fragment row of word pair p (swizzled by tig); + 64 for sub-block h = 1
    uint32_t sums;     // this lane group's sub-block sums
};
// Accumulates this lane's share of rows g, g + 8 (sub-blocks 2 tig, 2 tig + 1
// of every super-block): yq += d * sum_j sc_j * D_j (still carrying 2^-24) and
// ym += dmin * sum_j m_j * S_j; the row is 2^24 yq - ym summed over its four
// lanes (done by the caller after the K loop).
__device__ __forceinline__ void stage_mv(const uint8_t *st, const MvOff &o, int tig, float (&yq)[2], float (&ym)[2]) {
    uint4 q[4];
#pragma unroll
    for (int c = 0; c < 4; c++) q[c] = *reinterpret_cast<const uint4 *>(st + o.codes + c * 512);
    const uint2 mt = *reinterpret_cast<const uint2 *>(st + o.meta);
    // d, dmin of rows g, g+8 (four nibble quarters spread over the tig lanes)
    uint32_t dq = ((mt.x >> 12) & 0xFu) | ((mt.x >> 24) & 0xF0u) | ((mt.y >> 4) & 0xF00u) | ((mt.y >> 16) & 0xF000u);
    const uint32_t other = __shfl_xor_sync(FULL, dq, 1);
    const uint32_t pair = (tig & 1) ? (other | (dq << 16)) : (dq | (other << 16));
    const uint32_t pair2 = __shfl_xor_sync(FULL, pair, 2);
    const float2 fg = __half22float2(u32_as_h2(tig < 2 ? pair : pair2));
    const float2 f8 = __half22float2(u32_as_h2(tig < 2 ? pair2 : pair));
    float D[2][2][4];   // [sub-block h][chain][c fragment]
#pragma unroll
    for (int h = 0; h < 2; h++)
#pragma unroll
        for (int k = 0; k < 2; k++)
#pragma unroll
            for (int i = 0; i < 4; i++) D[h][k][i] = 0.0f;
#pragma unroll
    for (int c = 0; c < 4; c++) {
        const int h = c >> 1;
#pragma unroll
        for (int pp = 0; pp < 2; pp++) {
            const int pidx = (c & 1) * 2 + pp;
            const uint32_t w0 = pp ? q[c].z : q[c].x, w1 = pp ? q[c].w : q[c].y;
            const uint32_t s0 = w0 >> 8, s1 = w1 >> 8;
            const uint32_t a[4] = {w0 & 0x000F000Fu, w1 & 0x000F000Fu, s0 & 0x000F000Fu, s1 & 0x000F000Fu};
            const uint32_t a16[4] = {w0 & 0x00F000F0u, w1 & 0x00F000F0u, s0 & 0x00F000F0u, s1 & 0x00F000F0u};
            const uint4 xv = *reinterpret_cast<const uint4 *>(st + o.act[pidx] + h * 64);
            mma16816(D[h][c & 1], a, xv.x, xv.y, D[h][c & 1]);
            mma16816(D[h][c & 1], a16, xv.z, xv.w, D[h][c & 1]);
        }
    }
    const uint2 sv = *reinterpret_cast<const uint2 *>(st + o.sums);   // (S hi 2tig, 2tig+1, S lo 2tig, 2tig+1)
    const float2 shi = __half22float2(u32_as_h2(sv.x)), slo = __half22float2(u32_as_h2(sv.y));
    const float S0 = shi.x + slo.x, S1 = shi.y + slo.y;
#pragma unroll
    for (int r = 0; r < 2; r++) {   // row g (meta low word), row g + 8 (high word)
        const uint32_t w = r ? mt.y : mt.x;
        // sub-block 2tig: sc bits 0-5, m bits 6-11; 2tig+1: sc 16-21, m 22-27
        const float sc0 = (float)(w & 63u), m0 = (float)((w >> 6) & 63u);
        const float sc1 = (float)((w >> 16) & 63u), m1 = (float)((w >> 22) & 63u);
        const float v0 = (D[0][0][2 * r] + D[0][1][2 * r]) + (D[0][0][2 * r + 1] + D[0][1][2 * r + 1]) * LO_UNSCALE;
        const float v1 = (D[1][0][2 * r] + D[1][1][2 * r]) + (D[1][0][2 * r + 1] + D[1][1][2 * r + 1]) * LO_UNSCALE;
        const float dd = r ? f8.x : fg.x, dm = r ? f8.y : fg.y;
        yq[r] = fmaf(dd, fmaf(sc1, v1, sc0 * v0), yq[r]);
        ym[r] = fmaf(dm, fmaf(m1, S1, m0 * S0), ym[r]);
    }
}

}  // namespace zdec
