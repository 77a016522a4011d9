// attn_core.cuh -- one warp's share of one 32-token KV unit (flash-decode
// step with online softmax), shared by the attention kernel (attention.cu) and
// the persistent step kernel (step.cu).  The unit sits in shared memory exactly
// as the KV arena stores it (layout and swizzles in zdec_internal.cuh):
//   fp16: K [32 tokens][128] half at 0, V [128 dims][32 tokens] half at 8192;
//   Q8_0: K codes at 0, K scales [32][4] at 4096, V codes [128][32] at 4352,
//         V scales [4][32] at 8448.
#pragma once
#include "zdec_kernels.cuh"

namespace zdec {

constexpr uint32_t UNIT_BYTES_F16 = 16384;
constexpr uint32_t UNIT_BYTES_Q8 = 8704;

// One 32-token unit, one warp: scores of the unit's tokens for the 4 heads
// (rows 0-3 q hi, 8-11 q lo), online softmax, and P V for this warp's 64 head
// dims (dim half hh).  Tokens >= nv are masked (and their V zeroed).
template <int KVT>
__device__ __forceinline__ void att_unit(uint8_t *st, int nv, int hh, const uint32_t (&qa)[8][4], float &m_run,
                                         float &l_run, float (&oacc)[8][4]) {
    const int lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
    const float zero4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    constexpr uint32_t FULLM = 0xFFFFFFFFu;
    if (KVT == 0 && nv < KU) {   // fp16 V past the live tokens may hold anything: zero this warp's rows
        for (int i = lane; i < 64 * (KU - nv); i += 32) {
            const int dd = 64 * hh + i / (KU - nv), tt = nv + i % (KU - nv);
            *reinterpret_cast<uint16_t *>(st + 8192 + (size_t)kv_v16_off(dd, tt)) = 0;
        }
        __syncwarp();
    }
    float sc[2][4];
#pragma unroll
    for (int kg = 0; kg < 2; kg++) {
        float S[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; nt++) {
            const int tr = 16 * kg + 4 * (gid >> 1) + 2 * nt + (gid & 1);   // token of B column gid
#pragma unroll
            for (int i = 0; i < 4; i++) S[nt][i] = 0.0f;
            if (KVT == 0) {
#pragma unroll
                for (int s8 = 0; s8 < 8; s8++) {
                    const uint2 kb = *reinterpret_cast<const uint2 *>(
                        st + (size_t)tr * 256 + ((((2 * s8 + (tig >> 1)) ^ (tr & 7)) << 4) | ((tig & 1) << 3)));
                    mma16816(S[nt], qa[s8], kb.x, kb.y, S[nt]);
                }
            } else {
                const uint16_t *ks = reinterpret_cast<const uint16_t *>(st + 4096);
                const int ta = 16 * kg + 4 * tig + 2 * nt;   // tokens of C columns 2tig, 2tig+1
#pragma unroll
                for (int bl = 0; bl < 4; bl++) {
                    float tmp[4];
#pragma unroll
                    for (int hs = 0; hs < 2; hs++) {
                        const int s8 = 2 * bl + hs;
                        const uint32_t w = *reinterpret_cast<const uint32_t *>(
                            st + (size_t)tr * 128 + (((s8 ^ (tr & 7)) << 4) | (tig << 2)));
                        uint32_t b0, b1;
                        {
                            const uint32_t u = w ^ 0x80808080u;
                            const __half2 bias = __float2half2_rn(1152.0f);
                            b0 = h2_as_u32(__hsub2(u32_as_h2(__byte_perm(u, 0x64646464u, 0x4140)), bias));
                            b1 = h2_as_u32(__hsub2(u32_as_h2(__byte_perm(u, 0x64646464u, 0x4342)), bias));
                        }
                        if (hs) mma16816(tmp, qa[s8], b0, b1, tmp);
                        else mma16816(tmp, qa[s8], b0, b1, zero4);
                    }
                    const float ka = __half2float(__ushort_as_half(ks[ta * 4 + bl]));
                    const float kb = __half2float(__ushort_as_half(ks[(ta + 1) * 4 + bl]));
                    S[nt][0] += ka * tmp[0];
                    S[nt][1] += kb * tmp[1];
                    S[nt][2] += ka * tmp[2];
                    S[nt][3] += kb * tmp[3];
                }
            }
        }
        sc[kg][0] = S[0][0] + S[0][2];
        sc[kg][1] = S[0][1] + S[0][3];
        sc[kg][2] = S[1][0] + S[1][2];
        sc[kg][3] = S[1][1] + S[1][3];
#pragma unroll
        for (int e = 0; e < 4; e++)
            if (16 * kg + 4 * tig + e >= nv || gid >= GROUP) sc[kg][e] = -INFINITY;
    }
    float mt = -INFINITY;
#pragma unroll
    for (int kg = 0; kg < 2; kg++)
#pragma unroll
        for (int e = 0; e < 4; e++) mt = fmaxf(mt, sc[kg][e]);
    mt = fmaxf(mt, __shfl_xor_sync(FULLM, mt, 1));
    mt = fmaxf(mt, __shfl_xor_sync(FULLM, mt, 2));
    const float m_new = fmaxf(m_run, mt);
    float alpha = 1.0f, pr[2][4];
#pragma unroll
    for (int kg = 0; kg < 2; kg++)
#pragma unroll
        for (int e = 0; e < 4; e++) pr[kg][e] = 0.0f;
    if (m_new != -INFINITY) {
        alpha = expf(m_run - m_new);
#pragma unroll
        for (int kg = 0; kg < 2; kg++)
#pragma unroll
            for (int e = 0; e < 4; e++) pr[kg][e] = expf(sc[kg][e] - m_new);
    }
    m_run = m_new;
    l_run = l_run * alpha + ((pr[0][0] + pr[0][1]) + (pr[0][2] + pr[0][3])) + ((pr[1][0] + pr[1][1]) + (pr[1][2] + pr[1][3]));
#pragma unroll
    for (int dn = 0; dn < 8; dn++)
#pragma unroll
        for (int i = 0; i < 4; i++) oacc[dn][i] *= alpha;
#pragma unroll
    for (int kg = 0; kg < 2; kg++) {
        const int t0 = 16 * kg + 4 * tig;   // this lane's four tokens
        if (KVT == 0) {
            uint32_t pa[4];
            const __half2 h01 = __floats2half2_rn(pr[kg][0], pr[kg][1]), h23 = __floats2half2_rn(pr[kg][2], pr[kg][3]);
            const float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
            pa[0] = h2_as_u32(h01);
            pa[1] = h2_as_u32(__floats2half2_rn(pr[kg][0] - f01.x, pr[kg][1] - f01.y));
            pa[2] = h2_as_u32(h23);
            pa[3] = h2_as_u32(__floats2half2_rn(pr[kg][2] - f23.x, pr[kg][3] - f23.y));
#pragma unroll
            for (int dn = 0; dn < 8; dn++) {
                const int dd = 64 * hh + 8 * dn + gid;
                const uint2 vb = *reinterpret_cast<const uint2 *>(
                    st + 8192 + (size_t)dd * 64 + ((((t0 >> 3) ^ ((dd >> 1) & 3)) << 4) | ((t0 & 7) << 1)));
                mma16816(oacc[dn], pa, vb.x, vb.y, oacc[dn]);
            }
        } else {
            const uint16_t *vs = reinterpret_cast<const uint16_t *>(st + 8448);
#pragma unroll
            for (int bq = 0; bq < 2; bq++) {
                const int bl = 2 * hh + bq;   // this warp's 32-dim blocks
                float q4[4];
#pragma unroll
                for (int e = 0; e < 4; e++) q4[e] = pr[kg][e] * __half2float(__ushort_as_half(vs[bl * KU + t0 + e]));
                uint32_t pa[4];
                const __half2 h01 = __floats2half2_rn(q4[0], q4[1]), h23 = __floats2half2_rn(q4[2], q4[3]);
                const float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
                pa[0] = h2_as_u32(h01);
                pa[1] = h2_as_u32(__floats2half2_rn(q4[0] - f01.x, q4[1] - f01.y));
                pa[2] = h2_as_u32(h23);
                pa[3] = h2_as_u32(__floats2half2_rn(q4[2] - f23.x, q4[3] - f23.y));
#pragma unroll
                for (int dq = 0; dq < 4; dq++) {
                    const int dd = 32 * bl + 8 * dq + gid;
                    const uint32_t w = *reinterpret_cast<const uint32_t *>(
                        st + 4352 + (size_t)dd * 32 + ((((t0 >> 4) ^ ((dd >> 2) & 1)) << 4) | (t0 & 15)));
                    uint32_t b0, b1;
                    const uint32_t u = w ^ 0x80808080u;
                    const __half2 bias = __float2half2_rn(1152.0f);
                    b0 = h2_as_u32(__hsub2(u32_as_h2(__byte_perm(u, 0x64646464u, 0x4140)), bias));
                    b1 = h2_as_u32(__hsub2(u32_as_h2(__byte_perm(u, 0x64646464u, 0x4342)), bias));
                    mma16816(oacc[4 * bq + dq], pa, b0, b1, oacc[4 * bq + dq]);
                }
            }
        }
    }
}

}  // namespace zdec
