// gemm.cu -- the shared Q4_K weight stream times B activation rows.
//
// One read of every weight per decode step, multiplied against all B hidden
// states ("The weight read is the only term that does not scale": a step that
// advances eight sequences loads each weight tile once and multiplies eight
// hidden states against it).  Two kernels do this:
//   * gemm_mma_kernel: mma.sync.m16n8k16 with the weight rows in the MMA M
//     slot (16 rows per tile) and the batch in N (8 per tile, zero padded);
//     the dense-matrix-core path the pages switch to past about four
//     sequences ("RDNA4 pads the batch dimension to 16").
//   * gemm_matvec_kernel: the same tile blocks through CUDA-core fp32 FMAs,
//     the dequant-matvec of the batch-one path.
// Both dequantize in registers: one lop3 turns two 4-bit codes into the fp16
// pair (1024+q, 1024+q') (or 1024+16q for the high nibbles), one HFMA2 with
// (sc, sc) and (-1024 sc, -1024 sc) turns that into the exact integers q*sc
// (or 16*q*sc).  Sub-block scales therefore live in the A operand, a whole
// 256-column super-block accumulates in fp32 inside the tensor core, and the
// epilogue applies d and the min term: y += d*acc_q - dmin*acc_m, where
// acc_m = sum_j m_j * S_j comes from one more MMA against the per-sub-block
// activation sums S_j (split as hi + lo fp16).
#include "zdec_kernels.cuh"

namespace zdec {

constexpr uint32_t FULL = 0xFFFFFFFFu;

// ------------------------------------------------------------------ prep ---
// Block b converts fp32 row b into the GEMM operand: fp16 values (offsets 4..7
// of every group of 8 divided by 16, matching the tile-block nibble layout) and
// per-32 sub-block sums of the fp16 values, stored as hi + lo fp16 at
// sx[b][sb][tig] = {(hi_2tig, hi_2tig+1), (lo_2tig, lo_2tig+1)}.
template <bool NORM>
__global__ __launch_bounds__(512) void prep_kernel(const float *__restrict__ src, int lds, int K,
                                                   const float *__restrict__ gain, float eps, int B,
                                                   __half *__restrict__ x16, __half *__restrict__ sxh) {
    pdl_launch_dependents();
    pdl_wait();
    int b = blockIdx.x;
    int nsb = K / QK, nchunks = K / 8;
    __half *xo = x16 + (size_t)b * K;
    __half *so = sxh + (size_t)b * nsb * 16;
    if (b >= B) {   // padding row of the MMA N tile
        for (int c = threadIdx.x; c < nchunks; c += blockDim.x)
            *reinterpret_cast<uint4 *>(xo + 8 * c) = make_uint4(0, 0, 0, 0);
        for (int i = threadIdx.x; i < nsb * 16; i += blockDim.x) so[i] = __ushort_as_half(0);
        return;
    }
    const float *xr = src + (size_t)b * lds;
    float r = 1.0f;
    if (NORM) {
        __shared__ float red[32];
        float ss = 0.0f;
        for (int k = threadIdx.x; k < K; k += blockDim.x) ss = fmaf(xr[k], xr[k], ss);
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(FULL, ss, o);
        if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
        __syncthreads();
        if (threadIdx.x < 32) {
            float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.0f;
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
            if (threadIdx.x == 0) red[0] = v;
        }
        __syncthreads();
        r = 1.0f / sqrtf(red[0] / (float)K + eps);
    }
    const __half sixteenth = __float2half(0.0625f);
    for (int c = threadIdx.x; c < nchunks; c += blockDim.x) {   // nchunks % 32 == 0: warp-uniform
        float4 v0 = *reinterpret_cast<const float4 *>(xr + 8 * c);
        float4 v1 = *reinterpret_cast<const float4 *>(xr + 8 * c + 4);
        float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        __half h[8];
        float part = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; i++) {
            float y = NORM ? (v[i] * r) * gain[8 * c + i] : v[i];
            h[i] = __float2half_rn(y);
            part += __half2float(h[i]);
        }
#pragma unroll
        for (int i = 4; i < 8; i++) h[i] = __hmul(h[i], sixteenth);
        uint4 out;
        out.x = h2_as_u32(__halves2half2(h[0], h[1]));
        out.y = h2_as_u32(__halves2half2(h[2], h[3]));
        out.z = h2_as_u32(__halves2half2(h[4], h[5]));
        out.w = h2_as_u32(__halves2half2(h[6], h[7]));
        *reinterpret_cast<uint4 *>(xo + 8 * c) = out;
        part += __shfl_xor_sync(FULL, part, 1);
        part += __shfl_xor_sync(FULL, part, 2);
        if ((c & 3) == 0) {
            int sb = c >> 5, j = (c & 31) >> 2, tig = j >> 1, hh = j & 1;
            __half hi = __float2half_rn(part);
            __half lo = __float2half_rn(part - __half2float(hi));
            so[(sb * 4 + tig) * 4 + hh] = hi;
            so[(sb * 4 + tig) * 4 + 2 + hh] = lo;
        }
    }
}

cudaError_t launch_prep(const float *src, int lds, int K, const float *gain, float eps, int B,
                        int Bp, __half *x16, uint2 *sx, bool pdl, cudaStream_t stream) {
    int threads = K / 8 < 512 ? K / 8 : 512;
    __half *sxh = reinterpret_cast<__half *>(sx);
    if (gain)
        return launch_k(prep_kernel<true>, dim3(Bp), dim3(threads), 0, pdl, stream, src, lds, K,
                        gain, eps, B, x16, sxh);
    return launch_k(prep_kernel<false>, dim3(Bp), dim3(threads), 0, pdl, stream, src, lds, K,
                    gain, eps, B, x16, sxh);
}

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

// ------------------------------------------------------------ epilogue ---
// acc[nt][i] follows the mma C fragment: i = 0,1 -> row g, cols 2tig, 2tig+1;
// i = 2,3 -> row g+8.  Row tile rt, column tile nt covers batch rows 8nt..8nt+7.
template <int NT, int EPI>
__device__ __forceinline__ void gemm_epilogue(const GemmParams &p, float (&acc)[NT][4], bool active,
                                              int rt, int warp, int lane, float *s_amax_v,
                                              int *s_amax_i) {
    int g = lane >> 2, tig = lane & 3;
    if (EPI == EPI_STORE || EPI == EPI_RESID) {
        if (!active) return;
#pragma unroll
        for (int nt = 0; nt < NT; nt++)
#pragma unroll
            for (int i = 0; i < 4; i++) {
                int row = rt * 16 + g + (i >= 2 ? 8 : 0), col = 8 * nt + 2 * tig + (i & 1);
                if (col < p.B && row < p.N) {
                    float *o = p.out + (size_t)col * p.ldo + row;
                    if (EPI == EPI_STORE) *o = acc[nt][i];
                    else *o += acc[nt][i];
                }
            }
    } else if (EPI == EPI_SWIGLU) {
        if (!active) return;
        int f = rt * 8 + g;
#pragma unroll
        for (int nt = 0; nt < NT; nt++)
#pragma unroll
            for (int e = 0; e < 2; e++) {
                int col = 8 * nt + 2 * tig + e;
                if (col < p.B && f < p.N)
                    p.out[(size_t)col * p.ldo + f] = silu_f(acc[nt][e]) * acc[nt][2 + e];
            }
    } else {   // EPI_LMHEAD: logits and the CTA's argmax partial per batch row
#pragma unroll
        for (int nt = 0; nt < NT; nt++)
#pragma unroll
            for (int e = 0; e < 2; e++) {
                int col = 8 * nt + 2 * tig + e;
                int r0 = rt * 16 + g, r1 = r0 + 8;
                float v0 = (active && r0 < p.N) ? acc[nt][e] : -INFINITY;
                float v1 = (active && r1 < p.N) ? acc[nt][2 + e] : -INFINITY;
                if (active && p.out && col < p.B) {
                    if (r0 < p.N) p.out[(size_t)col * p.ldo + r0] = acc[nt][e];
                    if (r1 < p.N) p.out[(size_t)col * p.ldo + r1] = acc[nt][2 + e];
                }
                float bv = v0;
                int bi = r0;
                if (v1 > bv) { bv = v1; bi = r1; }
                for (int o = 4; o < 32; o <<= 1) {   // across g, lowest index on ties
                    float ov = __shfl_xor_sync(FULL, bv, o);
                    int oi = __shfl_xor_sync(FULL, bi, o);
                    if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
                }
                if (g == 0) {
                    s_amax_v[warp * (NT * 8) + col] = bv;
                    s_amax_i[warp * (NT * 8) + col] = bi;
                }
            }
    }
}

// K-split reduction through shared memory, then the epilogue on split 0.
template <int NT, int EPI>
__device__ __forceinline__ void gemm_finish(const GemmParams &p, float (&acc)[NT][4], bool valid,
                                            int rt) {
    __shared__ float red[8][NT][4][32];
    __shared__ float s_amax_v[8 * NT * 8];
    __shared__ int s_amax_i[8 * NT * 8];
    int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int RT = p.rt_per_cta, KS = p.ksplit;
    int rtl = warp % RT, ks = warp / RT;
    if (KS > 1) {
        if (ks > 0)
#pragma unroll
            for (int nt = 0; nt < NT; nt++)
#pragma unroll
                for (int i = 0; i < 4; i++) red[warp][nt][i][lane] = acc[nt][i];
        __syncthreads();
        if (ks == 0)
            for (int k2 = 1; k2 < KS; k2++) {
                int w2 = rtl + k2 * RT;
#pragma unroll
                for (int nt = 0; nt < NT; nt++)
#pragma unroll
                    for (int i = 0; i < 4; i++) acc[nt][i] += red[w2][nt][i][lane];
            }
    }
    gemm_epilogue<NT, EPI>(p, acc, valid && ks == 0, rt, warp, lane, s_amax_v, s_amax_i);
    if (EPI == EPI_LMHEAD) {
        __syncthreads();
        if ((int)threadIdx.x < NT * 8) {
            int col = threadIdx.x;
            float bv = -INFINITY;
            int bi = 0x7FFFFFFF;
            for (int w = 0; w < RT; w++) {   // split-0 warps, increasing rows
                float v = s_amax_v[w * (NT * 8) + col];
                int i = s_amax_i[w * (NT * 8) + col];
                if (v > bv || (v == bv && i < bi)) { bv = v; bi = i; }
            }
            if (col < p.B) {
                p.amax_val[blockIdx.x * MAX_B + col] = bv;
                p.amax_idx[blockIdx.x * MAX_B + col] = bi;
            }
        }
    }
}

// L2 prefetch of the CTA's contiguous run of tile blocks.  Weights never
// change during a step, so this is issued before the dependency wait.
__device__ __forceinline__ void prefetch_cta_weights(const GemmParams &p) {
    int rt0 = blockIdx.x * p.rt_per_cta;
    int n = min(p.rt_per_cta, p.nrt - rt0);
    const uint8_t *base = p.W + (size_t)rt0 * p.nsb * TILE_BYTES;
    size_t bytes = (size_t)n * p.nsb * TILE_BYTES;
    for (size_t off = (size_t)threadIdx.x * 4096; off < bytes; off += (size_t)blockDim.x * 4096)
        prefetch_l2(base + off, (uint32_t)min((size_t)4096, bytes - off));
}

// ---------------------------------------------------------- mma kernel ---
template <int NT, int EPI>
__global__ __launch_bounds__(256, (NT <= 2 ? 2 : 1)) void gemm_mma_kernel(const GemmParams p) {
    int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int g = lane >> 2, tig = lane & 3;
    int RT = p.rt_per_cta, KS = p.ksplit;
    int rtl = warp % RT, ks = warp / RT;
    int rt = blockIdx.x * RT + rtl;
    bool valid = rt < p.nrt;
    prefetch_cta_weights(p);
    pdl_launch_dependents();
    pdl_wait();

    const int K = p.nsb * QK;
    int sb0 = ks * p.nsb / KS, sb1 = (ks + 1) * p.nsb / KS;
    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; nt++)
#pragma unroll
        for (int i = 0; i < 4; i++) acc[nt][i] = 0.0f;
    const float zero4[4] = {0.0f, 0.0f, 0.0f, 0.0f};

    if (valid && sb0 < sb1) {
        const uint8_t *tile = p.W + ((size_t)rt * p.nsb + sb0) * TILE_BYTES;
        uint4 q[4];
        uint2 mt;
#pragma unroll
        for (int c = 0; c < 4; c++) q[c] = ld_stream_u4(tile + c * 512 + 16 * lane);
        mt = ld_stream_u2(tile + TILE_CODE_BYTES + 8 * lane);
        for (int sb = sb0; sb < sb1; sb++) {
            // issue the next tile block's loads before working on this one
            uint4 qn[4];
            uint2 mtn;
            if (sb + 1 < sb1) {
                const uint8_t *tn = tile + TILE_BYTES;
#pragma unroll
                for (int c = 0; c < 4; c++) qn[c] = ld_stream_u4(tn + c * 512 + 16 * lane);
                mtn = ld_stream_u2(tn + TILE_CODE_BYTES + 8 * lane);
            }
            TileMeta tm;
            decode_meta(mt, tig, tm);
            float tq[NT][4], tmin[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; nt++)
#pragma unroll
                for (int i = 0; i < 4; i++) tq[nt][i] = 0.0f;
#pragma unroll
            for (int c = 0; c < 4; c++) {
                const int h = c >> 1;
                const __half2 cg = h ? tm.cg1 : tm.cg0, og = h ? tm.og1 : tm.og0;
                const __half2 c8 = h ? tm.c81 : tm.c80, o8 = h ? tm.o81 : tm.o80;
#pragma unroll
                for (int pp = 0; pp < 2; pp++) {
                    const int pidx = (c & 1) * 2 + pp;
                    uint32_t w0 = pp ? q[c].z : q[c].x, w1 = pp ? q[c].w : q[c].y;
                    uint32_t at[4], at16[4];
                    decode_word(w0, cg, og, at[0], at16[0], at[2], at16[2]);
                    decode_word(w1, c8, o8, at[1], at16[1], at[3], at16[3]);
                    const int koff = sb * QK + 32 * (2 * tig + h) + 8 * pidx;
#pragma unroll
                    for (int nt = 0; nt < NT; nt++) {
                        uint4 xv = ld_u4(p.x16 + (size_t)(8 * nt + g) * K + koff);
                        mma16816(tq[nt], at, xv.x, xv.y, tq[nt]);
                        mma16816(tq[nt], at16, xv.z, xv.w, tq[nt]);
                    }
                }
            }
            const uint32_t am[4] = {tm.mg, tm.m8, tm.mg, tm.m8};
#pragma unroll
            for (int nt = 0; nt < NT; nt++) {
                uint2 s = p.sx[((size_t)(8 * nt + g) * p.nsb + sb) * 4 + tig];
                mma16816(tmin[nt], am, s.x, s.y, zero4);
                acc[nt][0] += tm.dg * tq[nt][0] - tm.dming * tmin[nt][0];
                acc[nt][1] += tm.dg * tq[nt][1] - tm.dming * tmin[nt][1];
                acc[nt][2] += tm.d8 * tq[nt][2] - tm.dmin8 * tmin[nt][2];
                acc[nt][3] += tm.d8 * tq[nt][3] - tm.dmin8 * tmin[nt][3];
            }
            if (sb + 1 < sb1) {
#pragma unroll
                for (int c = 0; c < 4; c++) q[c] = qn[c];
                mt = mtn;
                tile += TILE_BYTES;
            }
        }
    }
    gemm_finish<NT, EPI>(p, acc, valid, rt);
}

// ------------------------------------------------------- matvec kernel ---
__device__ __forceinline__ float dot2(uint32_t a, uint32_t x) {
    float2 fa = __half22float2(u32_as_h2(a)), fx = __half22float2(u32_as_h2(x));
    return fmaf(fa.x, fx.x, fa.y * fx.y);
}

template <int NB, int EPI>
__global__ __launch_bounds__(256, 2) void gemm_matvec_kernel(const GemmParams p) {
    int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int tig = lane & 3;
    int RT = p.rt_per_cta, KS = p.ksplit;
    int rtl = warp % RT, ks = warp / RT;
    int rt = blockIdx.x * RT + rtl;
    bool valid = rt < p.nrt;
    prefetch_cta_weights(p);
    pdl_launch_dependents();
    pdl_wait();

    const int K = p.nsb * QK;
    int sb0 = ks * p.nsb / KS, sb1 = (ks + 1) * p.nsb / KS;
    float accr[NB][2];
#pragma unroll
    for (int c = 0; c < NB; c++) accr[c][0] = accr[c][1] = 0.0f;
    if (valid) {
        for (int sb = sb0; sb < sb1; sb++) {
            const uint8_t *tile = p.W + ((size_t)rt * p.nsb + sb) * TILE_BYTES;
            uint4 q[4];
#pragma unroll
            for (int c = 0; c < 4; c++) q[c] = ld_stream_u4(tile + c * 512 + 16 * lane);
            TileMeta tm;
            decode_meta(ld_stream_u2(tile + TILE_CODE_BYTES + 8 * lane), tig, tm);
            float sq[NB][2];
#pragma unroll
            for (int c = 0; c < NB; c++) sq[c][0] = sq[c][1] = 0.0f;
#pragma unroll
            for (int c = 0; c < 4; c++) {
                const int h = c >> 1;
                const __half2 cg = h ? tm.cg1 : tm.cg0, og = h ? tm.og1 : tm.og0;
                const __half2 c8 = h ? tm.c81 : tm.c80, o8 = h ? tm.o81 : tm.o80;
#pragma unroll
                for (int pp = 0; pp < 2; pp++) {
                    const int pidx = (c & 1) * 2 + pp;
                    uint32_t w0 = pp ? q[c].z : q[c].x, w1 = pp ? q[c].w : q[c].y;
                    uint32_t a0, a016, a0h, a0h16, a1, a116, a1h, a1h16;
                    decode_word(w0, cg, og, a0, a016, a0h, a0h16);
                    decode_word(w1, c8, o8, a1, a116, a1h, a1h16);
                    const int koff = sb * QK + 32 * (2 * tig + h) + 8 * pidx;
#pragma unroll
                    for (int col = 0; col < NB; col++) {
                        uint4 xv = ld_u4(p.x16 + (size_t)col * K + koff);
                        sq[col][0] += dot2(a0, xv.x) + dot2(a0h, xv.y) + dot2(a016, xv.z) + dot2(a0h16, xv.w);
                        sq[col][1] += dot2(a1, xv.x) + dot2(a1h, xv.y) + dot2(a116, xv.z) + dot2(a1h16, xv.w);
                    }
                }
            }
            float2 mg = __half22float2(u32_as_h2(tm.mg)), m8 = __half22float2(u32_as_h2(tm.m8));
#pragma unroll
            for (int col = 0; col < NB; col++) {
                uint2 s = p.sx[((size_t)col * p.nsb + sb) * 4 + tig];
                float2 hi = __half22float2(u32_as_h2(s.x)), lo = __half22float2(u32_as_h2(s.y));
                float s1 = hi.x + lo.x, s2 = hi.y + lo.y;
                accr[col][0] += tm.dg * sq[col][0] - tm.dming * (mg.x * s1 + mg.y * s2);
                accr[col][1] += tm.d8 * sq[col][1] - tm.dmin8 * (m8.x * s1 + m8.y * s2);
            }
        }
    }
    // every lane of a quad holds a quarter of each row's sum: butterfly over tig
#pragma unroll
    for (int c = 0; c < NB; c++)
#pragma unroll
        for (int r = 0; r < 2; r++) {
            accr[c][r] += __shfl_xor_sync(FULL, accr[c][r], 1);
            accr[c][r] += __shfl_xor_sync(FULL, accr[c][r], 2);
        }
    // into the mma C-fragment layout so the epilogue is shared
    float acc[1][4];
#pragma unroll
    for (int i = 0; i < 4; i++) {
        int col = 2 * tig + (i & 1), r = i >> 1;
        float v = 0.0f;
#pragma unroll
        for (int c = 0; c < NB; c++)
            if (c == col) v = accr[c][r];
        acc[0][i] = v;
    }
    gemm_finish<1, EPI>(p, acc, valid, rt);
}

// ------------------------------------------------------------ dispatch ---
int gemm_grid(const GemmParams &p) { return (p.nrt + p.rt_per_cta - 1) / p.rt_per_cta; }

template <int EPI>
static cudaError_t launch_gemm_epi(const GemmParams &p, int impl, bool pdl, cudaStream_t s) {
    dim3 grid(gemm_grid(p)), block(256);
    if (impl == 1) {
        switch (p.B) {
            case 1: return launch_k(gemm_matvec_kernel<1, EPI>, grid, block, 0, pdl, s, p);
            case 2: return launch_k(gemm_matvec_kernel<2, EPI>, grid, block, 0, pdl, s, p);
            case 3: return launch_k(gemm_matvec_kernel<3, EPI>, grid, block, 0, pdl, s, p);
            case 4: return launch_k(gemm_matvec_kernel<4, EPI>, grid, block, 0, pdl, s, p);
            default: return cudaErrorInvalidValue;
        }
    }
    switch ((p.B + 7) / 8) {
        case 1: return launch_k(gemm_mma_kernel<1, EPI>, grid, block, 0, pdl, s, p);
        case 2: return launch_k(gemm_mma_kernel<2, EPI>, grid, block, 0, pdl, s, p);
        case 3: return launch_k(gemm_mma_kernel<3, EPI>, grid, block, 0, pdl, s, p);
        case 4: return launch_k(gemm_mma_kernel<4, EPI>, grid, block, 0, pdl, s, p);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_gemm(const GemmParams &p, int epi, int impl, bool pdl, cudaStream_t stream) {
    if (p.rt_per_cta * p.ksplit != 8) return cudaErrorInvalidValue;
    switch (epi) {
        case EPI_STORE: return launch_gemm_epi<EPI_STORE>(p, impl, pdl, stream);
        case EPI_RESID: return launch_gemm_epi<EPI_RESID>(p, impl, pdl, stream);
        case EPI_SWIGLU: return launch_gemm_epi<EPI_SWIGLU>(p, impl, pdl, stream);
        case EPI_LMHEAD: return launch_gemm_epi<EPI_LMHEAD>(p, impl, pdl, stream);
    }
    return cudaErrorInvalidValue;
}

// --------------------------------------------------------- argmax final ---
__global__ void argmax_final_kernel(const float *__restrict__ vals, const int *__restrict__ idxs,
                                    int nparts, int B, int32_t *ids, const int32_t *positions,
                                    int32_t *len_dev) {
    pdl_launch_dependents();
    pdl_wait();
    int b = blockIdx.x;
    __shared__ float sv[32];
    __shared__ int si[32];
    float bv = -INFINITY;
    int bi = 0x7FFFFFFF;
    for (int i = threadIdx.x; i < nparts; i += blockDim.x) {
        float v = vals[i * MAX_B + b];
        int ix = idxs[i * MAX_B + b];
        if (v > bv || (v == bv && ix < bi)) { bv = v; bi = ix; }
    }
    for (int o = 16; o > 0; o >>= 1) {
        float ov = __shfl_xor_sync(FULL, bv, o);
        int oi = __shfl_xor_sync(FULL, bi, o);
        if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
    }
    if ((threadIdx.x & 31) == 0) { sv[threadIdx.x >> 5] = bv; si[threadIdx.x >> 5] = bi; }
    __syncthreads();
    if (threadIdx.x == 0) {
        bv = sv[0]; bi = si[0];
        for (int w = 1; w < (int)(blockDim.x >> 5); w++)
            if (sv[w] > bv || (sv[w] == bv && si[w] < bi)) { bv = sv[w]; bi = si[w]; }
        ids[b] = bi == 0x7FFFFFFF ? 0 : bi;
        len_dev[b] = positions[b] + 1;
    }
}

cudaError_t launch_argmax_final(const float *amax_val, const int *amax_idx, int nparts, int B,
                                int32_t *ids, const int32_t *positions, int32_t *len_dev,
                                bool pdl, cudaStream_t stream) {
    return launch_k(argmax_final_kernel, dim3(B), dim3(256), 0, pdl, stream, amax_val, amax_idx,
                    nparts, B, ids, positions, len_dev);
}

}  // namespace zdec
