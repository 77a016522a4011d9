// gemm.cu -- the shared Q4_K weight stream times B activation rows.
//
// One read of every weight per decode step, multiplied against all B hidden
// states ("The weight read is the only term that does not scale": a step that
// advances eight sequences loads each weight tile once and multiplies eight
// hidden states against it).
//
// Kernel structure (gemm_kernel): a CTA owns one group of 8 row tiles
// (128 rows) and a range of 256-column super-blocks; warp w multiplies row
// tile w.  Stages of the range stream through a ring of shared-memory buffers
// with 1-D bulk copies (TMA) completing on one mbarrier per stage: each stage
// is the group's 18,432 contiguous bytes of tile blocks plus that
// super-block's activation rows.  Weight copies are issued before the
// programmatic-launch dependency wait (weights never depend on the previous
// kernel), activation copies after it.  Small matrices split K across a
// thread-block cluster: the peers store their partial tiles into rank 0's
// shared memory with st.async (counted on rank 0's mbarrier) and rank 0 sums
// them in rank order (no atomics).
//
// Arithmetic, per warp and super-block:
//   * dequant: one lop3 puts two 4-bit codes under the fp16 exponent of 1024;
//     one HFMA2 with (sc, sc) and (-1024 sc, -1024 sc) yields the exact
//     integers q*sc (16*q*sc for the high nibbles, whose activations are stored
//     divided by 16), so the sub-block scale lives in the A operand;
//   * IMPL 2: mma.sync.m16n8k16 with weight rows in M (16 per tile) and the
//     batch in N (8 per tile), fp32 accumulation over the whole super-block;
//     the batch is zero padded to 8 (the pages' 16-wide WMMA tile pads the
//     batch the same way, "RDNA4 pads the batch dimension to 16");
//     IMPL 1: the same operands through CUDA-core fp32 FMAs (the batch-one
//     dequant-matvec);
//   * epilogue: y += d*acc_q - dmin*acc_m, acc_m = sum_j m_j*S_j from one more
//     MMA against the per-sub-block activation sums S_j (hi + lo fp16).
// Activations arrive as fp16 hi + lo planes (~22 significant bits).
#include <cooperative_groups.h>

#include "gemm_core.cuh"

namespace cg = cooperative_groups;

namespace zdec {

// ------------------------------------------------------------------ prep ---
// Block b converts fp32 row b into the act planes (hi, lo) and sub-block sums.
// gain != nullptr applies RMSNorm: x * rsqrt(mean x^2 + eps) * gain.
template <bool NORM>
__global__ __launch_bounds__(512) void prep_kernel(const float *__restrict__ src, int lds, int K,
                                                   const float *__restrict__ gain, float eps, int Bp,
                                                   __half *__restrict__ hi, __half *__restrict__ lo,
                                                   __half *__restrict__ sums) {
    pdl_launch_dependents();
    pdl_wait();
    const int b = blockIdx.x, nchunks = K / 8;
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
    for (int c = threadIdx.x; c < nchunks; c += blockDim.x) {   // nchunks % 32 == 0: warp-uniform
        float4 v0 = *reinterpret_cast<const float4 *>(xr + 8 * c);
        float4 v1 = *reinterpret_cast<const float4 *>(xr + 8 * c + 4);
        float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        float y[8], part = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; i++) {
            y[i] = NORM ? (v[i] * r) * gain[8 * c + i] : v[i];
            part += y[i];
        }
        const int sb = c >> 5, cl = c & 31;
        store_act8(hi, lo, act_chunk(sb, b, cl, Bp), y);
        part += __shfl_xor_sync(FULL, part, 1);
        part += __shfl_xor_sync(FULL, part, 2);
        if ((c & 3) == 0) store_sum(sums, sb, b, cl >> 2, Bp, part);
    }
}

cudaError_t launch_prep(const float *src, int lds, int K, const float *gain, float eps, int B, int Bp,
                        __half *hi, __half *lo, __half *sums, bool pdl, cudaStream_t stream) {
    int threads = K / 8 < 512 ? K / 8 : 512;
    if (gain)
        return launch_k(prep_kernel<true>, dim3(B), dim3(threads), 0, pdl, 1, stream, src, lds, K, gain,
                        eps, Bp, hi, lo, sums);
    return launch_k(prep_kernel<false>, dim3(B), dim3(threads), 0, pdl, 1, stream, src, lds, K, gain, eps,
                    Bp, hi, lo, sums);
}

// CUDA-core dequant-matvec on the same stage (B <= 4); accr[col][rho] partial
// over this lane's quarter of the row (summed across tig at the end).
template <int NB>
__device__ __forceinline__ void stage_fma(const uint8_t *st, int warp, int lane, const StageLayout &L,
                                          float (&accr)[NB][2]) {
    const int tig = lane & 3;
    const uint8_t *tile = st + warp * TILE_BYTES;
    const uint8_t *ahi = st + L.hi, *alo = st + L.lo;
    const uint8_t *sums = st + L.sums;
    uint4 q[4];
#pragma unroll
    for (int c = 0; c < 4; c++) q[c] = *reinterpret_cast<const uint4 *>(tile + c * 512 + 16 * lane);
    TileMeta tm;
    decode_meta(*reinterpret_cast<const uint2 *>(tile + TILE_CODE_BYTES + 8 * lane), tig, tm);
    float sq[NB][2], sl[NB][2];
#pragma unroll
    for (int c = 0; c < NB; c++) sq[c][0] = sq[c][1] = sl[c][0] = sl[c][1] = 0.0f;
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
            const int chunk = tig * 8 + h * 4 + pidx;
#pragma unroll
            for (int col = 0; col < NB; col++) {
                const int off = (chunk ^ (tig | ((col & 1) << 2))) * 16;
                uint4 xv = *reinterpret_cast<const uint4 *>(ahi + col * 512 + off);
                uint4 xl = *reinterpret_cast<const uint4 *>(alo + col * 512 + off);
                sq[col][0] += dot2(a0, xv.x) + dot2(a0h, xv.y) + dot2(a016, xv.z) + dot2(a0h16, xv.w);
                sq[col][1] += dot2(a1, xv.x) + dot2(a1h, xv.y) + dot2(a116, xv.z) + dot2(a1h16, xv.w);
                sl[col][0] += dot2(a0, xl.x) + dot2(a0h, xl.y) + dot2(a016, xl.z) + dot2(a0h16, xl.w);
                sl[col][1] += dot2(a1, xl.x) + dot2(a1h, xl.y) + dot2(a116, xl.z) + dot2(a1h16, xl.w);
            }
        }
    }
    float2 mg = __half22float2(u32_as_h2(tm.mg)), m8 = __half22float2(u32_as_h2(tm.m8));
#pragma unroll
    for (int col = 0; col < NB; col++) {
        uint2 s = *reinterpret_cast<const uint2 *>(sums + col * 32 + tig * 8);
        float2 shi = __half22float2(u32_as_h2(s.x)), slo = __half22float2(u32_as_h2(s.y));
        float s1 = shi.x + slo.x, s2 = shi.y + slo.y;
        accr[col][0] += tm.dg * (sq[col][0] + sl[col][0] * LO_UNSCALE) - tm.dming * (mg.x * s1 + mg.y * s2);
        accr[col][1] += tm.d8 * (sq[col][1] + sl[col][1] * LO_UNSCALE) - tm.dmin8 * (m8.x * s1 + m8.y * s2);
    }
}

// ------------------------------------------------------------ epilogue ---
// y[nt][rho]: output row rt*16 + g + 8*rho, batch row b = 4nt + tig.
template <int NT, int EPI>
__device__ __forceinline__ void gemm_epilogue(const GemmParams &p, float (&y)[NT][2], int grp,
                                              const float (&xin)[NT][2], const float *sgain) {
    constexpr int NB = 4 * NT;   // batch rows this instance covers
    // SWIGLU: a[col][64 rows]; RESID with a next operand: x[col][128 rows]
    __shared__ float s_v[EPI == EPI_LMHEAD ? GT * NB : NB * 128];
    __shared__ int s_i[GT * NB];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, tig = lane & 3;
    const int rt = grp * GT + warp;
    const bool active = rt < p.nrt;
    if (EPI == EPI_STORE) {
        const bool qhead = p.q_frag && grp < p.q_heads;   // CTA-uniform
        if (active)
#pragma unroll
            for (int nt = 0; nt < NT; nt++)
#pragma unroll
                for (int r = 0; r < 2; r++) {
                    const int row = rt * 16 + g + 8 * r, b = 4 * nt + tig;
                    if (b < p.B && row < p.N) {
                        p.out[(size_t)b * p.ldo + row] = y[nt][r];
                        if (qhead) s_v[b * 128 + warp * 16 + g + 8 * r] = y[nt][r];
                    }
                }
        if (!qhead) return;
        // query head grp: rotate at its position, scale, split hi/lo, fragment order
        __syncthreads();
        const float qscale = 0.12751743082459868f;   // log2(e)/sqrt(128): the attention works in log2 units
        for (int task = threadIdx.x; task < p.B * 32; task += blockDim.x) {
            const int b = task >> 5, st = (task >> 2) & 7, tq = task & 3;
            // cos/sin of dims 16 st + 4 tq + {0..3} (mod 64); the row was
            // prefetched into L1 at the kernel's start
            const float4 *cs4 = reinterpret_cast<const float4 *>(p.q_rope + (size_t)p.q_pos[b] * 64 +
                                                                 ((16 * st + 4 * tq) & 63));
            const float4 r4[2] = {cs4[0], cs4[1]};
            const float2 cpair[4] = {make_float2(r4[0].x, r4[0].y), make_float2(r4[0].z, r4[0].w),
                                     make_float2(r4[1].x, r4[1].y), make_float2(r4[1].z, r4[1].w)};
            float v[4];
#pragma unroll
            for (int e = 0; e < 4; e++) {
                const int d = 16 * st + 4 * tq + e;
                const float x = s_v[b * 128 + d];
                const float2 c = cpair[e];
                v[e] = (d < 64 ? x * c.x - s_v[b * 128 + d + 64] * c.y : x * c.x + s_v[b * 128 + d - 64] * c.y) * qscale;
            }
            const __half2 h01 = __floats2half2_rn(v[0], v[1]), h23 = __floats2half2_rn(v[2], v[3]);
            const float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
            uint4 f;
            f.x = h2_as_u32(h01);
            f.y = h2_as_u32(__floats2half2_rn(v[0] - f01.x, v[1] - f01.y));
            f.z = h2_as_u32(h23);
            f.w = h2_as_u32(__floats2half2_rn(v[2] - f23.x, v[3] - f23.y));
            p.q_frag[(((size_t)b * p.q_heads + grp) * 8 + st) * 4 + tq] = f;
        }
    } else if (EPI == EPI_RESID) {
        // x += y; with next_gain set, the group's 128 updated rows also become the
        // next projection's operand g*x (act planes + sub-block sums) and one
        // partial sum of x^2 per column for that projection's RMSNorm scale
        if (active)
#pragma unroll
            for (int nt = 0; nt < NT; nt++)
#pragma unroll
                for (int r = 0; r < 2; r++) {
                    const int row = rt * 16 + g + 8 * r, b = 4 * nt + tig;
                    if (b < p.B && row < p.N) {
                        float *o = p.out + (size_t)b * p.ldo + row;
                        const float xn = xin[nt][r] + y[nt][r];   // x fetched at the kernel's start
                        *o = xn;
                        if (p.next_gain) s_v[b * 128 + warp * 16 + 8 * r + g] = xn;
                    }
                }
        if (!p.next_gain) return;
        __syncthreads();
        for (int task = threadIdx.x; task < NB * 16; task += blockDim.x) {   // (col, chunk of 8 rows)
            const int col = task >> 4, ch = task & 15;
            const int r0 = grp * 128 + ch * 8;
            const bool live = col < p.B && r0 < p.N;
            float part = 0.0f, sq = 0.0f;
            if (live) {
                float yy[8];
#pragma unroll
                for (int i = 0; i < 8; i++) {
                    const float xv = s_v[col * 128 + ch * 8 + i];
                    sq = fmaf(xv, xv, sq);
                    yy[i] = xv * sgain[ch * 8 + i];
                    part += yy[i];
                }
                store_act8(p.out16, p.out16lo, act_chunk(r0 >> 8, col, (r0 & 255) >> 3, p.out_Bp), yy);
            }
            part += __shfl_xor_sync(FULL, part, 1);   // four chunks = one sub-block
            part += __shfl_xor_sync(FULL, part, 2);
            if (live && (ch & 3) == 0) store_sum(p.out_sx, r0 >> 8, col, (r0 & 255) >> 5, p.out_Bp, part);
            // the 16 chunks of one column are 16 consecutive lanes
            sq += __shfl_xor_sync(FULL, sq, 1);
            sq += __shfl_xor_sync(FULL, sq, 2);
            sq += __shfl_xor_sync(FULL, sq, 4);
            sq += __shfl_xor_sync(FULL, sq, 8);
            if (live && ch == 0) p.part_out[grp * MAX_B + col] = sq;
        }
    } else if (EPI == EPI_SWIGLU) {
        // tile rows 0-7 gate, 8-15 up of ffn rows 8*rt .. 8*rt+7: a = silu(gate) * up,
        // then the group's 64 consecutive rows become the down projection's act planes
        if (active)
#pragma unroll
            for (int nt = 0; nt < NT; nt++) {
                const int b = 4 * nt + tig;
                s_v[b * 64 + warp * 8 + g] = silu_f(y[nt][0]) * y[nt][1];
            }
        __syncthreads();
        for (int task = threadIdx.x; task < NB * 8; task += blockDim.x) {   // 8 chunks of 8 rows per column
            const int col = task >> 3, ch = task & 7;
            const int f = grp * 64 + ch * 8;
            const bool live = col < p.B && f < p.N;
            float part = 0.0f;
            if (live) {
                float yy[8];
#pragma unroll
                for (int i = 0; i < 8; i++) {
                    yy[i] = s_v[col * 64 + ch * 8 + i];
                    part += yy[i];
                }
                store_act8(p.out16, p.out16lo, act_chunk(f >> 8, col, (f & 255) >> 3, p.out_Bp), yy);
            }
            part += __shfl_xor_sync(FULL, part, 1);   // four chunks = one 32-row sub-block
            part += __shfl_xor_sync(FULL, part, 2);
            if (live && (ch & 3) == 0) store_sum(p.out_sx, f >> 8, col, (f & 255) >> 5, p.out_Bp, part);
        }
    } else {   // EPI_LMHEAD: logits and the CTA's argmax partial per batch row
#pragma unroll
        for (int nt = 0; nt < NT; nt++) {
            const int b = 4 * nt + tig;
            const int r0 = rt * 16 + g, r1 = r0 + 8;
            const float v0 = (active && r0 < p.N) ? y[nt][0] : -INFINITY;
            const float v1 = (active && r1 < p.N) ? y[nt][1] : -INFINITY;
            if (active && p.out && b < p.B) {
                if (r0 < p.N) p.out[(size_t)b * p.ldo + r0] = y[nt][0];
                if (r1 < p.N) p.out[(size_t)b * p.ldo + r1] = y[nt][1];
            }
            float bv = v0;
            int bi = r0;
            if (v1 > bv) { bv = v1; bi = r1; }
            for (int o = 4; o < 32; o <<= 1) {   // across g, lowest index on ties
                const float ov = __shfl_xor_sync(FULL, bv, o);
                const int oi = __shfl_xor_sync(FULL, bi, o);
                if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
            }
            if (g == 0) {
                s_v[warp * NB + b] = bv;
                s_i[warp * NB + b] = bi;
            }
        }
        __syncthreads();
        if ((int)threadIdx.x < NB) {
            const int b = threadIdx.x;
            float bv = -INFINITY;
            int bi = 0x7FFFFFFF;
            for (int w = 0; w < GT; w++) {   // increasing rows
                const float v = s_v[w * NB + b];
                const int i = s_i[w * NB + b];
                if (v > bv || (v == bv && i < bi)) { bv = v; bi = i; }
            }
            if (b < p.B) {
                p.amax_val[grp * MAX_B + b] = bv;
                p.amax_idx[grp * MAX_B + b] = bi;
            }
        }
    }
}

// Bounded wait on a stage's mbarrier; on timeout the status word records it.
// limit: clock cycles (GEMM_WAIT_LIMIT, ~2 s: a copy that never lands).
constexpr long long GEMM_WAIT_LIMIT = 1LL << 32;
__device__ __forceinline__ bool wait_stage(uint64_t *bar, uint32_t parity, uint32_t *status,
                                           long long limit = GEMM_WAIT_LIMIT) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > limit) {
            if (status) atomicOr(status, STATUS_TIMEOUT);
            return false;
        }
    }
    return true;
}




// ------------------------------------------------------------- kernel ---
// NT n-tiles of 4 batch rows each (IMPL 2), or NT batch rows (IMPL 1, NT <= 4).
// Residency: three CTAs per SM for the mma kernels up to two n-tiles (B <= 8;
// <= 80 registers), one above.
template <int NT, int IMPL> struct GemmOcc { static constexpr int v = (IMPL >= 2 && NT <= 2) ? 3 : (NT <= 2 ? 2 : 1); };
// MMA accumulator chains per n-tile (stage_mma): all four where registers
// allow, one at NT = 2 (three CTAs per SM in 80 registers), two at NT = 8.
template <int NT> struct GemmChains { static constexpr int v = NT == 2 ? 1 : (NT == 8 ? 2 : 4); };
// Batch rows a stage holds: 4 per n-tile (IMPL 2), the four matvec columns
// (IMPL 1), or batch row 0 plus the zero row 1 that the idle B columns read
// (IMPL 3).
template <int NT, int IMPL> struct GemmBR { static constexpr int v = IMPL == 2 ? 4 * NT : (IMPL == 3 ? 2 : 4); };
// Bytes of one peer's partial tiles in rank 0's reduction area: every lane's
// y (IMPL 1, 2), or only the tig = 0 lanes, which hold the rows' sums (IMPL 3).
template <int NT, int IMPL> struct GemmRed {
    static constexpr uint32_t v = IMPL == 3 ? GT * 2 * 8 * 4 : GT * (IMPL == 2 ? NT : 1) * 2 * 32 * 4;
};

template <int NT, int EPI, int IMPL>
__global__ __launch_bounds__(256, (GemmOcc<NT, IMPL>::v)) void gemm_kernel(const GemmParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int s_bad;
    __shared__ uint64_t red_bar;   // rank 0 of a cluster: the peers' partial tiles have landed
    __shared__ int s_issued;        // stages whose copies have been issued
    __shared__ float s_gain[128];   // RESID with next_gain: the group's gain rows
    __shared__ float s_rms[MAX_B];  // RMSNorm scale per batch row (consumers of a folded norm)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tig = lane & 3;
    const int cs = p.cs, rank = blockIdx.x % cs, grp = blockIdx.x / cs;
    const int rt = grp * GT + warp;
    const int s0 = rank * p.nsb / cs, s1 = (rank + 1) * p.nsb / cs, n = s1 - s0;
    const int B = p.B, D = p.stages;
    constexpr int BR = GemmBR<NT, IMPL>::v;   // batch rows held per stage
    const StageLayout lay(BR);
    const uint32_t abytes = (uint32_t)B * 512u, sbytes = (uint32_t)B * 32u;
    const uint32_t tx = GROUP_BYTES + 2 * abytes + sbytes;
    const uint32_t sbyt = lay.bytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)D * sbyt);
    const uint8_t *gW = p.W + (size_t)grp * p.nsb * GROUP_BYTES;
    // Stage i of the CTA's range lives in ring slot i % D; the loop tracks
    // slot and phase parity incrementally, so no division runs per stage.
    auto slot_ptr = [&](int slot) { return smem + (uint32_t)slot * sbyt; };
    auto issue_w = [&](int slot, int i) {   // weights of stage i into `slot`
        mbar_expect_tx(&full[slot], tx);
        bulk_g2s(slot_ptr(slot), gW + (size_t)(s0 + i) * GROUP_BYTES, GROUP_BYTES, &full[slot]);
    };
    auto issue_act = [&](int slot, int i) {   // the activation rows of stage i into `slot`
        uint8_t *st = slot_ptr(slot);
        const size_t sb = (size_t)(s0 + i);
        bulk_g2s(st + lay.hi, p.x16 + sb * p.Bp * 256, abytes, &full[slot]);
        bulk_g2s(st + lay.lo, p.x16lo + sb * p.Bp * 256, abytes, &full[slot]);
        bulk_g2s(st + lay.sums, p.sx + sb * p.Bp * 16, sbytes, &full[slot]);
    };
    tl_min(p.tl, 0);
    if (threadIdx.x == 0) {
        s_bad = 0;
        for (int i = 0; i < D; i++) mbar_init(&full[i], 1);
        if (cs > 1 && rank == 0) {
            // the cs - 1 peers' partial tiles, stored asynchronously into the area
            mbar_init(&red_bar, 1);
            mbar_expect_tx(&red_bar, (uint32_t)(cs - 1) * GemmRed<NT, IMPL>::v);
        }
        mbar_fence_init();
    }
    // rank 0 receives the peers' partial tiles after the barriers (see the end):
    // behind the stage ring, or in it (red_alias) once rank 0's K loop is done
    const uint32_t red_off = p.red_off;
    // zero the batch rows the copies never write (rows B..BR-1 and the lo lanes'
    // min-term slots) in every stage buffer
    for (int i = threadIdx.x; i < D * BR * 8; i += blockDim.x) {
        const int st = i / (BR * 8), r = (i / 8) % BR, w = i % 8;   // 8 x 16 bytes per 128-byte unit
        uint8_t *base = smem + (size_t)st * sbyt;
        if (r >= B) {
            for (int k = 0; k < 4; k++) {
                *reinterpret_cast<uint4 *>(base + lay.hi + r * 512 + (w * 4 + k) * 16) = make_uint4(0, 0, 0, 0);
                *reinterpret_cast<uint4 *>(base + lay.lo + r * 512 + (w * 4 + k) * 16) = make_uint4(0, 0, 0, 0);
            }
            if (w < 2) *reinterpret_cast<uint4 *>(base + lay.sums + r * 32 + w * 16) = make_uint4(0, 0, 0, 0);
        }
        if (w < 2) *reinterpret_cast<uint4 *>(base + lay.zero + r * 32 + w * 16) = make_uint4(0, 0, 0, 0);
    }
    __syncthreads();
    // publishes red_bar's initialisation (waited on after the K loop); with an
    // aliased reduction area rank 0 arrives only when its stages are free
    if (cs > 1 && !(p.red_alias && rank == 0)) cluster_arrive_relaxed();
    // this lane's fixed offsets into a stage: virtual column g of n-tile 0 is the
    // hi (g even) or lo (g odd) plane of batch row g/2
    const int g = lane >> 2;
    uint32_t act_off = ((g & 1) ? lay.lo : lay.hi) + (uint32_t)(g >> 1) * 512u + (uint32_t)tig * 128u;
    const uint32_t swz = (uint32_t)tig | ((uint32_t)((g >> 1) & 1) << 2);
    uint32_t sum_off = (g & 1) ? lay.zero + (uint32_t)tig * 8u
                               : lay.sums + (uint32_t)(g >> 1) * 32u + (uint32_t)tig * 8u;
    MvOff mvo{};
    if (IMPL == 3) {   // B column g carries sub-block data only in lane group tig = g/2 (see stage_mv)
        act_off = (g == 2 * tig ? lay.hi : (g == 2 * tig + 1 ? lay.lo : lay.hi + 512u)) + (uint32_t)tig * 128u;
        sum_off = lay.sums + (uint32_t)tig * 8u;
        mvo.codes = (uint32_t)warp * TILE_BYTES + 16u * (uint32_t)lane;
        mvo.meta = (uint32_t)warp * TILE_BYTES + TILE_CODE_BYTES + 8u * (uint32_t)lane;
#pragma unroll
        for (int pw = 0; pw < 4; pw++) mvo.act[pw] = act_off + (((uint32_t)pw ^ (uint32_t)tig) << 4);
        mvo.sums = sum_off;
    }
    const int pre = min(D, n);
    if ((int)threadIdx.x < pre) issue_w(threadIdx.x, threadIdx.x);   // one issuing thread per stage
    if (threadIdx.x == 0) s_issued = pre;
    // epilogue inputs that no earlier kernel of the step writes (weights, the
    // rotary table, the step's positions), fetched before the dependency wait
    if (EPI == EPI_RESID && p.next_gain && threadIdx.x < 128)
        s_gain[threadIdx.x] = grp * 128 + (int)threadIdx.x < p.N ? p.next_gain[grp * 128 + threadIdx.x] : 0.0f;
    if (EPI == EPI_STORE && p.q_frag && grp < p.q_heads && (int)threadIdx.x < B * 4)   // 4 lines of 128 B per row
        prefetch_l1(p.q_rope + (size_t)p.q_pos[threadIdx.x >> 2] * 64 + (threadIdx.x & 3) * 16);
    pdl_launch_dependents();
    pdl_wait();
    tl_min(p.tl, 1);
    tl_max(p.tl, 4);
    // the activation rows of the first stages, one issuing thread per stage (a
    // copy that lands before thread 0's expect_tx only leaves the transaction
    // count negative until then: the phase still needs that arrival)
    if ((int)threadIdx.x < pre) issue_act(threadIdx.x, threadIdx.x);
    // the epilogue's inputs from earlier kernels, fetched now so that their
    // latency hides behind the K loop: this lane's partial sums of x^2 per
    // batch row (RMSNorm scale) and the residual rows it will update
    constexpr int NY = IMPL == 2 ? NT : 1;
    constexpr bool EARLY = NY == 1 || (NY == 2 && GemmOcc<NT, IMPL>::v < 3);   // registers hold the residual
    // RMSNorm sums of x^2 for the batch rows (warp w: rows w, w + 8, ...), only
    // in the CTA that runs the epilogue (rank 0).  Loaded now and reduced after
    // the K loop: the first partial of each lane is a plain load that nothing
    // uses before then, so its latency hides behind the loop.
    const bool rms_here = p.rms_part && rank == 0;
    float rms_ss[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    if (rms_here)
#pragma unroll
        for (int j = 0; j < 4; j++) {
            const int b = warp + 8 * j;
            if (b < B && b < 4 * NY && lane < p.rms_nparts) {
                rms_ss[j] = p.rms_part[lane * MAX_B + b];
                for (int i = lane + 32; i < p.rms_nparts; i += 32) rms_ss[j] += p.rms_part[i * MAX_B + b];
            }
        }
    float xin[NY][2];
    auto fetch_xin = [&]() {
#pragma unroll
        for (int nt = 0; nt < NY; nt++)
#pragma unroll
            for (int r = 0; r < 2; r++) {
                const int row = rt * 16 + (lane >> 2) + 8 * r, b = 4 * nt + tig;
                xin[nt][r] = (EPI == EPI_RESID && rank == 0 && rt < p.nrt && b < B && row < p.N)
                                 ? p.out[(size_t)b * p.ldo + row] : 0.0f;
            }
    };
    if (EARLY) fetch_xin();
    else if (EPI == EPI_RESID && rank == 0 && (int)threadIdx.x < 4 * B)   // the group's rows: 4 lines per batch row
        prefetch_l1(p.out + (size_t)(threadIdx.x >> 2) * p.ldo + grp * 128 + (threadIdx.x & 3) * 32);

    constexpr int NA = IMPL == 2 ? NT : 1;   // mma accumulator tiles
    constexpr int NB = IMPL == 1 ? NT : 1;   // matvec columns
    float acc[NA][4];
#pragma unroll
    for (int nt = 0; nt < NA; nt++)
#pragma unroll
        for (int i = 0; i < 4; i++) acc[nt][i] = 0.0f;
    float accr[NB][2];
#pragma unroll
    for (int c = 0; c < NB; c++) accr[c][0] = accr[c][1] = 0.0f;
    float ymq[2] = {0.0f, 0.0f}, ymm[2] = {0.0f, 0.0f};   // IMPL 3: code and min terms (stage_mv)
    // one stage per step (p.pair = 0): each slot is refilled as soon as every
    // warp is done with it, so the D - 1 stages ahead of the one computed stay
    // in flight; or two (p.pair = 1): their loads, dequant and MMAs are
    // independent, giving each warp two dependency chains, and the block-wide
    // syncs halve, but the pair's second slot refills one stage later
    bool ok = true;
    const long long wlim = p.wait_limit > 0 ? p.wait_limit : GEMM_WAIT_LIMIT;
    // wait_limit < 0 (tests): the first stage wait counts as run out at once,
    // so the give-up path (status, drain of the copies in flight, return)
    // runs deterministically, without racing the copies
    auto expired = [&](int i, int slot, uint32_t parity) {
        if (p.wait_limit < 0 && i == 0) {
            if (p.status) atomicOr(p.status, STATUS_TIMEOUT);
            return true;
        }
        return !wait_stage(&full[slot], parity, p.status, wlim);
    };
    const bool live = rt < p.nrt;   // the group's last row tiles may be padding
    int sa = 0;                     // ring slot of stage i
    uint32_t pa = 0;                // its phase parity
    const int step = p.pair ? 2 : 1;
    for (int i = 0; i < n; i += step) {
        const bool two = p.pair && i + 1 < n;
        int sb = sa + 1;            // stage i + 1
        uint32_t pb = pa;
        if (sb == D) { sb = 0; pb ^= 1u; }
        if (ok && expired(i, sa, pa)) { ok = false; s_bad = 1; }
        if (i == 0) tl_max(p.tl, 5);
        if (two && ok && expired(i + 1, sb, pb)) {
            ok = false;
            s_bad = 1;
        }
        if (ok && live) {
            const uint8_t *st_a = slot_ptr(sa), *st_b = slot_ptr(sb);
            if (IMPL == 2) {
                stage_mma<NA, GemmChains<NT>::v>(st_a, warp, lane, act_off, sum_off, swz, acc);
                if (two) stage_mma<NA, GemmChains<NT>::v>(st_b, warp, lane, act_off, sum_off, swz, acc);
            } else if (IMPL == 3) {
                stage_mv(st_a, mvo, tig, ymq, ymm);
                if (two) stage_mv(st_b, mvo, tig, ymq, ymm);
            } else {
                stage_fma<NB>(st_a, warp, lane, lay, accr);
                if (two) stage_fma<NB>(st_b, warp, lane, lay, accr);
            }
        }
        __syncthreads();   // every warp is done with both slots: refill them
        if (threadIdx.x == 0 && !s_bad) {
            if (i + D < n) { issue_w(sa, i + D); issue_act(sa, i + D); s_issued = i + D + 1; }
            if (two && i + 1 + D < n) { issue_w(sb, i + 1 + D); issue_act(sb, i + 1 + D); s_issued = i + D + 2; }
        }
        if (p.pair) {               // stage i + 2
            sa = sb + 1;
            pa = pb;
            if (sa == D) { sa = 0; pa ^= 1u; }
        } else {                    // stage i + 1
            sa = sb;
            pa = pb;
        }
    }
    tl_max(p.tl, 6);
    const bool bad = s_bad != 0;
    if (bad) {   // drain the last D issued stages, which may still be in flight (full bound); the result is abandoned
        if (threadIdx.x == 0)
            for (int i = max(0, s_issued - D); i < s_issued; i++) wait_stage(&full[i % D], (uint32_t)(i / D) & 1u, nullptr);
        __syncthreads();
        if (cs == 1) return;   // cluster members still take part in the reduction below
    }
    // per-lane outputs: y[nt][rho] for output row g + 8 rho, batch row 4nt + tig
    float y[NY][2];
    if (IMPL == 2) {
#pragma unroll
        for (int nt = 0; nt < NY; nt++) {
            y[nt][0] = acc[nt < NA ? nt : 0][0] + acc[nt < NA ? nt : 0][1] * LO_UNSCALE;
            y[nt][1] = acc[nt < NA ? nt : 0][2] + acc[nt < NA ? nt : 0][3] * LO_UNSCALE;
        }
    } else if (IMPL == 3) {   // the row's four lanes, then batch row 0 in lane tig 0
        float ymv[2];
#pragma unroll
        for (int r = 0; r < 2; r++) {
            ymv[r] = fmaf(16777216.0f, ymq[r], -ymm[r]);   // the codes carried 2^-24
            ymv[r] += __shfl_xor_sync(FULL, ymv[r], 1);
            ymv[r] += __shfl_xor_sync(FULL, ymv[r], 2);
        }
        y[0][0] = tig == 0 ? ymv[0] : 0.0f;
        y[0][1] = tig == 0 ? ymv[1] : 0.0f;
    } else {   // quad butterfly, then batch row tig
#pragma unroll
        for (int c = 0; c < NB; c++)
#pragma unroll
            for (int r = 0; r < 2; r++) {
                accr[c][r] += __shfl_xor_sync(FULL, accr[c][r], 1);
                accr[c][r] += __shfl_xor_sync(FULL, accr[c][r], 2);
            }
        y[0][0] = y[0][1] = 0.0f;
#pragma unroll
        for (int c = 0; c < NB; c++)
            if (c == tig) { y[0][0] = accr[c][0]; y[0][1] = accr[c][1]; }
    }
    if (cs > 1) {   // K split across the cluster: the peers push their partial tiles to rank 0
        if (p.red_alias && rank == 0) cluster_arrive_release();   // every copy into the ring has landed
        cluster_wait_acquire();   // every CTA of the cluster has initialised its barriers
        constexpr int SLOT = GemmRed<NT, IMPL>::v / 4;   // floats of one peer's partial tile set
        const uint32_t red_local = smem_u32(smem + red_off);
        if (rank != 0) {   // (y[nt][0], y[nt][1]) as one 8-byte store per lane
            const uint32_t dst = map_to_rank(red_local, 0) + (uint32_t)((rank - 1) * SLOT) * 4u;
            const uint32_t rbar = map_to_rank(smem_u32(&red_bar), 0);
            if (IMPL == 3) {
                if (tig == 0) st_async_v2(dst + (uint32_t)(warp * 8 + (lane >> 2)) * 8u, y[0][0], y[0][1], rbar);
            } else
#pragma unroll
            for (int nt = 0; nt < NY; nt++)
                st_async_v2(dst + (uint32_t)((warp * NY + nt) * 32 + lane) * 8u, y[nt][0], y[nt][1], rbar);
            tl_end(p.tl);
            return;
        }
        // rank 0: wait (bounded) for the cs - 1 pushes, then sum them in rank order
        if (!mbar_try_wait_cluster(&red_bar, 0)) {
            const long long t0 = clock64();
            while (!mbar_try_wait_cluster(&red_bar, 0))
                if (clock64() - t0 > (1LL << 32)) {
                    if (threadIdx.x == 0) atomicOr(p.status, STATUS_TIMEOUT);
                    s_bad = 1;
                    break;
                }
        }
        const float *red = reinterpret_cast<const float *>(smem + red_off);
        if (IMPL == 3) {
            if (tig == 0)
                for (int rr = 1; rr < cs; rr++) {
                    const float2 v = *reinterpret_cast<const float2 *>(red + (rr - 1) * SLOT + (warp * 8 + (lane >> 2)) * 2);
                    y[0][0] += v.x;
                    y[0][1] += v.y;
                }
        } else
        for (int rr = 1; rr < cs; rr++)
#pragma unroll
            for (int nt = 0; nt < NY; nt++) {
                const float2 v = *reinterpret_cast<const float2 *>(red + (rr - 1) * SLOT + ((warp * NY + nt) * 32 + lane) * 2);
                y[nt][0] += v.x;
                y[nt][1] += v.y;
            }
        __syncthreads();
        if (bad || s_bad) return;
        tl_max(p.tl, 7);
    }
    if (rms_here) {   // RMSNorm folded out of the operand: y = r_b * W (g * x_b)
#pragma unroll
        for (int j = 0; j < 4; j++) {
            const int b = warp + 8 * j;
            if (b < B && b < 4 * NY) {   // warp-uniform
                float ss = rms_ss[j];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(FULL, ss, o);
                if (lane == 0) s_rms[b] = 1.0f / sqrtf(ss / (float)p.rms_K + p.rms_eps);
            }
        }
        __syncthreads();
#pragma unroll
        for (int nt = 0; nt < NY; nt++) {
            const int b = 4 * nt + tig;
            const float r_b = b < B ? s_rms[b] : 1.0f;
            y[nt][0] *= r_b;
            y[nt][1] *= r_b;
        }
    }
    if (!EARLY) fetch_xin();
    gemm_epilogue<NY, EPI>(p, y, grp, xin, s_gain);
    if (p.tl) {
        __syncthreads();
        tl_end(p.tl);
    }
}

// ------------------------------------------------------------ dispatch ---
int gemm_grid(const GemmParams &p) { return n_groups(p.nrt) * p.cs; }

// Dynamic shared memory a CTA may take at `occ` CTAs per SM: its share of the
// SM's 228 KB (1 KB reserved per CTA) less the static arrays.
static uint32_t occ_budget(int occ) { return occ >= 3 ? 72u * 1024u : (occ == 2 ? 110u * 1024u : 200u * 1024u); }

static int stages_for(uint32_t stage_bytes, int occ, uint32_t reserved) {
    uint32_t budget = occ_budget(occ);
    budget = budget > reserved + 2 * stage_bytes ? budget - reserved : 2 * stage_bytes;
    int d = (int)(budget / stage_bytes);
    return d < 2 ? 2 : (d > 6 ? 6 : d);
}

// Shared-memory plan of a launch: ring depth, the reduction area and its
// place; may halve p.cs.  Returns the dynamic shared-memory bytes.
template <int NT, int IMPL>
static size_t plan_smem(GemmParams &p) {
    const StageLayout lay(GemmBR<NT, IMPL>::v);
    // rank 0 of a cluster holds the cs - 1 peers' partial tiles
    constexpr uint32_t NYB = GemmRed<NT, IMPL>::v;
    constexpr int OCC = GemmOcc<NT, IMPL>::v;
    // the peers' tiles go behind the ring when ring and tiles fit the CTA's
    // share of the SM together, else into the ring itself (rank 0 frees it
    // first); a split whose tiles fit neither way is halved
    const int d_plain = stages_for(lay.bytes, OCC, 0);
    while (p.cs > 1 && (uint32_t)(p.cs - 1) * NYB > (uint32_t)d_plain * lay.bytes &&
           (uint32_t)(p.cs - 1) * NYB + 2 * lay.bytes > 180u * 1024u)
        p.cs >>= 1;
    uint32_t red_bytes = p.cs > 1 ? (uint32_t)(p.cs - 1) * NYB : 0u;
    p.red_alias = 0;
    if (red_bytes && (size_t)d_plain * lay.bytes + 64 + red_bytes > occ_budget(OCC) &&
        red_bytes <= (uint32_t)d_plain * lay.bytes) {
        p.red_alias = 1;
        red_bytes = 0;
    }
    p.stages = p.red_alias ? d_plain : stages_for(lay.bytes, OCC, red_bytes);
    p.red_off = p.red_alias ? 0u : (uint32_t)p.stages * lay.bytes + 64u;
    return (size_t)p.stages * lay.bytes + 64 + red_bytes;
}

// Raise the dynamic shared-memory limit and allow clusters up to 16, once per instance.
template <int NT, int EPI, int IMPL>
static cudaError_t configure_one() {
    static bool configured = false;
    if (configured) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(gemm_kernel<NT, EPI, IMPL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         210 * 1024);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gemm_kernel<NT, EPI, IMPL>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e == cudaSuccess) configured = true;
    return e;
}

template <int NT, int EPI, int IMPL>
static cudaError_t launch_one(GemmParams p, bool pdl, cudaStream_t s) {
    const size_t smem = plan_smem<NT, IMPL>(p);
    cudaError_t e = configure_one<NT, EPI, IMPL>();
    if (e != cudaSuccess) return e;
    return launch_k(gemm_kernel<NT, EPI, IMPL>, dim3(gemm_grid(p)), dim3(256), smem, pdl, p.cs, s, p);
}

// CTAs of a split-cs launch that the GPU holds at once: the occupancy API's
// count of co-resident clusters (clusters must fit inside one GPC) times cs;
// 0 when the split cannot be launched as asked.
template <int NT, int EPI, int IMPL>
static int slots_one(int cs) {
    GemmParams p{};
    p.cs = cs;
    const size_t smem = plan_smem<NT, IMPL>(p);
    if (p.cs != cs || configure_one<NT, EPI, IMPL>() != cudaSuccess) return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(16 * cs);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_kernel<NT, EPI, IMPL>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n * cs;
}

template <int EPI>
static int slots_epi(int B, int impl, int cs) {
    if (impl == 3) return B == 1 ? slots_one<1, EPI, 3>(cs) : 0;
    if (impl == 1) {
        switch (B) {
            case 1: return slots_one<1, EPI, 1>(cs);
            case 2: return slots_one<2, EPI, 1>(cs);
            case 3: return slots_one<3, EPI, 1>(cs);
            case 4: return slots_one<4, EPI, 1>(cs);
            default: return 0;
        }
    }
    if (B <= 4) return slots_one<1, EPI, 2>(cs);
    if (B <= 8) return slots_one<2, EPI, 2>(cs);
    if (B <= 16) return slots_one<4, EPI, 2>(cs);
    return slots_one<8, EPI, 2>(cs);
}

int gemm_cluster_slots(int B, int impl, int epi, int cs) {
    if (cs < 1 || cs > 16 || B < 1 || B > MAX_B) return 0;
    switch (epi) {
        case EPI_STORE: return slots_epi<EPI_STORE>(B, impl, cs);
        case EPI_RESID: return slots_epi<EPI_RESID>(B, impl, cs);
        case EPI_SWIGLU: return slots_epi<EPI_SWIGLU>(B, impl, cs);
        case EPI_LMHEAD: return slots_epi<EPI_LMHEAD>(B, impl, cs);
    }
    return 0;
}

template <int EPI>
static cudaError_t launch_epi(const GemmParams &p, int impl, bool pdl, cudaStream_t s) {
    if (impl == 3) {
        if (p.B != 1) return cudaErrorInvalidValue;
        return launch_one<1, EPI, 3>(p, pdl, s);
    }
    if (impl == 1) {
        switch (p.B) {
            case 1: return launch_one<1, EPI, 1>(p, pdl, s);
            case 2: return launch_one<2, EPI, 1>(p, pdl, s);
            case 3: return launch_one<3, EPI, 1>(p, pdl, s);
            case 4: return launch_one<4, EPI, 1>(p, pdl, s);
            default: return cudaErrorInvalidValue;
        }
    }
    if (p.B <= 4) return launch_one<1, EPI, 2>(p, pdl, s);
    if (p.B <= 8) return launch_one<2, EPI, 2>(p, pdl, s);
    if (p.B <= 16) return launch_one<4, EPI, 2>(p, pdl, s);
    return launch_one<8, EPI, 2>(p, pdl, s);
}

cudaError_t launch_gemm(const GemmParams &p, int epi, int impl, bool pdl, cudaStream_t stream) {
    if (p.cs < 1 || p.cs > 16) return cudaErrorInvalidValue;
    if (p.B < 1 || p.B > MAX_B || p.B > p.Bp || !p.x16 || !p.x16lo || !p.sx) return cudaErrorInvalidValue;
    switch (epi) {
        case EPI_STORE: return launch_epi<EPI_STORE>(p, impl, pdl, stream);
        case EPI_RESID: return launch_epi<EPI_RESID>(p, impl, pdl, stream);
        case EPI_SWIGLU: return launch_epi<EPI_SWIGLU>(p, impl, pdl, stream);
        case EPI_LMHEAD: return launch_epi<EPI_LMHEAD>(p, impl, pdl, stream);
    }
    return cudaErrorInvalidValue;
}

// --------------------------------------------------------- argmax final ---
__global__ void argmax_final_kernel(const float *__restrict__ vals, const int *__restrict__ idxs,
                                    int nparts, int B, int32_t *ids, const int32_t *positions,
                                    const int32_t *slots, int32_t *len_dev, const uint32_t *status,
                                    unsigned long long *tl) {
    tl_min(tl, 0);
    pdl_launch_dependents();
    pdl_wait();
    tl_min(tl, 1);
    int b = blockIdx.x;
    __shared__ float sv[32];
    __shared__ int si[32];
    float bv = -INFINITY;
    int bi = 0x7FFFFFFF;
    // eight partials per thread per round, all loaded before any is compared
    // (one latency per round instead of one per partial)
    constexpr int U = 8;
    for (int i0 = threadIdx.x; i0 < nparts; i0 += U * blockDim.x) {
        float v[U];
        int ix[U];
#pragma unroll
        for (int k = 0; k < U; k++) {
            const int i = i0 + k * blockDim.x;
            v[k] = i < nparts ? vals[i * MAX_B + b] : -INFINITY;
            ix[k] = i < nparts ? idxs[i * MAX_B + b] : 0x7FFFFFFF;
        }
#pragma unroll
        for (int k = 0; k < U; k++)
            if (v[k] > bv || (v[k] == bv && ix[k] < bi)) { bv = v[k]; bi = ix[k]; }
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
        // the length advances only for a step no device check has flagged
        if ((*(volatile const uint32_t *)status & STATUS_STATE_ERRORS) == 0) len_dev[slots[b]] = positions[b] + 1;
        tl_end(tl);
    }
}

cudaError_t launch_argmax_final(const float *amax_val, const int *amax_idx, int nparts, int B,
                                int32_t *ids, const int32_t *positions, const int32_t *slots,
                                int32_t *len_dev, const uint32_t *status, bool pdl, cudaStream_t stream,
                                unsigned long long *tl) {
    return launch_k(argmax_final_kernel, dim3(B), dim3(256), 0, pdl, 1, stream, amax_val, amax_idx,
                    nparts, B, ids, positions, slots, len_dev, status, tl);
}

}  // namespace zdec
