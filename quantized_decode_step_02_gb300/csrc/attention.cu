// attention.cu -- per-sequence KV read: split-K flash-decode over an fp16 or
// Q8_0 cache, dequantized inside the kernel, plus the KV append paths.
//
// Each sequence reads its own cache every step; nothing here is shared across
// the batch ("Batched swarm: the KV read does not amortize", "The two halves
// of a decode-step memory bill").  A quantized cache only saves bytes if the
// attention kernel reads the compressed format and dequantizes on chip ("Q8
// KV cache pushes an RDNA4 swarm crossover...", "Why Q8 is close to free and
// where the sharp edges are"), which is what the Q8_0 instantiation does.
//
// Grid: (cluster rank r, kv head g, sequence b); 128 threads; the CS CTAs of
// one (b, g) form a thread-block cluster.  The 4 query heads of a kv head
// share one read of its K/V tiles.  The pos+1 tokens are cut into 64-token
// chunks; rank r takes a contiguous range of them (the rank that appends the
// new token one chunk fewer), streamed through a ring of 2-8 shared-memory
// stages with cp.async.  Both products run on
// mma.sync.m16n8k16 with fp32 accumulation:
//   scores: A = q (rows 0-3 the fp16 high parts of the 4 heads, rows 8-11 the
//           low parts, so q keeps ~22 bits), B = K^T (8 tokens per MMA);
//   output: A = p (same hi/lo split), B = V (8 head dims per MMA) read from a
//           V^T tile, whose layout makes each thread's four tokens adjacent.
// Q8_0: codes become exact fp16 integers in registers; K scales multiply the
// per-32-dim partial scores, V scales are folded into p per 32-dim block.
// Softmax runs in log2 units (q carries log2(e)/sqrt(128)).  Each CTA reduces
// its warps to one (max, sum, unnormalised output) partial in shared memory;
// rank 0 of the cluster merges the ranks' partials through distributed shared
// memory (fixed rank order) and writes the output.
#include <cooperative_groups.h>

#include "zdec_kernels.cuh"

namespace cg = cooperative_groups;

namespace zdec {

constexpr uint32_t AFULL = 0xFFFFFFFFu;

template <int KVT> struct AttnLayout;
template <> struct AttnLayout<0> {          // fp16
    static constexpr int K_STRIDE = 288;    // bytes per token row (256 + pad)
    static constexpr int V_STRIDE = 160;    // bytes per head-dim row of V^T (128 + pad)
    static constexpr int K_BYTES = ATT_CHUNK * K_STRIDE;
    static constexpr int V_BYTES = HD * V_STRIDE;
    static constexpr int KS_BYTES = 0, VS_BYTES = 0;
    static constexpr int STAGE = K_BYTES + V_BYTES;
};
template <> struct AttnLayout<1> {          // Q8_0
    static constexpr int K_STRIDE = 144;    // 128 codes + pad
    static constexpr int V_STRIDE = 80;     // 64 codes + pad
    static constexpr int K_BYTES = ATT_CHUNK * K_STRIDE;
    static constexpr int V_BYTES = HD * V_STRIDE;
    static constexpr int KS_BYTES = ATT_CHUNK * 4 * 2;   // [token][4] fp16
    static constexpr int VS_BYTES = 4 * ATT_CHUNK * 2;   // [blk][token] fp16
    static constexpr int STAGE = K_BYTES + V_BYTES + KS_BYTES + VS_BYTES;
};

// A CTA keeps `stages` chunks in flight.  With few CTAs per SM the chunk
// latency, not the SM's arithmetic, bounds a shallow ring: at two stages a
// Q8_0 cache ran at half the fp16 cache's bandwidth (the same chunks per
// latency, half the bytes).
constexpr int ATT_MAX_STAGES = 8;
static int att_max_stages(int kv_dtype) { return kv_dtype ? ATT_MAX_STAGES : 5; }   // <= 200 KB
int attention_default_stages(int kv_dtype) { return kv_dtype ? 4 : 2; }
size_t attention_smem_bytes(int kv_dtype, int ns) {
    if (ns < 2 || ns > att_max_stages(kv_dtype)) ns = attention_default_stages(kv_dtype);
    size_t stages = kv_dtype ? (size_t)ns * AttnLayout<1>::STAGE : (size_t)ns * AttnLayout<0>::STAGE;
    size_t merge = (4 * 4 * 2 + 4 * 4 * HD) * sizeof(float);
    return stages > merge ? stages : merge;
}

// Base of the (slot, layer, kv head) plane for a tensor of `per_token` bytes
// per token (K planes) or `per_dim` rows (V^T planes).
__device__ __forceinline__ size_t plane_index(const KvArena &a, int slot, int layer, int g) {
    return ((size_t)slot * a.n_layers + layer) * a.n_kv + g;
}

// -------------------------------------------------------- chunk staging ---
// Copy history tokens [c0, min(c0+64, H)) of the plane into a stage.  Partial
// 16-byte segments of V^T may pull in tokens >= H; those columns are zeroed
// by the fix-up before use.
template <int KVT>
__device__ __forceinline__ void issue_chunk(const AttnParams &p, uint8_t *stage, int b, int g, int c0,
                                            int H) {
    using Lay = AttnLayout<KVT>;
    int nt = min(ATT_CHUNK, H - c0);
    if (nt <= 0) return;
    size_t pi = plane_index(p.kv, b, p.layer, g);
    const int Lp = p.kv.Lp;
    uint8_t *sK = stage, *sV = stage + Lay::K_BYTES;
    if (KVT == 0) {
        // the arena's 16-byte segments are swizzled (kv_*_off); the padded
        // stage rows hold them in natural order
        const uint8_t *gK = p.kv.k + pi * Lp * (HD * 2);
        const uint8_t *gV = p.kv.v + pi * Lp * (HD * 2);
        for (int i = threadIdx.x; i < nt * 16; i += blockDim.x) {
            int t = i >> 4, sg = i & 15;
            cp_async16(sK + t * Lay::K_STRIDE + sg * 16, gK + kv_k16_off(c0 + t, 8 * sg));
        }
        if (nt == ATT_CHUNK) {   // whole chunk: 8 segments per head-dim row
            for (int i = threadIdx.x; i < HD * 8; i += blockDim.x) {
                const int d = i >> 3, sg = i & 7;
                cp_async16(sV + d * Lay::V_STRIDE + sg * 16, gV + kv_v16_off(d, c0 + 8 * sg));
            }
        } else {
            const int vseg = (nt + 7) >> 3;   // 8 tokens per 16 bytes
            for (int i = threadIdx.x; i < HD * vseg; i += blockDim.x) {
                const int d = i / vseg, sg = i % vseg;
                cp_async16(sV + d * Lay::V_STRIDE + sg * 16, gV + kv_v16_off(d, c0 + 8 * sg));
            }
        }
    } else {
        uint8_t *sKs = stage + Lay::K_BYTES + Lay::V_BYTES, *sVs = sKs + Lay::KS_BYTES;
        const uint8_t *gK = p.kv.k + pi * Lp * HD;
        const uint8_t *gKs = p.kv.ks + (pi * Lp + c0) * 8;
        const uint8_t *gV = p.kv.v + pi * Lp * HD;
        const uint8_t *gVs = p.kv.vs + pi * Lp * 8;
        for (int i = threadIdx.x; i < nt * 8; i += blockDim.x) {
            int t = i >> 3, sg = i & 7;
            cp_async16(sK + t * Lay::K_STRIDE + sg * 16, gK + kv_k8_off(c0 + t, 16 * sg));
        }
        for (int i = threadIdx.x; i < (nt + 1) / 2; i += blockDim.x)   // 2 tokens of scales per 16 B
            cp_async16(sKs + i * 16, gKs + (size_t)i * 16);
        if (nt == ATT_CHUNK) {   // whole chunk: 4 code segments per head-dim row, 8 per scale row
            for (int i = threadIdx.x; i < HD * 4; i += blockDim.x) {
                const int d = i >> 2, sg = i & 3;
                cp_async16(sV + d * Lay::V_STRIDE + sg * 16, gV + kv_v8_off(d, c0 + 16 * sg));
            }
            if (threadIdx.x < 32) {
                const int bl = threadIdx.x >> 3, sg = threadIdx.x & 7;
                cp_async16(sVs + bl * ATT_CHUNK * 2 + sg * 16, gVs + kv_vs_off(bl, c0 + 8 * sg));
            }
        } else {
            const int vseg = (nt + 15) >> 4;   // 16 tokens per 16 bytes
            for (int i = threadIdx.x; i < HD * vseg; i += blockDim.x) {
                const int d = i / vseg, sg = i % vseg;
                cp_async16(sV + d * Lay::V_STRIDE + sg * 16, gV + kv_v8_off(d, c0 + 16 * sg));
            }
            const int sseg = (nt + 7) >> 3;    // 8 tokens of one scale row per 16 B
            for (int i = threadIdx.x; i < 4 * sseg; i += blockDim.x) {
                const int bl = i / sseg, sg = i % sseg;
                cp_async16(sVs + bl * ATT_CHUNK * 2 + sg * 16, gVs + kv_vs_off(bl, c0 + 8 * sg));
            }
        }
    }
}

// Whole-chunk staging with the index arithmetic hoisted out of the chunk loop.
// A chunk starts at a multiple of 64 tokens, so every swizzle term depends on
// the thread alone and the arena offset of each 16-byte segment is
// c0 * (bytes per token) + a per-thread constant + an unrolled-copy constant.
// Thread tid copies segments i = tid + 128 j of each tensor (see issue_chunk
// for the segment order); ks / vs: threads 0-31 copy one scale segment each.
template <int KVT> struct ChunkPlan {
    const uint8_t *gK, *gV, *gS, *gT;   // plane bases: K, V codes, K scales, V scales
    uint32_t k_src, k_dst, v_src, v_dst, s_src, s_dst, t_src, t_dst;

    __device__ ChunkPlan(const AttnParams &p, int b, int g) {
        using Lay = AttnLayout<KVT>;
        const uint32_t tid = threadIdx.x;
        const size_t pi = plane_index(p.kv, b, p.layer, g);
        const int Lp = p.kv.Lp;
        if (KVT == 0) {
            gK = p.kv.k + pi * Lp * (HD * 2);
            gV = p.kv.v + pi * Lp * (HD * 2);
            gS = gT = nullptr;
            const uint32_t t = tid >> 4, sg = tid & 15;          // K: 16 segments per token
            k_src = t * 256 + ((sg ^ (t & 7)) << 4);
            k_dst = t * Lay::K_STRIDE + sg * 16;
            const uint32_t d = tid >> 3, vs = tid & 7;           // V^T: 8 segments per dim row
            v_src = ((vs >> 2) * HD + d) * 64 + (((vs & 3) ^ ((tid >> 4) & 3)) << 4);
            v_dst = Lay::K_BYTES + d * Lay::V_STRIDE + vs * 16;
            s_src = s_dst = t_src = t_dst = 0;
        } else {
            gK = p.kv.k + pi * Lp * HD;
            gV = p.kv.v + pi * Lp * HD;
            gS = p.kv.ks + pi * Lp * 8;
            gT = p.kv.vs + pi * Lp * 8;
            const uint32_t t = tid >> 3, sg = tid & 7;           // K: 8 segments per token
            k_src = t * 128 + ((sg ^ (t & 7)) << 4);
            k_dst = t * Lay::K_STRIDE + sg * 16;
            const uint32_t d = tid >> 2, vs = tid & 3;           // V^T: 4 segments per dim row
            v_src = ((vs >> 1) * HD + d) * 32 + (((vs & 1) ^ ((tid >> 4) & 1)) << 4);
            v_dst = Lay::K_BYTES + d * Lay::V_STRIDE + vs * 16;
            s_src = (tid & 31) * 16;                              // K scales: 512 contiguous bytes
            s_dst = Lay::K_BYTES + Lay::V_BYTES + (tid & 31) * 16;
            const uint32_t bl = (tid >> 3) & 3, ss = tid & 7;     // V scales: 4 rows of 8 segments
            t_src = (((ss >> 2) * 4 + bl) * KU + 8 * (ss & 3)) * 2;
            t_dst = Lay::K_BYTES + Lay::V_BYTES + Lay::KS_BYTES + bl * ATT_CHUNK * 2 + ss * 16;
        }
    }

    // tokens [c0, c0 + 64) of the plane into the stage at shared address st
    __device__ __forceinline__ void issue(uint32_t st, int c0) const {
        using Lay = AttnLayout<KVT>;
        if (KVT == 0) {
            const uint8_t *k = gK + (size_t)c0 * 256 + k_src, *v = gV + (size_t)c0 * 256 + v_src;
#pragma unroll
            for (int j = 0; j < 8; j++) {   // tokens t + 8 j; dims d + 16 j
                cp_async16_s(st + k_dst + j * 8 * Lay::K_STRIDE, k + j * 8 * 256);
                cp_async16_s(st + v_dst + j * 16 * Lay::V_STRIDE, v + j * 16 * 64);
            }
        } else {
            const uint8_t *k = gK + (size_t)c0 * 128 + k_src, *v = gV + (size_t)c0 * 128 + v_src;
#pragma unroll
            for (int j = 0; j < 4; j++) {   // tokens t + 16 j; dims d + 32 j
                cp_async16_s(st + k_dst + j * 16 * Lay::K_STRIDE, k + j * 16 * 128);
                cp_async16_s(st + v_dst + j * 32 * Lay::V_STRIDE, v + j * 32 * 32);
            }
            if (threadIdx.x < 32) {
                cp_async16_s(st + s_dst, gS + (size_t)c0 * 8 + s_src);
                cp_async16_s(st + t_dst, gT + (size_t)c0 * 8 + t_src);
            }
        }
    }
};

__device__ __forceinline__ void codes4_to_h2(uint32_t w, uint32_t &lo, uint32_t &hi) {
    // bytes b0..b3 (int8) -> (b0, b1), (b2, b3) as exact fp16 integers:
    // flip the sign bit, place each byte under exponent 0x64 (value 1024 + byte),
    // subtract 1024 + 128
    uint32_t u = w ^ 0x80808080u;
    const __half2 bias = __float2half2_rn(1152.0f);
    lo = h2_as_u32(__hsub2(u32_as_h2(__byte_perm(u, 0x64646464u, 0x4140)), bias));
    hi = h2_as_u32(__hsub2(u32_as_h2(__byte_perm(u, 0x64646464u, 0x4342)), bias));
}

// Q8_0 of 32 fp16 values held one per lane: returns this lane's code, and the
// fp16 scale bits.  amax/127 by IEEE division, codes by IEEE division by the
// fp32 scale, round half to even, clamp to +-127; all-zero blocks -> 0, 0.
__device__ __forceinline__ int8_t q8_0_lane(__half xh, uint16_t &scale_bits) {
    float x = __half2float(xh);
    float amax = fabsf(x);
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(AFULL, amax, o));
    if (amax == 0.0f) { scale_bits = 0; return 0; }
    float d = __fdiv_rn(amax, 127.0f);
    scale_bits = __half_as_ushort(__float2half_rn(d));
    int q = __float2int_rn(__fdiv_rn(x, d));
    q = max(-127, min(127, q));
    return (int8_t)q;
}

// --------------------------------------------------------------- kernel ---
template <int KVT>
__global__ __launch_bounds__(128) void attention_kernel(const AttnParams p) {
    using Lay = AttnLayout<KVT>;
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ __align__(16) uint8_t s_newk[HD * 2], s_newv[HD * 2];   // new token (fp16 or codes)
    __shared__ uint16_t s_newks[4], s_newvs[4];
    __shared__ float s_part[GROUP][HD + 4];   // this CTA's (max, sum, output) per head

    const int rank = blockIdx.x, g = blockIdx.y, b = blockIdx.z, CS = p.cs;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
    tl_min(p.tl, 0);
    const int pos = p.positions[b];       // staged before the step: not a predecessor output
    if (pos < 0 || pos >= p.max_L) return;   // bad device input (whole cluster); flagged by the embedding kernel
    const int ntok = pos + 1;
    const int nch = (ntok + ATT_CHUNK - 1) / ATT_CHUNK;
    // the rank holding the new token also appends it and patches its chunk:
    // one virtual chunk of extra work, so its range is one chunk shorter
    const int nw = nch + (p.append ? 1 : 0);
    const int c_lo = min(nch, rank * nw / CS), c_hi = min(nch, (rank + 1) * nw / CS);
    const int T0 = c_lo * ATT_CHUNK;
    const int T1 = min(c_hi * ATT_CHUNK, ntok);
    const bool empty = c_lo >= c_hi;       // still takes part in the cluster merge
    const int H = p.append ? min(T1, pos) : T1;   // tokens read from the arena
    const int nchunks = c_hi - c_lo;
    const bool has_new = p.append && !empty && T1 == ntok;

    const int NS = p.stages;   // 2..ATT_MAX_STAGES (checked at launch)
    const ChunkPlan<KVT> plan(p, b, g);
    const uint32_t smem_s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    // whole chunks through the plan, the history's ragged end through issue_chunk
    auto load_chunk = [&](int slot, int c0) {
        if (H - c0 >= ATT_CHUNK) plan.issue(smem_s + (uint32_t)(slot * Lay::STAGE), c0);
        else issue_chunk<KVT>(p, smem + slot * Lay::STAGE, b, g, c0, H);
    };
    // ring of NS slots: chunks 0..NS-2 now (the history is no predecessor's
    // output: loaded before the wait); chunk ci + NS - 1 goes out at the top of
    // iteration ci, into the slot chunk ci - 1 has just freed, so that one
    // block barrier per chunk covers both the landing and the reuse
#pragma unroll 1
    for (int s = 0; s < NS - 1; s++) {
        if (s < nchunks) load_chunk(s, T0 + s * ATT_CHUNK);
        cp_async_commit();
    }

    // the rotary row of the new token: a constant table, read before the wait
    float2 rope_new[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
    if (has_new && warp == 0 && p.append) {
        const float2 *cs = p.rope + (size_t)pos * (HD / 2);
        rope_new[0] = cs[lane];
        rope_new[1] = cs[lane + 32];
    }

    pdl_launch_dependents();
    pdl_wait();
    tl_min(p.tl, 1);
    tl_max(p.tl, 4);

    // ---- query fragments: head 4g+gid (gid < 4), dims 16s' + 4tig + {0..3}
    uint32_t qa[8][4];
    if (p.q_frag) {   // prepared by the QKV projection's epilogue (rotated, scaled, hi/lo)
        const uint4 *qf = p.q_frag + ((size_t)b * p.nq + GROUP * g + (gid < GROUP ? gid : 0)) * 32 + tig;
#pragma unroll
        for (int st = 0; st < 8; st++) {
            const uint4 f = gid < GROUP ? qf[st * 4] : make_uint4(0, 0, 0, 0);
            qa[st][0] = f.x;
            qa[st][1] = f.y;
            qa[st][2] = f.z;
            qa[st][3] = f.w;
        }
    } else {
        const float qscale = 0.12751743082459868f;   // log2(e)/sqrt(128): scores in log2 units
        const int hq = GROUP * g + gid;
        const float *qrow = p.qkv + (size_t)b * p.qkv_ld + (size_t)hq * HD;
        const float2 *cs = p.rope + (size_t)pos * (HD / 2);
#pragma unroll
        for (int st = 0; st < 8; st++) {
            float v[4];
#pragma unroll
            for (int e = 0; e < 4; e++) {
                int d = 16 * st + 4 * tig + e;
                float x = 0.0f;
                if (gid < GROUP) {
                    x = qrow[d];
                    if (p.append) {
                        int i = d & 63;
                        float2 c = cs[i];
                        x = d < 64 ? x * c.x - qrow[d + 64] * c.y : x * c.x + qrow[d - 64] * c.y;
                    }
                }
                v[e] = x * qscale;
            }
            __half2 h01 = __floats2half2_rn(v[0], v[1]), h23 = __floats2half2_rn(v[2], v[3]);
            float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
            qa[st][0] = h2_as_u32(h01);
            qa[st][1] = h2_as_u32(__floats2half2_rn(v[0] - f01.x, v[1] - f01.y));
            qa[st][2] = h2_as_u32(h23);
            qa[st][3] = h2_as_u32(__floats2half2_rn(v[2] - f23.x, v[3] - f23.y));
        }
    }

    tl_max(p.tl, 5);
    // ---- the new token (warp 0 of the CTA that holds it): its k and v rows
    // are loaded now, but rotated, rounded, quantized (Q8_0) and appended only
    // at the chunk that holds it, so that the load latency hides behind the
    // earlier chunks
    float kx[4], vx[4];
    if (has_new && warp == 0) {
        const float *krow = p.qkv + (size_t)b * p.qkv_ld + (size_t)(p.nq + g) * HD;
        const float *vrow = p.qkv + (size_t)b * p.qkv_ld + (size_t)(p.nq + p.kv.n_kv + g) * HD;
#pragma unroll
        for (int i = 0; i < 4; i++) { kx[i] = krow[lane + 32 * i]; vx[i] = vrow[lane + 32 * i]; }
    }
    auto append_new = [&]() {
        float kr[4];
#pragma unroll
        for (int i = 0; i < 2; i++) {   // pairs (d, d+64): d = lane + 32 i
            const float2 c = rope_new[i];
            kr[i] = kx[i] * c.x - kx[i + 2] * c.y;
            kr[i + 2] = kx[i + 2] * c.x + kx[i] * c.y;
        }
#pragma unroll
        for (int i = 0; i < 4; i++) {
            int d = lane + 32 * i;
            __half kh = __float2half_rn(kr[i]), vh = __float2half_rn(vx[i]);
            if (KVT == 0) {
                reinterpret_cast<__half *>(s_newk)[d] = kh;
                reinterpret_cast<__half *>(s_newv)[d] = vh;
            } else {
                uint16_t ksb, vsb;
                int8_t kc = q8_0_lane(kh, ksb), vc = q8_0_lane(vh, vsb);
                reinterpret_cast<int8_t *>(s_newk)[d] = kc;
                reinterpret_cast<int8_t *>(s_newv)[d] = vc;
                if (lane == 0) {
                    s_newks[i] = ksb;
                    s_newvs[i] = vsb;
                }
            }
        }
    };
    // the appended token into the arena, from shared memory, once the cluster
    // no longer waits on this CTA (no global store is then outstanding at the
    // cluster barriers' release)
    auto store_new = [&]() {
        const size_t pi = plane_index(p.kv, b, p.layer, g);
        const int Lp = p.kv.Lp;
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const int d = lane + 32 * i;
            if (KVT == 0) {
                *reinterpret_cast<__half *>(p.kv.k + pi * Lp * (HD * 2) + kv_k16_off(pos, d)) =
                    reinterpret_cast<const __half *>(s_newk)[d];
                *reinterpret_cast<__half *>(p.kv.v + pi * Lp * (HD * 2) + kv_v16_off(d, pos)) =
                    reinterpret_cast<const __half *>(s_newv)[d];
            } else {
                *reinterpret_cast<int8_t *>(p.kv.k + pi * Lp * HD + kv_k8_off(pos, d)) =
                    reinterpret_cast<const int8_t *>(s_newk)[d];
                *reinterpret_cast<int8_t *>(p.kv.v + pi * Lp * HD + kv_v8_off(d, pos)) =
                    reinterpret_cast<const int8_t *>(s_newv)[d];
                if (lane == 0) {
                    *reinterpret_cast<uint16_t *>(p.kv.ks + pi * Lp * 8 + kv_ks_off(pos, i)) = s_newks[i];
                    *reinterpret_cast<uint16_t *>(p.kv.vs + pi * Lp * 8 + kv_vs_off(i, pos)) = s_newvs[i];
                }
            }
        }
    };

    // ---- online softmax state (meaningful on lanes gid < 4: head 4g+gid)
    float m_run = -INFINITY, l_run = 0.0f;
    float oacc[16][4];
#pragma unroll
    for (int dn = 0; dn < 16; dn++)
#pragma unroll
        for (int i = 0; i < 4; i++) oacc[dn][i] = 0.0f;
    const float zero4[4] = {0.0f, 0.0f, 0.0f, 0.0f};

    int slot = 0, rslot = NS - 1;
    for (int ci = 0; ci < nchunks; ci++) {
        uint8_t *st = smem + slot * Lay::STAGE;
        const int c0 = T0 + ci * ATT_CHUNK;
        switch (NS) {   // NS - 1 + ci groups committed; chunk ci's is group ci
            case 2: cp_async_wait<0>(); break;
            case 3: cp_async_wait<1>(); break;
            case 4: cp_async_wait<2>(); break;
            case 5: cp_async_wait<3>(); break;
            case 6: cp_async_wait<4>(); break;
            case 7: cp_async_wait<5>(); break;
            default: cp_async_wait<6>(); break;
        }
        __syncthreads();   // chunk ci has landed; every warp is done with chunk ci - 1
        if (ci + NS - 1 < nchunks) load_chunk(rslot, T0 + (ci + NS - 1) * ATT_CHUNK);
        cp_async_commit();
        rslot = rslot + 1 == NS ? 0 : rslot + 1;
        // fix-up (only the chunk at the end of the loaded history): zero V columns
        // past it and insert the new token; whole-history chunks skip both barriers
        const int zfrom = max(H, c0) - c0;
        if (zfrom < ATT_CHUNK) {
            if (has_new && warp == 0) append_new();   // before the barrier that publishes s_new*
            uint8_t *sV = st + Lay::K_BYTES;
            {   // thread d clears row d of V^T from column zfrom on (128 threads, 128 rows)
                // element stores up to a 16-byte boundary, then whole 16-byte stores
                // (rows start 16-byte aligned: strides 160 / 80 / 128 bytes)
                const int d = threadIdx.x;
                const uint4 z4 = make_uint4(0, 0, 0, 0);
                if (KVT == 0) {
                    __half *row = reinterpret_cast<__half *>(sV + d * Lay::V_STRIDE);
                    int t = zfrom;
                    for (; t < ATT_CHUNK && (t & 7); t++) row[t] = __ushort_as_half(0);
                    for (; t < ATT_CHUNK; t += 8) *reinterpret_cast<uint4 *>(row + t) = z4;
                } else {
                    uint8_t *row = sV + d * Lay::V_STRIDE;
                    int t = zfrom;
                    for (; t < ATT_CHUNK && (t & 15); t++) row[t] = 0;
                    for (; t < ATT_CHUNK; t += 16) *reinterpret_cast<uint4 *>(row + t) = z4;
                    if (d < 4) {
                        uint16_t *srow = reinterpret_cast<uint16_t *>(st + Lay::K_BYTES + Lay::V_BYTES + Lay::KS_BYTES) +
                                         d * ATT_CHUNK;
                        int u = zfrom;
                        for (; u < ATT_CHUNK && (u & 7); u++) srow[u] = 0;
                        for (; u < ATT_CHUNK; u += 8) *reinterpret_cast<uint4 *>(srow + u) = z4;
                    }
                }
            }
            __syncthreads();
            if (has_new && pos >= c0 && pos < c0 + ATT_CHUNK) {
                int t = pos - c0;
                uint8_t *sK = st;
                int d = threadIdx.x;   // 128 threads, one head dim each
                if (KVT == 0) {
                    reinterpret_cast<__half *>(sK + t * Lay::K_STRIDE)[d] = reinterpret_cast<__half *>(s_newk)[d];
                    reinterpret_cast<__half *>(sV + d * Lay::V_STRIDE)[t] = reinterpret_cast<__half *>(s_newv)[d];
                } else {
                    sK[t * Lay::K_STRIDE + d] = s_newk[d];
                    sV[d * Lay::V_STRIDE + t] = s_newv[d];
                    if (d < 4) {
                        uint16_t *sKs = reinterpret_cast<uint16_t *>(st + Lay::K_BYTES + Lay::V_BYTES);
                        uint16_t *sVs = sKs + ATT_CHUNK * 4;
                        sKs[t * 4 + d] = s_newks[d];
                        sVs[d * ATT_CHUNK + t] = s_newvs[d];
                    }
                }
            }
            __syncthreads();
        }

        const int tb = c0 + 16 * warp;   // this warp's 16 tokens
        if (tb < T1) {
            const uint8_t *sK = st;
            const uint8_t *sV = st + Lay::K_BYTES;
            // ---- scores S[head][token], tokens of n-tile nt, slot c: 4(c>>1) + 2nt + (c&1)
            float S[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; nt++) {
                const int tr = 16 * warp + 4 * (gid >> 1) + 2 * nt + (gid & 1);
#pragma unroll
                for (int i = 0; i < 4; i++) S[nt][i] = 0.0f;
                if (KVT == 0) {
#pragma unroll
                    for (int st8 = 0; st8 < 8; st8++) {
                        uint2 kb = *reinterpret_cast<const uint2 *>(sK + tr * Lay::K_STRIDE + (16 * st8 + 4 * tig) * 2);
                        mma16816(S[nt], qa[st8], kb.x, kb.y, S[nt]);
                    }
                } else {
                    const uint16_t *sKs = reinterpret_cast<const uint16_t *>(st + Lay::K_BYTES + Lay::V_BYTES);
                    const int ta = 16 * warp + 4 * tig + 2 * nt;   // tokens of columns 2tig, 2tig+1
                    // the four block scales of tokens ta and ta + 1
                    const uint2 ksa = *reinterpret_cast<const uint2 *>(sKs + ta * 4);
                    const uint2 ksb = *reinterpret_cast<const uint2 *>(sKs + (ta + 1) * 4);
                    const float2 ka01 = __half22float2(u32_as_h2(ksa.x)), ka23 = __half22float2(u32_as_h2(ksa.y));
                    const float2 kb01 = __half22float2(u32_as_h2(ksb.x)), kb23 = __half22float2(u32_as_h2(ksb.y));
                    const float kas[4] = {ka01.x, ka01.y, ka23.x, ka23.y};
                    const float kbs[4] = {kb01.x, kb01.y, kb23.x, kb23.y};
#pragma unroll
                    for (int bl = 0; bl < 4; bl++) {
                        float tmp[4];
#pragma unroll
                        for (int hs = 0; hs < 2; hs++) {
                            const int st8 = 2 * bl + hs;
                            uint32_t w = *reinterpret_cast<const uint32_t *>(sK + tr * Lay::K_STRIDE + 16 * st8 + 4 * tig);
                            uint32_t b0, b1;
                            codes4_to_h2(w, b0, b1);
                            if (hs) mma16816(tmp, qa[st8], b0, b1, tmp);
                            else mma16816(tmp, qa[st8], b0, b1, zero4);
                        }
                        const float ka = kas[bl], kb = kbs[bl];
                        S[nt][0] += ka * tmp[0];
                        S[nt][1] += kb * tmp[1];
                        S[nt][2] += ka * tmp[2];
                        S[nt][3] += kb * tmp[3];
                    }
                }
            }
            // ---- online softmax on this tile (head gid, tokens 4tig + {0,1,2,3})
            float sc[4];
            sc[0] = S[0][0] + S[0][2];
            sc[1] = S[0][1] + S[0][3];
            sc[2] = S[1][0] + S[1][2];
            sc[3] = S[1][1] + S[1][3];
            if (gid >= GROUP) sc[0] = sc[1] = sc[2] = sc[3] = -INFINITY;   // zero A rows: no head
            if (tb + 16 > T1)   // the range's last tile may end early
#pragma unroll
                for (int e = 0; e < 4; e++)
                    if (tb + 4 * tig + e >= T1) sc[e] = -INFINITY;
            float mt = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
            mt = fmaxf(mt, __shfl_xor_sync(AFULL, mt, 1));
            mt = fmaxf(mt, __shfl_xor_sync(AFULL, mt, 2));
            // scores are in log2 units (q carries log2(e)/sqrt(128)); the output
            // is rescaled only when some head's running max grew (alpha = 1
            // exactly otherwise), which after the first tiles is rare
            const float m_new = fmaxf(m_run, mt);
            const bool grow = m_new > m_run;
            const float alpha = grow ? exp2f(m_run - m_new) : 1.0f;   // m_run = -inf -> 0
            float pr[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            if (m_new != -INFINITY) {
#pragma unroll
                for (int e = 0; e < 4; e++) pr[e] = exp2f(sc[e] - m_new);
            }
            m_run = m_new;
            l_run = l_run * alpha + (pr[0] + pr[1]) + (pr[2] + pr[3]);
            if (__any_sync(AFULL, grow))
#pragma unroll
                for (int dn = 0; dn < 16; dn++)
#pragma unroll
                    for (int i = 0; i < 4; i++) oacc[dn][i] *= alpha;
            // ---- output += P V
            if (KVT == 0) {
                uint32_t pa[4];
                __half2 h01 = __floats2half2_rn(pr[0], pr[1]), h23 = __floats2half2_rn(pr[2], pr[3]);
                float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
                pa[0] = h2_as_u32(h01);
                pa[1] = h2_as_u32(__floats2half2_rn(pr[0] - f01.x, pr[1] - f01.y));
                pa[2] = h2_as_u32(h23);
                pa[3] = h2_as_u32(__floats2half2_rn(pr[2] - f23.x, pr[3] - f23.y));
#pragma unroll
                for (int dn = 0; dn < 16; dn++) {
                    const int d = 8 * dn + gid;
                    uint2 vb = *reinterpret_cast<const uint2 *>(sV + d * Lay::V_STRIDE + (16 * warp + 4 * tig) * 2);
                    mma16816(oacc[dn], pa, vb.x, vb.y, oacc[dn]);
                }
            } else {
                const uint16_t *sVs = reinterpret_cast<const uint16_t *>(st + Lay::K_BYTES + Lay::V_BYTES + Lay::KS_BYTES);
                const int tl = 16 * warp + 4 * tig;
#pragma unroll
                for (int bl = 0; bl < 4; bl++) {
                    const uint2 vsc = *reinterpret_cast<const uint2 *>(sVs + bl * ATT_CHUNK + tl);   // tokens tl..tl+3
                    const float2 v01 = __half22float2(u32_as_h2(vsc.x)), v23 = __half22float2(u32_as_h2(vsc.y));
                    const float q4[4] = {pr[0] * v01.x, pr[1] * v01.y, pr[2] * v23.x, pr[3] * v23.y};
                    uint32_t pa[4];
                    __half2 h01 = __floats2half2_rn(q4[0], q4[1]), h23 = __floats2half2_rn(q4[2], q4[3]);
                    float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
                    pa[0] = h2_as_u32(h01);
                    pa[1] = h2_as_u32(__floats2half2_rn(q4[0] - f01.x, q4[1] - f01.y));
                    pa[2] = h2_as_u32(h23);
                    pa[3] = h2_as_u32(__floats2half2_rn(q4[2] - f23.x, q4[3] - f23.y));
#pragma unroll
                    for (int dq = 0; dq < 4; dq++) {
                        const int dn = 4 * bl + dq, d = 8 * dn + gid;
                        uint32_t w = *reinterpret_cast<const uint32_t *>(sV + d * Lay::V_STRIDE + tl);
                        uint32_t b0, b1;
                        codes4_to_h2(w, b0, b1);
                        mma16816(oacc[dn], pa, b0, b1, oacc[dn]);
                    }
                }
            }
        }
        slot = slot + 1 == NS ? 0 : slot + 1;
    }
    cp_async_wait<0>();
    tl_max(p.tl, 6);

    // ---- merge the 4 warps of this CTA (smem reused after the stages)
    float *wm = reinterpret_cast<float *>(smem);          // [4 warps][4 heads]
    float *wl = wm + 16;
    float *wo = wl + 16;                                   // [4][4][128]
    float l_tot = l_run;
    l_tot += __shfl_xor_sync(AFULL, l_tot, 1);
    l_tot += __shfl_xor_sync(AFULL, l_tot, 2);
    __syncthreads();
    if (gid < GROUP) {
        if (tig == 0) { wm[warp * 4 + gid] = m_run; wl[warp * 4 + gid] = l_tot; }
#pragma unroll
        for (int dn = 0; dn < 16; dn++)
#pragma unroll
            for (int e = 0; e < 2; e++)
                wo[(warp * 4 + gid) * HD + 8 * dn + 2 * tig + e] = oacc[dn][e] + oacc[dn][2 + e];
    }
    __syncthreads();
    const int head = threadIdx.x >> 5, d0 = (threadIdx.x & 31) * 4;
    {
        float M = -INFINITY;
        for (int w = 0; w < 4; w++) M = fmaxf(M, wm[w * 4 + head]);
        float L = 0.0f, O[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        for (int w = 0; w < 4; w++) {
            float mw = wm[w * 4 + head];
            float f = mw == -INFINITY ? 0.0f : exp2f(mw - M);
            L += f * wl[w * 4 + head];
            for (int e = 0; e < 4; e++) O[e] += f * wo[(w * 4 + head) * HD + d0 + e];
        }
        if ((threadIdx.x & 31) == 0) { s_part[head][0] = M; s_part[head][1] = L; }
        for (int e = 0; e < 4; e++) s_part[head][4 + d0 + e] = O[e];
    }
    // ---- rank 0 merges the cluster's partials through distributed shared memory
    cg::cluster_group cluster = cg::this_cluster();
    cluster_arrive_release();   // the partials in s_part (shared memory only)
    cluster_wait_acquire();
    if (rank == 0) {
        // issue every peer's loads before using any (distributed shared memory
        // latency is paid once, not once per rank)
        float mr[16], lr[16];
        float4 orr[16];
#pragma unroll
        for (int r = 0; r < 16; r++) {
            mr[r] = -INFINITY;
            lr[r] = 0.0f;
            orr[r] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            if (r < CS) {
                const float *ps = cluster.map_shared_rank(&s_part[0][0], r) + head * (HD + 4);
                mr[r] = ps[0];
                lr[r] = ps[1];
                orr[r] = *reinterpret_cast<const float4 *>(ps + 4 + d0);
            }
        }
        float M = -INFINITY;
#pragma unroll
        for (int r = 0; r < 16; r++) M = fmaxf(M, mr[r]);
        float L = 0.0f, O[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int r = 0; r < 16; r++) {
            const float f = mr[r] == -INFINITY ? 0.0f : exp2f(mr[r] - M);
            L += f * lr[r];
            O[0] += f * orr[r].x; O[1] += f * orr[r].y; O[2] += f * orr[r].z; O[3] += f * orr[r].w;
        }
        const float inv = 1.0f / L;
        const int qd = p.nq * HD;
        const int kcol = (GROUP * g + head) * HD + d0;   // column of o, the O projection's input
        float y[4];
        for (int e = 0; e < 4; e++) y[e] = O[e] * inv;
        float *o = p.o + (size_t)b * qd + kcol;
        for (int e = 0; e < 4; e++) o[e] = y[e];
        // the O projection's operand as fp16 hi + lo parts (elements 4..7 of every
        // 8 stored /16) and the per-32 sub-block sums, as the GEMM prep writes them
        __half h[4], hl[4];
        float part = 0.0f;
        for (int e = 0; e < 4; e++) {
            h[e] = __float2half_rn(y[e]);
            hl[e] = __float2half_rn((y[e] - __half2float(h[e])) * LO_SCALE);
            part += y[e];
        }
        if (d0 & 4)
            for (int e = 0; e < 4; e++) {
                h[e] = __hmul(h[e], __float2half(0.0625f));
                hl[e] = __hmul(hl[e], __float2half(0.0625f));
            }
        const size_t ai = act_chunk(kcol >> 8, b, (kcol & 255) >> 3, p.oBp) + (kcol & 7);
        *reinterpret_cast<uint2 *>(p.o16 + ai) =
            make_uint2(h2_as_u32(__halves2half2(h[0], h[1])), h2_as_u32(__halves2half2(h[2], h[3])));
        *reinterpret_cast<uint2 *>(p.o16lo + ai) =
            make_uint2(h2_as_u32(__halves2half2(hl[0], hl[1])), h2_as_u32(__halves2half2(hl[2], hl[3])));
        part += __shfl_xor_sync(AFULL, part, 1);
        part += __shfl_xor_sync(AFULL, part, 2);
        part += __shfl_xor_sync(AFULL, part, 4);
        if ((lane & 7) == 0) store_sum(p.osx, kcol >> 8, b, (kcol >> 5) & 7, p.oBp, part);
    }
    tl_max(p.tl, 7);
    // peers keep their partials alive until rank 0 has read them (its reads
    // have returned by the time it arrives; nothing needs ordering)
    cluster_arrive_relaxed();
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
    // a step whose inputs a device check flagged (or that follows one before
    // zdec_sync) changes no cache state: the status word is final by now,
    // every kernel that sets it having completed before this kernel's wait
    if (has_new && warp == 0 && (*(volatile uint32_t *)p.status & STATUS_STATE_ERRORS) == 0) store_new();
    tl_end(p.tl);
}

cudaError_t attention_setup(int kv_dtype) {
    int smem = (int)attention_smem_bytes(kv_dtype, att_max_stages(kv_dtype));
    cudaError_t e;
    if (kv_dtype == 0) {
        e = cudaFuncSetAttribute(attention_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(attention_kernel<0>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    } else {
        e = cudaFuncSetAttribute(attention_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(attention_kernel<1>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    }
    return e;
}

int attention_max_clusters(int kv_dtype, int stages, int cs) {
    if (cs < 1 || cs > 16 || stages < 2 || stages > att_max_stages(kv_dtype)) return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cs, 8, 1);
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = attention_smem_bytes(kv_dtype, stages);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    cudaError_t e = kv_dtype ? cudaOccupancyMaxActiveClusters(&n, attention_kernel<1>, &cfg)
                             : cudaOccupancyMaxActiveClusters(&n, attention_kernel<0>, &cfg);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

cudaError_t launch_attention(const AttnParams &p0, bool pdl, cudaStream_t stream) {
    AttnParams p = p0;
    if (p.cs < 1 || p.cs > 16) return cudaErrorInvalidValue;
    if (p.stages == 0) p.stages = attention_default_stages(p.kv.kv_dtype);
    if (p.stages < 2 || p.stages > att_max_stages(p.kv.kv_dtype)) return cudaErrorInvalidValue;
    dim3 grid(p.cs, p.kv.n_kv, p.B), block(128);
    size_t smem = attention_smem_bytes(p.kv.kv_dtype, p.stages);
    if (p.kv.kv_dtype == 0) return launch_k(attention_kernel<0>, grid, block, smem, pdl, p.cs, stream, p);
    return launch_k(attention_kernel<1>, grid, block, smem, pdl, p.cs, stream, p);
}

// ------------------------------------------------------------ bulk append ---
// One warp per (layer, token, kv head); lane holds dims lane + 32 i, i.e.
// element `lane` of Q8_0 block i.
__global__ void kv_append_kernel(const KvArena a, int slot, int t0, int n,
                                 const uint16_t *__restrict__ k16, const uint16_t *__restrict__ v16) {
    long w = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    int lane = threadIdx.x & 31;
    if (w >= (long)a.n_layers * n * a.n_kv) return;
    int g = (int)(w % a.n_kv);
    int t = (int)((w / a.n_kv) % n);
    int l = (int)(w / ((long)a.n_kv * n));
    const uint16_t *ks = k16 + (((size_t)l * n + t) * a.n_kv + g) * HD;
    const uint16_t *vs = v16 + (((size_t)l * n + t) * a.n_kv + g) * HD;
    size_t pi = plane_index(a, slot, l, g);
    int pos = t0 + t;
    for (int i = 0; i < 4; i++) {
        int d = lane + 32 * i;
        uint16_t kb = ks[d], vb = vs[d];
        if (a.kv_dtype == 0) {
            *reinterpret_cast<uint16_t *>(a.k + pi * a.Lp * (HD * 2) + kv_k16_off(pos, d)) = kb;
            *reinterpret_cast<uint16_t *>(a.v + pi * a.Lp * (HD * 2) + kv_v16_off(d, pos)) = vb;
        } else {
            uint16_t ksb, vsb;
            int8_t kc = q8_0_lane(__ushort_as_half(kb), ksb);
            int8_t vc = q8_0_lane(__ushort_as_half(vb), vsb);
            *reinterpret_cast<int8_t *>(a.k + pi * a.Lp * HD + kv_k8_off(pos, d)) = kc;
            *reinterpret_cast<int8_t *>(a.v + pi * a.Lp * HD + kv_v8_off(d, pos)) = vc;
            if (lane == 0) {
                *reinterpret_cast<uint16_t *>(a.ks + pi * a.Lp * 8 + kv_ks_off(pos, i)) = ksb;
                *reinterpret_cast<uint16_t *>(a.vs + pi * a.Lp * 8 + kv_vs_off(i, pos)) = vsb;
            }
        }
    }
}

cudaError_t launch_kv_append(const KvArena &a, int slot, int t0, int n, const uint16_t *k16,
                             const uint16_t *v16, cudaStream_t stream) {
    long warps = (long)a.n_layers * n * a.n_kv;
    if (warps == 0) return cudaSuccess;
    kv_append_kernel<<<(unsigned)((warps * 32 + 255) / 256), 256, 0, stream>>>(a, slot, t0, n, k16, v16);
    return cudaGetLastError();
}

// One thread per (token, kv head, dim) of one layer.
__global__ void kv_read_kernel(const KvArena a, int slot, int layer, int t0, int n, uint8_t *k,
                               uint8_t *v, uint16_t *ks, uint16_t *vs) {
    long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long)n * a.n_kv * HD) return;
    int d = (int)(i % HD), g = (int)((i / HD) % a.n_kv), t = (int)(i / ((long)HD * a.n_kv));
    size_t pi = plane_index(a, slot, layer, g);
    int pos = t0 + t;
    if (a.kv_dtype == 0) {
        reinterpret_cast<uint16_t *>(k)[i] = *reinterpret_cast<const uint16_t *>(a.k + pi * a.Lp * (HD * 2) + kv_k16_off(pos, d));
        reinterpret_cast<uint16_t *>(v)[i] = *reinterpret_cast<const uint16_t *>(a.v + pi * a.Lp * (HD * 2) + kv_v16_off(d, pos));
    } else {
        k[i] = a.k[pi * a.Lp * HD + kv_k8_off(pos, d)];
        v[i] = a.v[pi * a.Lp * HD + kv_v8_off(d, pos)];
        if ((d & 31) == 0) {
            size_t o = ((size_t)t * a.n_kv + g) * 4 + (d >> 5);
            ks[o] = *reinterpret_cast<const uint16_t *>(a.ks + pi * a.Lp * 8 + kv_ks_off(pos, d >> 5));
            vs[o] = *reinterpret_cast<const uint16_t *>(a.vs + pi * a.Lp * 8 + kv_vs_off(d >> 5, pos));
        }
    }
}

cudaError_t launch_kv_read(const KvArena &a, int slot, int layer, int t0, int n, uint8_t *k,
                           uint8_t *v, uint16_t *ks, uint16_t *vs, cudaStream_t stream) {
    long total = (long)n * a.n_kv * HD;
    if (total == 0) return cudaSuccess;
    kv_read_kernel<<<(unsigned)((total + 255) / 256), 256, 0, stream>>>(a, slot, layer, t0, n, k, v, ks, vs);
    return cudaGetLastError();
}

}  // namespace zdec
