// kv_pool.cuh -- the paged KV cache: page geometry, per-tensor storage types
// and the byte layout of one 64-token chunk, shared by the attention kernel
// and the append / read-back kernels.
//
// The cache is a pool of pages.  A page holds 64 consecutive tokens of one
// sequence for every layer and kv head, K and V.  Each sequence slot owns a
// block table (page index per 64 tokens of its history, -1 where none), so
// sequences of any length share one pool and a freed slot's pages go to the
// next admitted sequence ("Eight concurrent agents pull 5.6x more tokens from
// one RX 9070 XT", "Where it stops, and the argument I got wrong in May": the
// KV budget, not the arithmetic, bounds the swarm; "Q8 KV cache pushes an
// RDNA4 swarm crossover...", "The storage format is the last cheap lever").
//
// Inside a page the (layer, kv head) chunks follow each other; a chunk is the
// K region then the V region.  K and V each take one of three storage types
// ("Q8 KV cache pushes...", "Why Q8 is close to free and where the sharp
// edges are": K and V cache types are chosen independently):
//   F16   K [64 tokens][128] half, the 16-byte segment s (8 dims) of token t
//         at s ^ (t & 7)                                         16384 B
//         V [2 units][128 dims][32 tokens] half (V^T per 32-token unit), the
//         segment s (8 tokens) of dim row d at s ^ ((d >> 1) & 3) 16384 B
//   Q8_0  K codes [64][128] int8, segment s (16 dims) at s ^ (t & 7), then
//         scales [64][4] fp16 (one per 32 dims)                    8704 B
//         V codes [2][128][32] int8, segment s (16 tokens) of dim row d at
//         s ^ ((d >> 2) & 1), then scales [2][4][32] fp16          8704 B
//         Codes are stored offset by 128 (byte = code ^ 0x80) so that one
//         byte_perm puts them under an fp16 exponent.
//   FP8   e4m3 codes, laid out as the Q8_0 codes, no scales        8192 B
// The swizzles place the rows that the attention's mma fragments read
// together in distinct shared-memory banks once a chunk is copied verbatim.
#pragma once
#include "zdec_internal.cuh"

namespace zdec {

enum KvType : int { KV_T_F16 = 0, KV_T_Q8 = 1, KV_T_FP8 = 2 };
constexpr int PAGE_TOKENS = 64;              // tokens per page (= the attention's chunk)

__host__ __device__ constexpr uint32_t kv_region_bytes(int type) {
    return type == KV_T_F16 ? 16384u : (type == KV_T_Q8 ? 8704u : 8192u);
}

struct KvPool {
    uint8_t *base;          // n_pages pages
    size_t page_bytes;      // n_layers * n_kv * (K region + V region)
    int n_pages;
    int k_type, v_type;     // KvType of K and V
    int n_layers, n_kv;
    const int32_t *table;   // [max_slots][max_pages]: page of each 64 tokens of a slot, -1: none
    int max_pages;          // table entries per slot
};

// Byte offset of the (layer, kv head) chunk inside a page.
__host__ __device__ __forceinline__ size_t kv_chunk_off(const KvPool &p, int layer, int g) {
    return (size_t)(layer * p.n_kv + g) * (kv_region_bytes(p.k_type) + kv_region_bytes(p.v_type));
}
// Page of token t of a slot (-1 if none).
__device__ __forceinline__ int kv_page(const KvPool &p, int slot, int t) {
    return p.table[(size_t)slot * p.max_pages + (t >> 6)];
}
__device__ __forceinline__ bool kv_page_ok(const KvPool &p, int page) { return page >= 0 && page < p.n_pages; }

// Offsets inside a K region, t = token within the chunk (0..63), d = dim.
__host__ __device__ __forceinline__ uint32_t k16_off(int t, int d) {
    return (uint32_t)t * 256u + ((((uint32_t)(d >> 3) ^ (uint32_t)(t & 7)) << 4) | ((uint32_t)(d & 7) << 1));
}
__host__ __device__ __forceinline__ uint32_t k8_off(int t, int d) {
    return (uint32_t)t * 128u + ((((uint32_t)(d >> 4) ^ (uint32_t)(t & 7)) << 4) | (uint32_t)(d & 15));
}
__host__ __device__ __forceinline__ uint32_t ks_off(int t, int blk) { return 8192u + (uint32_t)t * 8u + (uint32_t)blk * 2u; }
// Offsets inside a V region.
__host__ __device__ __forceinline__ uint32_t v16_off(int t, int d) {
    const uint32_t tt = (uint32_t)(t & 31);
    return ((uint32_t)(t >> 5) * 128u + (uint32_t)d) * 64u +
           ((((tt >> 3) ^ ((uint32_t)(d >> 1) & 3u)) << 4) | ((tt & 7u) << 1));
}
__host__ __device__ __forceinline__ uint32_t v8_off(int t, int d) {
    const uint32_t tt = (uint32_t)(t & 31);
    return ((uint32_t)(t >> 5) * 128u + (uint32_t)d) * 32u +
           ((((tt >> 4) ^ ((uint32_t)(d >> 2) & 1u)) << 4) | (tt & 15u));
}
__host__ __device__ __forceinline__ uint32_t vs_off(int t, int blk) {
    return 8192u + (((uint32_t)(t >> 5) * 4u + (uint32_t)blk) * 32u + (uint32_t)(t & 31)) * 2u;
}

// ------------------------------------------------------- conversions ---
// Q8_0 of 32 fp16 values held one per lane (all 32 lanes): returns this
// lane's code and the block's fp16 scale bits.  amax / 127 by IEEE division,
// codes by IEEE division by that fp32 scale, rounded half to even and clamped
// to +-127; an all-zero block stores scale 0 and codes 0.
__device__ __forceinline__ int8_t q8_0_lane(__half xh, uint16_t &scale_bits) {
    const float x = __half2float(xh);
    float amax = fabsf(x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    if (amax == 0.0f) { scale_bits = 0; return 0; }
    const float d = __fdiv_rn(amax, 127.0f);
    scale_bits = __half_as_ushort(__float2half_rn(d));
    int q = __float2int_rn(__fdiv_rn(x, d));
    q = max(-127, min(127, q));
    return (int8_t)q;
}
// fp16 -> e4m3: nearest, ties to even, saturating at +-448 (hardware cvt).
__device__ __forceinline__ uint8_t e4m3_from_half(__half x) {
    uint16_t out;
    const uint32_t in = (uint32_t)__half_as_ushort(x);   // low half converts to the low byte
    asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(out) : "r"(in));
    return (uint8_t)(out & 0xFFu);
}
// Two e4m3 codes (low byte first) -> two fp16 values (exact).
__device__ __forceinline__ uint32_t e4m3x2_to_h2(uint16_t c2) {
    uint32_t out;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(out) : "h"(c2));
    return out;
}

}  // namespace zdec
