// zdec_internal.cuh -- layouts and device helpers shared by the zdec kernels.
//
// Repacked Q4_K layout ("tile blocks").  A matrix of N rows x K columns is cut
// into row tiles of 16 rows; each (row tile, super-block of 256 columns) is one
// 2304-byte tile block (= 16 canonical 144-byte blocks).  Eight consecutive row
// tiles form a group (128 rows); the eight tile blocks of one (group,
// super-block) are adjacent, so a GEMM stage is one 18,432-byte bulk copy:
//   offset(rt, sb) = ((rt / 8) * nsb + sb) * 18432 + (rt % 8) * 2304,
// nsb = K / 256.  The row count is padded to a whole group with zero blocks.
// Inside a tile block the bytes are arranged for the warp that multiplies it
// with mma.sync.m16n8k16 (lane = 4*g + tig, g = lane/4, tig = lane%4):
//   [0, 2048)    codes: 4 chunks of 512 B; chunk c, lane l -> 16 bytes at
//                c*512 + 16*l, i.e. one uint4 load per lane per chunk.
//   [2048, 2304) meta: one uint64 per lane at 2048 + 8*l.
// Lane (g, tig) owns rows g and g+8 of the tile and, in every super-block,
// the two 32-weight sub-blocks j1 = 2*tig and j2 = 2*tig+1 of both rows.
// Within sub-block j = 2*tig + h the lane's 32 weights are 4 groups of 8
// (p = 0..3): k = 256*sb + 32*j + 8*p + o, o = 0..7.  Group (h, p) of row
// rho (0: row g, 1: row g+8) is one 32-bit word; chunk c = 2*h + (p >> 1),
// word index (p & 1)*2 + rho.  Nibble n of the word (bits 4n..4n+3) holds
// offset o = {0,4,2,6,1,5,3,7}[n].  With the masks 0x000F000F / 0x00F000F0
// (and the same after >> 8) one lop3 yields the half2 pairs the mma A
// fragment wants: offsets (0,1) and (2,3) as 1024+q, offsets (4,5) and (6,7)
// as 1024+16q.  The activation operand stores the elements at offsets 4..7
// divided by 16 so both kinds of pair multiply to q*x.
// Meta uint64 of lane (g, tig): low word = row g, high word = row g+8, each
//   bits 0-5 sc[j1], 16-21 sc[j2], 6-11 m[j1], 22-27 m[j2],
//   bits 12-15, 28-31 (both words): four nibbles of one fp16 value: tig 0 ->
//   d of row g, 1 -> dmin of row g, 2 -> d of row g+8, 3 -> dmin of row g+8
//   (value bits 0-3 low word 12-15, 4-7 low 28-31, 8-11 high 12-15, 12-15 high 28-31).
#pragma once
#include <cstdint>
#include <cuda_fp16.h>

namespace zdec {

constexpr int QK = 256;                 // weights per super-block
constexpr int CANON_BLOCK = 144;        // canonical bytes per super-block
constexpr int TILE_BYTES = 2304;        // 16 rows x 144
constexpr int TILE_CODE_BYTES = 2048;
constexpr int HD = 128;                 // head_dim the attention kernel implements
constexpr int GROUP = 4;                // query heads per kv head the kernel implements
constexpr int ATT_CHUNK = 64;           // tokens per attention smem chunk
constexpr int MAX_B = 32;
constexpr int GT = 8;                   // row tiles per group (one per GEMM warp)
constexpr int GROUP_BYTES = GT * TILE_BYTES;

__host__ __device__ __forceinline__ size_t tile_offset(int rt, int sb, int nsb) {
    return ((size_t)(rt >> 3) * nsb + sb) * GROUP_BYTES + (size_t)(rt & 7) * TILE_BYTES;
}
__host__ __device__ __forceinline__ int n_groups(int n_rowtiles) { return (n_rowtiles + GT - 1) / GT; }

// GEMM activation operand ("act planes").  For every super-block sb the rows
// b = 0..Bp-1 hold that super-block's 256 values as fp16, elements 4..7 of
// every 8 divided by 16 (matching the nibble layout), in 32 chunks of 8.  Chunk
// c of row b sits at chunk position c ^ ((c >> 3) | ((b & 1) << 2)) so that the
// eight lanes of a shared-memory phase (two rows, four tigs) hit eight
// different bank groups.  A plane is [nsb][Bp][256] halves; the hi and lo
// parts of a split operand are two planes.  The sub-block sums are
// [nsb][Bp][4 tig][4] halves: (hi_2tig, hi_2tig+1, lo_2tig, lo_2tig+1) where
// hi + lo is the fp32 sum of the 32 values of sub-block j.
__host__ __device__ __forceinline__ size_t act_chunk(int sb, int b, int c, int Bp) {
    int pc = c ^ ((c >> 3) | ((b & 1) << 2));
    return ((size_t)sb * Bp + b) * 256 + (size_t)pc * 8;
}
__host__ __device__ __forceinline__ size_t act_sum(int sb, int b, int j, int lo, int Bp) {
    return (((size_t)sb * Bp + b) * 4 + (j >> 1)) * 4 + (lo ? 2 : 0) + (j & 1);
}

// offset -> nibble position inside a lane word, and back
__host__ __device__ constexpr int nib_of_off(int o) {
    return o == 0 ? 0 : o == 4 ? 1 : o == 2 ? 2 : o == 6 ? 3 : o == 1 ? 4 : o == 5 ? 5 : o == 3 ? 6 : 7;
}
__host__ __device__ constexpr int off_of_nib(int n) {
    return n == 0 ? 0 : n == 1 ? 4 : n == 2 ? 2 : n == 3 ? 6 : n == 4 ? 1 : n == 5 ? 5 : n == 6 ? 3 : 7;
}

// ----------------------------------------------------------------- PTX ---
__device__ __forceinline__ void pdl_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Hint: bring the 128-byte line holding p into this SM's L1.
__device__ __forceinline__ void prefetch_l1(const void *p) {
    asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
}
__device__ __forceinline__ uint4 ld_stream_u4(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}
__device__ __forceinline__ uint2 ld_stream_u2(const void *p) {
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
                 : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}
__device__ __forceinline__ uint4 ld_u4(const void *p) {
    return *reinterpret_cast<const uint4 *>(p);
}
__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t mask, uint32_t orv) {
    uint32_t r;
    // (a & mask) | orv
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(a), "r"(mask), "r"(orv));
    return r;
}
// D = A(16x16 f16, row) * B(16x8 f16, col) + C(16x8 f32)
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1, const float (&c)[4]) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1),
          "f"(c[0]), "f"(c[1]), "f"(c[2]), "f"(c[3]));
}
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async16_s(uint32_t s, const void *gmem) {   // s: shared-window address
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// ------------------------------------------------- mbarrier + bulk copy ---
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}
// 1-D bulk copy global -> this CTA's shared memory, completing on `bar`.
// Addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}

// ------------------------------------------------------------- clusters ---
__device__ __forceinline__ void cluster_arrive_release() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Arrive without a release of this thread's memory operations: for a barrier
// that only publishes mbarrier initialisations, which thread 0 has already
// released with fence.mbarrier_init.release.cluster.
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
// Shared-memory address `a` of this CTA -> the same address in cluster rank r.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t a, uint32_t r) {
    uint32_t out;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(a), "r"(r));
    return out;
}
// Asynchronous store of registers into another CTA's shared memory (cluster
// addresses), counted as bytes of a transaction on that CTA's mbarrier `bar`
// (which expects them): no fence or separate arrive needed.  addr aligned to
// the vector size.
__device__ __forceinline__ void st_async_v4(uint32_t addr, float4 v, uint32_t bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];"
                 ::"r"(addr), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(bar)
                 : "memory");
}
__device__ __forceinline__ void st_async_v2(uint32_t addr, float a, float b, uint32_t bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];"
                 ::"r"(addr), "f"(a), "f"(b), "r"(bar)
                 : "memory");
}
// Wait on this CTA's mbarrier, acquiring what other CTAs of the cluster released.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }
__device__ __forceinline__ __half2 u32_as_h2(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }

// The lo plane holds (y - fp16(y)) * LO_SCALE: the residual is ~2^-11 |y|, and
// scaling it by 2^10 keeps it out of the fp16 subnormal range for small
// activations (the GEMM divides its lo accumulator by the same power of two).
constexpr float LO_SCALE = 1024.0f;
constexpr float LO_UNSCALE = 1.0f / 1024.0f;

// fp16 hi + lo of eight values into act planes at element index idx (a chunk
// start); elements 4..7 are stored divided by 16.  lo may be null.
__device__ __forceinline__ void store_act8(__half *hi, __half *lo, size_t idx, const float (&y)[8]) {
    __half h[8], l[8];
#pragma unroll
    for (int i = 0; i < 8; i++) {
        h[i] = __float2half_rn(y[i]);
        l[i] = __float2half_rn((y[i] - __half2float(h[i])) * LO_SCALE);
    }
    const __half sixteenth = __float2half(0.0625f);
#pragma unroll
    for (int i = 4; i < 8; i++) {
        h[i] = __hmul(h[i], sixteenth);
        l[i] = __hmul(l[i], sixteenth);
    }
    uint4 v;
    v.x = h2_as_u32(__halves2half2(h[0], h[1]));
    v.y = h2_as_u32(__halves2half2(h[2], h[3]));
    v.z = h2_as_u32(__halves2half2(h[4], h[5]));
    v.w = h2_as_u32(__halves2half2(h[6], h[7]));
    *reinterpret_cast<uint4 *>(hi + idx) = v;
    if (lo) {
        v.x = h2_as_u32(__halves2half2(l[0], l[1]));
        v.y = h2_as_u32(__halves2half2(l[2], l[3]));
        v.z = h2_as_u32(__halves2half2(l[4], l[5]));
        v.w = h2_as_u32(__halves2half2(l[6], l[7]));
        *reinterpret_cast<uint4 *>(lo + idx) = v;
    }
}
// Sub-block sum `part` (fp32) of sub-block j of super-block sb, row b.
__device__ __forceinline__ void store_sum(__half *sums, int sb, int b, int j, int Bp, float part) {
    __half hi = __float2half_rn(part);
    __half lo = __float2half_rn(part - __half2float(hi));
    sums[act_sum(sb, b, j, 0, Bp)] = hi;
    sums[act_sum(sb, b, j, 1, Bp)] = lo;
}

// ------------------------------------------------------ launch timeline ---
// Optional per-launch timestamps (%globaltimer, ns): tl[0] earliest CTA start,
// tl[1] earliest CTA past the dependency wait, tl[2] latest CTA end, tl[3] the
// launch's kind (written by the host), tl[4..7] the latest CTA to reach a
// kernel's own milestones (projection: past the wait, first stage landed, K
// loop done, cluster reduction done).  Null: off.  Recorded by thread 0 of
// every CTA with atomic min / max.
__device__ __forceinline__ unsigned long long gtimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void tl_min(unsigned long long *tl, int k) {
    if (tl && threadIdx.x == 0) atomicMin(tl + k, gtimer());
}
__device__ __forceinline__ void tl_end(unsigned long long *tl) {
    if (tl && threadIdx.x == 0) atomicMax(tl + 2, gtimer());
}
// Latest CTA to reach milestone k (4..7; what each means is up to the kernel).
__device__ __forceinline__ void tl_max(unsigned long long *tl, int k) {
    if (tl && threadIdx.x == 0) atomicMax(tl + k, gtimer());
}

// ------------------------------------------------------- device status ---
enum : uint32_t { STATUS_POSITION = 1u, STATUS_CAPACITY = 2u, STATUS_TIMEOUT = 4u, STATUS_TOKEN = 8u,
                  STATUS_PAGE = 16u /* a cached token without a KV page */ };
// Any of these makes the step (and every later step until the host clears the
// word) leave the KV cache and the device lengths untouched.
constexpr uint32_t STATUS_STATE_ERRORS = STATUS_POSITION | STATUS_CAPACITY | STATUS_TIMEOUT | STATUS_TOKEN | STATUS_PAGE;


}  // namespace zdec
