// attention.cu -- per-sequence KV read: split-K flash-decode over a paged
// cache whose K and V each hold fp16, Q8_0 or FP8 (e4m3), dequantized inside
// the kernel, plus the KV append and read-back paths.
//
// Each sequence reads its own cache every step; nothing here is shared across
// the batch ("Batched swarm: the KV read does not amortize", "The two halves
// of a decode-step memory bill").  A quantized cache only saves bytes if the
// attention kernel reads the compressed format and dequantizes on chip ("Q8
// KV cache pushes an RDNA4 swarm crossover...", "Why Q8 is close to free and
// where the sharp edges are"); K and V choose their formats independently, and
// FP8 is the scale-free one-byte format ("Batched swarm...", "What a
// long-running swarm should actually tune").
//
// Work split.  Grid (cluster rank, kv head, segment slot); 128 threads; the
// CS CTAs of one (segment, kv head) form a thread-block cluster.  The batch's
// rows are cut into segments of at most S 64-token chunks, S the smallest
// that gives every row ceil(chunks / S) segments within the launch's segment
// slots, so a long row takes several clusters and a short one few ("Where it
// stops, and the argument I got wrong in May": agents hold 800 to 30,000
// tokens).  Within a segment the ranks take contiguous chunk ranges (the rank
// holding the new token one chunk fewer).  A chunk is one page's (layer, kv
// head) region: one bulk copy (TMA) per tensor lands it in a ring of
// shared-memory stages exactly as stored.
//
// Arithmetic (4 warps, 16 tokens each per chunk; the 4 query heads of the kv
// head share every K/V tile): scores and P V run on mma.sync.m16n8k16 with
// fp32 accumulation, the chunk's tokens as M and the 4 heads as N (column n:
// head n >> 1, fp16 part n & 1 of q or p split into hi + lo, ~22 bits).  Q8_0
// codes become exact fp16 integers in registers (byte_perm under exponent
// 1024, minus 1152) with K scales applied to 32-dim partial scores and V
// scales folded into p per 32-dim block; FP8 codes convert exactly with the
// hardware's e4m3x2 -> f16x2 cvt.  Softmax in log2 units (q carries
// log2(e)/sqrt(128)).  The warps run through the chunks without a block
// barrier; the last warp done with a ring slot refills it.
//
// Merge: warps -> CTA (shared memory), ranks -> rank 0 (each peer stores its
// partial into rank 0's shared memory with st.async, counted on rank 0's
// mbarrier; merged in fixed rank order), segments -> the last segment to
// finish (global partials and a ticket per (row, kv head), merged in segment
// order), so the result never depends on timing.

#include "kv_pool.cuh"
#include "zdec_kernels.cuh"


namespace zdec {

constexpr uint32_t AFULL = 0xFFFFFFFFu;
constexpr int ATT_MAX_STAGES = 8;
constexpr int SEG_PART = 4 * (HD + 4);          // floats of one segment's partial per kv head
constexpr long long ATT_WAIT_LIMIT = 1LL << 32;   // clock cycles (~2 s): a copy that never lands
constexpr int ATT_PAGE_CACHE = 64;              // block-table entries a CTA stages in shared memory
constexpr int ATT_MAX_CS = 16;                  // CTAs of a cluster (one segment of a row)
constexpr uint32_t ATT_PEER_BYTES = 128 * 16 + GROUP * 8;   // one peer's partial as pushed to rank 0

__host__ __device__ constexpr uint32_t att_stage_bytes(int kt, int vt) { return kv_region_bytes(kt) + kv_region_bytes(vt); }
static int att_max_stages(int kt, int vt) {
    // 227 KB of dynamic shared memory per CTA, less the static arrays (< 2 KB)
    // and a 16-CTA cluster's receive area
    const uint32_t budget = 227u * 1024u - 2048u - (uint32_t)(ATT_MAX_CS - 1) * GROUP * (HD + 4) * 4u;
    const int n = (int)(budget / att_stage_bytes(kt, vt));
    return n < ATT_MAX_STAGES ? n : ATT_MAX_STAGES;
}
int attention_default_stages(int kt, int vt) { return att_max_stages(kt, vt) < 3 ? att_max_stages(kt, vt) : 3; }
// Shared memory of a CTA: the chunk ring (reused by the warp merge after the
// loop), then rank 0's area for its cs - 1 peers' partials, which is never
// aliased, so a peer may push as soon as its own loop is done.
__host__ __device__ __forceinline__ uint32_t att_recv_off(int kt, int vt, int ns) {
    const uint32_t stages = (uint32_t)ns * att_stage_bytes(kt, vt);
    const uint32_t merge = (4 * 4 * 2 + 4 * 4 * (HD + 4)) * (uint32_t)sizeof(float);   // the CTA's warp merge
    return ((stages > merge ? stages : merge) + 15u) & ~15u;
}
size_t attention_smem_bytes(int kt, int vt, int ns, int cs) {
    if (ns < 2 || ns > att_max_stages(kt, vt)) ns = attention_default_stages(kt, vt);
    cs = std::max(1, std::min(ATT_MAX_CS, cs));
    return att_recv_off(kt, vt, ns) + (size_t)(cs - 1) * GROUP * (HD + 4) * sizeof(float);
}

__device__ __forceinline__ void mbar_arrive_local(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool att_wait(uint64_t *bar, uint32_t parity, long long limit) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > limit) return false;
    return true;
}
// Q8_0 codes (stored + 128) of four consecutive elements -> two exact fp16 pairs.
__device__ __forceinline__ void q8x4_to_h2(uint32_t w, uint32_t &lo, uint32_t &hi) {
    const __half2 bias = __float2half2_rn(1152.0f);
    lo = h2_as_u32(__hsub2(u32_as_h2(__byte_perm(w, 0x64646464u, 0x4140)), bias));
    hi = h2_as_u32(__hsub2(u32_as_h2(__byte_perm(w, 0x64646464u, 0x4342)), bias));
}
// The chunk's tokens are the mma's M dimension and the group's 4 query heads
// its N: column n of a B operand or an accumulator is head n >> 1, fp16 part
// n & 1 (the query is carried as hi + lo parts, ~22 bits).  A warp takes 16
// tokens of a chunk, 16 w .. 16 w + 15.  Along the mma's k index, the lane
// positions 2 tig + {0, 1, 8, 9} stand for four adjacent dims (scores) or
// tokens (output), 4 tig + {0, 1, 2, 3}, on both operands alike, so that
// every lane reads four adjacent elements of a K row or a V^T row.

// Scores S^T = K q^T of this warp's 16 tokens: returns the scores of head tig
// for tokens ta = 16 w + gid and tb = ta + 8 (hi and lo parts summed).
template <int KT>
__device__ __forceinline__ void qk_tile(const uint8_t *sK, int warp, int gid, int tig, const uint32_t (&qb)[8][2],
                                        float &sa, float &sb) {
    const int ta = 16 * warp + gid, tb = ta + 8;
    float c[4];
    if (KT == KV_T_Q8) {
        const uint2 sca = *reinterpret_cast<const uint2 *>(sK + ks_off(ta, 0));   // 4 block scales
        const uint2 scb = *reinterpret_cast<const uint2 *>(sK + ks_off(tb, 0));
        const float2 a01 = __half22float2(u32_as_h2(sca.x)), a23 = __half22float2(u32_as_h2(sca.y));
        const float2 b01 = __half22float2(u32_as_h2(scb.x)), b23 = __half22float2(u32_as_h2(scb.y));
        const float ka[4] = {a01.x, a01.y, a23.x, a23.y}, kb[4] = {b01.x, b01.y, b23.x, b23.y};
        const float zero4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int i = 0; i < 4; i++) c[i] = 0.0f;
#pragma unroll
        for (int bl = 0; bl < 4; bl++) {   // one 32-dim block: two k steps, then its scales
            float tmp[4];
#pragma unroll
            for (int hs = 0; hs < 2; hs++) {
                const int s8 = 2 * bl + hs;
                const uint32_t wa = *reinterpret_cast<const uint32_t *>(sK + k8_off(ta, 16 * s8 + 4 * tig));
                const uint32_t wb = *reinterpret_cast<const uint32_t *>(sK + k8_off(tb, 16 * s8 + 4 * tig));
                uint32_t a[4];
                q8x4_to_h2(wa, a[0], a[2]);
                q8x4_to_h2(wb, a[1], a[3]);
                if (hs) mma16816(tmp, a, qb[s8][0], qb[s8][1], tmp);
                else mma16816(tmp, a, qb[s8][0], qb[s8][1], zero4);
            }
            c[0] += ka[bl] * tmp[0];
            c[1] += ka[bl] * tmp[1];
            c[2] += kb[bl] * tmp[2];
            c[3] += kb[bl] * tmp[3];
        }
    } else {
        // two independent accumulator chains (even / odd k steps)
        float ce[4] = {0.0f, 0.0f, 0.0f, 0.0f}, co[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int s8 = 0; s8 < 8; s8++) {
            uint32_t a[4];
            if (KT == KV_T_F16) {
                const uint2 va = *reinterpret_cast<const uint2 *>(sK + k16_off(ta, 16 * s8 + 4 * tig));
                const uint2 vb = *reinterpret_cast<const uint2 *>(sK + k16_off(tb, 16 * s8 + 4 * tig));
                a[0] = va.x; a[2] = va.y;
                a[1] = vb.x; a[3] = vb.y;
            } else {
                const uint32_t wa = *reinterpret_cast<const uint32_t *>(sK + k8_off(ta, 16 * s8 + 4 * tig));
                const uint32_t wb = *reinterpret_cast<const uint32_t *>(sK + k8_off(tb, 16 * s8 + 4 * tig));
                a[0] = e4m3x2_to_h2((uint16_t)(wa & 0xFFFFu)); a[2] = e4m3x2_to_h2((uint16_t)(wa >> 16));
                a[1] = e4m3x2_to_h2((uint16_t)(wb & 0xFFFFu)); a[3] = e4m3x2_to_h2((uint16_t)(wb >> 16));
            }
            if (s8 & 1) mma16816(co, a, qb[s8][0], qb[s8][1], co);
            else mma16816(ce, a, qb[s8][0], qb[s8][1], ce);
        }
#pragma unroll
        for (int i = 0; i < 4; i++) c[i] = ce[i] + co[i];
    }
    sa = c[0] + c[1];
    sb = c[2] + c[3];
}

// fp16 part `lo` (0: hi = fp16(x), 1: lo = fp16(x - hi)) of two values, packed.
__device__ __forceinline__ uint32_t part2(float x0, float x1, bool lo) {
    const __half2 h = __floats2half2_rn(x0, x1);
    const float2 f = __half22float2(h);
    const __half2 l = __floats2half2_rn(x0 - f.x, x1 - f.y);
    return h2_as_u32(lo ? l : h);
}

// out^T += V^T P^T for this warp's 16 tokens.  pa, pb: this lane's
// probabilities of head tig for tokens 16 w + gid and + 8.  Accumulator mt
// holds dims 16 mt + gid (c0, c1) and + 8 (c2, c3), columns head tig hi, lo.
template <int VT>
__device__ __forceinline__ void pv_tile(const uint8_t *sV, int warp, int gid, int tig, float pa, float pb,
                                        float (&oacc)[8][4]) {
    // the P^T operand: lane (gid, tig) carries head gid >> 1, part gid & 1, of
    // tokens 4 tig + e (e = 0..3) of the warp's 16; token j of head h is in
    // lane (j & 7, h), as its first score for j < 8 and its second above
    const int h = gid >> 1;
    const bool lo = gid & 1;
    float pv[4];
#pragma unroll
    for (int e = 0; e < 4; e++) {
        const int src = ((4 * (tig & 1) + e) << 2) | h;
        const float x = __shfl_sync(AFULL, pa, src), y = __shfl_sync(AFULL, pb, src);
        pv[e] = tig < 2 ? x : y;
    }
    const int t0 = 16 * warp + 4 * tig;   // the lane's four tokens along k
    if (VT == KV_T_Q8) {
        // V's block scales (per token and 32 dims) go into the P^T operand
#pragma unroll
        for (int bl = 0; bl < 4; bl++) {
            const uint2 s4 = *reinterpret_cast<const uint2 *>(sV + vs_off(t0, bl));   // tokens t0..t0+3
            const float2 s01 = __half22float2(u32_as_h2(s4.x)), s23 = __half22float2(u32_as_h2(s4.y));
            const uint32_t b0 = part2(pv[0] * s01.x, pv[1] * s01.y, lo);
            const uint32_t b1 = part2(pv[2] * s23.x, pv[3] * s23.y, lo);
#pragma unroll
            for (int mh = 0; mh < 2; mh++) {
                const int mt = 2 * bl + mh, da = 16 * mt + gid;
                const uint32_t wa = *reinterpret_cast<const uint32_t *>(sV + v8_off(t0, da));
                const uint32_t wb = *reinterpret_cast<const uint32_t *>(sV + v8_off(t0, da + 8));
                uint32_t a[4];
                q8x4_to_h2(wa, a[0], a[2]);
                q8x4_to_h2(wb, a[1], a[3]);
                mma16816(oacc[mt], a, b0, b1, oacc[mt]);
            }
        }
    } else {
        const uint32_t b0 = part2(pv[0], pv[1], lo), b1 = part2(pv[2], pv[3], lo);
#pragma unroll
        for (int mt = 0; mt < 8; mt++) {
            const int da = 16 * mt + gid;
            uint32_t a[4];
            if (VT == KV_T_F16) {
                const uint2 va = *reinterpret_cast<const uint2 *>(sV + v16_off(t0, da));
                const uint2 vb = *reinterpret_cast<const uint2 *>(sV + v16_off(t0, da + 8));
                a[0] = va.x; a[2] = va.y;
                a[1] = vb.x; a[3] = vb.y;
            } else {
                const uint32_t wa = *reinterpret_cast<const uint32_t *>(sV + v8_off(t0, da));
                const uint32_t wb = *reinterpret_cast<const uint32_t *>(sV + v8_off(t0, da + 8));
                a[0] = e4m3x2_to_h2((uint16_t)(wa & 0xFFFFu)); a[2] = e4m3x2_to_h2((uint16_t)(wa >> 16));
                a[1] = e4m3x2_to_h2((uint16_t)(wb & 0xFFFFu)); a[3] = e4m3x2_to_h2((uint16_t)(wb >> 16));
            }
            mma16816(oacc[mt], a, b0, b1, oacc[mt]);
        }
    }
}

// Store one element d of a row at token t of a K or V region, `x` in storage
// form (fp16 bits, Q8_0 code + 128, or an e4m3 byte).
template <int T>
__device__ __forceinline__ void put_k(uint8_t *reg, int t, int d, uint16_t x) {
    if (T == KV_T_F16) *reinterpret_cast<uint16_t *>(reg + k16_off(t, d)) = x;
    else reg[k8_off(t, d)] = (uint8_t)x;
}
template <int T>
__device__ __forceinline__ void put_v(uint8_t *reg, int t, int d, uint16_t x) {
    if (T == KV_T_F16) *reinterpret_cast<uint16_t *>(reg + v16_off(t, d)) = x;
    else reg[v8_off(t, d)] = (uint8_t)x;
}
// One element of a row of fp16 values held by the 32 lanes of a warp (dims
// lane + 32 i) in storage form; a Q8_0 block's scale comes from the whole
// warp (every lane must call this together).
template <int T>
__device__ __forceinline__ uint16_t encode_lane(__half h, uint16_t &scale_bits) {
    if (T == KV_T_F16) return __half_as_ushort(h);
    if (T == KV_T_Q8) return (uint16_t)(uint8_t)(q8_0_lane(h, scale_bits) ^ 0x80);
    return e4m3_from_half(h);
}

// ------------------------------------------------------------------ kernel ---
template <int KT, int VT>
__global__ __launch_bounds__(128, 3) void attention_kernel(const AttnParams p) {
    constexpr uint32_t KB = kv_region_bytes(KT), VB = kv_region_bytes(VT), SB = KB + VB;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ uint16_t s_newk[HD], s_newv[HD];          // the new token in storage form
    __shared__ uint16_t s_newks[4], s_newvs[4];
    __shared__ __align__(8) uint64_t full[ATT_MAX_STAGES];
    __shared__ __align__(8) uint64_t merge_bar;           // rank 0: the peers' partials have landed
    __shared__ int s_map[4];                             // row, segment, segments of the row, chunks per segment
    __shared__ int s_bad, s_last;
    __shared__ int s_done[ATT_MAX_STAGES];               // warps done with the chunk in each ring slot
    __shared__ int s_issued;                             // chunks whose copies have been issued
    __shared__ int s_pages[ATT_PAGE_CACHE];              // pages of this CTA's first chunks

    const int rank = blockIdx.x, g = blockIdx.y, z = blockIdx.z, CS = p.cs;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
    tl_min(p.tl, 0);
    // ---- which row and segment this cluster takes.  Positions, slots and
    // block tables are step inputs written before the step's first kernel,
    // so this runs before the dependency wait.  One segment slot per row
    // (gridDim.z == B) needs no search: row z, whole.
    if (gridDim.z == (unsigned)p.B) {
        if (threadIdx.x == 0) {
            const int pos = p.positions[z];
            const bool valid = pos >= 0 && pos < p.max_L;
            s_map[0] = valid ? z : -1;
            s_map[1] = 0;
            s_map[2] = 1;
            s_map[3] = valid ? (pos + PAGE_TOKENS) / PAGE_TOKENS : 1;
            s_bad = 0;
        }
    } else if (warp == 0) {
        int nch = 0;
        if (lane < p.B) {
            const int pos = p.positions[lane];
            nch = (pos >= 0 && pos < p.max_L) ? (pos + PAGE_TOKENS) / PAGE_TOKENS : 0;
        }
        int tot = nch, mx = nch;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            tot += __shfl_xor_sync(AFULL, tot, o);
            mx = max(mx, __shfl_xor_sync(AFULL, mx, o));
        }
        const int NZ = (int)gridDim.z;
        int lo = max(1, (tot + NZ - 1) / NZ), hi = max(1, mx);
        lo = min(hi, max(lo, p.seg_min));
        while (lo < hi) {   // the smallest S whose segment count fits the launch
            const int mid = (lo + hi) >> 1;
            int cnt = nch ? (nch + mid - 1) / mid : 0;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(AFULL, cnt, o);
            if (cnt <= NZ) hi = mid;
            else lo = mid + 1;
        }
        const int S = lo;
        const int segs = nch ? (nch + S - 1) / S : 0;
        int incl = segs;   // inclusive prefix sum over the rows
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(AFULL, incl, o);
            if (lane >= o) incl += v;
        }
        const unsigned hit = __ballot_sync(AFULL, lane < p.B && incl > z);
        if (lane == 0) {
            s_map[0] = -1;
            s_bad = 0;
        }
        __syncwarp();
        if (hit) {
            const int r = __ffs(hit) - 1;
            if (lane == r) {
                s_map[0] = r;
                s_map[1] = z - (incl - segs);
                s_map[2] = segs;
                s_map[3] = S;
            }
        }
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < p.stages; i++) {
            mbar_init(&full[i], 1);
            s_done[i] = 0;
        }
        mbar_init(&merge_bar, 1);
        // rank 0 expects its peers' partials: per peer 128 threads x 16 B of
        // output and 4 heads x 8 B of (max, sum), stored asynchronously
        if (rank == 0 && CS > 1) mbar_expect_tx(&merge_bar, (uint32_t)(CS - 1) * ATT_PEER_BYTES);
        mbar_fence_init();
    }
    __syncthreads();
    // publishes rank 0's merge barrier to the peers (waited on before they push)
    if (CS > 1) cluster_arrive_relaxed();
    const int b = s_map[0];
    if (b < 0) {   // an idle segment slot: every CTA of the cluster leaves here
        pdl_launch_dependents();
        return;
    }
    const int seg = s_map[1], nseg = s_map[2], S = s_map[3];
    const int pos = p.positions[b];
    const int slot = p.slots[b];
    const int ntok = pos + 1;
    const int nch = (ntok + PAGE_TOKENS - 1) / PAGE_TOKENS;
    const int sc0 = seg * S, nseg_ch = min(nch, sc0 + S) - sc0;   // this segment's chunks
    const bool seg_new = p.append && sc0 + nseg_ch == nch;         // it holds the new token
    const int nw = nseg_ch + (seg_new ? 1 : 0);   // the appending rank counts one chunk more
    const int c_lo = sc0 + min(nseg_ch, rank * nw / CS), c_hi = sc0 + min(nseg_ch, (rank + 1) * nw / CS);
    const int T1 = min(c_hi * PAGE_TOKENS, ntok);
    const bool empty = c_lo >= c_hi;          // still takes part in the cluster merge
    const int H = p.append ? min(T1, pos) : T1;   // tokens read from the cache
    const int nchunks = c_hi - c_lo;
    const bool has_new = p.append && !empty && T1 == ntok;
    const int NS = p.stages;
    const size_t coff = kv_chunk_off(p.kv, p.layer, g);
    auto stage = [&](int i) { return smem + (size_t)(i % NS) * SB; };
    // the block-table entries of this CTA's chunks, loaded in parallel
    for (int t = threadIdx.x; t < nchunks && t < ATT_PAGE_CACHE; t += blockDim.x)
        s_pages[t] = kv_page(p.kv, slot, (c_lo + t) * PAGE_TOKENS);
    __syncthreads();
    // chunk i of this CTA's range into ring slot i % NS; a chunk with no
    // cached token (only the new one) or without a page completes its stage
    // with no copy
    auto issue = [&](int i) {
        const int c = c_lo + i;
        uint64_t *bar = &full[i % NS];
        const int page = i < ATT_PAGE_CACHE ? s_pages[i] : kv_page(p.kv, slot, c * PAGE_TOKENS);
        if (c * PAGE_TOKENS < H && kv_page_ok(p.kv, page)) {
            const uint8_t *src = p.kv.base + (size_t)page * p.kv.page_bytes + coff;
            mbar_expect_tx(bar, SB);
            bulk_g2s(stage(i), src, KB, bar);
            bulk_g2s(stage(i) + KB, src + KB, VB, bar);
        } else {
            if (c * PAGE_TOKENS < H) atomicOr(p.status, STATUS_PAGE);
            mbar_arrive_local(bar);
        }
    };
    // the cached history does not depend on the previous kernel: the first
    // NS chunks (the whole ring) go out before the dependency wait, one
    // issuing thread each
    if ((int)threadIdx.x < NS && (int)threadIdx.x < nchunks) issue(threadIdx.x);
    // read only after the loop; the later writes come from the warp that
    // releases a slot last, after every warp (thread 0's included) is past it
    if (threadIdx.x == 0) s_issued = min(NS, nchunks);

    // the rotary row of the new token: a constant table, read before the wait
    float2 rope_new[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
    if (has_new && warp == 0) {
        const float2 *cs = p.rope + (size_t)pos * (HD / 2);
        rope_new[0] = cs[lane];
        rope_new[1] = cs[lane + 32];
    }

    pdl_launch_dependents();
    pdl_wait();
    tl_min(p.tl, 1);
    tl_max(p.tl, 4);

    // ---- the query as the scores' B operand: lane (gid, tig) carries head
    // 4 g + (gid >> 1), fp16 part gid & 1, of dims 16 s + 4 tig + {0..3}
    uint32_t qb[8][2];
    const bool qlo = gid & 1;
    if (p.q_frag) {   // prepared by the QKV projection's epilogue (rotated, scaled, hi/lo)
        const uint4 *qf = p.q_frag + ((size_t)b * p.nq + GROUP * g + (gid >> 1)) * 32 + tig;
#pragma unroll
        for (int st = 0; st < 8; st++) {
            const uint4 f = qf[st * 4];   // hi(d0, d1), lo(d0, d1), hi(d2, d3), lo(d2, d3)
            qb[st][0] = qlo ? f.y : f.x;
            qb[st][1] = qlo ? f.w : f.z;
        }
    } else {
        const float qscale = 0.12751743082459868f;   // log2(e)/sqrt(128): scores in log2 units
        const int hq = GROUP * g + (gid >> 1);
        const float *qrow = p.qkv + (size_t)b * p.qkv_ld + (size_t)hq * HD;
        const float2 *cs = p.rope + (size_t)pos * (HD / 2);
#pragma unroll
        for (int st = 0; st < 8; st++) {
            float v[4];
#pragma unroll
            for (int e = 0; e < 4; e++) {
                const int d = 16 * st + 4 * tig + e;
                float x = qrow[d];
                if (p.append) {
                    const float2 c = cs[d & 63];
                    x = d < 64 ? x * c.x - qrow[d + 64] * c.y : x * c.x + qrow[d - 64] * c.y;
                }
                v[e] = x * qscale;
            }
            qb[st][0] = part2(v[0], v[1], qlo);
            qb[st][1] = part2(v[2], v[3], qlo);
        }
    }

    // ---- the new token (warp 0 of the CTA that holds it): its k and v rows
    // are loaded now, and rotated, rounded and encoded at the chunk that holds
    // it, so that the load latency hides behind the earlier chunks
    float kx[4], vx[4];
    if (has_new && warp == 0) {
        const float *krow = p.qkv + (size_t)b * p.qkv_ld + (size_t)(p.nq + g) * HD;
        const float *vrow = p.qkv + (size_t)b * p.qkv_ld + (size_t)(p.nq + p.kv.n_kv + g) * HD;
#pragma unroll
        for (int i = 0; i < 4; i++) { kx[i] = krow[lane + 32 * i]; vx[i] = vrow[lane + 32 * i]; }
    }
    auto encode_new = [&]() {   // warp 0: rotate-half pairs (d, d + 64), d = lane + 32 i
        float kr[4];
#pragma unroll
        for (int i = 0; i < 2; i++) {
            const float2 c = rope_new[i];
            kr[i] = kx[i] * c.x - kx[i + 2] * c.y;
            kr[i + 2] = kx[i + 2] * c.x + kx[i] * c.y;
        }
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const int d = lane + 32 * i;
            uint16_t ksb = 0, vsb = 0;
            s_newk[d] = encode_lane<KT>(__float2half_rn(kr[i]), ksb);
            s_newv[d] = encode_lane<VT>(__float2half_rn(vx[i]), vsb);
            if (lane == 0) {
                s_newks[i] = ksb;
                s_newvs[i] = vsb;
            }
        }
    };

    // ---- online softmax state of head 4 g + tig (l_run: this lane's tokens)
    float m_run = -INFINITY, l_run = 0.0f;
    float oacc[8][4];
#pragma unroll
    for (int mt = 0; mt < 8; mt++)
#pragma unroll
        for (int i = 0; i < 4; i++) oacc[mt][i] = 0.0f;
    bool ok = true;

    // Each warp runs through the chunks on its own: no block barrier per
    // chunk.  The last of the 4 warps done with a ring slot refills it with
    // the chunk NS further on (a warp's loads of the slot are complete once
    // their values have entered its MMAs; __syncwarp orders the lanes' loads
    // before lane 0's release).  Only the chunks at the end of the history,
    // which every thread edits first, take block barriers.
    for (int ci = 0; ci < nchunks; ci++) {
        const int c0 = (c_lo + ci) * PAGE_TOKENS;
        const int zfrom = max(H, c0) - c0;   // first local token not read from the cache
        const bool fixup = zfrom < PAGE_TOKENS;   // the same on every warp
        if (fixup) {
            if (has_new && warp == 0) encode_new();
            __syncthreads();   // the new token's codes, for every thread
        }
        if (ok && !att_wait(&full[ci % NS], (uint32_t)(ci / NS) & 1u, ATT_WAIT_LIMIT)) {
            ok = false;
            s_bad = 1;
            atomicOr(p.status, STATUS_TIMEOUT);
        }
        uint8_t *sK = stage(ci), *sV = stage(ci) + KB;
        if (fixup) {
            // the chunk holding the end of the history: clear what lies past
            // it (stale values of the page's earlier use may be Inf or NaN, and
            // 0 * NaN would reach the output) and insert the new token
            const int d = threadIdx.x;   // 128 threads, one head dim each
            for (int t = zfrom; t < PAGE_TOKENS; t++) put_v<VT>(sV, t, d, VT == KV_T_Q8 ? 0x80 : 0);
            if (VT == KV_T_Q8 && d < 4)
                for (int t = zfrom; t < PAGE_TOKENS; t++) *reinterpret_cast<uint16_t *>(sV + vs_off(t, d)) = 0;
            if (has_new && pos >= c0 && pos < c0 + PAGE_TOKENS) {
                const int t = pos - c0;
                put_k<KT>(sK, t, d, s_newk[d]);
                put_v<VT>(sV, t, d, s_newv[d]);
                if (KT == KV_T_Q8 && d < 4) *reinterpret_cast<uint16_t *>(sK + ks_off(t, d)) = s_newks[d];
                if (VT == KV_T_Q8 && d < 4) *reinterpret_cast<uint16_t *>(sV + vs_off(t, d)) = s_newvs[d];
            }
            __syncthreads();
        }
        const int tw = c0 + 16 * warp;   // this warp's 16 tokens
        if (ok && tw < T1) {
            float sa, sb;   // head tig, tokens tw + gid and tw + gid + 8
            qk_tile<KT>(sK, warp, gid, tig, qb, sa, sb);
            if (tw + gid >= T1) sa = -INFINITY;   // the range's last tile may end early
            if (tw + gid + 8 >= T1) sb = -INFINITY;
            float mt = fmaxf(sa, sb);
            mt = fmaxf(mt, __shfl_xor_sync(AFULL, mt, 4));
            mt = fmaxf(mt, __shfl_xor_sync(AFULL, mt, 8));
            mt = fmaxf(mt, __shfl_xor_sync(AFULL, mt, 16));
            // the output is rescaled only when some head's running max grew
            // (alpha = 1 exactly otherwise), which after the first tiles is rare
            const float m_new = fmaxf(m_run, mt);
            const bool grow = m_new > m_run;
            const float alpha = grow ? exp2f(m_run - m_new) : 1.0f;   // m_run = -inf -> 0
            float pa = 0.0f, pb = 0.0f;
            if (m_new != -INFINITY) {
                pa = exp2f(sa - m_new);
                pb = exp2f(sb - m_new);
            }
            m_run = m_new;
            l_run = l_run * alpha + (pa + pb);
            if (__any_sync(AFULL, grow))
#pragma unroll
                for (int m = 0; m < 8; m++)
#pragma unroll
                    for (int i = 0; i < 4; i++) oacc[m][i] *= alpha;
            pv_tile<VT>(sV, warp, gid, tig, pa, pb, oacc);
        }
        // this warp is done with slot ci % NS
        __syncwarp();
        if (lane == 0) {
            const int slot = ci % NS;
            __threadfence_block();
            if (atomicAdd(&s_done[slot], 1) == 3) {   // the last of the 4 warps
                s_done[slot] = 0;
                if (ci + NS < nchunks && !s_bad) {
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // the reads before the copy's writes
                    issue(ci + NS);
                    s_issued = ci + NS + 1;
                }
            }
        }
    }
    tl_max(p.tl, 6);
    __syncthreads();
    if (s_bad && threadIdx.x == 0)   // copies still in flight land before the ring is reused
        for (int i = max(0, s_issued - NS); i < s_issued; i++)
            att_wait(&full[i % NS], (uint32_t)(i / NS) & 1u, ATT_WAIT_LIMIT);

    // ---- merge the 4 warps of this CTA (shared memory reused after the stages)
    float *wm = reinterpret_cast<float *>(smem);   // [4 warps][4 heads]
    float *wl = wm + 16;
    float *wo = wl + 16;                            // [4][4][HD + 4] (padded: no bank conflicts)
    float l_tot = l_run;   // over the warp's tokens: the lanes of head tig
    l_tot += __shfl_xor_sync(AFULL, l_tot, 4);
    l_tot += __shfl_xor_sync(AFULL, l_tot, 8);
    l_tot += __shfl_xor_sync(AFULL, l_tot, 16);
    __syncthreads();
    if (gid == 0) { wm[warp * 4 + tig] = m_run; wl[warp * 4 + tig] = l_tot; }
#pragma unroll
    for (int m = 0; m < 8; m++) {
        wo[(warp * 4 + tig) * (HD + 4) + 16 * m + gid] = oacc[m][0] + oacc[m][1];
        wo[(warp * 4 + tig) * (HD + 4) + 16 * m + gid + 8] = oacc[m][2] + oacc[m][3];
    }
    __syncthreads();
    const int head = threadIdx.x >> 5, d0 = (threadIdx.x & 31) * 4;
    float cta_m, cta_l, cta_o[4];   // this CTA's (max, sum, output) of head `head`, dims d0..d0+3
    {
        float M = -INFINITY;
        for (int w = 0; w < 4; w++) M = fmaxf(M, wm[w * 4 + head]);
        float L = 0.0f, O[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        for (int w = 0; w < 4; w++) {
            const float mw = wm[w * 4 + head];
            const float f = mw == -INFINITY ? 0.0f : exp2f(mw - M);
            L += f * wl[w * 4 + head];
            for (int e = 0; e < 4; e++) O[e] += f * wo[(w * 4 + head) * (HD + 4) + d0 + e];
        }
        cta_m = M;
        cta_l = L;
#pragma unroll
        for (int e = 0; e < 4; e++) cta_o[e] = O[e];
    }
    // ---- the cluster's partials meet in rank 0's shared memory: each peer
    // stores its (max, sum, output) per head into rank 0's receive area as
    // soon as its own loop is done, and arrives on rank 0's merge barrier
    if (CS > 1) cluster_wait_acquire();   // every CTA has initialised its barriers (long ago)
    float *recv = reinterpret_cast<float *>(smem + att_recv_off(KT, VT, NS));   // [peer rank - 1][head][HD + 4]
    if (rank != 0) {
        const uint32_t dst = map_to_rank(smem_u32(recv + ((rank - 1) * GROUP + head) * (HD + 4)), 0);
        const uint32_t rbar = map_to_rank(smem_u32(&merge_bar), 0);
        if ((threadIdx.x & 31) == 0) st_async_v2(dst, cta_m, cta_l, rbar);
        st_async_v4(dst + (uint32_t)(4 + d0) * 4u, make_float4(cta_o[0], cta_o[1], cta_o[2], cta_o[3]), rbar);
    } else {
        bool landed = CS == 1 || mbar_try_wait_cluster(&merge_bar, 0);
        if (!landed) {
            const long long t0 = clock64();
            while (!(landed = mbar_try_wait_cluster(&merge_bar, 0)))
                if (clock64() - t0 > ATT_WAIT_LIMIT) break;
            if (!landed && threadIdx.x == 0) atomicOr(p.status, STATUS_TIMEOUT);
        }
        tl_max(p.tl, 5);
        // in rank order, two passes over the partials in shared memory
        const int nrecv = landed ? CS - 1 : 0;
        float M = cta_m;
        for (int r = 0; r < nrecv; r++) M = fmaxf(M, recv[(r * GROUP + head) * (HD + 4)]);
        const float f0 = cta_m == -INFINITY ? 0.0f : exp2f(cta_m - M);
        float L = f0 * cta_l, O[4];
#pragma unroll
        for (int e = 0; e < 4; e++) O[e] = f0 * cta_o[e];
        for (int r = 0; r < nrecv; r++) {
            const float *ps = recv + (r * GROUP + head) * (HD + 4);
            const float mr = ps[0];
            const float f = mr == -INFINITY ? 0.0f : exp2f(mr - M);
            L += f * ps[1];
            const float4 o4 = *reinterpret_cast<const float4 *>(ps + 4 + d0);
            O[0] += f * o4.x; O[1] += f * o4.y; O[2] += f * o4.z; O[3] += f * o4.w;
        }
        bool finish = nseg == 1;
        if (!finish) {
            // several segments: this one's partial goes to global memory; the
            // last segment of the (row, kv head) to arrive merges them all, in
            // segment order
            float *mine = p.seg_part + ((size_t)z * p.kv.n_kv + g) * SEG_PART + head * (HD + 4);
            if ((threadIdx.x & 31) == 0) { mine[0] = M; mine[1] = L; }
            *reinterpret_cast<float4 *>(mine + 4 + d0) = make_float4(O[0], O[1], O[2], O[3]);
            __threadfence();
            __syncthreads();
            if (threadIdx.x == 0) {
                int *ticket = p.seg_ticket + b * p.kv.n_kv + g;
                s_last = atomicAdd(ticket, 1) == nseg - 1;
                if (s_last) *ticket = 0;   // every segment has arrived: ready for the next launch
                __threadfence();
            }
            __syncthreads();
            finish = s_last != 0;
            if (finish) {
                const int z0 = z - seg;
                M = -INFINITY;
                for (int s = 0; s < nseg; s++)
                    M = fmaxf(M, __ldcg(p.seg_part + ((size_t)(z0 + s) * p.kv.n_kv + g) * SEG_PART + head * (HD + 4)));
                L = 0.0f;
                O[0] = O[1] = O[2] = O[3] = 0.0f;
                for (int s = 0; s < nseg; s++) {
                    const float *ps = p.seg_part + ((size_t)(z0 + s) * p.kv.n_kv + g) * SEG_PART + head * (HD + 4);
                    const float ms = __ldcg(ps);
                    const float f = ms == -INFINITY ? 0.0f : exp2f(ms - M);
                    L += f * __ldcg(ps + 1);
                    const float4 os = __ldcg(reinterpret_cast<const float4 *>(ps + 4 + d0));
                    O[0] += f * os.x; O[1] += f * os.y; O[2] += f * os.z; O[3] += f * os.w;
                }
            }
        }
        if (finish) {
            const float inv = 1.0f / L;
            const int qd = p.nq * HD;
            const int kcol = (GROUP * g + head) * HD + d0;   // column of o, the O projection's input
            float y[4];
            for (int e = 0; e < 4; e++) y[e] = O[e] * inv;
            if (p.o) {   // the fp32 output (read-back paths; the step reads only the planes)
                float *o = p.o + (size_t)b * qd + kcol;
                for (int e = 0; e < 4; e++) o[e] = y[e];
            }
            // the O projection's operand as fp16 hi + lo parts (elements 4..7 of
            // every 8 stored / 16) and the per-32 sub-block sums, as the GEMM
            // prep writes them
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
    }
    tl_max(p.tl, 7);
    // the appended token into its page, unless a device check flagged the step
    // (the status word is final by now: every kernel that sets it completed
    // before this kernel's dependency wait)
    if (has_new && warp == 0 && (*(volatile uint32_t *)p.status & STATUS_STATE_ERRORS) == 0) {
        const int page = kv_page(p.kv, slot, pos);
        if (kv_page_ok(p.kv, page)) {
            uint8_t *k = p.kv.base + (size_t)page * p.kv.page_bytes + coff, *v = k + KB;
            const int t = pos & (PAGE_TOKENS - 1);
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const int d = lane + 32 * i;
                put_k<KT>(k, t, d, s_newk[d]);
                put_v<VT>(v, t, d, s_newv[d]);
                if (lane == 0) {
                    if (KT == KV_T_Q8) *reinterpret_cast<uint16_t *>(k + ks_off(t, i)) = s_newks[i];
                    if (VT == KV_T_Q8) *reinterpret_cast<uint16_t *>(v + vs_off(t, i)) = s_newvs[i];
                }
            }
        }
    }
    tl_end(p.tl);
}

// ------------------------------------------------------------------ dispatch ---
template <int KT, int VT>
static cudaError_t set_attrs() {
    const int smem = (int)attention_smem_bytes(KT, VT, att_max_stages(KT, VT), ATT_MAX_CS);
    cudaError_t e = cudaFuncSetAttribute(attention_kernel<KT, VT>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(attention_kernel<KT, VT>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    return e;
}
template <int KT, int VT>
static int max_clusters(int stages, int cs, int nkv) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cs, nkv, 8);
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = attention_smem_bytes(KT, VT, stages, cs);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, attention_kernel<KT, VT>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}
template <int KT, int VT>
static cudaError_t launch_kt(const AttnParams &p, bool pdl, cudaStream_t s, int nz) {
    return launch_k(attention_kernel<KT, VT>, dim3(p.cs, p.kv.n_kv, nz), dim3(128),
                    attention_smem_bytes(KT, VT, p.stages, p.cs), pdl, p.cs, s, p);
}

// Evaluates CALL(KT, VT) for the runtime type pair (kt, vt) and returns it.
#define ZDEC_KV_DISPATCH(kt, vt, CALL)                                                   \
    switch ((kt) * 3 + (vt)) {                                                           \
        case 0: return CALL(0, 0); case 1: return CALL(0, 1); case 2: return CALL(0, 2); \
        case 3: return CALL(1, 0); case 4: return CALL(1, 1); case 5: return CALL(1, 2); \
        case 6: return CALL(2, 0); case 7: return CALL(2, 1); case 8: return CALL(2, 2); \
        default: break;                                                                  \
    }

cudaError_t attention_setup(int kt, int vt) {
#define ZDEC_SET(a, b) set_attrs<a, b>()
    ZDEC_KV_DISPATCH(kt, vt, ZDEC_SET)
#undef ZDEC_SET
    return cudaErrorInvalidValue;
}

int attention_max_clusters(int kt, int vt, int stages, int cs, int nkv) {
    if (cs < 1 || cs > 16 || kt < 0 || kt > 2 || vt < 0 || vt > 2 || stages < 2 || stages > att_max_stages(kt, vt))
        return 0;
#define ZDEC_MC(a, b) max_clusters<a, b>(stages, cs, nkv)
    ZDEC_KV_DISPATCH(kt, vt, ZDEC_MC)
#undef ZDEC_MC
    return 0;
}

int attention_stage_limit(int kt, int vt) { return att_max_stages(kt, vt); }

cudaError_t launch_attention(const AttnParams &p0, int nz, bool pdl, cudaStream_t stream) {
    AttnParams p = p0;
    const int kt = p.kv.k_type, vt = p.kv.v_type;
    if (p.cs < 1 || p.cs > 16 || kt < 0 || kt > 2 || vt < 0 || vt > 2 || p.B < 1 || p.B > MAX_B)
        return cudaErrorInvalidValue;
    if (nz < p.B || (nz > p.B && (!p.seg_part || !p.seg_ticket))) return cudaErrorInvalidValue;
    if (p.stages == 0) p.stages = attention_default_stages(kt, vt);
    if (p.stages < 2 || p.stages > att_max_stages(kt, vt)) return cudaErrorInvalidValue;
    if (p.seg_min < 1) p.seg_min = 1;
#define ZDEC_LA(a, b) launch_kt<a, b>(p, pdl, stream, nz)
    ZDEC_KV_DISPATCH(kt, vt, ZDEC_LA)
#undef ZDEC_LA
    return cudaErrorInvalidValue;
}

// ------------------------------------------------------------ bulk append ---
// One warp per (layer, token, kv head); lane holds dims lane + 32 i, i.e.
// element `lane` of Q8_0 block i.  Every page the tokens land in is already
// assigned to the slot (the host allocates pages before it enqueues this).
template <int KT, int VT>
__global__ void kv_append_kernel(const KvPool a, int slot, int t0, int n, const uint16_t *__restrict__ k16,
                                 const uint16_t *__restrict__ v16, uint32_t *status) {
    constexpr uint32_t KB = kv_region_bytes(KT);
    const long w = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (w >= (long)a.n_layers * n * a.n_kv) return;   // whole warps: the grid covers 32 lanes per item
    const int g = (int)(w % a.n_kv);
    const int t = (int)((w / a.n_kv) % n);
    const int l = (int)(w / ((long)a.n_kv * n));
    const uint16_t *ks = k16 + (((size_t)l * n + t) * a.n_kv + g) * HD;
    const uint16_t *vs = v16 + (((size_t)l * n + t) * a.n_kv + g) * HD;
    const int pos = t0 + t;
    const int page = kv_page(a, slot, pos);
    if (!kv_page_ok(a, page)) {
        if (lane == 0) atomicOr(status, STATUS_PAGE);
        return;
    }
    uint8_t *k = a.base + (size_t)page * a.page_bytes + kv_chunk_off(a, l, g), *v = k + KB;
    const int tl = pos & (PAGE_TOKENS - 1);
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const int d = lane + 32 * i;
        uint16_t ksb = 0, vsb = 0;
        const uint16_t kc = encode_lane<KT>(__ushort_as_half(ks[d]), ksb);
        const uint16_t vc = encode_lane<VT>(__ushort_as_half(vs[d]), vsb);
        put_k<KT>(k, tl, d, kc);
        put_v<VT>(v, tl, d, vc);
        if (lane == 0) {
            if (KT == KV_T_Q8) *reinterpret_cast<uint16_t *>(k + ks_off(tl, i)) = ksb;
            if (VT == KV_T_Q8) *reinterpret_cast<uint16_t *>(v + vs_off(tl, i)) = vsb;
        }
    }
}

template <int KT, int VT>
static cudaError_t append_kt(const KvPool &a, int slot, int t0, int n, const uint16_t *k16, const uint16_t *v16,
                             uint32_t *status, cudaStream_t stream) {
    const long warps = (long)a.n_layers * n * a.n_kv;
    kv_append_kernel<KT, VT><<<(unsigned)((warps * 32 + 255) / 256), 256, 0, stream>>>(a, slot, t0, n, k16, v16, status);
    return cudaGetLastError();
}

cudaError_t launch_kv_append(const KvPool &a, int slot, int t0, int n, const uint16_t *k16, const uint16_t *v16,
                             uint32_t *status, cudaStream_t stream) {
    if ((long)a.n_layers * n * a.n_kv == 0) return cudaSuccess;
#define ZDEC_AP(x, y) append_kt<x, y>(a, slot, t0, n, k16, v16, status, stream)
    ZDEC_KV_DISPATCH(a.k_type, a.v_type, ZDEC_AP)
#undef ZDEC_AP
    return cudaErrorInvalidValue;
}

// ------------------------------------------------------------------ read-back ---
// One thread per (token, kv head, dim) of one layer: canonical token-major
// rows; fp16 bits, Q8_0 codes (the stored offset removed) with their scales
// [n][n_kv][4], or e4m3 codes.  Tokens without a page read as zero.
__global__ void kv_read_kernel(const KvPool a, int slot, int layer, int t0, int n, uint8_t *k, uint8_t *v,
                               uint16_t *ks, uint16_t *vs) {
    const long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long)n * a.n_kv * HD) return;
    const int d = (int)(i % HD), g = (int)((i / HD) % a.n_kv), t = (int)(i / ((long)HD * a.n_kv));
    const int pos = t0 + t;
    const int page = kv_page(a, slot, pos);
    const bool ok = kv_page_ok(a, page);
    const uint8_t *kr = ok ? a.base + (size_t)page * a.page_bytes + kv_chunk_off(a, layer, g) : nullptr;
    const uint8_t *vr = ok ? kr + kv_region_bytes(a.k_type) : nullptr;
    const int tl = pos & (PAGE_TOKENS - 1);
    const size_t so = ((size_t)t * a.n_kv + g) * 4 + (d >> 5);
    if (a.k_type == KV_T_F16) reinterpret_cast<uint16_t *>(k)[i] = ok ? *reinterpret_cast<const uint16_t *>(kr + k16_off(tl, d)) : 0;
    else k[i] = ok ? (uint8_t)(kr[k8_off(tl, d)] ^ (a.k_type == KV_T_Q8 ? 0x80 : 0)) : 0;
    if (a.v_type == KV_T_F16) reinterpret_cast<uint16_t *>(v)[i] = ok ? *reinterpret_cast<const uint16_t *>(vr + v16_off(tl, d)) : 0;
    else v[i] = ok ? (uint8_t)(vr[v8_off(tl, d)] ^ (a.v_type == KV_T_Q8 ? 0x80 : 0)) : 0;
    if ((d & 31) == 0) {
        if (a.k_type == KV_T_Q8) ks[so] = ok ? *reinterpret_cast<const uint16_t *>(kr + ks_off(tl, d >> 5)) : 0;
        if (a.v_type == KV_T_Q8) vs[so] = ok ? *reinterpret_cast<const uint16_t *>(vr + vs_off(tl, d >> 5)) : 0;
    }
}

cudaError_t launch_kv_read(const KvPool &a, int slot, int layer, int t0, int n, uint8_t *k, uint8_t *v,
                           uint16_t *ks, uint16_t *vs, cudaStream_t stream) {
    const long total = (long)n * a.n_kv * HD;
    if (total == 0) return cudaSuccess;
    kv_read_kernel<<<(unsigned)((total + 255) / 256), 256, 0, stream>>>(a, slot, layer, t0, n, k, v, ks, vs);
    return cudaGetLastError();
}

}  // namespace zdec
