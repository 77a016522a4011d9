// repack.cu -- canonical Q4_K rows <-> tile blocks (layout in
// zdec_internal.cuh), exact dequantization read-backs, and the embedding
// gather that starts every decode step.
#include "tiles.cuh"

namespace zdec {

// ---------------------------------------------------- canonical parsing ---
struct CanonBlock {
    uint16_t d, dmin;   // fp16 bits
    uint8_t sc[8], m[8];
};

__device__ __forceinline__ int field6(const uint8_t *f, int i) {
    int bit = 6 * i;
    // a 6-bit field spans at most two bytes; reading f[12] for field 15 stays
    // inside the 144-byte block (it is the first code byte, masked out)
    uint32_t w = (uint32_t)f[bit >> 3] | ((uint32_t)f[(bit >> 3) + 1] << 8);
    return (int)((w >> (bit & 7)) & 63u);
}

__device__ __forceinline__ void parse_canon(const uint8_t *blk, CanonBlock &c) {
    c.d = (uint16_t)(blk[0] | (blk[1] << 8));
    c.dmin = (uint16_t)(blk[2] | (blk[3] << 8));
    for (int i = 0; i < 8; i++) {
        c.sc[i] = (uint8_t)field6(blk + 4, i);
        c.m[i] = (uint8_t)field6(blk + 4, 8 + i);
    }
}
__device__ __forceinline__ int canon_q(const uint8_t *blk, int i) {
    uint8_t b = blk[16 + (i >> 1)];
    return (i & 1) ? (b >> 4) : (b & 15);
}

// Local tile row of logical row `row` under a row map (0 plain, 1 gate half,
// 2 up half of a gate/up interleaved matrix) and its row tile.
__device__ __forceinline__ void map_row(int row_map, int row, int &rt, int &lr) {
    if (row_map == 0) { rt = row >> 4; lr = row & 15; }
    else { rt = row >> 3; lr = (row & 7) + (row_map == 2 ? 8 : 0); }
}

// --------------------------------------------------------------- repack ---
// One warp per tile block; lane (g, tig) writes its 64 code bytes and meta word.
__global__ void repack_kernel(const uint8_t *__restrict__ src0, const uint8_t *__restrict__ src1,
                              int interleave8, int src_rows, int n_rowtiles, int nsb,
                              uint8_t *__restrict__ dst) {
    __shared__ uint8_t zero_block[CANON_BLOCK + 16];
    for (int i = threadIdx.x; i < CANON_BLOCK + 16; i += blockDim.x) zero_block[i] = 0;
    __syncthreads();
    long warp = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    int lane = threadIdx.x & 31;
    if (warp >= (long)n_rowtiles * nsb) return;
    int rt = (int)(warp / nsb), sb = (int)(warp % nsb);
    int g = lane >> 2, tig = lane & 3;
    const uint8_t *blk[2];
    for (int rho = 0; rho < 2; rho++) {
        int lr = g + 8 * rho;
        const uint8_t *src;
        int row;
        if (interleave8) { src = rho ? src1 : src0; row = 8 * rt + g; }
        else { src = src0; row = 16 * rt + lr; }
        blk[rho] = row < src_rows ? src + ((size_t)row * nsb + sb) * CANON_BLOCK : zero_block;
    }
    CanonBlock cb[2];
    parse_canon(blk[0], cb[0]);
    parse_canon(blk[1], cb[1]);

    uint8_t *tile = dst + tile_offset(rt, sb, nsb);
    int j1 = 2 * tig, j2 = 2 * tig + 1;
    for (int c = 0; c < 4; c++) {
        int h = c >> 1;
        uint32_t words[4];
        for (int wi = 0; wi < 4; wi++) {
            int p = (c & 1) * 2 + (wi >> 1);
            int rho = wi & 1;
            uint32_t w = 0;
            for (int n = 0; n < 8; n++) {
                int k = 32 * (2 * tig + h) + 8 * p + off_of_nib(n);
                w |= (uint32_t)canon_q(blk[rho], k) << (4 * n);
            }
            words[wi] = w;
        }
        *reinterpret_cast<uint4 *>(tile + c * 512 + 16 * lane) =
            make_uint4(words[0], words[1], words[2], words[3]);
    }
    uint32_t mw[2];
    for (int rho = 0; rho < 2; rho++)
        mw[rho] = (uint32_t)cb[rho].sc[j1] | ((uint32_t)cb[rho].sc[j2] << 16) |
                  ((uint32_t)cb[rho].m[j1] << 6) | ((uint32_t)cb[rho].m[j2] << 22);
    uint32_t dq = (tig == 0) ? cb[0].d : (tig == 1) ? cb[0].dmin : (tig == 2) ? cb[1].d : cb[1].dmin;
    mw[0] |= ((dq & 0xFu) << 12) | (((dq >> 4) & 0xFu) << 28);
    mw[1] |= (((dq >> 8) & 0xFu) << 12) | (((dq >> 12) & 0xFu) << 28);
    *reinterpret_cast<uint2 *>(tile + TILE_CODE_BYTES + 8 * lane) = make_uint2(mw[0], mw[1]);
}

cudaError_t launch_repack(const uint8_t *src0, const uint8_t *src1, int interleave8, int src_rows,
                          int n_rowtiles, int nsb, uint8_t *dst, cudaStream_t stream) {
    n_rowtiles = n_groups(n_rowtiles) * GT;   // pad to whole groups with zero blocks
    long warps = (long)n_rowtiles * nsb;
    int threads = 256;
    long blocks = (warps * 32 + threads - 1) / threads;
    repack_kernel<<<(unsigned)blocks, threads, 0, stream>>>(src0, src1, interleave8, src_rows,
                                                            n_rowtiles, nsb, dst);
    return cudaGetLastError();
}

// One thread per (row, super-block): rebuild the canonical 144 bytes.
__global__ void export_canonical_kernel(const uint8_t *__restrict__ tiles, int row_map, int nsb,
                                        int row0, int nrows, uint8_t *__restrict__ dst) {
    long t = (long)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= (long)nrows * nsb) return;
    int r = (int)(t / nsb), sb = (int)(t % nsb);
    int rt, lr;
    map_row(row_map, row0 + r, rt, lr);
    const uint8_t *tile = tiles + tile_offset(rt, sb, nsb);
    uint16_t d, dmin;
    int sc[8], m[8];
    tile_row_fields(tile, lr, d, dmin, sc, m);
    uint8_t *o = dst + ((size_t)r * nsb + sb) * CANON_BLOCK;
    o[0] = d & 0xFF; o[1] = d >> 8; o[2] = dmin & 0xFF; o[3] = dmin >> 8;
    uint8_t f[12] = {0};
    for (int i = 0; i < 16; i++) {
        uint32_t v = (uint32_t)(i < 8 ? sc[i] : m[i - 8]);
        for (int b = 0; b < 6; b++) {
            int bit = 6 * i + b;
            if (v & (1u << b)) f[bit >> 3] |= (uint8_t)(1u << (bit & 7));
        }
    }
    for (int i = 0; i < 12; i++) o[4 + i] = f[i];
    for (int k = 0; k < 256; k += 2)
        o[16 + (k >> 1)] = (uint8_t)(tile_q(tile, lr, k) | (tile_q(tile, lr, k + 1) << 4));
}

cudaError_t launch_export_canonical(const uint8_t *tiles, int row_map, int nsb, int row0,
                                    int nrows, uint8_t *dst, cudaStream_t stream) {
    long n = (long)nrows * nsb;
    export_canonical_kernel<<<(unsigned)((n + 127) / 128), 128, 0, stream>>>(tiles, row_map, nsb,
                                                                            row0, nrows, dst);
    return cudaGetLastError();
}

// One thread per (row, super-block, sub-block): 32 exact fp32 weights.
__global__ void dequant_rows_kernel(const uint8_t *__restrict__ tiles, int row_map, int nsb,
                                    int row0, int nrows, float *__restrict__ dst) {
    long t = (long)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= (long)nrows * nsb * 8) return;
    int r = (int)(t / (nsb * 8));
    int rem = (int)(t % (nsb * 8));
    int sb = rem >> 3, j = rem & 7;
    int rt, lr;
    map_row(row_map, row0 + r, rt, lr);
    const uint8_t *tile = tiles + tile_offset(rt, sb, nsb);
    uint16_t dbits, mbits;
    int sc[8], m[8];
    tile_row_fields(tile, lr, dbits, mbits, sc, m);
    float d = __half2float(__ushort_as_half(dbits)), dmin = __half2float(__ushort_as_half(mbits));
    float *o = dst + (size_t)r * nsb * 256 + sb * 256 + 32 * j;
    for (int i = 0; i < 32; i++) o[i] = dq_value(d, sc[j], dmin, m[j], tile_q(tile, lr, 32 * j + i));
}

cudaError_t launch_dequant_rows(const uint8_t *tiles, int row_map, int nsb, int row0, int nrows,
                                float *dst, cudaStream_t stream) {
    long n = (long)nrows * nsb * 8;
    dequant_rows_kernel<<<(unsigned)((n + 127) / 128), 128, 0, stream>>>(tiles, row_map, nsb, row0,
                                                                        nrows, dst);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- embed ---
// Block b gathers row tokens[b] of the tied embedding: one thread per 8
// elements (super-block sb, sub-block j, quarter c), so the row's loads go out
// at once.
__global__ void embed_kernel(const uint8_t *__restrict__ E, int nsb, int vocab,
                             const int32_t *tokens, const int32_t *positions, const int32_t *slots,
                             const int32_t *len_dev, uint32_t *status, int B,
                             float *__restrict__ x, int ldx, const float *__restrict__ gain,
                             __half *u, __half *ulo, __half *usx, int Bp, float *part,
                             unsigned long long *tl) {
    tl_min(tl, 0);
    pdl_launch_dependents();
    pdl_wait();
    tl_min(tl, 1);
    __shared__ float red[32];
    const int b = blockIdx.x;   // the grid is B blocks
    int tok = tokens[b];
    if (threadIdx.x == 0 && positions[b] != len_dev[slots[b]]) atomicOr(status, STATUS_POSITION);
    if (tok < 0 || tok >= vocab) {               // flagged; row 0 keeps the step well defined
        if (threadIdx.x == 0) atomicOr(status, STATUS_TOKEN);
        tok = 0;
    }
    const int rt = tok >> 4, lr = tok & 15;
    float ss = 0.0f;
    // blockDim.x is a multiple of 32 and nsb * 32 items are whole warps, so the
    // 4 quarters of a sub-block are 4 adjacent lanes of one warp
    for (int t = threadIdx.x; t < nsb * 32; t += blockDim.x) {
        const int sb = t >> 5, j = (t >> 2) & 7, c = t & 3;
        const uint8_t *tile = E + tile_offset(rt, sb, nsb);
        uint16_t dbits, mbits;
        int sc[8], m[8];
        tile_row_fields(tile, lr, dbits, mbits, sc, m);
        const float d = __half2float(__ushort_as_half(dbits)), dmin = __half2float(__ushort_as_half(mbits));
        float *o = x + (size_t)b * ldx + sb * 256 + 32 * j + 8 * c;
        float y[8], w[8], usum = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; i++) {
            const int k = 32 * j + 8 * c + i;
            w[i] = dq_value(d, sc[j], dmin, m[j], tile_q(tile, lr, k));
            ss = fmaf(w[i], w[i], ss);
            y[i] = w[i] * gain[sb * 256 + k];
            usum += y[i];
        }
        reinterpret_cast<float4 *>(o)[0] = make_float4(w[0], w[1], w[2], w[3]);
        reinterpret_cast<float4 *>(o)[1] = make_float4(w[4], w[5], w[6], w[7]);
        store_act8(u, ulo, act_chunk(sb, b, 4 * j + c, Bp), y);
        usum += __shfl_xor_sync(0xFFFFFFFFu, usum, 1);   // the sub-block's 4 quarters
        usum += __shfl_xor_sync(0xFFFFFFFFu, usum, 2);
        if (c == 0) store_sum(usx, sb, b, j, Bp, usum);
    }
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x == 0) {
        float tot = 0.0f;
        for (int w = 0; w < (int)(blockDim.x >> 5); w++) tot += red[w];
        part[b] = tot;
        tl_end(tl);
    }
}

cudaError_t launch_embed(const uint8_t *E, int nsb, int vocab, const int32_t *tokens,
                         const int32_t *positions, const int32_t *slots, const int32_t *len_dev,
                         uint32_t *status, int B, float *x, int ldx, const float *gain, __half *u,
                         __half *ulo, __half *usx, int Bp, float *part, bool pdl, cudaStream_t stream,
                         unsigned long long *tl) {
    return launch_k(embed_kernel, dim3(B), dim3(512), 0, pdl, 1, stream, E, nsb, vocab, tokens,
                    positions, slots, len_dev, status, B, x, ldx, gain, u, ulo, usx, Bp, part, tl);
}

}  // namespace zdec
