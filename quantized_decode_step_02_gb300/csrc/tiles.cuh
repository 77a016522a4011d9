// tiles.cuh -- scalar reads of single rows out of the repacked Q4_K tile
// blocks (layout in zdec_internal.cuh): the fields, codes and exact values
// of one row, used by the read-backs and by the embedding gather.
#pragma once
#include "zdec_kernels.cuh"

namespace zdec {

// ------------------------------------------------------ tile-block reads ---
__device__ __forceinline__ uint16_t tile_dq(const uint8_t *tile, int lane) {
    const uint32_t *mw = reinterpret_cast<const uint32_t *>(tile + TILE_CODE_BYTES + 8 * lane);
    uint32_t lo = mw[0], hi = mw[1];
    return (uint16_t)(((lo >> 12) & 0xFu) | (((lo >> 28) & 0xFu) << 4) |
                      (((hi >> 12) & 0xFu) << 8) | (((hi >> 28) & 0xFu) << 12));
}

// Fields of local row lr of a tile block.
__device__ __forceinline__ void tile_row_fields(const uint8_t *tile, int lr, uint16_t &d, uint16_t &dmin,
                                int sc[8], int m[8]) {
    int g = lr & 7, rho = lr >> 3;
    d = tile_dq(tile, 4 * g + 2 * rho);
    dmin = tile_dq(tile, 4 * g + 2 * rho + 1);
    for (int tig = 0; tig < 4; tig++) {
        const uint32_t *mw =
            reinterpret_cast<const uint32_t *>(tile + TILE_CODE_BYTES + 8 * (4 * g + tig));
        uint32_t w = mw[rho];
        sc[2 * tig] = w & 63;
        sc[2 * tig + 1] = (w >> 16) & 63;
        m[2 * tig] = (w >> 6) & 63;
        m[2 * tig + 1] = (w >> 22) & 63;
    }
}

// Code of element k (0..255) of local row lr.
__device__ __forceinline__ int tile_q(const uint8_t *tile, int lr, int k) {
    int g = lr & 7, rho = lr >> 3;
    int j = k >> 5, tig = j >> 1, h = j & 1;
    int p = (k >> 3) & 3, o = k & 7;
    int lane = 4 * g + tig;
    int c = 2 * h + (p >> 1);
    int wi = (p & 1) * 2 + rho;
    const uint32_t *words = reinterpret_cast<const uint32_t *>(tile + c * 512 + 16 * lane);
    return (int)((words[wi] >> (4 * nib_of_off(o))) & 15u);
}

// Exact dequantization, the canonical rule: ((d*sc)*q) - (dmin*m), each a
// separately rounded fp32 operation.
__device__ __forceinline__ float dq_value(float d, int sc, float dmin, int m, int q) {
    float step = __fmul_rn(d, (float)sc);
    float off = __fmul_rn(dmin, (float)m);
    return __fsub_rn(__fmul_rn(step, (float)q), off);
}

}  // namespace zdec
