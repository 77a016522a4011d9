// zdec_kernels.cuh -- host-side launchers of the zdec kernels.  Every launcher
// enqueues on `stream`; `pdl` asks for programmatic dependent launch (the
// kernel may start while its predecessor drains and waits in-kernel with
// griddepcontrol.wait before touching the predecessor's outputs).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>
#include <utility>

#include "kv_pool.cuh"
#include "zdec_internal.cuh"

namespace zdec {

// ------------------------------------------------------------- repack.cu
// Canonical rows -> tile blocks.  interleave8 == 0: tile row r of row tile rt
// is source row 16*rt + r of src0.  interleave8 == 1: rows 0-7 of tile rt are
// rows 8*rt..8*rt+7 of src0 and rows 8-15 the same rows of src1 (gate/up).
// Source rows >= src_rows are zero blocks (padding).
cudaError_t launch_repack(const uint8_t *src0, const uint8_t *src1, int interleave8, int src_rows,
                          int n_rowtiles, int nsb, uint8_t *dst, cudaStream_t stream);
// Tile blocks -> canonical blocks for logical rows [row0, row0+nrows) of a
// matrix stored at `tiles`.  row_map: 0 plain rows, 1 the gate half and 2 the
// up half of a gate/up interleaved matrix.
cudaError_t launch_export_canonical(const uint8_t *tiles, int row_map, int nsb, int row0,
                                    int nrows, uint8_t *dst, cudaStream_t stream);
cudaError_t launch_dequant_rows(const uint8_t *tiles, int row_map, int nsb, int row0, int nrows,
                                float *dst, cudaStream_t stream);
// x[b][:] = dequant(E[tokens[b]]) for b < B; also checks each row's position
// against the device length of its slot, len_dev[slots[b]] (status bit
// STATUS_POSITION on mismatch) and its token against the vocabulary.
// It also writes the first projection's operand gain*x (act planes, row pitch
// Bp) and the sum of x^2 of each row into part[b] (one partial per row).
cudaError_t launch_embed(const uint8_t *E, int nsb, int vocab, const int32_t *tokens,
                         const int32_t *positions, const int32_t *slots, const int32_t *len_dev,
                         uint32_t *status, int B, float *x, int ldx, const float *gain, __half *u,
                         __half *ulo, __half *usx, int Bp, float *part, bool pdl, cudaStream_t stream,
                         unsigned long long *tl = nullptr);

// --------------------------------------------------------------- gemm.cu
enum Epi : int { EPI_STORE = 0, EPI_RESID = 1, EPI_SWIGLU = 2, EPI_LMHEAD = 3 };

struct GemmParams {
    const uint8_t *W;      // grouped tile blocks
    int N;                 // valid output rows (SWIGLU: ffn rows)
    int nrt;               // row tiles (16 rows each; the storage is padded to groups of 8)
    int nsb;               // K / 256
    const __half *x16;     // act plane (hi) [nsb][Bp][256]
    const __half *x16lo;   // act plane (lo) or nullptr
    const __half *sx;      // sub-block sums [nsb][Bp][4][4]
    int B;                 // batch rows used
    int Bp;                // row pitch of the act planes
    float *out;            // STORE: y[b*ldo + n]; RESID: x[b*ldo + n] += y; LMHEAD: logits or null
    int ldo;
    __half *out16;         // SWIGLU, RESID with next_gain: act planes of the next
    __half *out16lo;       //   projection (hi, lo) and its sub-block sums
    __half *out_sx;
    int out_Bp;
    const float *next_gain;   // RESID: RMSNorm gain of the next projection (nullptr: none)
    float *part_out;          // RESID: per-group sum of x^2 per column [grid][MAX_B]
    const float *rms_part;    // consumer: partial sums of x^2 of its operand (nullptr: no norm)
    int rms_nparts;
    int rms_K;
    float rms_eps;
    float *amax_val;       // LMHEAD: per-CTA argmax partials [grid][MAX_B]
    int *amax_idx;
    int cs;                // K split over a cluster of cs CTAs (1..16)
    int stages;            // pipeline depth (set by the launcher)
    int pair;              // 1: stages consumed two at a time; 0: one at a time
    uint32_t red_off;      // cluster rank 0's area for the peers' partial tiles (set by the launcher)
    int red_alias;         // 1: that area is rank 0's stage ring, written once its K loop is done
    uint32_t *status;      // device status word (bounded-wait timeouts)
    long long wait_limit;  // clock cycles a stage wait may take before it gives up (0: ~2 s;
                           // < 0: the first stage wait gives up at once, for tests); the drain
                           // of copies in flight after a give-up always takes the full bound
    unsigned long long *tl;   // launch timeline slot (zdec_internal.cuh) or null
    // STORE of a QKV projection: the query heads (groups < q_heads, one 128-row
    // group each) also go out rotated (RoPE at q_pos[b]), scaled by log2(e)/sqrt(128)
    // and split into fp16 hi + lo, in the attention's mma A-fragment order:
    // q_frag[((b * q_heads + head) * 8 + st) * 4 + tig] = (hi, lo) of dims
    // 16 st + 4 tig + {0,1} and (hi, lo) of dims + {2,3} (null: off)
    uint4 *q_frag;
    const int32_t *q_pos;
    const float2 *q_rope;
    int q_heads;
};
// impl 1: CUDA-core dequant-matvec (B <= 4); impl 2: mma.sync swap-AB GEMM.
cudaError_t launch_gemm(const GemmParams &p, int epi, int impl, bool pdl, cudaStream_t stream);
int gemm_grid(const GemmParams &p);
// CTAs of the (B, impl, epi) projection kernel split cs ways that the GPU holds
// at once (the occupancy API's co-resident clusters times cs); 0: not launchable.
int gemm_cluster_slots(int B, int impl, int epi, int cs);

// prep: fp32 rows -> fp16 operand + sub-block sums.  gain != nullptr applies
// RMSNorm (x * rsqrt(mean x^2 + eps) * gain).  Rows B..Bp-1 are zeroed.
cudaError_t launch_prep(const float *src, int lds, int K, const float *gain, float eps, int B, int Bp,
                        __half *hi, __half *lo, __half *sums, bool pdl, cudaStream_t stream);
// ids[b] = argmax over the per-CTA partials (lowest index on ties); also
// advances the device length of each row's slot, len_dev[slots[b]] =
// positions[b] + 1, unless the status word holds an error (then the step
// changes no length).
cudaError_t launch_argmax_final(const float *amax_val, const int *amax_idx, int nparts, int B,
                                int32_t *ids, const int32_t *positions, const int32_t *slots,
                                int32_t *len_dev, const uint32_t *status, bool pdl, cudaStream_t stream,
                                unsigned long long *tl = nullptr);

// ---------------------------------------------------------- attention.cu
struct AttnParams {
    KvPool kv;
    int layer;
    int nq;                // query heads (= 4 * n_kv)
    const int32_t *positions;   // [B] position of each row's new token
    const int32_t *slots;       // [B] cache slot of each row
    const float *qkv;      // [B][qkv_ld]: q (nq*128), k (n_kv*128), v (n_kv*128)
    int qkv_ld;
    const float2 *rope;    // [max_L][64] (cos, sin)
    int append;            // 1: rotate q/k at pos and append k, v; 0: q already rotated, no append
    int cs;                // CTAs per (segment, kv head): one thread-block cluster (1..16)
    int seg_min;           // fewest 64-token chunks a segment takes (when rows are long enough)
    float *o;              // [B][nq*128] fp32 output, or null (then only the planes below)
    __half *o16;           // act planes (hi, lo) and sums of the O projection's input
    __half *o16lo;
    __half *osx;
    int oBp;               // their row pitch
    int B;
    int max_L;             // positions >= max_L are ignored (the step is flagged elsewhere)
    uint32_t *status;      // device status word
    unsigned long long *tl;   // launch timeline slot (zdec_internal.cuh) or null
    const uint4 *q_frag;   // query fragments prepared by the QKV projection (GemmParams), or null
    int stages;            // 64-token chunks in flight per CTA (2..; 0: the type pair's default)
    float *seg_part;       // [segment slots][n_kv][4][132] partials of rows cut into several segments
    int *seg_ticket;       // [MAX_B][n_kv] arrival counters, zero between launches
};
// grid (cs, n_kv, nz): nz >= B segment slots (nz > B needs seg_part / seg_ticket).
cudaError_t launch_attention(const AttnParams &p, int nz, bool pdl, cudaStream_t stream);
// Raise the attention kernel's dynamic shared-memory limit for a (K, V) type
// pair (once, before capture).
cudaError_t attention_setup(int k_type, int v_type);
// Dynamic shared memory of a launch with `stages` chunks in flight (0: default)
// and clusters of cs CTAs.
size_t attention_smem_bytes(int k_type, int v_type, int stages, int cs);
int attention_default_stages(int k_type, int v_type);
int attention_stage_limit(int k_type, int v_type);
// Clusters of cs attention CTAs (with `stages` chunks in flight) the GPU holds
// at once, from the occupancy API (0: not launchable).  Needs attention_setup.
int attention_max_clusters(int k_type, int v_type, int stages, int cs, int n_kv);
// Bulk append of fp16 K/V [n_layers][n][n_kv][128] (device) at tokens t0.. of
// a slot, encoded per tensor type; every page must be assigned already.
cudaError_t launch_kv_append(const KvPool &a, int slot, int t0, int n, const uint16_t *k16,
                             const uint16_t *v16, uint32_t *status, cudaStream_t stream);
// Canonical read-back of one layer: [n][n_kv][128] fp16 bits, or one-byte
// codes (Q8_0 without its storage offset, e4m3), plus Q8_0 scales [n][n_kv][4].
cudaError_t launch_kv_read(const KvPool &a, int slot, int layer, int t0, int n, uint8_t *k,
                           uint8_t *v, uint16_t *ks, uint16_t *vs, cudaStream_t stream);

// Launch helper: optional programmatic stream serialization and a 1-D cluster
// of `cluster` CTAs along x (1 = no cluster).
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, bool pdl,
                     int cluster, cudaStream_t stream, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        n++;
    }
    if (cluster > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = cluster;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        n++;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace zdec
