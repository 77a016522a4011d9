/*
 * zdec.h -- C ABI of a batched, Q4_K-quantized decode step for one GB300.
 *
 * The operation: one decode step of a grouped-query-attention decoder for B
 * sequences at once.  The Q4_K weight stream is read once per step and shared
 * by all B sequences; each sequence reads its own KV cache (fp16, Q8_0 or FP8
 * e4m3, chosen separately for K and V) from a paged pool.
 * Source: the blog pages "Eight concurrent agents pull 5.6x more tokens from
 * one RX 9070 XT" (sections "The weight read is the only term that does not
 * scale", "RDNA4 pads the batch dimension to 16"), "Batched swarm: the KV read
 * does not amortize" ("The two halves of a decode-step memory bill") and "Q8
 * KV cache pushes an RDNA4 swarm crossover from 5k to 10k tokens" ("Why Q8 is
 * close to free and where the sharp edges are": quantized KV is dequantized
 * inside the fused attention kernel).
 *
 * Conventions for every call:
 *   - No exception crosses this ABI.  Every call returns a zdec_status; on
 *     failure zdec_last_error(ctx) holds a message (per context; calls that
 *     take no context report through zdec_last_global_error()).
 *   - A failed call changes no state unless its comment says otherwise.
 *   - All GPU work is enqueued on the CUDA stream given at create (or, for
 *     the stateless op entry points, on the stream argument; NULL means the
 *     legacy default stream).  Calls are asynchronous unless noted.
 *   - "dev" pointers are CUDA device pointers; "host" pointers are ordinary
 *     (pageable or pinned) host memory.  The library never frees caller
 *     memory and never keeps caller pointers past the call, except the
 *     output pointers of a decode step, which it writes asynchronously.
 *   - fp16 means IEEE binary16 bit patterns (uint16_t).
 */
#ifndef ZDEC_H
#define ZDEC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ZDEC_OK = 0,
    ZDEC_ERR_ARG = -1,          /* bad argument: null pointer, out-of-range index, bad shape  */
    ZDEC_ERR_OOM = -2,          /* device or host allocation failed; nothing was created        */
    ZDEC_ERR_CAPACITY = -3,     /* a sequence would exceed max_L, or the KV pool has no page   */
    ZDEC_ERR_POSITION = -4,     /* positions[b] != number of tokens cached for row b's slot    */
    ZDEC_ERR_UNSUPPORTED = -5,  /* shape outside what the kernels implement (see zdec_create)  */
    ZDEC_ERR_CUDA = -6,         /* a CUDA runtime call failed; message has cudaGetErrorString  */
    ZDEC_ERR_TIMEOUT = -7,      /* a bounded device wait gave up (reported by zdec_sync)       */
    ZDEC_ERR_DEVICE = -8        /* a device-side check flagged an error (reported by zdec_sync) */
} zdec_status;

/* Storage type of a cached tensor (K or V), per "Q8 KV cache pushes an RDNA4
 * swarm crossover from 5k to 10k tokens", section "Why Q8 is close to free
 * and where the sharp edges are" (independent K and V cache types) and
 * "Batched swarm: the KV read does not amortize", section "What a
 * long-running swarm should actually tune" (fp8 or int8 KV):
 *   F16   2 bytes per element.
 *   Q8_0  32-element blocks: one fp16 scale d = fp16(amax/127) (IEEE fp32
 *         division) and 32 int8 codes clamp(rint(x/d), -127, 127), ties to
 *         even, dividing by the fp32 d; an all-zero block stores 0 and 0.
 *         34 bytes per 32 elements.
 *   FP8   e4m3 (4 exponent bits, bias 7, 3 mantissa bits), nearest value,
 *         ties to the even code, saturating at +-448; 1 byte per element. */
typedef enum { ZDEC_KV_F16 = 0, ZDEC_KV_Q8_0 = 1, ZDEC_KV_FP8 = 2 } zdec_kv_dtype;

/* Model shape.  Supported: hidden and ffn multiples of 512, n_q_heads*head_dim
 * a multiple of 512, head_dim == 128, n_q_heads/n_kv_heads == 4 (the grouped
 * attention kernel handles groups of four query heads), vocab >= 1. */
typedef struct {
    int n_layers, hidden, n_q_heads, n_kv_heads, head_dim, ffn, vocab;
    float rope_theta;   /* RoPE base; rotate-half pairs (i, i+head_dim/2)  */
    float rms_eps;      /* RMSNorm epsilon                                 */
} zdec_model_desc;

/* Weights as HOST pointers to canonical Q4_K rows.  A canonical Q4_K block
 * holds 256 consecutive weights of one row in 144 bytes:
 *   [0:2] d (fp16) [2:4] dmin (fp16) [4:16] sixteen 6-bit fields, field i at
 *   bits 6i..6i+5 of the little-endian 96-bit word: fields 0-7 sub-block
 *   scales sc_j, 8-15 sub-block mins m_j; [16:144] codes, byte t = element 2t
 *   (low nibble) | element 2t+1 (high nibble).  Weight i (sub-block j = i/32)
 *   is (d*sc_j)*q_i - dmin*m_j.
 * A rows x cols matrix is row-major: row r is cols/256 consecutive blocks.
 * Shapes: embed [vocab x hidden] (also the tied LM head), wq [n_q*hd x hidden],
 * wk, wv [n_kv*hd x hidden], wo [hidden x n_q*hd], w_gate, w_up [ffn x hidden],
 * w_down [hidden x ffn]; norms are fp32 [hidden].  Per-layer arrays have
 * n_layers entries.  The library copies and repacks everything at create;
 * the caller may free these afterwards. */
typedef struct {
    const void *embed;
    const float *final_norm;
    const float *const *attn_norm;
    const float *const *ffn_norm;
    const void *const *wq, *const *wk, *const *wv, *const *wo;
    const void *const *w_gate, *const *w_up, *const *w_down;
} zdec_weights;

/* The KV cache of a context.  Its memory is a pool of pages of 64 tokens
 * (every layer and kv head, K and V); each sequence slot owns a block table
 * of pages, taken from the pool as the slot grows and returned by
 * zdec_reset_seq, so slots of very different lengths share one budget
 * ("Eight concurrent agents pull 5.6x more tokens from one RX 9070 XT",
 * section "Where it stops, and the argument I got wrong in May": agents hold
 * 800 to 30,000 tokens and VRAM, not arithmetic, bounds the swarm). */
typedef struct {
    int k_type;              /* zdec_kv_dtype of K                                     */
    int v_type;              /* zdec_kv_dtype of V                                     */
    int max_B;               /* sequence slots, also the largest batch of a step (<= 32) */
    int max_L;               /* tokens one slot may hold                               */
    long long pool_tokens;   /* pool capacity in tokens, rounded up to whole pages
                                (0: max_B slots of max_L tokens each)                  */
} zdec_cache_desc;

typedef struct zdec_ctx zdec_ctx;

/* Create a decoder: validate the shape, allocate on the current CUDA device
 * (repacked weights ~0.5625 B/weight, the KV pool, the block tables, the
 * per-step workspace), repack the weights on the GPU and wait for it.
 * Defined by: "Eight concurrent agents pull 5.6x more tokens from one RX 9070
 * XT", sections "The weight read is the only term that does not scale" (one
 * copy of the weights, shared by every sequence of a step) and "Where it
 * stops, and the argument I got wrong in May" (the KV budget, not the
 * arithmetic, bounds how many sequences fit).
 * cuda_stream is a cudaStream_t (NULL: a new non-blocking stream owned by the
 * context).  Returns ZDEC_ERR_OOM (nothing allocated is kept) if the pool does
 * not fit; ZDEC_ERR_ARG for a bad type, max_B outside [1, 32], max_L < 1 or
 * pool_tokens < 0. */
zdec_status zdec_create_cache(const zdec_model_desc *desc, const zdec_weights *weights,
                              const zdec_cache_desc *cache, void *cuda_stream, zdec_ctx **out);
/* Shorthand: one type for K and V, a pool of max_B x max_L tokens. */
zdec_status zdec_create(const zdec_model_desc *desc, const zdec_weights *weights,
                        zdec_kv_dtype kv_dtype, int max_B, int max_L, void *cuda_stream,
                        zdec_ctx **out);
void zdec_destroy(zdec_ctx *ctx);

/* Defined by: "Q8 KV cache pushes an RDNA4 swarm crossover from 5k to 10k
 * tokens", sections "The crossover is just a byte count" (the cache holds K
 * and V of every cached token) and "Why Q8 is close to free and where the
 * sharp edges are" (the cache is quantized where it is written).
 * Append n_tokens already-rotated K/V rows to sequence slot `seq`, starting at
 * its current length, taking pool pages as needed.  k_f16 / v_f16:
 * [n_layers][n_tokens][n_kv_heads][head_dim] fp16, host memory (on_device = 0)
 * or device memory (on_device = 1); the call waits for the copy either way.
 * Each tensor is encoded on write by its type (zdec_kv_dtype).
 * ZDEC_ERR_CAPACITY if len + n_tokens > max_L or the pool lacks pages (nothing
 * is appended and no page is taken). */
zdec_status zdec_append_kv(zdec_ctx *ctx, int seq, int n_tokens, const void *k_f16,
                           const void *v_f16, int on_device);

/* Flags of zdec_decode_step. */
#define ZDEC_STEP_HOST_IO  1   /* tokens/positions are host, logits/ids host; the call
                                  copies in, runs, copies out and waits */
#define ZDEC_STEP_EAGER    2   /* launch kernel by kernel instead of replaying a CUDA graph */

/* Defined by: "Eight concurrent agents pull 5.6x more tokens from one RX 9070
 * XT", section "The workload stopped being one person typing" (advance B
 * in-flight sequences by one token each per step, reading the weights once)
 * and "Batched swarm: the KV read does not amortize", section "The two halves
 * of a decode-step memory bill" (each sequence reads its own KV cache).
 * One decode step for rows b = 0..B-1, row b being sequence slot b, B <= max_B.
 *   tokens [B] int32 token ids, positions [B] int32: position b must equal the
 *   number of tokens cached for slot b.  With host I/O the check happens
 *   before anything is enqueued (ZDEC_ERR_POSITION); with device inputs the
 *   first kernel checks it (and the token ids), the step then writes no KV
 *   row and advances no length, and zdec_sync reports ZDEC_ERR_DEVICE.
 *   logits [B][vocab] fp32 (may be NULL), ids [B] int32 greedy argmax (lowest
 *   index on ties).
 * The step embeds each token, runs every layer (RMSNorm, QKV, RoPE, KV append,
 * split-K attention, O projection + residual, RMSNorm, SwiGLU FFN + residual),
 * the final RMSNorm and the tied LM head, appends each row's new K/V at its
 * position (taking a pool page when the position starts one) and advances
 * its slot's length by one.  ZDEC_ERR_CAPACITY (nothing enqueued) if a slot
 * is full or the pool has no page for a new token.  Without ZDEC_STEP_HOST_IO
 * the call is asynchronous; outputs are valid after zdec_sync or a stream
 * sync. */
zdec_status zdec_decode_step(zdec_ctx *ctx, int B, const int32_t *tokens,
                             const int32_t *positions, float *logits, int32_t *ids, int flags);
/* The same step with row b reading and extending slot slots[b] (host array of
 * B distinct slots in [0, max_B)), so that sequences are admitted and retired
 * between steps in any slot ("Eight concurrent agents...", section "What I am
 * building next": continuous batching over server slots).  A map different
 * from the previous step's waits for the steps in flight first.  ZDEC_ERR_ARG
 * for a repeated or out-of-range slot. */
zdec_status zdec_decode_step_slots(zdec_ctx *ctx, int B, const int32_t *slots, const int32_t *tokens,
                                   const int32_t *positions, float *logits, int32_t *ids, int flags);

/* Wait for the context's stream and report any device-side status
 * (ZDEC_ERR_DEVICE / ZDEC_ERR_TIMEOUT), clearing it.  A step whose device
 * check failed, and every step enqueued after it until this call, wrote no
 * KV row and advanced no length; on either error this call also resets the
 * host's lengths (zdec_seq_len) to the device's.  The pages define no such
 * call: it is the asynchronous ABI's error channel. */
zdec_status zdec_sync(zdec_ctx *ctx);

/* Sequence slots, per "Eight concurrent agents pull 5.6x more tokens from one
 * RX 9070 XT", section "The workload stopped being one person typing" (server
 * slots that admit and retire agents between steps): reset_seq empties slot
 * `seq` and returns its pages to the pool (length := 0; waits for the
 * stream); seq_len reads the host's copy of its length.  ZDEC_ERR_ARG for a
 * slot outside [0, max_B). */
zdec_status zdec_reset_seq(zdec_ctx *ctx, int seq);
zdec_status zdec_seq_len(const zdec_ctx *ctx, int seq, int *len);
const char *zdec_last_error(const zdec_ctx *ctx);
const char *zdec_last_global_error(void);

/* Defined by: "Eight concurrent agents pull 5.6x more tokens from one RX 9070
 * XT", section "RDNA4 pads the batch dimension to 16" (a dequant-matvec for
 * one sequence, a tensor-core GEMM past a few sequences).
 * Which dense kernel runs the Q4_K projections:
 * 0 = default (B = 1: the sub-block-column mma matvec, impl 3; 2 <= B <= 4 by
 * the measured switch point between the CUDA-core matvec and the GEMM),
 * 1 = always the CUDA-core dequant-matvec (B <= 4 only), 2 = always the
 * mma.sync GEMM (batch in the mma N dimension, sub-block scales folded into
 * the A operand), 3 = the sub-block-column mma matvec at B = 1 (raw codes as
 * the A operand, one mma column per sub-block; the GEMM above B = 1).  Takes
 * effect at the next step (cached CUDA graphs are rebuilt). */
zdec_status zdec_set_gemm_impl(zdec_ctx *ctx, int impl);

/* Tracing.  on = 1 makes every later step run without graph replay and
 * record a timeline of the GPU global timer (ns): [launches][8] entries per
 * step: the first CTA's start, the first CTA past its dependency wait, the
 * last CTA's end, the launch's kind (ZDEC_KERNEL_*), then the latest CTA to
 * reach the kernel's milestones (for the projections: past the wait, first
 * stage landed, K loop done, cluster reduction done; for the attention: past
 * the wait, the cluster's partials landed in rank 0, chunk loop done, merge
 * done; zero where a kernel records none).  on = 0 stops and frees it. */
zdec_status zdec_set_trace(zdec_ctx *ctx, int on);
/* Copy the trace of the last traced step (waits for the stream).  *n gets the
 * entry count (0 when tracing is off); out_host needs that many uint64
 * (out_host = NULL: only the size query). */
zdec_status zdec_debug_step_trace(zdec_ctx *ctx, uint64_t *out_host, size_t cap, size_t *n);

typedef struct {
    size_t weight_bytes;      /* repacked weights on the device              */
    size_t arena_bytes;       /* KV pool                                     */
    size_t workspace_bytes;   /* per-step activations, partials, logits     */
    size_t kv_bytes_per_token;/* per sequence, K+V over all layers           */
    int kernels_per_step;     /* kernel launches of one step (last B used)   */
    int attn_splits;          /* attention CTAs per (segment, kv head), last step */
    int matvec_max_B;         /* switch point in use                         */
    int attn_segments;        /* attention segment slots per row, last step  */
    int k_type, v_type;       /* zdec_kv_dtype of K and V                    */
    int page_tokens;          /* tokens per pool page                        */
    int pool_pages;           /* pages in the pool                           */
    int free_pages;           /* pages no slot holds                         */
} zdec_info;
zdec_status zdec_get_info(const zdec_ctx *ctx, zdec_info *info);

/* Per-kernel timing: runs one eager step (like ZDEC_STEP_EAGER, device inputs,
 * rows 0..B-1 in slots 0..B-1) with a CUDA event pair around every launch on
 * the context stream, waits, and writes up to `cap` records: kind[i] (see
 * ZDEC_KERNEL_*), ms[i].  *n receives the number of launches.  The step is a
 * real step (lengths advance). */
enum { ZDEC_KERNEL_EMBED = 0, ZDEC_KERNEL_GEMM_QKV = 2, ZDEC_KERNEL_ATTENTION = 3, ZDEC_KERNEL_GEMM_O = 4,
       ZDEC_KERNEL_GEMM_GATEUP = 5, ZDEC_KERNEL_GEMM_DOWN = 6, ZDEC_KERNEL_GEMM_LMHEAD = 7,
       ZDEC_KERNEL_ARGMAX = 8 };
zdec_status zdec_profile_step(zdec_ctx *ctx, int B, const int32_t *tokens_dev,
                              const int32_t *positions_dev, float *logits_dev, int32_t *ids_dev,
                              int *kind, float *ms, int cap, int *n);

/* ------------------------------------------------------------ debug ---
 * Read-backs used by the parity tests.  All synchronous; host outputs. */
enum { ZDEC_T_EMBED = 0, ZDEC_T_WQ = 1, ZDEC_T_WK = 2, ZDEC_T_WV = 3, ZDEC_T_WO = 4,
       ZDEC_T_GATE = 5, ZDEC_T_UP = 6, ZDEC_T_DOWN = 7 };
/* Rows [row0, row0+nrows) of tensor `which` (layer ignored for EMBED),
 * unpacked from the device's repacked layout back to canonical 144-byte
 * blocks (out: nrows * cols/256 * 144 bytes). */
zdec_status zdec_debug_export_q4k(zdec_ctx *ctx, int which, int layer, int row0, int nrows,
                                  void *out_host);
/* The same rows dequantized on the device, fp32 (out: nrows * cols floats). */
zdec_status zdec_debug_dequant(zdec_ctx *ctx, int which, int layer, int row0, int nrows,
                               float *out_host);
/* Stored KV of slot `seq`, layer `layer`, tokens [t0, t0+n) in canonical
 * token-major layout [n][n_kv_heads][head_dim], each tensor in its own type:
 * F16 -> fp16 (uint16); Q8_0 -> int8 codes, and its scales [n][n_kv_heads]
 * [head_dim/32] fp16 in ks (K) or vs (V); FP8 -> e4m3 codes (uint8).  ks / vs
 * may be NULL for a tensor that is not Q8_0.  Tokens without a page read 0. */
zdec_status zdec_debug_read_kv(zdec_ctx *ctx, int seq, int layer, int t0, int n, void *k,
                               void *v, void *ks, void *vs);
/* The block table of slot `seq` as the device holds it (waits for the
 * stream): *n = entries per slot (ceil(max_L / 64)); pages_host (if not NULL,
 * cap >= *n) receives the page of each 64 tokens, -1 where none. */
zdec_status zdec_debug_block_table(zdec_ctx *ctx, int seq, int32_t *pages_host, int cap, int *n);
/* Arm a capture of the fp32 residual stream for the next decode step, which
 * then runs eagerly, waits, and fills out [B][n_layers+1][hidden] (after the
 * embedding and after each layer) before it returns.  out must hold
 * B*(n_layers+1)*hidden floats for the B of that step; host memory. */
zdec_status zdec_debug_capture_hidden(zdec_ctx *ctx, float *out_host);
/* Bound of the projection kernels' stage waits, in GPU clock cycles (0: the
 * default, about 2 s; -1: every projection's first stage wait counts as run
 * out at once, which tests use to take the give-up path deterministically).
 * A wait that runs out sets the device status that zdec_sync reports as
 * ZDEC_ERR_TIMEOUT; the kernel first waits (with the full bound) for its own
 * copies still in flight, then returns, and the step writes no KV row and
 * advances no length.  Waits for the stream; cached CUDA graphs are rebuilt
 * at the next step.  ZDEC_ERR_ARG for cycles < -1. */
zdec_status zdec_debug_set_wait_limit(zdec_ctx *ctx, long long cycles);
/* Attention alone on the cached tokens 0..positions[b] of slot b, layer
 * `layer` (nothing appended): q [B][n_q_heads][head_dim] fp32 already
 * rotated, o [B][n_q_heads][head_dim] fp32.  Host memory. */
zdec_status zdec_debug_attention(zdec_ctx *ctx, int layer, int B, const float *q_host,
                                 const int32_t *positions_host, float *o_host);

/* ------------------------------------------------------- stateless ops ---
 * The dense Q4_K projection on its own (used for kernel-level parity and the
 * GEMM roofline).  N multiple of 16, K multiple of 512, 1 <= B <= 32. */

/* Bytes of the repacked layout of an N x K matrix: the canonical bytes with
 * the row count rounded up to a multiple of 128 (zero blocks pad the last
 * group of eight 16-row tiles). */
size_t zdec_q4k_repacked_bytes(int N, int K);
/* canonical_dev (N*K/256 blocks, row-major) -> repacked_dev.  Device memory. */
zdec_status zdec_q4k_repack(const void *canonical_dev, int N, int K, void *repacked_dev,
                            void *stream);
/* Scratch bytes zdec_q4k_gemm needs for B rows of length K: fp16 high and
 * low parts of the activations (exactly B rows, no padding) and their per-32
 * sub-block sums. */
size_t zdec_q4k_gemm_workspace_bytes(int K, int B);
/* Defined by: "Eight concurrent agents pull 5.6x more tokens from one RX 9070
 * XT", section "The weight read is the only term that does not scale" (one
 * read of each weight tile multiplied against every row of the batch).
 * y[b][n] = sum_k W[n][k] x[b][k] for b < B.  x_dev fp32 [B][K], y_dev fp32
 * [B][N], workspace_dev >= zdec_q4k_gemm_workspace_bytes(K, B) bytes, 16-byte
 * aligned, owned by the caller.  impl: 1 = dequant-matvec (B <= 4),
 * 2 = mma.sync GEMM, 3 = sub-block-column mma matvec (B = 1).  Activations
 * enter as fp16 high + low parts (about 22 significant bits); weights are
 * exact; accumulation is fp32. */
zdec_status zdec_q4k_gemm(const void *repacked_dev, int N, int K, const float *x_dev, int B,
                          float *y_dev, int impl, void *workspace_dev, size_t workspace_bytes,
                          void *stream);

/* ---------------------------------------------- allocation-free variant ---
 * The pages have no counterpart to this call: it is zdec_q4k_gemm without a
 * workspace argument, for callers that cannot provide device memory (a plain
 * C host with no device allocator of its own, or code that must not call
 * cudaMalloc/cudaFree, which waits for the whole device).  It allocates
 * nothing: its scratch is one array of 1,081,600 bytes per device that the
 * library's module image holds, sized for K*B <= ZDEC_Q4K_GEMM_STATIC_MAX_KB.
 * Arguments, layouts and results are those of zdec_q4k_gemm (the same
 * kernels, so the outputs are bitwise equal).  Errors: K*B above the limit
 * returns ZDEC_ERR_ARG, with the limit in zdec_last_global_error(), before
 * any CUDA call; the other checks are zdec_q4k_gemm's.
 * - The first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress, which may load the module); make that first call
 *   before any stream capture begins on that device.  The address is kept
 *   per device ordinal for the life of the process: after cudaDeviceReset
 *   (or anything else that destroys the device's primary context) it no
 *   longer names the array, so do not call this entry point after that.
 * - Calls whose kernels may overlap in time (different streams with no
 *   ordering between them, or different host threads) share the array and
 *   race on it: order them, e.g. on one stream or with events.  Consecutive
 *   calls on one stream are safe. */
#define ZDEC_Q4K_GEMM_STATIC_MAX_KB 262144
zdec_status zdec_q4k_gemm_static(const void *repacked_dev, int N, int K, const float *x_dev, int B,
                                 float *y_dev, int impl, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* ZDEC_H */
